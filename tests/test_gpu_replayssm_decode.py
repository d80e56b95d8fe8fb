"""Non-speculative ReplaySSM decode with the flush fused into the decode call (ReplaySSM notes,
"Motivation and method" and "Core equations": a refresh folds the committed records into the anchor
and recasts the read copy; outputs read the copy).  The fused call equals ers_refresh with T = 1
followed by the plain decode bit for bit (outputs, anchors, read copies, buffers, positions), on
the warp-per-head kernel (bf16, FP8 and NVFP4 copies) and on the engines that run the two steps as two
launches; outputs match the oracle's protocol model (verify of one draft, commit one)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import torch_io
from gpu_helpers import (MAX_REL_BF16, MAX_REL_NARROW, OUT_TOL_BF16, STATE_TOL, StepCheck, dev, layer, same_bits,
                         state_err)

pytestmark = pytest.mark.gpu


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _run(dims, read_dtype, S, K, seed, samples):
    ers = _ers()
    w = dataclasses.replace(synth.workload("decode_b256_h64"), dims=dims)
    d, L = w.dims, w.dims.chunk
    params, hist, h0, stream = synth.decode_inputs(w, seed=seed, batch=S, steps=K)
    prm = layer(params)
    ht = synth.Tokens.concat(hist)
    lens = [h.ntokens for h in hist]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev())
    hx, hdt, hB, hC = torch_io.tokens_to(ht, dev())
    _, fin = ers.ssd_scan_fwd(hx, hdt, prm, hB, hC, chunk=L, cu_seqlens=cu)
    tok = torch_io.tokens_to(stream, dev(), lead=(K, S))

    def fresh():
        c = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, L, torch.bfloat16, read_copy=True,
                            read_dtype=read_dtype)
        c.state.copy_(fin)
        ers.refresh(c, prm, replayssm=True, drafts_T=L + 1)
        return c

    c1, c2 = fresh(), fresh()
    # the oracle's protocol model on sampled sequences, anchored at the same prefix
    starts = np.concatenate([[0], np.cumsum(lens)])
    parts = [(ht.x[starts[i]:starts[i + 1]], ht.dt[starts[i]:starts[i + 1]], ht.B[starts[i]:starts[i + 1]],
              ht.C[starts[i]:starts[i + 1]]) for i in samples]
    cat = [np.concatenate([p[f] for p in parts]) for f in range(4)]
    _, anchor = oracle.recurrence(*cat[:2], params.A, *cat[2:], params.D, params.dt_bias,
                                  np.concatenate([[0], np.cumsum([len(p[0]) for p in parts])]))
    cast = {"fp8": oracle.fp8_rows_round, "nvfp4": oracle.nvfp4_rows_round}.get(read_dtype)
    model = oracle.ReplaySSMModel(params, anchor, L, read_cast=cast)
    flushes = 0
    chk = StepCheck(OUT_TOL_BF16, keep=(0, 1), max_rel=MAX_REL_BF16 if read_dtype == "bf16" else MAX_REL_NARROW,
                    what=f"ReplaySSM decode ({read_dtype} copy)")   # per (sequence, head)
    for k in range(K):
        x, dt, B, C = (t[k] for t in tok)
        flushes += int((c1.pos == L).sum())
        y1 = ers.replay_decode(c1, prm, x, dt, B, C, replayssm=True, fuse_refresh=True)
        ers.refresh(c2, prm, replayssm=True, drafts_T=1)
        y2 = ers.replay_decode(c2, prm, x, dt, B, C, replayssm=True, fuse_refresh=False)
        assert same_bits(y1, y2), k
        rows = [k * S + i for i in samples]
        y_o = model.verify([(stream.x[r:r + 1], stream.dt[r:r + 1], stream.B[r:r + 1], stream.C[r:r + 1])
                            for r in rows])
        model.commit([1] * len(samples))
        chk.step(y1[samples], y_o[:, 0], f"step {k}")
    chk.finish()
    assert flushes > 0
    assert torch.equal(c1.pos, c2.pos) and same_bits(c1.state, c2.state)
    assert torch.equal(c1.read_copy.view(torch.uint8), c2.read_copy.view(torch.uint8))
    if read_dtype != "bf16":
        assert same_bits(c1.read_scale, c2.read_scale)
    if read_dtype == "nvfp4":
        assert torch.equal(c1.read_block_scale, c2.read_block_scale)
    for f in ("buf_x", "buf_dt", "buf_B", "buf_C"):
        assert same_bits(getattr(c1, f), getattr(c2, f)), f
    assert np.array_equal(c1.pos.cpu().numpy()[samples], model.h())
    assert state_err(c1.state[samples], model.anchor) <= STATE_TOL


@pytest.mark.parametrize("read_dtype", ["bf16", "fp8", "nvfp4"])
def test_fused_flush_warp_per_head(read_dtype):
    _run(synth.Dims(64, 8, 64, 128, 16), read_dtype, 48, 40, 21, [0, 17, 47])


@pytest.mark.parametrize("dims", [synth.Dims(16, 2, 64, 128, 64), synth.Dims(8, 2, 32, 32, 16)],
                         ids=["tensor-core-chunk64", "fma-p32n32"])
def test_fused_flush_two_launch_engines(dims):
    _run(dims, "bf16", 12, 2 * dims.chunk + 5, 22, [0, 11])


@pytest.mark.parametrize("read_dtype", ["bf16", "fp8", "nvfp4"])
def test_fused_flush_group_spread_over_several_ctas(read_dtype):
    """32 heads in one group: the group's heads span four CTAs of the decode kernel, all of which
    fold the group's committed B rows while the flushing step stores the new token as buffer row 0.
    Fused and separate refreshes still agree bit for bit, and outputs match the protocol model."""
    _run(synth.Dims(32, 1, 64, 128, 16), read_dtype, 96, 40, 23, [0, 41, 95])


@pytest.mark.parametrize("read_dtype", ["bf16", "fp8", "nvfp4"])
def test_fused_flush_full_size_sampled(read_dtype):
    """The bench's launch configuration (256 sequences, 64 heads / 8 groups, headdim 64, dstate 128,
    L 16) for 20 steps, so that every slot passes a fused flush: fused and separate refreshes agree
    bit for bit over every sequence, and sampled sequences match the protocol model."""
    _run(synth.Dims(64, 8, 64, 128, 16), read_dtype, 256, 20, 24, [0, 128, 255])
