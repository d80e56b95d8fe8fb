"""Output-only speculative verify + commit on the GPU (ReplaySSM notes, "Motivation and method",
"Core equations"): verify outputs of accepted drafts equal non-speculative ReplaySSM-mode decode
bit for bit over the same committed stream and refresh points; the anchor never sees the read
copy; parity with the oracle's dual-precision protocol model."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import torch_io
from gpu_helpers import STATE_TOL, StepCheck, dev, layer, same_bits, state_err

pytestmark = pytest.mark.gpu


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _prefilled(w, S, steps, seed, history=32):
    ers = _ers()
    d = w.dims
    params, hist, drafts, acc = synth.verify_inputs(w, seed=seed, batch=S, steps=steps, history=history)
    prm = layer(params)
    hx, hdt, hB, hC = torch_io.tokens_to(hist, dev())
    cu = torch.arange(0, S * history + 1, history, dtype=torch.int32, device=dev())
    _, fin = ers.ssd_scan_fwd(hx, hdt, prm, hB, hC, chunk=d.chunk, cu_seqlens=cu)
    io = torch.bfloat16 if w.bf16 else torch.float32
    cache = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, io, read_copy=True)
    cache.state.copy_(fin)
    ers.refresh(cache, prm, replayssm=True, drafts_T=d.chunk + 1)   # h = 0 everywhere: cast the read copy
    return params, prm, hist, drafts, acc, cache


def _verify_vs_nonspec(w, S, K, seed, samples):
    ers = _ers()
    T, L = w.drafts, w.dims.chunk
    params, prm, hist, drafts, acc, cache = _prefilled(w, S, K, seed=seed)
    ref = _prefilled(w, S, K, seed=seed)[-1]                  # identical starting cache for the comparator
    assert same_bits(cache.read_copy, ref.read_copy)
    dx, ddt, dB, dC = torch_io.tokens_to(drafts, dev(), lead=(K, S, T))
    acc_t = torch.from_numpy(acc).to(dev())
    model = oracle.ReplaySSMModel(params, _oracle_anchor(params, hist, samples, 32), L)
    chk = StepCheck(2e-3, keep=(0, 2), what="verify")   # per (sequence, head) over all steps and drafts
    for k in range(K):
        y = ers.spec_verify(cache, prm, dx[k], ddt[k], dB[k], dC[k])
        ers.commit(cache, acc_t[k], T)
        # non-speculative comparator: same flush decisions, then one accepted token at a time
        ers.refresh(ref, prm, replayssm=True, drafts_T=T)
        a = acc[k]
        for j in range(T):
            sel = np.nonzero(a > j)[0]
            if sel.size == 0:
                break
            sel_t = torch.from_numpy(sel.astype(np.int32)).to(dev())
            sl = sel_t.long()
            yd = ers.replay_decode(ref, prm, dx[k, sl, j], ddt[k, sl, j], dB[k, sl, j], dC[k, sl, j], slot=sel_t,
                                   replayssm=True)
            assert same_bits(yd, y[sl, j]), f"step {k} draft {j}"
        # the oracle's protocol model on sampled sequences
        dr = [tuple(np.ascontiguousarray(getattr(drafts, f).reshape(K, S, T, *getattr(drafts, f).shape[1:])[k, i])
                    for f in ("x", "dt", "B", "C")) for i in samples]
        y_o = model.verify(dr)
        model.commit([int(acc[k, i]) for i in samples])
        chk.step(y[samples], y_o, f"step {k}")
    chk.finish()
    assert torch.equal(cache.pos, ref.pos)
    assert same_bits(cache.state, ref.state) and same_bits(cache.read_copy, ref.read_copy)
    assert np.array_equal(cache.pos.cpu().numpy()[samples], model.h())
    assert state_err(cache.state[samples], model.anchor) <= STATE_TOL
    assert model.flushes > 0


def test_verify_b512_matches_nonspec_decode_and_oracle():
    w = synth.workload("verify_b512_t4")
    _verify_vs_nonspec(w, w.batch, w.steps, 0, [0, 1, 200, 511])


def test_verify_tensor_core_engine_chunk64():
    """Chunk 64 runs verify, commit, flush and ReplaySSM decode on the tensor-core engine."""
    import dataclasses
    base = synth.workload("verify_b512_t4")
    w = dataclasses.replace(base, dims=synth.Dims(16, 2, 64, 128, 64))
    _verify_vs_nonspec(w, 12, 40, 3, [0, 5, 11])


def _oracle_anchor(params, hist, samples, history):
    rows = np.concatenate([np.arange(i * history, (i + 1) * history) for i in samples])
    cu = np.arange(0, len(samples) * history + 1, history)
    _, fin = oracle.recurrence(hist.x[rows], hist.dt[rows], params.A, hist.B[rows], hist.C[rows], params.D,
                               params.dt_bias, cu)
    return fin


def test_zero_acceptance_keeps_anchor_bits():
    ers = _ers()
    w = synth.workload("verify_b512_t4")
    S, K, T = 8, 6, w.drafts
    params, prm, hist, drafts, acc, cache = _prefilled(w, S, K, seed=1)
    anchor0 = cache.state.clone()
    dx, ddt, dB, dC = torch_io.tokens_to(drafts, dev(), lead=(K, S, T))
    zero = torch.zeros(S, dtype=torch.int32, device=dev())
    for k in range(K):
        ers.spec_verify(cache, prm, dx[k], ddt[k], dB[k], dC[k])
        ers.commit(cache, zero, T)
    assert same_bits(cache.state, anchor0) and int(cache.pos.abs().sum()) == 0


def test_anchor_independent_of_read_copy():
    """Corrupting the read copy changes outputs but never the anchor (dual precision)."""
    ers = _ers()
    w = synth.workload("verify_b512_t4")
    S, K, T = 8, 12, w.drafts
    params, prm, hist, drafts, acc, c1 = _prefilled(w, S, K, seed=2)
    c2 = _prefilled(w, S, K, seed=2)[-1]
    dx, ddt, dB, dC = torch_io.tokens_to(drafts, dev(), lead=(K, S, T))
    acc_t = torch.from_numpy(acc).to(dev())
    differ = False
    for k in range(K):
        c2.read_copy.mul_(1.0078125)          # perturb the read copy between refreshes
        y1 = ers.spec_verify(c1, prm, dx[k], ddt[k], dB[k], dC[k]); ers.commit(c1, acc_t[k], T)
        y2 = ers.spec_verify(c2, prm, dx[k], ddt[k], dB[k], dC[k]); ers.commit(c2, acc_t[k], T)
        differ |= not same_bits(y1, y2)
    assert differ
    assert same_bits(c1.state, c2.state)


@pytest.mark.parametrize("heads,groups,bf16,drafts", [(16, 2, False, 4), (32, 2, True, 4), (16, 2, True, 6)])
def test_verify_fp32_io_wide_groups_and_long_drafts(heads, groups, bf16, drafts):
    """Verify with fp32 io on the warp-per-head kernel, and on the per-(sequence, head) kernels it
    hands over to when a group has more than 8 heads or there are more than 4 drafts."""
    import dataclasses
    base = synth.workload("verify_b512_t4")
    w = dataclasses.replace(base, dims=synth.Dims(heads, groups, 64, 128, 16), bf16=bf16, drafts=drafts)
    _verify_vs_nonspec(w, 8, 24, 4, [0, 7])


@pytest.mark.parametrize("heads,groups", [(8, 2), (12, 2), (3, 3)])
def test_verify_tensor_core_partial_head_blocks(heads, groups):
    """ReplaySSM verify and decode on the tensor-core kernel with fewer than 8 heads per group: one
    operand chain of 4 heads, a second chain whose box reaches past the group (6 heads), one head per
    group; bitwise against non-speculative decode and within tolerance of the protocol model."""
    import dataclasses
    base = synth.workload("verify_b512_t4")
    w = dataclasses.replace(base, dims=synth.Dims(heads, groups, 64, 128, 16))
    _verify_vs_nonspec(w, 8, 24, 5, [0, 7])

