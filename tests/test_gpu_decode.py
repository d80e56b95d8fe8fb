"""Exact-replay decode on the GPU (exact-replay RFC section 3; Evidence 5): outputs equal a
single-shot SSD prefill of the same tokens bit for bit, across chunk boundaries, at the
256-sequence x 64-step decode workload; fused and separate refresh agree; parity with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import torch_io
from gpu_helpers import STATE_TOL, check_out, dev, layer, same_bits, state_err

pytestmark = pytest.mark.gpu


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _setup(w, batch, steps, seed=0):
    ers = _ers()
    d = w.dims
    params, hist, p0, stream = synth.decode_inputs(w, seed=seed, batch=batch, steps=steps)
    prm = layer(params)
    cache = ers.ReplayCache(batch, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, torch.bfloat16)
    htoks = synth.Tokens.concat(hist)
    lens = [h.ntokens for h in hist]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev())
    hx, hdt, hB, hC = torch_io.tokens_to(htoks, dev())
    ers.chunked_prefill(cache, prm, hx, hdt, hB, hC, cu)
    sx, sdt, sB, sC = torch_io.tokens_to(stream, dev(), lead=(steps, batch))
    return params, prm, hist, p0, stream, cache, (sx, sdt, sB, sC)


def _single_shot(w, prm, hist, stream, batch, steps):
    """Per sequence: history + its stream tokens, packed, one ssd_scan_fwd call."""
    ers = _ers()
    parts = []
    for i in range(batch):
        rows = [k * batch + i for k in range(steps)]
        parts.append(synth.Tokens.concat([hist[i], synth.Tokens(stream.x[rows], stream.dt[rows], stream.B[rows],
                                                                 stream.C[rows], stream.bf16)]))
    allt = synth.Tokens.concat(parts)
    lens = [p.ntokens for p in parts]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x, dt, B, C = torch_io.tokens_to(allt, dev())
    y, fin = ers.ssd_scan_fwd(x, dt, prm, B, C, chunk=w.dims.chunk, cu_seqlens=torch.from_numpy(cu).to(dev()))
    return parts, cu, y, fin


def test_decode_b256_bitwise_equals_single_shot_and_oracle():
    ers = _ers()
    w = synth.workload("decode_b256_h64")
    S, K = w.batch, w.steps
    params, prm, hist, p0, stream, cache, (sx, sdt, sB, sC) = _setup(w, S, K)
    assert torch.equal(cache.pos.cpu(), torch.from_numpy(p0))
    ys = torch.stack([ers.replay_decode(cache, prm, sx[k], sdt[k], sB[k], sC[k]) for k in range(K)])  # [K,S,H,P]
    parts, cu, y_ss, _ = _single_shot(w, prm, hist, stream, S, K)
    for i in range(S):
        hl = hist[i].ntokens
        ref = y_ss[int(cu[i]) + hl:int(cu[i + 1])]
        assert same_bits(ys[:, i], ref), f"sequence {i} (p0={p0[i]})"
    # the oracle on every sequence: each (sequence, head)'s decoded outputs, and the boundary
    # checkpoint after the last step
    _oracle_all(w, params, parts, hist, ys, cache)


def _oracle_all(w, params, parts, hist, ys, cache):
    """Every sequence against the oracle: decoded outputs ys [K, S, H, P] per (sequence, head) and
    as a whole, checkpoints per (sequence, head), positions."""
    Q = w.dims.chunk
    S = len(parts)
    allt = synth.Tokens.concat(parts)
    cu = np.concatenate([[0], np.cumsum([p.ntokens for p in parts])]).astype(np.int64)
    y_o, _ = oracle.recurrence(allt.x, allt.dt, params.A, allt.B, allt.C, params.D, params.dt_bias, cu)
    ref = np.stack([y_o[cu[i] + hist[i].ntokens:cu[i + 1]] for i in range(S)])      # [S, K, H, P]
    check_out(ys.transpose(0, 1), ref, 2e-3, keep=(0, 2), what="decode vs oracle")
    nb = [(p.ntokens // Q) * Q for p in parts]
    sel = np.concatenate([np.arange(cu[i], cu[i] + nb[i]) for i in range(S)]).astype(np.int64)
    _, s_o = oracle.recurrence(allt.x[sel], allt.dt[sel], params.A, allt.B[sel], allt.C[sel], params.D,
                               params.dt_bias, np.concatenate([[0], np.cumsum(nb)]))
    assert state_err(cache.state[:S], s_o) <= STATE_TOL
    assert np.array_equal(cache.pos[:S].cpu().numpy(), np.array([p.ntokens % Q for p in parts]))


def test_fused_and_separate_refresh_agree():
    ers = _ers()
    w = synth.workload("decode_b256_h64")
    S, K = 32, 40
    _, prm, _, _, _, c1, (sx, sdt, sB, sC) = _setup(w, S, K, seed=5)
    _, _, _, _, _, c2, _ = _setup(w, S, K, seed=5)
    for k in range(K):
        y1 = ers.replay_decode(c1, prm, sx[k], sdt[k], sB[k], sC[k], fuse_refresh=True)
        y2 = ers.replay_decode(c2, prm, sx[k], sdt[k], sB[k], sC[k], fuse_refresh=False)
        ers.refresh(c2, prm)
        assert same_bits(y1, y2), k
    assert same_bits(c1.state, c2.state) and torch.equal(c1.pos, c2.pos)


def test_decode_from_empty_state_tiny_fp32():
    """fp32 io: decode-by-replay from token 0 equals single-shot prefill bitwise (tiny case)."""
    ers = _ers()
    w = synth.workload("tiny_fp32")
    d = w.dims
    params, toks, _ = synth.prefill_inputs(w, seed=0)
    prm = layer(params)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    y_ref, fin = ers.ssd_scan_fwd(x, dt, prm, B, C, chunk=d.chunk)
    cache = ers.ReplayCache(1, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, torch.float32)
    ys = [ers.replay_decode(cache, prm, x[t:t + 1], dt[t:t + 1], B[t:t + 1], C[t:t + 1]) for t in range(64)]
    assert same_bits(torch.cat(ys), y_ref)
    assert same_bits(cache.state[0], fin[0])


def test_decode_slot_indirection_and_subset():
    """Decoding a subset of slots through `slot` touches only those slots."""
    ers = _ers()
    w = synth.workload("decode_b256_h64")
    S, K = 16, 3
    _, prm, _, _, _, c1, (sx, sdt, sB, sC) = _setup(w, S, K, seed=7)
    _, _, _, _, _, c2, _ = _setup(w, S, K, seed=7)
    sel = torch.tensor([9, 2, 14], dtype=torch.int32, device=dev())
    before = c2.state.clone()
    ya = ers.replay_decode(c1, prm, sx[0], sdt[0], sB[0], sC[0])
    yb = ers.replay_decode(c2, prm, sx[0][sel.long()], sdt[0][sel.long()], sB[0][sel.long()], sC[0][sel.long()],
                           slot=sel)
    assert same_bits(yb, ya[sel.long()])
    others = [i for i in range(S) if i not in (9, 2, 14)]
    assert same_bits(c2.state[others], before[others])
    assert torch.equal(c2.pos[sel.long()], c1.pos[sel.long()])


@pytest.mark.parametrize("chunk", [32, 64, 128])
def test_decode_bitwise_across_engines_and_chunk_sizes(chunk):
    """Chunk 32 runs on the CUDA-core engine's bandwidth-shaped decode, chunks >= 64 on the
    tensor-core engine: in each, decode by replay equals single-shot prefill bit for bit and
    matches the oracle, across several refreshes."""
    import dataclasses
    ers = _ers()
    base = synth.workload("decode_b256_h64")
    w = dataclasses.replace(base, dims=synth.Dims(16, 2, 64, 128, chunk), batch=12, steps=chunk + 40,
                            history_chunks=1)
    S, K = w.batch, w.steps
    params, prm, hist, p0, stream, cache, (sx, sdt, sB, sC) = _setup(w, S, K, seed=11)
    ys = torch.stack([ers.replay_decode(cache, prm, sx[k], sdt[k], sB[k], sC[k]) for k in range(K)])
    parts, cu, y_ss, fin = _single_shot(w, prm, hist, stream, S, K)
    for i in range(S):
        ref = y_ss[int(cu[i]) + hist[i].ntokens:int(cu[i + 1])]
        assert same_bits(ys[:, i], ref), f"sequence {i} (p0={p0[i]})"
    _oracle_all(w, params, parts, hist, ys, cache)


@pytest.mark.parametrize("heads,groups,bf16", [(32, 2, True), (16, 2, False), (20, 2, True)])
def test_decode_head_blocks_and_fp32_io(heads, groups, bf16):
    """The warp-per-head decode with 16 heads per group (two head blocks per group), with fp32 io,
    and with 10 heads per group (a partly idle second head block): bitwise equal to single-shot
    prefill, and within tolerance of the oracle."""
    import dataclasses
    ers = _ers()
    base = synth.workload("decode_b256_h64")
    w = dataclasses.replace(base, dims=synth.Dims(heads, groups, 64, 128, 16), batch=6, steps=40, bf16=bf16,
                            history_chunks=1)
    S, K = w.batch, w.steps
    d = w.dims
    params, hist, p0, stream = synth.decode_inputs(w, seed=21, batch=S, steps=K)
    prm = layer(params)
    io = torch.bfloat16 if bf16 else torch.float32
    cache = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, io)
    htoks = synth.Tokens.concat(hist)
    cu = torch.tensor(np.concatenate([[0], np.cumsum([h.ntokens for h in hist])]), dtype=torch.int32, device=dev())
    ers.chunked_prefill(cache, prm, *torch_io.tokens_to(htoks, dev()), cu)
    sx, sdt, sB, sC = torch_io.tokens_to(stream, dev(), lead=(K, S))
    ys = torch.stack([ers.replay_decode(cache, prm, sx[k], sdt[k], sB[k], sC[k]) for k in range(K)])
    parts, cu_ss, y_ss, _ = _single_shot(w, prm, hist, stream, S, K)
    for i in range(S):
        ref = y_ss[int(cu_ss[i]) + hist[i].ntokens:int(cu_ss[i + 1])]
        assert same_bits(ys[:, i], ref), f"sequence {i} (p0={p0[i]})"
    tol = 2e-3 if bf16 else 1e-5
    allt = synth.Tokens.concat(parts)
    y_o, _ = oracle.recurrence(allt.x, allt.dt, params.A, allt.B, allt.C, params.D, params.dt_bias, cu_ss)
    ref = np.stack([y_o[cu_ss[i] + hist[i].ntokens:cu_ss[i + 1]] for i in range(S)])
    check_out(ys.transpose(0, 1), ref, tol, keep=(0, 2), max_rel=2.0 ** -6 if bf16 else 1e-4, what="head blocks")
