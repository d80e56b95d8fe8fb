"""Chunked SSD prefill on the GPU: parity with the fp64 oracle, and bit-identity of single-shot,
aligned/unaligned chunked prefill and varlen packing (exact-replay RFC, Evidence 3-5)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import torch_io
from gpu_helpers import STATE_TOL, check_out, dev, layer, max_rel, out_tol, same_bits, state_err

pytestmark = pytest.mark.gpu


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _run_splits(w, params, toks, splits):
    ers = _ers()
    d = w.dims
    cache = ers.ReplayCache(1, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, torch_io.io_dtype(toks))
    prm = layer(params)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    ys, lo = [], 0
    for n in splits:
        ys.append(ers.chunked_prefill(cache, prm, x[lo:lo + n], dt[lo:lo + n], B[lo:lo + n], C[lo:lo + n]))
        lo += n
    assert lo == toks.ntokens
    return torch.cat(ys), cache


@pytest.mark.parametrize("name", ["tiny_fp32", "prefill_2048_h32"])
def test_scan_matches_oracle(name):
    ers = _ers()
    w = synth.workload(name)
    params, toks, cu = synth.prefill_inputs(w, seed=0)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    y, fin, cs = ers.ssd_scan_fwd(x, dt, layer(params), B, C, chunk=w.dims.chunk, return_chunk_states=True)
    y_o, s_o = oracle.recurrence(toks.x, toks.dt, params.A, toks.B, toks.C, params.D, params.dt_bias)
    check_out(y, y_o, out_tol(toks), keep=1, max_rel=max_rel(toks), what=name)   # per head, and whole
    assert state_err(fin, s_o) <= STATE_TOL
    # intermediate chunk-end states equal the oracle state after each chunk
    Q = w.dims.chunk
    for c in (0, toks.ntokens // Q - 1):
        _, s_c = oracle.recurrence(toks.x[:(c + 1) * Q], toks.dt[:(c + 1) * Q], params.A, toks.B[:(c + 1) * Q],
                                   toks.C[:(c + 1) * Q], params.D, params.dt_bias)
        assert state_err(cs[:, c], s_c) <= STATE_TOL


def test_scan_varlen_packing_bitwise_and_oracle():
    ers = _ers()
    w = synth.workload("varlen_4seq_h64")
    params, toks, cu = synth.prefill_inputs(w, seed=0)
    prm = layer(params)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    cu_t = torch.from_numpy(cu).to(dev())
    y, fin = ers.ssd_scan_fwd(x, dt, prm, B, C, chunk=w.dims.chunk, cu_seqlens=cu_t)
    y_o, s_o = oracle.recurrence(toks.x, toks.dt, params.A, toks.B, toks.C, params.D, params.dt_bias, cu)
    # per (sequence, head), so that the one-token sequence is held to the bar on its own
    check_out(y, y_o, out_tol(toks), keep=1, cu=cu, max_rel=max_rel(toks), what="varlen")
    assert state_err(fin, s_o) <= STATE_TOL
    for i in range(len(cu) - 1):
        lo, hi = int(cu[i]), int(cu[i + 1])
        ys, fs = ers.ssd_scan_fwd(x[lo:hi], dt[lo:hi], prm, B[lo:hi], C[lo:hi], chunk=w.dims.chunk)
        assert same_bits(ys, y[lo:hi]), f"sequence {i} differs from its solo run"
        assert same_bits(fs[0], fin[i])


def test_scan_prefix_invariance():
    ers = _ers()
    w = synth.workload("prefill_2048_h32")
    params, toks, _ = synth.prefill_inputs(w, seed=1, seqlens=(600,))
    prm = layer(params)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    y, _ = ers.ssd_scan_fwd(x, dt, prm, B, C, chunk=256)
    for n in (1, 2, 255, 256, 257, 511, 599):
        yp, _ = ers.ssd_scan_fwd(x[:n], dt[:n], prm, B[:n], C[:n], chunk=256)
        assert same_bits(yp, y[:n]), n


@pytest.mark.parametrize("name,splits", [
    ("tiny_fp32", [16, 48]),
    ("tiny_fp32", [7, 57]),
    ("tiny_fp32", [1] * 64),
    ("prefill_2048_h32", [256, 257, 1535]),
    ("prefill_2048_h32", [100] * 20 + [48]),
    ("prefill_2048_h32", [256] * 8),
])
def test_chunked_prefill_splits_bitwise(name, splits):
    ers = _ers()
    w = synth.workload(name)
    params, toks, _ = synth.prefill_inputs(w, seed=0)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    y_ref, fin_ref = ers.ssd_scan_fwd(x, dt, layer(params), B, C, chunk=w.dims.chunk)
    y, cache = _run_splits(w, params, toks, splits)
    assert same_bits(y, y_ref)
    T, Q = toks.ntokens, w.dims.chunk
    assert int(cache.pos[0]) == T % Q
    if T % Q == 0:
        assert same_bits(cache.state[0], fin_ref[0])


def test_chunked_prefill_varlen_resume_mixed_offsets():
    """Several sequences resumed at different buffered offsets in one call equal their single-shot runs."""
    ers = _ers()
    w = synth.workload("varlen_4seq_h64")
    d = w.dims
    lens1 = [300, 17, 513, 1, 0, 256]
    lens2 = [5, 600, 1, 255, 40, 256]
    S = len(lens1)
    params, toks, _ = synth.prefill_inputs(w, seed=2, seqlens=[a + b for a, b in zip(lens1, lens2)])
    prm = layer(params)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    starts = np.concatenate([[0], np.cumsum([a + b for a, b in zip(lens1, lens2)])])
    cache = ers.ReplayCache(S + 2, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, torch.bfloat16)
    slot = torch.tensor([3, 0, 7, 1, 5, 2], dtype=torch.int32, device=dev())
    outs = []
    for part, lens in ((0, lens1), (1, lens2)):
        idx = []
        for i in range(S):
            lo = int(starts[i]) + (0 if part == 0 else lens1[i])
            idx.extend(range(lo, lo + lens[i]))
        idx_t = torch.tensor(idx, dtype=torch.long, device=dev())
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev())
        outs.append((idx, ers.chunked_prefill(cache, prm, x[idx_t], dt[idx_t], B[idx_t], C[idx_t], cu, slot=slot)))
    for i in range(S):
        lo, hi = int(starts[i]), int(starts[i + 1])
        ys, fs = ers.ssd_scan_fwd(x[lo:hi], dt[lo:hi], prm, B[lo:hi], C[lo:hi], chunk=d.chunk)
        got = []
        for idx, y in outs:
            sel = [k for k, t in enumerate(idx) if lo <= t < hi]
            got.append(y[torch.tensor(sel, dtype=torch.long, device=dev())] if sel else y[:0])
        assert same_bits(torch.cat(got), ys), f"sequence {i}"
        assert int(cache.pos[int(slot[i])]) == (hi - lo) % d.chunk
    # the oracle: every sequence's outputs over both calls, and each slot's boundary checkpoint
    cu_all = starts.astype(np.int64)
    y_o, _ = oracle.recurrence(toks.x, toks.dt, params.A, toks.B, toks.C, params.D, params.dt_bias, cu_all)
    y_all = torch.empty_like(x)
    for idx, y in outs:
        if idx:
            y_all[torch.tensor(idx, dtype=torch.long, device=dev())] = y
    check_out(y_all, y_o, 2e-3, keep=1, cu=cu_all, what="mixed offsets")
    Q = d.chunk
    nb = [((hi - lo) // Q) * Q for lo, hi in zip(starts[:-1], starts[1:])]
    sel = np.concatenate([np.arange(int(starts[i]), int(starts[i]) + nb[i]) for i in range(S)]).astype(np.int64)
    _, s_o = oracle.recurrence(toks.x[sel], toks.dt[sel], params.A, toks.B[sel], toks.C[sel], params.D,
                               params.dt_bias, np.concatenate([[0], np.cumsum(nb)]))
    assert state_err(cache.state[slot.long()], s_o) <= STATE_TOL


def test_empty_and_single_token_sequences():
    ers = _ers()
    w = synth.workload("varlen_4seq_h64")
    params, toks, cu = synth.prefill_inputs(w, seed=4, seqlens=(0, 1, 0, 3, 0))
    prm = layer(params)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    init_np = np.random.Generator(np.random.PCG64(41)).standard_normal((5, 64, 64, 128)).astype(np.float32)
    init = torch.from_numpy(init_np).to(dev())
    y, fin = ers.ssd_scan_fwd(x, dt, prm, B, C, chunk=256, cu_seqlens=torch.from_numpy(cu).to(dev()), init_state=init)
    y_o, s_o = oracle.recurrence(toks.x, toks.dt, params.A, toks.B, toks.C, params.D, params.dt_bias, cu, init_np)
    check_out(y, y_o, 2e-3, keep=1, cu=cu, what="empty and one-token sequences")
    assert state_err(fin, s_o) <= STATE_TOL
    assert same_bits(fin[0], init[0]) and same_bits(fin[2], init[2])
