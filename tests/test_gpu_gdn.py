"""Gated-delta-rule (GDN) output-only verify on the GPU (ReplaySSM notes, "Core equations": GDN
residuals from the triangular system, outputs from the checkpoint and the residuals; "Data
protocol and entry point": zero, partial and full acceptance, window refresh, no empty solve).  Verify outputs equal
non-speculative (T = 1) verification over the same committed stream and refresh points bit for bit;
the anchor never sees the read copy; parity with the oracle's stepwise recurrence."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_helpers import OUT_TOL_BF16, STATE_TOL, StepCheck, dev, same_bits, state_err

pytestmark = pytest.mark.gpu


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _cache(ers, anchor, d, io=torch.bfloat16):
    c = ers.GdnCache(anchor.shape[0], d.nheads, d.ngroups, d.dk, d.dv, d.window, io)
    c.anchor.copy_(torch.from_numpy(anchor))
    c.read_copy.copy_(c.anchor)                     # bf16 RNE of the same fp32 values
    return c


def _drafts(toks, K, S, T, io):
    to = lambda a, dt: torch.from_numpy(a).to(dev()).to(dt)
    return (to(toks.q, io).view(K, S, T, *toks.q.shape[1:]), to(toks.k, io).view(K, S, T, *toks.k.shape[1:]),
            to(toks.v, io).view(K, S, T, *toks.v.shape[1:]), to(toks.g, torch.float32).view(K, S, T, -1),
            to(toks.beta, torch.float32).view(K, S, T, -1))


def _run(d, S, K, T, seed, samples, io=torch.bfloat16):
    ers = _ers()
    anchor, toks, acc = synth.gdn_verify_inputs(seed, S, K, d, T)
    cache, ref = _cache(ers, anchor, d, io), _cache(ers, anchor, d, io)
    q, k, v, g, beta = _drafts(toks, K, S, T, io)
    acc_t = torch.from_numpy(acc).to(dev())
    model = oracle.GdnReplayModel(anchor[samples].astype(np.float64), d.window)
    flushes = 0
    chk = StepCheck(OUT_TOL_BF16, keep=(0, 2), what="GDN verify")   # per (sequence, head) over all steps
    for st in range(K):
        flushes += int(((cache.pos + T) > d.window).sum())
        o = ers.gdn_verify(cache, q[st], k[st], v[st], g[st], beta[st])
        ers.gdn_commit(cache, acc_t[st].clone(), T)          # a fresh, aligned row
        # non-speculative comparator: the same refresh points, then one accepted token at a time
        ers.gdn_refresh(ref, T)
        a = acc[st]
        for j in range(T):
            sel = np.nonzero(a > j)[0]
            if sel.size == 0:
                break
            sel_t = torch.from_numpy(sel.astype(np.int32)).to(dev())
            sl = sel_t.long()
            oj = ers.gdn_verify(ref, *(t[st][sl, j:j + 1].contiguous() for t in (q, k, v, g, beta)), slot=sel_t)
            ers.gdn_commit(ref, torch.ones(sel.size, dtype=torch.int32, device=dev()), 1, slot=sel_t)
            assert same_bits(oj[:, 0], o[sl, j]), f"step {st} draft {j}"
        dr = [tuple(np.ascontiguousarray(getattr(toks, f).reshape(K, S, T, *getattr(toks, f).shape[1:])[st, i])
                    for f in ("q", "k", "v", "g", "beta")) for i in samples]
        o_ref = model.verify(dr)
        model.commit([int(acc[st, i]) for i in samples])
        chk.step(o[samples], o_ref, f"step {st}")
    chk.finish()
    assert flushes > 0
    assert torch.equal(cache.pos, ref.pos)
    assert same_bits(cache.anchor, ref.anchor) and same_bits(cache.read_copy, ref.read_copy)
    assert np.array_equal(cache.pos.cpu().numpy()[samples], model.h())
    assert state_err(cache.anchor[samples], model.anchor) <= STATE_TOL
    return cache


def test_gdn_verify_equals_nonspec_and_oracle():
    _run(synth.GdnDims(32, 16, 128, 128, 16), 24, 20, 4, 71, [0, 11, 23])


def test_gdn_verify_full_size_sampled():
    """The bench's launch configuration (512 sequences x 4 drafts, 32 value heads / 16 key groups,
    dk = dv = 128, window 16): bitwise equal to non-speculative verification for every sequence, and
    within the tolerances of the oracle for sampled sequences."""
    w = synth.GDN_VERIFY
    _run(w["dims"], w["batch"], 8, w["drafts"], 75, [0, 257, 511])


def test_gdn_verify_bf16_eight_drafts():
    """Eight drafts with bf16 io: the 8-wide variant, its tensor-core dot products over 16 operand rows."""
    _run(synth.GdnDims(8, 2, 128, 128, 16), 6, 10, 8, 77, [0, 5])


def test_gdn_verify_window_32():
    """The widest window (L = 32): flushes fold up to 32 records, so the fold's first pass takes its
    one-row-per-reduce-scatter branch (more than 16 records)."""
    _run(synth.GdnDims(8, 2, 128, 128, 32), 8, 22, 4, 78, [0, 7])


def test_gdn_verify_fp32_io_short_window_long_drafts():
    _run(synth.GdnDims(8, 2, 128, 128, 8), 6, 14, 6, 72, [0, 5], io=torch.float32)


def test_gdn_zero_acceptance_and_read_copy_isolation():
    ers = _ers()
    d = synth.GdnDims(8, 4, 128, 128, 16)
    S, K, T = 6, 12, 4
    anchor, toks, acc = synth.gdn_verify_inputs(73, S, K, d, T)
    q, k, v, g, beta = _drafts(toks, K, S, T, torch.bfloat16)
    c0 = _cache(ers, anchor, d)
    zero = torch.zeros(S, dtype=torch.int32, device=dev())
    for st in range(K):
        ers.gdn_verify(c0, q[st], k[st], v[st], g[st], beta[st]); ers.gdn_commit(c0, zero, T)
    assert same_bits(c0.anchor, torch.from_numpy(anchor).to(dev())) and int(c0.pos.abs().sum()) == 0
    c1, c2 = _cache(ers, anchor, d), _cache(ers, anchor, d)
    acc_t = torch.from_numpy(acc).to(dev())
    differ = False
    for st in range(K):
        c2.read_copy.mul_(1.0078125)                 # perturb the read copy between refreshes
        o1 = ers.gdn_verify(c1, q[st], k[st], v[st], g[st], beta[st]); ers.gdn_commit(c1, acc_t[st].clone(), T)
        o2 = ers.gdn_verify(c2, q[st], k[st], v[st], g[st], beta[st]); ers.gdn_commit(c2, acc_t[st].clone(), T)
        differ |= not same_bits(o1, o2)
    assert differ and same_bits(c1.anchor, c2.anchor)


def test_gdn_overflow_without_auto_flush():
    ers = _ers()
    d = synth.GdnDims(8, 4, 128, 128, 4)
    anchor, toks, _ = synth.gdn_verify_inputs(74, 2, 2, d, 4)
    q, k, v, g, beta = _drafts(toks, 2, 2, 4, torch.bfloat16)
    c = _cache(ers, anchor, d)
    ers.gdn_verify(c, q[0], k[0], v[0], g[0], beta[0]); ers.gdn_commit(c, torch.full((2,), 3, dtype=torch.int32,
                                                                                       device=dev()), 4)
    st = ers.Status(dev())
    ers.gdn_verify(c, q[1], k[1], v[1], g[1], beta[1], auto_flush=False, status=st, check=False)
    assert st.read() == 6                                          # ERS_EOVERFLOW


def test_gdn_device_errors_are_reported_without_side_effects():
    """Device-detected conditions go to the status word and leave the cache as it was: a slot index
    out of range (ERS_ESLOT), a committed count out of [0, L] (ERS_EALIGN), an accepted count above
    T (ERS_ECOMMIT)."""
    ers = _ers()
    d = synth.GdnDims(8, 4, 128, 128, 16)
    S, T = 4, 4
    anchor, toks, _ = synth.gdn_verify_inputs(76, S, 1, d, T)
    q, k, v, g, beta = _drafts(toks, 1, S, T, torch.bfloat16)
    c = _cache(ers, anchor, d)
    before = (c.anchor.clone(), c.read_copy.clone(), c.pos.clone())
    st = ers.Status(dev())
    bad = torch.tensor([0, 1, 2, 99], dtype=torch.int32, device=dev())
    ers.gdn_verify(c, q[0], k[0], v[0], g[0], beta[0], slot=bad, status=st, check=False)
    assert st.read() == 8                                          # ERS_ESLOT
    assert same_bits(c.anchor, before[0]) and same_bits(c.read_copy, before[1])
    c.pos[1] = d.window + 3
    st = ers.Status(dev())
    ers.gdn_verify(c, q[0], k[0], v[0], g[0], beta[0], status=st, check=False)
    assert st.read() == 5                                          # ERS_EALIGN
    c.pos.copy_(before[2])
    st = ers.Status(dev())
    ers.gdn_commit(c, torch.tensor([0, T + 1, 1, 2], dtype=torch.int32, device=dev()), T, status=st, check=False)
    assert st.read() == 7                                          # ERS_ECOMMIT
    assert int(c.pos[1]) == 0
