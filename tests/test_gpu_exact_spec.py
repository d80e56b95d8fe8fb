"""Exact-mode speculative verify and commit, which keep the chunk grid (exact-replay RFC section 6,
speculative decoding on the exact-replay path; ReplaySSM notes, "Motivation and method": outputs of
drafts from the checkpoint and buffered inputs, rejected drafts never enter the state).  Drafts end
before, exactly at, and past the chunk boundary; verify outputs equal exact-mode decode of the same
tokens bit for bit and leave the cache unchanged; a commit leaves the state that decoding the
accepted drafts leaves; the committed stream matches the oracle."""
import ctypes
import dataclasses

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


def _caches(w, S, KT, seed, n):
    """n identical caches prefilled with each sequence's history (2 chunks + p0 ~ U{0..Q-1})."""
    ers = _ers()
    d = w.dims
    params, hist, p0, stream = synth.decode_inputs(w, seed=seed, batch=S, steps=KT)
    prm = layer(params)
    cu = torch.tensor(np.concatenate([[0], np.cumsum([h.ntokens for h in hist])]), dtype=torch.int32, device=dev())
    hx, hdt, hB, hC = torch_io.tokens_to(synth.Tokens.concat(hist), dev())
    caches = []
    for _ in range(n):
        c = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk,
                            torch.bfloat16 if w.bf16 else torch.float32)
        ers.chunked_prefill(c, prm, hx, hdt, hB, hC, cu)
        caches.append(c)
    return params, prm, hist, p0, stream, caches


def _drafts(stream, K, T, S):
    """Draft j of sequence i at step k is stream row (k T + j) S + i: tensors [K, S, T, ...]."""
    tok = torch_io.tokens_to(stream, dev(), lead=(K, T, S))
    return [t.transpose(1, 2).contiguous() for t in tok]


def _cache_state(c):
    return (c.state.clone(), c.pos.clone(), c.buf_x.clone(), c.buf_dt.clone(), c.buf_B.clone(), c.buf_C.clone())


def _same_cache(c, snap, S, Q):
    state, pos, bx, bdt, bB, bC = snap
    assert same_bits(c.state, state) and torch.equal(c.pos, pos)
    for i in range(S):
        p = int(pos[i])
        for got, want in ((c.buf_x, bx), (c.buf_dt, bdt), (c.buf_B, bB), (c.buf_C, bC)):
            assert same_bits(got[i, :p], want[i, :p])


def _decode_accepted(ers, c, prm, dr, acc, T):
    """Non-speculative exact decode of the accepted drafts (sequence i decodes acc[i] tokens)."""
    dx, ddt, dB, dC = dr
    outs = []
    for j in range(T):
        sel = np.nonzero(acc > j)[0]
        if sel.size == 0:
            break
        sl = torch.from_numpy(sel.astype(np.int32)).to(dev())
        l = sl.long()
        outs.append((sel, j, ers.replay_decode(c, prm, dx[l, j], ddt[l, j], dB[l, j], dC[l, j], slot=sl)))
    return outs


@pytest.mark.parametrize("dims,T,bf16", [(synth.Dims(64, 8, 64, 128, 16), 4, True), (synth.Dims(64, 8, 64, 128, 16), 16, True),
                                         (synth.Dims(16, 2, 64, 128, 64), 4, True), (synth.Dims(12, 3, 64, 128, 16), 3, True),
                                         (synth.Dims(16, 2, 64, 128, 16), 4, False)],
                         ids=["chunk16-T4", "chunk16-T16", "tensor-core-chunk64-T4", "chunk16-T3-4heads", "chunk16-T4-fp32"])
def test_verify_equals_decode_and_commit_equals_decode(dims, T, bf16):
    ers = _ers()
    w = dataclasses.replace(synth.workload("decode_b256_h64"), dims=dims, bf16=bf16)
    Q = dims.chunk
    S = 40
    params, prm, hist, p0, stream, (c_spec, c_dec, c_ref) = _caches(w, S, T, 61, 3)
    dr = [t[0] for t in _drafts(stream, 1, T, S)]
    # positions that make drafts end before, exactly at and past the boundary, and start a new chunk
    assert (p0 + T > Q).any() and (T == Q or (p0 + T < Q).any())
    snap = _cache_state(c_spec)
    y = ers.spec_verify_exact(c_spec, prm, *dr)
    torch.cuda.synchronize()
    _same_cache(c_spec, snap, S, Q)                     # verify changes nothing
    # every draft of every sequence against exact decode of drafts 0..j
    for j in range(T):
        yd = ers.replay_decode(c_dec, prm, *(t[:, j].contiguous() for t in dr))
        assert same_bits(y[:, j], yd), f"draft {j}"
    # accepted counts covering: none, ending short of, exactly at and past the boundary, all
    rng = np.random.Generator(np.random.PCG64(62))
    acc = rng.integers(0, T + 1, size=S).astype(np.int32)
    acc[0], acc[1] = 0, T
    for i in range(2, S):
        if p0[i] + T >= Q and i % 3 == 0:
            acc[i] = Q - p0[i]                            # exactly fills the chunk
    ers.commit_exact(c_spec, prm, torch.from_numpy(acc).to(dev()), *dr)
    outs = _decode_accepted(ers, c_ref, prm, dr, acc, T)
    torch.cuda.synchronize()
    _same_cache(c_spec, _cache_state(c_ref), S, Q)
    for sel, j, yd in outs:
        assert same_bits(yd, y[torch.from_numpy(sel).long().to(dev()), j])
    assert np.array_equal(c_spec.pos.cpu().numpy(), (p0 + acc) % Q)


def _spec_loop(S, K, seeds, sample=None):
    """K steps of verify + commit at 4 drafts with accepted ~ U{0..4} on S sequences of the decode
    workload: every accepted draft's output equals non-speculative exact decode of the committed
    stream bit for bit, the caches end identical, and outputs and checkpoints of the sampled
    sequences (all when sample is None) match the fp64 oracle per (sequence, head)."""
    ers = _ers()
    w = synth.workload("decode_b256_h64")
    d = w.dims
    Q, T = d.chunk, 4
    params, prm, hist, p0, stream, (c_spec, c_ref) = _caches(w, S, K * T, seeds[0], 2)
    drafts = _drafts(stream, K, T, S)
    acc_all = np.random.Generator(np.random.PCG64(seeds[1])).integers(0, T + 1, size=(K, S)).astype(np.int32)
    from exact_replay_decode_gb300 import _abi
    ws = torch.empty(_abi.lib().ers_spec_verify_exact_workspace_size(ctypes.byref(c_spec.dims), S),
                     dtype=torch.uint8, device=dev())
    committed = [[] for _ in range(S)]                   # stream rows of each sequence's committed drafts
    ys = [[] for _ in range(S)]
    for k in range(K):
        dr = [t[k] for t in drafts]
        y = ers.spec_verify_exact(c_spec, prm, *dr, workspace=ws)
        acc = acc_all[k]
        ers.commit_exact(c_spec, prm, torch.from_numpy(acc).to(dev()), *dr, workspace=ws)
        for sel, j, yd in _decode_accepted(ers, c_ref, prm, dr, acc, T):
            l = torch.from_numpy(sel).long().to(dev())
            assert same_bits(y[l, j], yd), f"step {k} draft {j}"
        for i in range(S):
            for j in range(int(acc[i])):
                committed[i].append((k * T + j) * S + i)
                ys[i].append(y[i, j])
    torch.cuda.synchronize()
    _same_cache(c_spec, _cache_state(c_ref), S, Q)
    assert np.array_equal(c_spec.pos.cpu().numpy(), np.array([(hist[i].ntokens + len(committed[i])) % Q
                                                              for i in range(S)]))
    # the oracle over history + committed drafts, per (sequence, head) of the sampled sequences
    idx = list(range(S)) if sample is None else list(sample)
    parts = [synth.Tokens.concat([hist[i], synth.Tokens(stream.x[committed[i]], stream.dt[committed[i]],
                                                         stream.B[committed[i]], stream.C[committed[i]], True)])
             for i in idx]
    allt = synth.Tokens.concat(parts)
    cu = np.concatenate([[0], np.cumsum([p.ntokens for p in parts])]).astype(np.int64)
    y_o, _ = oracle.recurrence(allt.x, allt.dt, params.A, allt.B, allt.C, params.D, params.dt_bias, cu)
    got = torch.stack([yy for i in idx for yy in ys[i]])
    ref = np.concatenate([y_o[cu[n] + hist[i].ntokens:cu[n + 1]] for n, i in enumerate(idx)])
    cu_c = np.concatenate([[0], np.cumsum([len(ys[i]) for i in idx])])
    check_out(got, ref, 2e-3, keep=1, cu=cu_c, what="exact speculative outputs")
    nb = [(p.ntokens // Q) * Q for p in parts]
    sel = np.concatenate([np.arange(cu[n], cu[n] + nb[n]) for n in range(len(idx))]).astype(np.int64)
    _, s_o = oracle.recurrence(allt.x[sel], allt.dt[sel], params.A, allt.B[sel], allt.C[sel], params.D,
                               params.dt_bias, np.concatenate([[0], np.cumsum(nb)]))
    assert state_err(c_spec.state[torch.tensor(idx, device=dev())], s_o) <= STATE_TOL


def test_speculative_loop_matches_decode_and_oracle():
    """32 steps on 24 sequences, the oracle on every one."""
    _spec_loop(24, 32, (63, 64))


def test_speculative_loop_full_size_sampled():
    """The bench's launch configuration (256 sequences x 4 drafts, 64 heads / 8 groups, headdim 64,
    dstate 128, chunk 16) for 8 steps: every accepted draft bitwise against exact decode, the oracle
    on sampled sequences."""
    _spec_loop(256, 8, (65, 66), sample=[0, 101, 255])


def test_commit_exact_rejects_bad_counts_and_positions():
    ers = _ers()
    w = synth.workload("decode_b256_h64")
    S, T = 4, 4
    params, prm, hist, p0, stream, (c,) = _caches(w, S, T, 65, 1)
    dr = [t[0] for t in _drafts(stream, 1, T, S)]
    before = _cache_state(c)
    st = ers.Status(dev())
    ers.commit_exact(c, prm, torch.tensor([0, 5, 1, 0], dtype=torch.int32, device=dev()), *dr, status=st, check=False)
    assert st.read() == 7                                  # ERS_ECOMMIT for the count above T
    assert int(c.pos[1]) == int(before[1][1])              # that sequence is left as it was
