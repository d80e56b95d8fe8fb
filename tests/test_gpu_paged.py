"""Paged partial-chunk buffers (exact-replay RFC §6: the buffers live in the paged cache, slot and
position indexed separately; the kernel tests cover contiguous and paged layouts).  A cache whose
buffers are pages in a shuffled page table gives the same bits as the contiguous layout through
chunked prefill, exact-mode decode with fused refresh, ReplaySSM verify + commit + flush, and the
tensor-core engine; a page index out of range is reported and clamped."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import torch_io
from gpu_helpers import STATE_TOL, StepCheck, check_out, dev, layer, same_bits, state_err

pytestmark = pytest.mark.gpu


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _paged(ers, S, d, io, page_rows, seed, **kw):
    ppl = d.chunk // page_rows
    npages = S * ppl + 7
    c = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, io, paged=(page_rows, npages), **kw)
    perm = np.random.Generator(np.random.PCG64(seed)).permutation(npages)[:S * ppl].astype(np.int32)
    c.buf_pages.copy_(torch.from_numpy(perm.reshape(S, ppl)))
    return c


def _logical(c, name):
    """The paged buffer `name` gathered into the contiguous [S, Q, ...] layout."""
    t = getattr(c, name)
    S, ppl = c.buf_pages.shape
    g = t[c.buf_pages.long().flatten()]                      # [S * ppl, page_rows, ...]
    return g.reshape(S, ppl * c.page_rows, *t.shape[2:])


@pytest.mark.parametrize("chunk,page_rows", [(16, 4), (16, 1), (64, 16)])
def test_exact_decode_paged_equals_contiguous(chunk, page_rows):
    ers = _ers()
    w = dataclasses.replace(synth.workload("decode_b256_h64"), dims=synth.Dims(16, 2, 64, 128, chunk))
    d = w.dims
    S, K = 12, chunk + 9
    params, hist, _, stream = synth.decode_inputs(w, seed=51, batch=S, steps=K)
    prm = layer(params)
    c0 = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, torch.bfloat16)
    c1 = _paged(ers, S, d, torch.bfloat16, page_rows, 52)
    ht = synth.Tokens.concat(hist)
    cu = torch.tensor(np.concatenate([[0], np.cumsum([h.ntokens for h in hist])]), dtype=torch.int32, device=dev())
    hx, hdt, hB, hC = torch_io.tokens_to(ht, dev())
    y0 = ers.chunked_prefill(c0, prm, hx, hdt, hB, hC, cu)
    y1 = ers.chunked_prefill(c1, prm, hx, hdt, hB, hC, cu)
    assert same_bits(y0, y1)
    tok = torch_io.tokens_to(stream, dev(), lead=(K, S))
    ys = []
    for k in range(K):
        a = ers.replay_decode(c0, prm, *(t[k] for t in tok))
        b = ers.replay_decode(c1, prm, *(t[k] for t in tok))
        assert same_bits(a, b), k
        ys.append(b)
    assert same_bits(c0.state, c1.state) and torch.equal(c0.pos, c1.pos)
    # the paged cache against the oracle: history outputs, decoded outputs per (sequence, head), and
    # the boundary checkpoints
    parts = [synth.Tokens.concat([hist[i]] + [stream.slice(k * S + i, k * S + i + 1) for k in range(K)])
             for i in range(S)]
    allt = synth.Tokens.concat(parts)
    cu_o = np.concatenate([[0], np.cumsum([q.ntokens for q in parts])]).astype(np.int64)
    y_o, _ = oracle.recurrence(allt.x, allt.dt, params.A, allt.B, allt.C, params.D, params.dt_bias, cu_o)
    hl = [h.ntokens for h in hist]
    y_hist = np.concatenate([y_o[cu_o[i]:cu_o[i] + hl[i]] for i in range(S)])
    check_out(y1, y_hist, 2e-3, keep=1, cu=cu.cpu().numpy(), what="paged chunked prefill")
    ref = np.stack([y_o[cu_o[i] + hl[i]:cu_o[i + 1]] for i in range(S)])                  # [S, K, H, P]
    check_out(torch.stack(ys).transpose(0, 1), ref, 2e-3, keep=(0, 2), what="paged decode")
    Q = d.chunk
    nb = [(q.ntokens // Q) * Q for q in parts]
    sel = np.concatenate([np.arange(cu_o[i], cu_o[i] + nb[i]) for i in range(S)]).astype(np.int64)
    _, s_o = oracle.recurrence(allt.x[sel], allt.dt[sel], params.A, allt.B[sel], allt.C[sel], params.D,
                               params.dt_bias, np.concatenate([[0], np.cumsum(nb)]))
    assert state_err(c1.state, s_o) <= STATE_TOL
    for name in ("buf_x", "buf_dt", "buf_B", "buf_C"):
        for i in range(S):
            p = int(c0.pos[i])
            assert same_bits(getattr(c0, name)[i, :p], _logical(c1, name)[i, :p]), name


def test_verify_paged_equals_contiguous():
    ers = _ers()
    w = synth.workload("verify_b512_t4")
    d = w.dims
    S, K, T, L = 24, 14, w.drafts, d.chunk
    params, hist, drafts, acc = synth.verify_inputs(w, seed=53, batch=S, steps=K)
    prm = layer(params)
    hx, hdt, hB, hC = torch_io.tokens_to(hist, dev())
    cu = torch.arange(0, S * 32 + 1, 32, dtype=torch.int32, device=dev())
    _, fin = ers.ssd_scan_fwd(hx, hdt, prm, hB, hC, chunk=L, cu_seqlens=cu)
    c0 = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, L, torch.bfloat16, read_copy=True)
    c1 = _paged(ers, S, d, torch.bfloat16, 2, 54, read_copy=True)
    for c in (c0, c1):
        c.state.copy_(fin)
        ers.refresh(c, prm, replayssm=True, drafts_T=L + 1)
    dx, ddt, dB, dC = torch_io.tokens_to(drafts, dev(), lead=(K, S, T))
    acc_t = torch.from_numpy(acc).to(dev())
    # the oracle's protocol model (fp64 anchor, bf16 read copy) on every sequence of the paged cache
    _, anchor = oracle.recurrence(hist.x, hist.dt, params.A, hist.B, hist.C, params.D, params.dt_bias,
                                  np.arange(0, S * 32 + 1, 32))
    model = oracle.ReplaySSMModel(params, anchor, L)
    chk = StepCheck(2e-3, keep=(0, 2), what="paged verify")
    shp = {f: getattr(drafts, f).reshape(K, S, T, *getattr(drafts, f).shape[1:]) for f in ("x", "dt", "B", "C")}
    for k in range(K):
        a = ers.spec_verify(c0, prm, dx[k], ddt[k], dB[k], dC[k]); ers.commit(c0, acc_t[k], T)
        b = ers.spec_verify(c1, prm, dx[k], ddt[k], dB[k], dC[k]); ers.commit(c1, acc_t[k], T)
        assert same_bits(a, b), k
        y_o = model.verify([tuple(np.ascontiguousarray(shp[f][k, i]) for f in ("x", "dt", "B", "C"))
                            for i in range(S)])
        model.commit([int(v) for v in acc[k]])
        chk.step(b, y_o, f"step {k}")
    chk.finish()
    assert same_bits(c0.state, c1.state) and torch.equal(c0.pos, c1.pos)
    assert same_bits(c0.read_copy, c1.read_copy)
    assert np.array_equal(c1.pos.cpu().numpy(), model.h())
    assert state_err(c1.state, model.anchor) <= STATE_TOL


def test_bad_page_index_is_reported_and_clamped():
    ers = _ers()
    w = dataclasses.replace(synth.workload("decode_b256_h64"), dims=synth.Dims(16, 2, 64, 128, 16))
    d = w.dims
    S = 4
    params, _, _, stream = synth.decode_inputs(w, seed=55, batch=S, steps=1)
    prm = layer(params)
    c = _paged(ers, S, d, torch.bfloat16, 4, 56)
    c.buf_pages[2, 0] = c.npages + 3
    st = ers.Status(dev())
    tok = torch_io.tokens_to(stream, dev(), lead=(1, S))
    ers.replay_decode(c, prm, *(t[0] for t in tok), status=st, check=False)
    assert st.read() == 8                                         # ERS_ESLOT
