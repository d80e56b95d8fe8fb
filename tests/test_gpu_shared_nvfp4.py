"""The shared NVFP4 state (ReplaySSM notes, "Paper-reported results": the shared-FP4 recurrence mode;
the stochastic rounding of the codes and the random words are this library's reading: Philox4x32-10
at counter (nonce, slot, h * P + d, n / 4), as for fp16 anchors).  The NVFP4 read copy is the only
state: a refresh folds from its values and writes it back with stochastically rounded codes.

* With exact folds (A = 0, dt far above softplus's pass-through, dyadic x and B: every product and
  sum is exact in fp32 and in fp64) the refreshed state is a value the oracle reaches exactly: after
  two rounds of refreshes the GPU's state equals the oracle model's, value for value.
* Fused flush in decode == ers_refresh + decode, verify == non-speculative decode, bit for bit.
* Parity with the oracle's protocol model on the decode workload's inputs; an empty history leaves
  the state's bytes as they are."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import torch_io
from gpu_helpers import MAX_REL_NARROW, OUT_TOL_BF16, StepCheck, dev, layer, same_bits, read_values

pytestmark = pytest.mark.gpu

KEY = (0x2468ACE0, 0x13579BDF)
DIMS = synth.Dims(64, 8, 64, 128, 16)


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _shared(ers, S, d, prm, fin):
    c = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, torch.bfloat16, read_copy=True,
                        read_dtype="nvfp4", anchor="nvfp4_sr_shared", sr_key=KEY)
    c.seed(fin, prm)
    return c


def _copy_bytes(c):
    return (c.read_copy.clone(), c.read_block_scale.clone(), c.read_scale.clone())


def _same_copy(a, b):
    return all(torch.equal(x.view(torch.uint8), y.view(torch.uint8)) for x, y in zip(a, b))


def test_shared_state_refreshes_equal_the_oracle_exactly():
    ers = _ers()
    S, L = 6, DIMS.chunk
    K1, K2 = 11, 7
    params, stream, st0 = synth.exact_fold_inputs(81, S, K1 + K2, DIMS)
    prm = layer(params)
    c = _shared(ers, S, DIMS, prm, torch.from_numpy(st0).to(dev()))
    a0 = oracle.nvfp4_rows_round(st0)                                   # the seed: round-to-nearest cast
    assert np.array_equal(read_values(c).cpu().numpy().astype(np.float64), a0)
    nonce = {"v": 0}
    model = oracle.ReplaySSMModel(params, a0, L, shared=True,
                                  anchor_round=lambda i, fin: oracle.nvfp4_sr_state(fin, KEY, nonce["v"], i))
    tok = torch_io.tokens_to(stream, dev(), lead=(K1 + K2, S))
    for k in range(K1 + K2):
        ers.replay_decode(c, prm, *(t[k] for t in tok), replayssm=True, fuse_refresh=False)
        rows = slice(k * S, (k + 1) * S)
        model.verify([(stream.x[r:r + 1], stream.dt[r:r + 1], stream.B[r:r + 1], stream.C[r:r + 1])
                      for r in range(rows.start, rows.stop)])
        model.commit([1] * S)
        if k + 1 in (K1, K1 + K2):                                      # refresh every slot
            nonce["v"] = 500 + k
            c.sr_nonce = 500 + k
            ers.refresh(c, prm, replayssm=True, drafts_T=L)
            model.refresh(list(range(S)))
            got = read_values(c).cpu().numpy().astype(np.float64)
            assert np.array_equal(got, model.anchor), k
    assert model.flushes == 2 * S


def test_fused_flush_equals_refresh_and_decode_and_matches_the_model():
    ers = _ers()
    S, K, L = 32, 40, DIMS.chunk
    samples = [0, 13, 31]
    w = dataclasses.replace(synth.workload("decode_b256_h64"), dims=DIMS)
    params, hist, _, stream = synth.decode_inputs(w, seed=82, batch=S, steps=K)
    prm = layer(params)
    ht = synth.Tokens.concat(hist)
    cu = np.concatenate([[0], np.cumsum([h.ntokens for h in hist])])
    _, fin = oracle.recurrence(ht.x, ht.dt, params.A, ht.B, ht.C, params.D, params.dt_bias, cu)
    fin32 = fin.astype(np.float32)                     # the oracle's state after the history starts both
    c1, c2 = (_shared(ers, S, DIMS, prm, torch.from_numpy(fin32).to(dev())) for _ in range(2))
    a0 = oracle.nvfp4_rows_round(fin32[samples])
    assert np.array_equal(read_values(c1)[samples].cpu().numpy().astype(np.float64), a0)
    nonce = {"v": 0}
    model = oracle.ReplaySSMModel(params, a0, L, shared=True,
                                  anchor_round=lambda i, f: oracle.nvfp4_sr_state(f, KEY, nonce["v"], samples[i]))
    tok = torch_io.tokens_to(stream, dev(), lead=(K, S))
    chk = StepCheck(OUT_TOL_BF16, keep=(0, 1), max_rel=MAX_REL_NARROW, what="ReplaySSM decode")
    flushes = 0
    for k in range(K):
        nonce["v"] = c1.sr_nonce = c2.sr_nonce = 3000 + k
        flushes += int((c1.pos == L).sum())
        y1 = ers.replay_decode(c1, prm, *(t[k] for t in tok), replayssm=True, fuse_refresh=True)
        ers.refresh(c2, prm, replayssm=True, drafts_T=1)
        y2 = ers.replay_decode(c2, prm, *(t[k] for t in tok), replayssm=True, fuse_refresh=False)
        assert same_bits(y1, y2), k
        rows = [k * S + i for i in samples]
        y_o = model.verify([(stream.x[r:r + 1], stream.dt[r:r + 1], stream.B[r:r + 1], stream.C[r:r + 1])
                            for r in rows])
        model.commit([1] * len(samples))
        chk.step(y1[samples], y_o[:, 0], f"step {k}")
    chk.finish()
    assert flushes > 0 and model.flushes > 0
    assert torch.equal(c1.pos, c2.pos) and _same_copy(_copy_bytes(c1), _copy_bytes(c2))
    # the GPU folds in fp32 and the model in fp64: a stochastic decision flips only where the two
    # fp32 values straddle the threshold of a word (about 2^-23 relative per value and flush), so
    # almost every value is the model's and none is more than a few code steps away
    got = read_values(c1)[samples].cpu().numpy().astype(np.float64)
    assert np.mean(got != model.anchor) < 1e-3


def test_verify_equals_nonspec_decode_and_empty_history_keeps_the_state():
    ers = _ers()
    w = synth.workload("verify_b512_t4")
    d = w.dims
    S, K, T, L = 48, 20, w.drafts, d.chunk
    params, hist, drafts, acc = synth.verify_inputs(w, seed=83, batch=S, steps=K)
    prm = layer(params)
    hx, hdt, hB, hC = torch_io.tokens_to(hist, dev())
    cu = torch.arange(0, S * 32 + 1, 32, dtype=torch.int32, device=dev())
    _, fin = ers.ssd_scan_fwd(hx, hdt, prm, hB, hC, chunk=L, cu_seqlens=cu)
    cache, ref = _shared(ers, S, d, prm, fin), _shared(ers, S, d, prm, fin)
    before = _copy_bytes(cache)
    cache.sr_nonce = 1
    ers.refresh(cache, prm, replayssm=True, drafts_T=L + 1)            # every slot has pos = 0
    assert _same_copy(before, _copy_bytes(cache))
    dx, ddt, dB, dC = torch_io.tokens_to(drafts, dev(), lead=(K, S, T))
    acc_t = torch.from_numpy(acc).to(dev())
    flushed = 0
    for k in range(K):
        cache.sr_nonce = ref.sr_nonce = 7000 + k
        flushed += int(((cache.pos + T) > L).sum())
        y = ers.spec_verify(cache, prm, dx[k], ddt[k], dB[k], dC[k])
        ers.commit(cache, acc_t[k], T)
        ers.refresh(ref, prm, replayssm=True, drafts_T=T)
        a = acc[k]
        for j in range(T):
            sel = np.nonzero(a > j)[0]
            if sel.size == 0:
                break
            sel_t = torch.from_numpy(sel.astype(np.int32)).to(dev())
            sl = sel_t.long()
            yd = ers.replay_decode(ref, prm, dx[k, sl, j], ddt[k, sl, j], dB[k, sl, j], dC[k, sl, j], slot=sel_t,
                                   replayssm=True, fuse_refresh=False)
            assert same_bits(yd, y[sl, j]), f"step {k} draft {j}"
    assert flushed > 0
    assert torch.equal(cache.pos, ref.pos) and _same_copy(_copy_bytes(cache), _copy_bytes(ref))
