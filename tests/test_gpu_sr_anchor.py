"""fp16 ReplaySSM anchors written by stochastic rounding (ReplaySSM notes, "Paper-reported results":
"NVFP4 read / FP16+SR recurrence"; the rounding rule and the random words are this library's
reading: Philox4x32-10 at counter (nonce, slot, h * P + d, n / 4)).

* Anchor writes equal the oracle's, value for value, under exact folds (A = 0, dt far above
  softplus's pass-through, dyadic x and B, so both sides round the same exact sum once to fp32),
  across the fp16 range (subnormals, smallest normals, saturation); the read copy cast from the
  same values equals the oracle's too.
* Fused flush in decode == ers_refresh + decode, verify == non-speculative decode, bit for bit, with
  fp16 anchors and an NVFP4 copy (the paper's tp4_hi16_sr configuration).
* Parity with the oracle's protocol model run with the same rounding (anchors within a few fp16
  steps, outputs within the bf16 output tolerance)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from synth import torch_io
from gpu_helpers import MAX_REL_NARROW, OUT_TOL_BF16, StepCheck, dev, layer, same_bits, read_values

pytestmark = pytest.mark.gpu

KEY = (0x1234ABCD, 0x0BADF00D)
# fp16 anchors: the GPU's fp32 refresh result and the oracle's differ in their last fp32 bits, which
# flips an occasional stochastic-rounding decision by one fp16 step (2^-10 relative); a few refreshes
# accumulate a few such steps.
ANCHOR_TOL_F16 = 4 * 2.0 ** -10


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _anchor_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.float().cpu().numpy().astype(np.float64)
    P, N = ref.shape[-2], ref.shape[-1]
    d = np.abs(g - ref).reshape(-1, P * N).max(axis=1)
    r = np.abs(ref).reshape(-1, P * N).max(axis=1)
    return float((d / np.maximum(r, 1e-30)).max())


def _oracle_start(params, hist) -> np.ndarray:
    """The oracle's state after each sequence's history (fp64 [S, H, P, N]): the starting anchor of
    both the oracle model and the caches (which get its fp16 cast)."""
    ht = synth.Tokens.concat(hist)
    cu = np.concatenate([[0], np.cumsum([h.ntokens for h in hist])])
    _, fin = oracle.recurrence(ht.x, ht.dt, params.A, ht.B, ht.C, params.D, params.dt_bias, cu)
    return fin


def _setup(S, K, seed, read_dtype, anchor, dims=synth.Dims(64, 8, 64, 128, 16)):
    ers = _ers()
    w = dataclasses.replace(synth.workload("decode_b256_h64"), dims=dims)
    d, L = w.dims, w.dims.chunk
    params, hist, h0, stream = synth.decode_inputs(w, seed=seed, batch=S, steps=K)
    prm = layer(params)
    st16 = _oracle_start(params, hist).astype(np.float32).astype(np.float16)   # on the fp16 grid

    def fresh(anc=anchor):
        c = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, L, torch.bfloat16, read_copy=True,
                            read_dtype=read_dtype, anchor=anc, sr_key=KEY)
        c.state.copy_(torch.from_numpy(st16 if anc == "fp16_sr" else st16.astype(np.float32)))
        ers.refresh(c, prm, replayssm=True, drafts_T=L + 1)    # h = 0: the anchor keeps its bits
        return c
    return params, prm, stream, torch_io.tokens_to(stream, dev(), lead=(K, S)), st16, fresh


def _exact_model(params, anchor0, L, read_dtype, nonce):
    cast = oracle.nvfp4_rows_round if read_dtype == "nvfp4" else oracle.bf16_round
    return oracle.ReplaySSMModel(params, anchor0, L, read_cast=cast,
                                 anchor_round=lambda i, fin: oracle.sr_fp16_anchor(fin, KEY, nonce, i))


def _run_exact(ers, params, stream, st16, S, K, read_dtype, nonce):
    """K decodes of every slot from the fp16 anchor st16, then a refresh of every slot; returns the
    cache and the oracle model run over the same records (the fold is exact on both sides, so the
    stochastic rounding sees the same fp32 values)."""
    d, L = DIMS, DIMS.chunk
    prm = layer(params)
    c = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, L, torch.bfloat16, read_copy=True,
                        read_dtype=read_dtype, anchor="fp16_sr", sr_key=KEY)
    c.state.copy_(st16)
    ers.refresh(c, prm, replayssm=True, drafts_T=L + 1)        # h = 0: the anchor keeps its bits
    model = _exact_model(params, st16.float().cpu().numpy().astype(np.float64), L, read_dtype, nonce)
    tok = torch_io.tokens_to(stream, dev(), lead=(K, S))
    for k in range(K):
        ers.replay_decode(c, prm, *(t[k] for t in tok), replayssm=True, fuse_refresh=False)
        model.verify([(stream.x[r:r + 1], stream.dt[r:r + 1], stream.B[r:r + 1], stream.C[r:r + 1])
                      for r in range(k * S, (k + 1) * S)])
        model.commit([1] * S)
    c.sr_nonce = nonce
    ers.refresh(c, prm, replayssm=True, drafts_T=L)            # h + L > L: every slot folds
    model.refresh(list(range(S)))
    return c, model


DIMS = synth.Dims(64, 8, 64, 128, 16)


@pytest.mark.parametrize("read_dtype", ["bf16", "nvfp4"])
def test_sr_anchor_write_matches_oracle(read_dtype):
    """Exact folds (A = 0, dt far above softplus's pass-through, dyadic x and B): the fp32 value each
    rounding sees is the single rounding of an exact sum on both sides, so the fp16 anchor and the
    read copy equal the oracle's, value for value."""
    ers = _ers()
    S, K = 6, 9
    params, stream, st0 = synth.exact_fold_inputs(31, S, K, DIMS)
    st16 = torch.from_numpy(st0.astype(np.float16)).to(dev())
    c, model = _run_exact(ers, params, stream, st16, S, K, read_dtype, 77)
    got = c.state.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, model.anchor)
    assert np.array_equal(read_values(c).cpu().numpy().astype(np.float64), model.read)
    plain = oracle.ReplaySSMModel(params, st16.float().cpu().numpy().astype(np.float64), DIMS.chunk)
    for k in range(K):
        plain.verify([(stream.x[r:r + 1], stream.dt[r:r + 1], stream.B[r:r + 1], stream.C[r:r + 1])
                      for r in range(k * S, (k + 1) * S)])
        plain.commit([1] * S)
    plain.refresh(list(range(S)))
    moved = got != plain.anchor.astype(np.float32).astype(np.float64)
    assert moved.mean() > 0.5                                   # rounding did happen


def test_fused_flush_and_verify_with_sr_anchors():
    """tp4_hi16_sr: NVFP4 copy, fp16 SR anchor.  Fused flush == refresh + decode; verify == the
    non-speculative decode; anchors and outputs match the oracle's protocol model."""
    ers = _ers()
    S, K, L = 32, 40, 16
    samples = [0, 9, 31]
    params, prm, stream, tok, st16, fresh = _setup(S, K, 32, "nvfp4", "fp16_sr")
    c1, c2 = fresh(), fresh()
    anchor0 = st16.astype(np.float64)[samples]
    nonce = {"v": 0}
    model = oracle.ReplaySSMModel(params, anchor0, L, read_cast=oracle.nvfp4_rows_round,
                                  anchor_round=lambda i, fin: oracle.sr_fp16_anchor(fin, KEY, nonce["v"],
                                                                                    samples[i]))
    chk = StepCheck(OUT_TOL_BF16, keep=(0, 1), max_rel=MAX_REL_NARROW, what="ReplaySSM decode")
    flushes = 0
    for k in range(K):
        nonce["v"] = 1000 + k
        c1.sr_nonce = c2.sr_nonce = 1000 + k
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
    assert flushes > 0
    assert same_bits(c1.state, c2.state) and torch.equal(c1.pos, c2.pos)
    assert torch.equal(c1.read_copy, c2.read_copy) and torch.equal(c1.read_block_scale, c2.read_block_scale)
    assert _anchor_err(c1.state[samples], model.anchor) <= ANCHOR_TOL_F16


def test_verify_equals_nonspec_decode_with_sr_anchors():
    ers = _ers()
    w = synth.workload("verify_b512_t4")
    d = w.dims
    S, K, T, L = 48, 20, w.drafts, d.chunk
    params, hist, drafts, acc = synth.verify_inputs(w, seed=33, batch=S, steps=K)
    prm = layer(params)
    hx, hdt, hB, hC = torch_io.tokens_to(hist, dev())
    cu = torch.arange(0, S * 32 + 1, 32, dtype=torch.int32, device=dev())
    _, fin = ers.ssd_scan_fwd(hx, hdt, prm, hB, hC, chunk=L, cu_seqlens=cu)

    def fresh():
        c = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, L, torch.bfloat16, read_copy=True,
                            read_dtype="nvfp4", anchor="fp16_sr", sr_key=KEY)
        c.state.copy_(fin.half())
        ers.refresh(c, prm, replayssm=True, drafts_T=L + 1)
        return c
    cache, ref = fresh(), fresh()
    dx, ddt, dB, dC = torch_io.tokens_to(drafts, dev(), lead=(K, S, T))
    acc_t = torch.from_numpy(acc).to(dev())
    for k in range(K):
        cache.sr_nonce = ref.sr_nonce = 5000 + k
        y = ers.spec_verify(cache, prm, dx[k], ddt[k], dB[k], dC[k])
        ers.commit(cache, acc_t[k], T)
        ers.refresh(ref, prm, replayssm=True, drafts_T=T)
        ref.sr_nonce = 0                                        # decodes write no anchors
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
    assert torch.equal(cache.pos, ref.pos) and same_bits(cache.state, ref.state)
    assert torch.equal(cache.read_copy, ref.read_copy)


def test_sr_anchor_unsupported_calls_raise():
    ers = _ers()
    H, G, P, N = 8, 2, 64, 128
    prm = layer(synth.make_params(np.random.Generator(np.random.PCG64(0)), H))
    x = torch.zeros(2, H, P, dtype=torch.bfloat16, device=dev())
    dt = torch.zeros(2, H, dtype=torch.float32, device=dev())
    B = torch.zeros(2, G, N, dtype=torch.bfloat16, device=dev())
    c = ers.ReplayCache(2, H, G, P, N, 16, torch.bfloat16, read_copy=True, anchor="fp16_sr")
    with pytest.raises(ers.ErsError) as e:
        ers.replay_decode(c, prm, x, dt, B, B.clone())                 # exact mode
    assert e.value.code == 12
    c32 = ers.ReplayCache(2, H, G, P, N, 16, torch.float32, read_copy=True, anchor="fp16_sr")
    with pytest.raises(ers.ErsError) as e:
        ers.replay_decode(c32, prm, x.float(), dt, B.float(), B.float(), replayssm=True)   # fp32 io
    assert e.value.code == 12


def test_sr_anchor_write_edge_values():
    """Anchors spanning the fp16 range (subnormals, the smallest normals, values near 65504) under
    exact folds whose increments are scaled per head to the anchor's own spacing (x times 2^-27 on
    the subnormal head, 2^-17 on the smallest normals): the fp16 writes equal the oracle's rounding,
    value for value, on every path (subnormal, normal, saturation)."""
    ers = _ers()
    S, K, H, P, N = 6, 5, 64, 64, 128
    params, stream, _ = synth.exact_fold_inputs(34, S, K, DIMS)
    stream.x[:, 1] *= np.float32(2.0 ** -27)
    stream.x[:, 2] *= np.float32(2.0 ** -17)
    st = synth.quant_probe_state(35, (S, H, P, N))
    st = np.clip(st, -60000.0, 60000.0)
    st[0, 1] = np.float32(2.0 ** -20) * np.sign(st[0, 1])                 # a head of fp16 subnormals
    st[0, 2] = np.float32(2.0 ** -14) * (1 + (np.arange(N) % 7) / 8.0)     # the smallest normals
    st[1, 3] = np.float32(65472.0) * np.where(st[1, 3] < 0, -1, 1)          # next to the fp16 maximum
    st16 = torch.from_numpy(st.astype(np.float16)).to(dev())
    c, model = _run_exact(ers, params, stream, st16, S, K, "nvfp4", 91)
    got = c.state.float().cpu().numpy().astype(np.float64)
    assert np.array_equal(got, model.anchor)
    sub = np.abs(got[0, 1]) < 2.0 ** -14
    assert sub.mean() > 0.9 and np.any(got[0, 1] != 0)                   # the subnormal path ran
    assert np.any(np.abs(got) == 65504.0)                                 # and the saturation
