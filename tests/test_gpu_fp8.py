"""FP8 e4m3 and NVFP4 read copies on the GPU (ReplaySSM notes, "Paper-reported results": FP8 or
NVFP4 reads over an FP32 recurrence; the page gives no quantiser, so the library defines them:
FP8 with a power-of-two scale per state row; NVFP4 with e2m1 codes, an e4m3 scale per 16 values
and a power-of-two scale per row).

The copies the kernels cast equal the oracle's FP8 rounding of the same fp32 state bit for bit
(refresh, fused refresh in decode, verify flush); verify outputs equal non-speculative FP8 decode
bit for bit; the anchor does not depend on the read precision; parity with the oracle's protocol
model run with the FP8 read cast."""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import torch_io
from gpu_helpers import OUT_TOL_BF16, dev, layer, same_bits, read_values

pytestmark = pytest.mark.gpu


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _params(H, seed=0):
    return synth.make_params(np.random.Generator(np.random.PCG64(seed)), H)


_CAST = {"fp8": oracle.fp8_rows_round, "nvfp4": oracle.nvfp4_rows_round}


@pytest.mark.parametrize("read_dtype", ["fp8", "nvfp4"])
def test_refresh_cast_matches_oracle(read_dtype):
    """ReplaySSM refresh of an empty history only recasts: the copy is the oracle's FP8 / NVFP4
    rounding of the fp32 anchor as stored (edge rows: zero, subnormal codes, constant, single entry,
    rows spanning 60 binades)."""
    ers = _ers()
    S, H, G, P, N, L = 6, 16, 2, 64, 128, 16
    st = synth.quant_probe_state(11, (S, H, P, N))
    cache = ers.ReplayCache(S, H, G, P, N, L, torch.bfloat16, read_copy=True, read_dtype=read_dtype)
    cache.state.copy_(torch.from_numpy(st))
    prm = layer(_params(H))
    ers.refresh(cache, prm, replayssm=True, drafts_T=L + 1)   # h = 0 + T > L everywhere
    got = read_values(cache).cpu().numpy()
    want = _CAST[read_dtype](st).astype(np.float32)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert same_bits(cache.state, torch.from_numpy(st).to(dev()))     # the anchor is untouched
    assert int(cache.pos.abs().sum()) == 0


def test_fp8_cast_untouched_without_flush():
    """A refresh whose flush rule does not fire leaves codes and scales as they were."""
    ers = _ers()
    S, H, G, P, N, L = 3, 8, 1, 64, 128, 16
    cache = ers.ReplayCache(S, H, G, P, N, L, torch.bfloat16, read_copy=True, read_dtype="fp8")
    cache.read_copy.fill_(0x5A)
    cache.read_scale.fill_(2.0)
    ers.refresh(cache, layer(_params(H)), replayssm=True, drafts_T=4)  # h + T = 4 <= L
    assert int((cache.read_copy != 0x5A).sum()) == 0 and bool((cache.read_scale == 2.0).all())


def _exact_mode_cache(S, K, seed, read_dtype, dims=synth.Dims(64, 8, 64, 128, 16)):
    """An exact-mode cache at position 0 holding an fp32 checkpoint, with exact-fold tokens (A = 0,
    dt far above softplus's pass-through, dyadic x and B): every refresh rounds one exact sum to fp32,
    as the oracle's fold taken through fp32 does."""
    ers = _ers()
    params, stream, st0 = synth.exact_fold_inputs(seed, S, K, dims)
    prm = layer(params)
    cache = ers.ReplayCache(S, dims.nheads, dims.ngroups, dims.headdim, dims.dstate, dims.chunk, torch.bfloat16,
                            read_copy=True, read_dtype=read_dtype)
    cache.state.copy_(torch.from_numpy(st0))
    return params, prm, cache, stream, st0, torch_io.tokens_to(stream, dev(), lead=(K, S))


def test_fp8_exact_mode_fused_refresh_casts_and_matches_separate():
    """Exact-mode decode keeps an FP8 copy: every checkpoint a filled chunk writes equals the oracle's
    fold (value for value) and the copy its FP8 rounding; fused and separate refresh agree bit for
    bit; the outputs (which read the fp32 checkpoint) equal those of a run with a bf16 copy."""
    ers = _ers()
    S, K, Q = 24, 40, 16
    params, prm, c1, stream, st0, (sx, sdt, sB, sC) = _exact_mode_cache(S, K, 3, "fp8")
    c2 = _exact_mode_cache(S, K, 3, "fp8")[2]
    c3 = _exact_mode_cache(S, K, 3, "bf16")[2]
    ck = st0.astype(np.float64)
    casts = 0
    for k in range(K):
        y1 = ers.replay_decode(c1, prm, sx[k], sdt[k], sB[k], sC[k], fuse_refresh=True)
        y2 = ers.replay_decode(c2, prm, sx[k], sdt[k], sB[k], sC[k], fuse_refresh=False)
        ers.refresh(c2, prm)
        y3 = ers.replay_decode(c3, prm, sx[k], sdt[k], sB[k], sC[k], fuse_refresh=True)
        assert same_bits(y1, y2) and same_bits(y1, y3), k
        assert torch.equal(c1.read_copy, c2.read_copy) and same_bits(c1.read_scale, c2.read_scale), k
        if (k + 1) % Q == 0:                            # every slot filled its chunk at this step
            r = (np.arange(k + 1 - Q, k + 1)[None, :] * S + np.arange(S)[:, None]).ravel()   # slot-major rows
            _, ck = oracle.recurrence(stream.x[r], stream.dt[r], params.A, stream.B[r], stream.C[r], params.D,
                                      params.dt_bias, np.arange(0, S * Q + 1, Q), ck)
            want = ck.astype(np.float32)
            assert np.array_equal(c1.state.cpu().numpy().view(np.uint32), want.view(np.uint32)), k
            got = read_values(c1).cpu().numpy()
            assert np.array_equal(got.view(np.uint32), oracle.fp8_rows_round(ck).astype(np.float32).view(np.uint32))
            casts += S
    assert casts > 0
    assert same_bits(c1.state, c3.state) and torch.equal(c1.pos, c3.pos)


def _verify_run(w, S, K, seed, read_dtype):
    ers = _ers()
    d = w.dims
    params, hist, drafts, acc = synth.verify_inputs(w, seed=seed, batch=S, steps=K)
    prm = layer(params)
    history = 32
    hx, hdt, hB, hC = torch_io.tokens_to(hist, dev())
    cu = torch.arange(0, S * history + 1, history, dtype=torch.int32, device=dev())
    _, fin = ers.ssd_scan_fwd(hx, hdt, prm, hB, hC, chunk=d.chunk, cu_seqlens=cu)

    def fresh():
        c = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, d.chunk, torch.bfloat16, read_copy=True,
                            read_dtype=read_dtype)
        c.state.copy_(fin)
        ers.refresh(c, prm, replayssm=True, drafts_T=d.chunk + 1)
        return c
    return params, prm, hist, drafts, acc, fresh


@pytest.mark.parametrize("read_dtype", ["fp8", "nvfp4"])
def test_verify_equals_nonspec_decode_and_oracle(read_dtype):
    """Verify + commit with an FP8 / NVFP4 copy: accepted drafts equal non-speculative ReplaySSM
    decode over the same committed stream bit for bit, and outputs match the oracle's protocol model
    run with the same read cast."""
    ers = _ers()
    w = synth.workload("verify_b512_t4")
    S, K, T, L = 64, 24, w.drafts, w.dims.chunk
    samples = [0, 13, 63]
    params, prm, hist, drafts, acc, fresh = _verify_run(w, S, K, 7, read_dtype)
    cache, ref = fresh(), fresh()
    dx, ddt, dB, dC = torch_io.tokens_to(drafts, dev(), lead=(K, S, T))
    acc_t = torch.from_numpy(acc).to(dev())
    rows = np.concatenate([np.arange(i * 32, (i + 1) * 32) for i in samples])
    _, anchor = oracle.recurrence(hist.x[rows], hist.dt[rows], params.A, hist.B[rows], hist.C[rows], params.D,
                                  params.dt_bias, np.arange(0, len(samples) * 32 + 1, 32))
    model = oracle.ReplaySSMModel(params, anchor, L, read_cast=_CAST[read_dtype])
    flushes = 0
    for k in range(K):
        flushing = ((cache.pos + T) > L).nonzero().flatten().tolist()
        y = ers.spec_verify(cache, prm, dx[k], ddt[k], dB[k], dC[k])
        flushes += len(flushing)
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
        dr = [tuple(np.ascontiguousarray(getattr(drafts, f).reshape(K, S, T, *getattr(drafts, f).shape[1:])[k, i])
                    for f in ("x", "dt", "B", "C")) for i in samples]
        y_o = model.verify(dr)
        model.commit([int(acc[k, i]) for i in samples])
        g = y[samples].float().cpu().numpy().astype(np.float64)
        assert np.abs(g - y_o).mean() <= OUT_TOL_BF16 * np.abs(y_o).mean(), k
    assert flushes > 0
    assert torch.equal(cache.pos, ref.pos)
    assert same_bits(cache.state, ref.state)
    assert torch.equal(cache.read_copy, ref.read_copy) and same_bits(cache.read_scale, ref.read_scale)
    if read_dtype == "nvfp4":
        assert torch.equal(cache.read_block_scale, ref.read_block_scale)


@pytest.mark.parametrize("read_dtype", ["fp8", "nvfp4"])
def test_verify_flush_casts_equal_the_oracle_under_exact_folds(read_dtype):
    """Verify + commit with exact-fold drafts: after every step the anchors equal the oracle model's
    and the copies its FP8 / NVFP4 rounding of them, value for value."""
    ers = _ers()
    d = synth.Dims(64, 8, 64, 128, 16)
    S, K, T, L = 16, 14, 4, d.chunk
    params, stream, st0 = synth.exact_fold_inputs(21, S, K * T, d)
    prm = layer(params)
    acc = np.random.Generator(np.random.PCG64(22)).integers(0, T + 1, (K, S)).astype(np.int32)
    cache = ers.ReplayCache(S, d.nheads, d.ngroups, d.headdim, d.dstate, L, torch.bfloat16, read_copy=True,
                            read_dtype=read_dtype)
    cache.state.copy_(torch.from_numpy(st0))
    ers.refresh(cache, prm, replayssm=True, drafts_T=L + 1)
    model = oracle.ReplaySSMModel(params, st0.astype(np.float64), L, read_cast=_CAST[read_dtype])
    sh = lambda a: a.reshape(K, S, T, *a.shape[1:])
    dx, ddt, dB, dC = (torch.from_numpy(sh(a)).to(dev()) for a in (stream.x, stream.dt, stream.B, stream.C))
    dx, dB, dC = dx.to(torch.bfloat16), dB.to(torch.bfloat16), dC.to(torch.bfloat16)
    acc_t = torch.from_numpy(acc).to(dev())
    flushes = 0
    for k in range(K):
        ers.spec_verify(cache, prm, dx[k], ddt[k], dB[k], dC[k])
        ers.commit(cache, acc_t[k], T)
        model.verify([tuple(sh(a)[k, i] for a in (stream.x, stream.dt, stream.B, stream.C)) for i in range(S)])
        model.commit(acc[k])
        assert np.array_equal(cache.state.cpu().numpy().view(np.uint32),
                              model.anchor.astype(np.float32).view(np.uint32)), k
        assert np.array_equal(read_values(cache).cpu().numpy().astype(np.float64), model.read), k
    assert model.flushes > 0


def test_anchor_independent_of_read_precision():
    """The same verify/commit run with a bf16, an FP8 and an NVFP4 copy: outputs differ, the anchors
    and committed pointers are bit-identical (refresh folds the fp32 anchor, never the copy)."""
    ers = _ers()
    w = synth.workload("verify_b512_t4")
    S, K, T = 32, 20, w.drafts
    _, prm, _, drafts, acc, fresh16 = _verify_run(w, S, K, 9, "bf16")
    c16, c8, c4 = fresh16(), _verify_run(w, S, K, 9, "fp8")[-1](), _verify_run(w, S, K, 9, "nvfp4")[-1]()
    dx, ddt, dB, dC = torch_io.tokens_to(drafts, dev(), lead=(K, S, T))
    acc_t = torch.from_numpy(acc).to(dev())
    differ = False
    for k in range(K):
        y16 = ers.spec_verify(c16, prm, dx[k], ddt[k], dB[k], dC[k]); ers.commit(c16, acc_t[k], T)
        y8 = ers.spec_verify(c8, prm, dx[k], ddt[k], dB[k], dC[k]); ers.commit(c8, acc_t[k], T)
        y4 = ers.spec_verify(c4, prm, dx[k], ddt[k], dB[k], dC[k]); ers.commit(c4, acc_t[k], T)
        differ |= not same_bits(y16, y8) and not same_bits(y8, y4)
    assert differ
    assert same_bits(c16.state, c8.state) and torch.equal(c16.pos, c8.pos)
    assert same_bits(c16.state, c4.state) and torch.equal(c16.pos, c4.pos)


def test_fp8_unsupported_shapes_raise():
    ers = _ers()
    H, G, P, N = 8, 2, 64, 128
    prm = layer(_params(H))
    cache = ers.ReplayCache(2, H, G, P, N, 32, torch.bfloat16, read_copy=True, read_dtype="fp8")
    x = torch.zeros(2, H, P, dtype=torch.bfloat16, device=dev())
    dt = torch.zeros(2, H, dtype=torch.float32, device=dev())
    B = torch.zeros(2, G, N, dtype=torch.bfloat16, device=dev())
    with pytest.raises(ers.ErsError) as e:
        ers.replay_decode(cache, prm, x, dt, B, B.clone(), replayssm=True)
    assert e.value.code == 12                                           # ERS_EUNSUPPORTED
    c4 = ers.ReplayCache(2, H, G, P, N, 16, torch.bfloat16, read_copy=True, read_dtype="nvfp4")
    with pytest.raises(ers.ErsError) as e:
        ers.replay_decode(c4, prm, x, dt, B, B.clone())                # exact mode keeps no NVFP4 copy
    assert e.value.code == 12
