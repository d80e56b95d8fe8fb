"""The per-token state-writeback (SSU) comparison kernel, and device-side error reporting."""
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


def test_ssu_matches_oracle_and_is_batch_invariant():
    ers = _ers()
    w = synth.workload("decode_b256_h64")
    d = w.dims
    S, K = 256, 8
    rng = np.random.Generator(np.random.PCG64(11))
    params = synth.make_params(rng, d.nheads)
    toks = synth.make_tokens(rng, K * S, d, True)
    init = rng.standard_normal((S, d.nheads, d.headdim, d.dstate)).astype(np.float32)
    prm = layer(params)
    x, dt, B, C = torch_io.tokens_to(toks, dev(), lead=(K, S))
    state = torch.from_numpy(init).to(dev())
    ys = torch.stack([ers.ssu_update(state, prm, x[k], dt[k], B[k], C[k]) for k in range(K)])
    for i in (0, 3, 255):
        rows = [k * S + i for k in range(K)]
        y_o, s_o = oracle.recurrence(toks.x[rows], toks.dt[rows], params.A, toks.B[rows], toks.C[rows], params.D,
                                     params.dt_bias, init_state=init[i:i + 1])
        check_out(ys[:, i], y_o, 2e-3, keep=1, what=f"SSU sequence {i}")
        assert state_err(state[i], s_o[0]) <= STATE_TOL
    # batch invariance: the first b sequences run alone give the same bits
    for b in (1, 4, 16, 64):
        st = torch.from_numpy(init[:b].copy()).to(dev())
        yb = torch.stack([ers.ssu_update(st, prm, x[k, :b], dt[k, :b], B[k, :b], C[k, :b]) for k in range(K)])
        assert same_bits(yb, ys[:, :b]) and same_bits(st, state[:b]), b


def _cache(S=4):
    ers = _ers()
    return ers.ReplayCache(S, 8, 2, 64, 128, 16, torch.bfloat16, read_copy=True)


def _tok(S, lead=()):
    g = torch.Generator(device="cpu").manual_seed(0)
    x = torch.randn(S, *lead, 8, 64, generator=g).to(torch.bfloat16).to(dev())
    dt = torch.randn(S, *lead, 8, generator=g).to(dev())
    B = torch.randn(S, *lead, 2, 128, generator=g).to(torch.bfloat16).to(dev())
    C = torch.randn(S, *lead, 2, 128, generator=g).to(torch.bfloat16).to(dev())
    return x, dt, B, C


def _prm():
    ers = _ers()
    return ers.LayerParams(-torch.rand(8, device=dev()) - 1, torch.randn(8, device=dev()),
                           torch.full((8,), -3.0, device=dev()))


def test_device_errors_are_reported_not_trapped():
    ers = _ers()
    prm = _prm()
    c = _cache()
    st = ers.Status()
    # buffered position outside [0, Q)
    c.pos.fill_(16)
    ers.replay_decode(c, prm, *_tok(4), status=st, check=False)
    assert st.read() == 5  # ERS_EALIGN
    c.pos.zero_()
    # slot out of range
    st.reset()
    bad = torch.tensor([0, 9], dtype=torch.int32, device=dev())
    ers.replay_decode(c, prm, *_tok(2), slot=bad, status=st, check=False)
    assert st.read() == 8  # ERS_ESLOT
    # verify overflow without auto flush
    st.reset()
    c.pos.fill_(14)
    ers.spec_verify(c, prm, *_tok(4, (4,)), auto_flush=False, status=st, check=False)
    assert st.read() == 6  # ERS_EOVERFLOW
    # accepted > T
    st.reset()
    c.pos.zero_()
    ers.commit(c, torch.tensor([0, 5, 1, 1], dtype=torch.int32, device=dev()), 4, status=st, check=False)
    assert st.read() == 7  # ERS_ECOMMIT
    # raising wrapper
    with pytest.raises(ers.ErsError):
        c.pos.fill_(-1)
        ers.replay_decode(c, prm, *_tok(4))
    # the context is still usable
    c.pos.zero_()
    y = ers.replay_decode(c, prm, *_tok(4))
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all()


def test_empty_batches_through_the_binding():
    """Zero sequences through the Python binding: empty outputs of the right shape, no error, and no
    cache byte changes (decode, verify, commit and refresh of a ReplaySSM cache; GDN verify and
    commit; the conv1d update)."""
    ers = _ers()
    prm = _prm()
    c = _cache()
    c.pos.copy_(torch.tensor([3, 15, 0, 9], dtype=torch.int32, device=dev()))
    snap = [t.clone() for t in (c.state, c.read_copy, c.pos, c.buf_x, c.buf_B)]
    assert ers.replay_decode(c, prm, *_tok(0), replayssm=True).shape == (0, 8, 64)
    assert ers.spec_verify(c, prm, *_tok(0, (4,))).shape == (0, 4, 8, 64)
    ers.commit(c, torch.zeros(0, dtype=torch.int32, device=dev()), 4)
    ers.refresh(c, prm, nseq=0, replayssm=True, drafts_T=4)
    gc = ers.GdnCache(4, 8, 4, window=16)
    q = torch.zeros(0, 4, 4, 128, dtype=torch.bfloat16, device=dev())
    v = torch.zeros(0, 4, 8, 128, dtype=torch.bfloat16, device=dev())
    gb = torch.zeros(0, 4, 8, dtype=torch.float32, device=dev())
    assert ers.gdn_verify(gc, q, q, v, gb, gb).shape == (0, 4, 8, 128)
    ers.gdn_commit(gc, torch.zeros(0, dtype=torch.int32, device=dev()), 4)
    w = torch.randn(64, 4, device=dev()).to(torch.bfloat16)
    cs = torch.randn(4, 3, 64, device=dev()).to(torch.bfloat16)
    cs0 = cs.clone()
    assert ers.conv1d_update(torch.zeros(0, 64, dtype=torch.bfloat16, device=dev()), w, None, cs).shape == (0, 64)
    torch.cuda.synchronize()
    for a, b in zip((c.state, c.read_copy, c.pos, c.buf_x, c.buf_B), snap):
        assert same_bits(a, b)
    assert same_bits(cs, cs0) and int(gc.pos.abs().sum()) == 0


def test_host_validation_errors_launch_nothing():
    ers = _ers()
    prm = _prm()
    c = _cache()
    x, dt, B, C = _tok(4, (4,))
    with pytest.raises(ers.ErsError):
        ers.spec_verify(c, prm, x[:, :0], dt[:, :0], B[:, :0], C[:, :0])   # T = 0
    with pytest.raises(TypeError):
        ers.replay_decode(c, prm, x[:, 0].float(), dt[:, 0], B[:, 0], C[:, 0])
