"""Pins for the fp64 oracle: it is checked against things other than itself.

Each test uses a different route to the same numbers: a hand-worked fixture,
closed forms (geometric series, no-decay linear attention, one token), the
chunked SSD form and the ReplaySSM reassociated output form written out from
their own equations, a library IIR filter, linearity, and invariants (prefix,
packing, group mapping).  A dropped term, a wrong sign, swapped B/C, a wrong
group index or a wrong decay would fail at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


def _rand_case(rng, T, H, G, P, N, A_scale=(1.0, 16.0)):
    x = rng.standard_normal((T, H, P))
    dt = rng.standard_normal((T, H))
    B = rng.standard_normal((T, G, N))
    C = rng.standard_normal((T, G, N))
    A = -rng.uniform(*A_scale, size=H)
    D = rng.standard_normal(H)
    dt_bias = np.log(np.expm1(rng.uniform(1e-3, 1e-1, size=H)))
    return x, dt, A, B, C, D, dt_bias


def _delta(dt, dt_bias):
    # softplus written as log(1 + e^z) directly; inputs here stay in |z| < 30.
    return np.log1p(np.exp(dt + dt_bias[None, :]))


def _relerr(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# -- softplus ------------------------------------------------------------------------------------

def test_softplus_identities():
    assert oracle.softplus(0.0) == pytest.approx(math.log(2.0), rel=0, abs=1e-16)
    for z in (-30.0, -3.5, -0.25, 0.7, 4.0, 25.0):
        # softplus(z) - softplus(-z) = z  and  softplus(z) > max(z, 0)
        assert oracle.softplus(z) - oracle.softplus(-z) == pytest.approx(z, rel=1e-14, abs=1e-14)
        assert oracle.softplus(z) > max(z, 0.0)
    assert oracle.softplus(700.0) == 700.0          # no overflow for large arguments
    assert oracle.softplus(-40.0) == pytest.approx(math.exp(-40.0), rel=1e-12)


# -- hand-worked fixture ---------------------------------------------------------------------------

def test_golden_scalar_two_token():
    with open(os.path.join(HERE, "golden", "scalar_two_token.json")) as f:
        g = json.load(f)
    env = {"log": math.log, "exp": math.exp}
    inp = g["inputs"]
    x = np.array(inp["x"]).reshape(2, 1, 1)
    dt = np.array(inp["dt"]).reshape(2, 1)
    B = np.array(inp["B"]).reshape(2, 1, 1)
    C = np.array(inp["C"]).reshape(2, 1, 1)
    A = np.array([eval(inp["A"], env)])
    y, fin = oracle.recurrence(x, dt, A, B, C, np.array([inp["D"]]), np.array([inp["dt_bias"]]))
    exp_y = [eval(e, env) for e in g["expected_y"]]
    assert y[:, 0, 0] == pytest.approx(exp_y, rel=1e-14)
    assert fin[0, 0, 0, 0] == pytest.approx(eval(g["expected_final_state"], env), rel=1e-14)


# -- closed forms ------------------------------------------------------------------------------------

def test_single_token_closed_form():
    rng = np.random.default_rng(1)
    x, dt, A, B, C, D, dtb = _rand_case(rng, 1, 3, 1, 5, 7)
    y, fin = oracle.recurrence(x, dt, A, B, C, D, dtb)
    delta = _delta(dt, dtb)[0]
    bc = float(B[0, 0] @ C[0, 0])
    want = delta[:, None] * bc * x[0] + D[:, None] * x[0]
    assert _relerr(y[0], want) < 1e-14
    want_state = delta[:, None, None] * x[0][:, :, None] * B[0, 0][None, None, :]
    assert _relerr(fin[0], want_state) < 1e-14


def test_geometric_series_constant_inputs():
    """Constant inputs: S_T = v k^T (1 - a^T) / (1 - a) with a = exp(delta A)."""
    rng = np.random.default_rng(2)
    T, H, P, N = 37, 2, 3, 4
    x1 = rng.standard_normal((H, P))
    B1 = rng.standard_normal(N)
    C1 = rng.standard_normal(N)
    dt1 = rng.standard_normal(H)
    A = -rng.uniform(0.05, 2.0, size=H)
    D = rng.standard_normal(H)
    dtb = np.zeros(H)
    x = np.broadcast_to(x1, (T, H, P)).copy()
    B = np.broadcast_to(B1, (T, 1, N)).copy()
    C = np.broadcast_to(C1, (T, 1, N)).copy()
    dt = np.broadcast_to(dt1, (T, H)).copy()
    y, fin = oracle.recurrence(x, dt, A, B, C, D, dtb)
    delta = np.log1p(np.exp(dt1))
    a = np.exp(delta * A)
    for t in (0, 5, T - 1):
        geo = (1 - a ** (t + 1)) / (1 - a)
        S = (delta * geo)[:, None, None] * x1[:, :, None] * B1[None, None, :]
        want = S @ C1 + D[:, None] * x1
        assert _relerr(y[t], want) < 1e-13
    S = (delta * (1 - a ** T) / (1 - a))[:, None, None] * x1[:, :, None] * B1[None, None, :]
    assert _relerr(fin[0], S) < 1e-13


def test_no_decay_is_causal_linear_attention():
    """A = 0: y_t = sum_{s<=t} delta_s (B_s . C_t) x_s + D x_t (+ init C_t)."""
    rng = np.random.default_rng(3)
    T, H, G, P, N = 23, 4, 2, 3, 5
    x, dt, _, B, C, D, dtb = _rand_case(rng, T, H, G, P, N)
    A = np.zeros(H)
    init = rng.standard_normal((1, H, P, N))
    y, fin = oracle.recurrence(x, dt, A, B, C, D, dtb, init_state=init)
    delta = _delta(dt, dtb)
    for h in range(H):
        g = h // (H // G)
        att = np.tril(C[:, g] @ B[:, g].T) * delta[None, :, h]     # [t, s]
        want = att @ x[:, h] + (C[:, g] @ init[0, h].T) + D[h] * x[:, h]
        assert _relerr(y[:, h], want) < 1e-13
        want_state = init[0, h] + np.einsum("s,sp,sn->pn", delta[:, h], x[:, h], B[:, g])
        assert _relerr(fin[0, h], want_state) < 1e-13


def test_scalar_case_matches_scipy_lfilter():
    """P = N = 1 with constant delta is a first-order IIR filter."""
    signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(4)
    T = 200
    xs = rng.standard_normal(T)
    Cs = rng.standard_normal(T)
    dt = np.full((T, 1), 0.3)
    A = np.array([-1.7])
    D = np.array([0.25])
    y, _ = oracle.recurrence(xs.reshape(T, 1, 1), dt, A, np.ones((T, 1, 1)), Cs.reshape(T, 1, 1), D,
                             np.array([0.0]))
    delta = math.log1p(math.exp(0.3))
    a = math.exp(delta * A[0])
    state = signal.lfilter([delta], [1.0, -a], xs)
    assert _relerr(y[:, 0, 0], state * Cs + D[0] * xs) < 1e-13


# -- the chunked SSD form, written from its own equations --------------------------------------------

def _ssd_chunked(x, dt, A, B, C, D, dtb, Q, init):
    T, H, P = x.shape
    G = B.shape[1]
    delta = _delta(dt, dtb)
    y = np.zeros_like(x)
    state = init.copy()
    for c0 in range(0, T, Q):
        c1 = min(T, c0 + Q)
        for h in range(H):
            g = h // (H // G)
            dA = delta[c0:c1, h] * A[h]
            acum = np.cumsum(dA)
            seg = acum[:, None] - acum[None, :]                      # Acum_t - Acum_s
            Lmask = np.where(np.tril(np.ones((c1 - c0, c1 - c0), bool)), np.exp(np.where(
                np.tril(np.ones((c1 - c0, c1 - c0), bool)), seg, 0.0)), 0.0)
            Gm = C[c0:c1, g] @ B[c0:c1, g].T                          # [t, s]
            M = Gm * Lmask * delta[None, c0:c1, h]
            y_diag = M @ x[c0:c1, h]                                 # [t, P]
            y_off = np.exp(acum)[:, None] * (C[c0:c1, g] @ state[h].T)
            y[c0:c1, h] = y_diag + y_off + D[h] * x[c0:c1, h]
            w = np.exp(acum[-1] - acum) * delta[c0:c1, h]
            state[h] = np.exp(acum[-1]) * state[h] + np.einsum("s,sp,sn->pn", w, x[c0:c1, h], B[c0:c1, g])
    return y, state


@pytest.mark.parametrize("Q", [1, 7, 16, 64])
def test_chunked_ssd_form_matches(Q):
    rng = np.random.default_rng(10 + Q)
    T, H, G, P, N = 64, 4, 1, 16, 16
    x, dt, A, B, C, D, dtb = _rand_case(rng, T, H, G, P, N)
    init = rng.standard_normal((H, P, N))
    want_y, want_s = _ssd_chunked(x, dt, A, B, C, D, dtb, Q, init)
    y, fin = oracle.recurrence(x, dt, A, B, C, D, dtb, init_state=init[None])
    assert _relerr(y, want_y) < 1e-12
    assert _relerr(fin[0], want_s) < 1e-12


# -- ReplaySSM reassociated output form (explicit gamma products) --------------------------------------

def test_reassociated_output_only_form():
    """S_h = gamma_{1:h} S_ckpt + sum_j gamma_{j+1:h} v_j k_j^T and
    O = S_ckpt Q D + V (W . K^T Q) with W_js = 1[j <= h+s] gamma_{j+1:h+s}."""
    rng = np.random.default_rng(5)
    h, T = 9, 4                      # committed records, drafts
    H, G, P, N = 2, 1, 3, 5
    x, dt, A, B, C, D, dtb = _rand_case(rng, h + T, H, G, P, N, A_scale=(0.1, 3.0))
    S_ckpt = rng.standard_normal((1, H, P, N))
    y, _ = oracle.recurrence(x, dt, A, B, C, D, dtb, init_state=S_ckpt)
    _, S_h = oracle.recurrence(x[:h], dt[:h], A, B[:h], C[:h], D, dtb, init_state=S_ckpt)
    delta = _delta(dt, dtb)
    for hd in range(H):
        alpha = np.exp(delta[:, hd] * A[hd])              # alpha_i, i = 1..h+T  (0-based here)
        gam = lambda a, b: float(np.prod(alpha[a - 1:b])) if b >= a else 1.0  # gamma_{a:b}, 1-based
        V = delta[:, hd, None] * x[:, hd]                  # v_j  [j, P]
        K = B[:, 0]                                        # k_j  [j, N]
        Qm = C[:, 0]                                       # q    [j, N]
        Sh = gam(1, h) * S_ckpt[0, hd] + sum(gam(j + 2, h) * np.outer(V[j], K[j]) for j in range(h))
        assert _relerr(S_h[0, hd], Sh) < 1e-13
        for s in range(1, T + 1):
            col = h + s                                    # 1-based position of draft s
            q = Qm[col - 1]
            O = gam(1, col) * (S_ckpt[0, hd] @ q)
            for j in range(1, col + 1):
                O = O + V[j - 1] * gam(j + 1, col) * float(K[j - 1] @ q)
            want = O + D[hd] * x[col - 1, hd]
            assert _relerr(y[col - 1, hd], want) < 1e-13


# -- invariants --------------------------------------------------------------------------------------

def test_linearity_in_x_and_initial_state():
    rng = np.random.default_rng(6)
    T, H, G, P, N = 19, 2, 1, 4, 3
    x1, dt, A, B, C, D, dtb = _rand_case(rng, T, H, G, P, N)
    x2 = rng.standard_normal(x1.shape)
    i1, i2 = rng.standard_normal((2, 1, H, P, N))
    a, b = 0.75, -1.3
    y1, s1 = oracle.recurrence(x1, dt, A, B, C, D, dtb, init_state=i1)
    y2, s2 = oracle.recurrence(x2, dt, A, B, C, D, dtb, init_state=i2)
    y, s = oracle.recurrence(a * x1 + b * x2, dt, A, B, C, D, dtb, init_state=a * i1 + b * i2)
    assert _relerr(y, a * y1 + b * y2) < 1e-12
    assert _relerr(s, a * s1 + b * s2) < 1e-12


def test_group_mapping_contiguous_heads():
    """Heads h use group h // (H/G): compare with G = H and B/C replicated per head."""
    rng = np.random.default_rng(7)
    T, H, G, P, N = 11, 6, 2, 3, 4
    x, dt, A, B, C, D, dtb = _rand_case(rng, T, H, G, P, N)
    y, s = oracle.recurrence(x, dt, A, B, C, D, dtb)
    idx = np.arange(H) // (H // G)
    y2, s2 = oracle.recurrence(x, dt, A, B[:, idx], C[:, idx], D, dtb)
    assert np.array_equal(y, y2) and np.array_equal(s, s2)


def test_prefix_and_packing_invariance():
    rng = np.random.default_rng(8)
    H, G, P, N = 4, 2, 3, 5
    x, dt, A, B, C, D, dtb = _rand_case(rng, 30, H, G, P, N)
    y, _ = oracle.recurrence(x, dt, A, B, C, D, dtb)
    for t in (1, 7, 29):
        yp, _ = oracle.recurrence(x[:t], dt[:t], A, B[:t], C[:t], D, dtb)
        assert np.array_equal(yp, y[:t])
    cu = np.array([0, 12, 13, 30])
    yk, sk = oracle.recurrence(x, dt, A, B, C, D, dtb, cu_seqlens=cu)
    for i in range(3):
        lo, hi = cu[i], cu[i + 1]
        ys, ss = oracle.recurrence(x[lo:hi], dt[lo:hi], A, B[lo:hi], C[lo:hi], D, dtb)
        assert np.array_equal(yk[lo:hi], ys) and np.array_equal(sk[i], ss[0])


def test_thread_count_does_not_change_bits():
    rng = np.random.default_rng(9)
    x, dt, A, B, C, D, dtb = _rand_case(rng, 40, 8, 2, 8, 8)
    cu = np.array([0, 17, 40])
    y1, s1 = oracle.recurrence(x, dt, A, B, C, D, dtb, cu, nthreads=1)
    y8, s8 = oracle.recurrence(x, dt, A, B, C, D, dtb, cu, nthreads=8)
    assert np.array_equal(y1, y8) and np.array_equal(s1, s8)


# -- the ReplaySSM protocol model ------------------------------------------------------------------------

def _protocol_case(seed, S=3, steps=9, T=4, L=16, N=4):
    rng = np.random.default_rng(seed)
    H, G, P = 2, 1, 3
    params = synth.Params(-rng.uniform(0.2, 3.0, H).astype(np.float32), rng.standard_normal(H).astype(np.float32),
                          np.log(np.expm1(rng.uniform(1e-3, 1e-1, H))).astype(np.float32))
    anchor = rng.standard_normal((S, H, P, N))
    drafts = [[(rng.standard_normal((T, H, P)), rng.standard_normal((T, H)), rng.standard_normal((T, G, N)),
                rng.standard_normal((T, G, N))) for _ in range(S)] for _ in range(steps)]
    acc = rng.integers(0, T + 1, size=(steps, S))
    return params, anchor, drafts, acc, L


def test_protocol_flush_rule_hand_worked():
    """The flush rule h + T > L (ReplaySSM "Core equations"; commit h = (flushed ? 0 : h) + accepted),
    worked by hand for L = 5, T = 3 and acceptances 3, 0, 2, 3, 1, 3: the committed counts after
    each commit are 3, 0, 2, 5, 1, 4 and flushes happen at steps 2 and 5 only (step 4 has h + T = L:
    no flush).  Both protocol models (Mamba2 and GDN) follow it."""
    L, T, acc = 5, 3, [3, 0, 2, 3, 1, 3]
    want_h, want_flushes = [3, 0, 2, 5, 1, 4], [0, 1, 1, 1, 2, 2]
    params, anchor, drafts, _, _ = _protocol_case(19, S=1, steps=len(acc), T=T, L=L)
    m = oracle.ReplaySSMModel(params, anchor, L)
    d = synth.GdnDims(2, 1, 4, 3, L)
    rng = np.random.Generator(np.random.PCG64(20))
    g = oracle.GdnReplayModel(rng.standard_normal((1, 2, 3, 4)), L)
    for k, a in enumerate(acc):
        m.verify(drafts[k]); m.commit([a])
        t = synth.make_gdn_tokens(rng, T, d, False)
        g.verify([(t.q, t.k, t.v, t.g, t.beta)]); g.commit([a])
        assert int(m.h()[0]) == want_h[k] and m.flushes == want_flushes[k], k
        assert int(g.h()[0]) == want_h[k] and g.flushes == want_flushes[k], k


def test_protocol_zero_acceptance_keeps_anchor():
    params, anchor, drafts, _, L = _protocol_case(11)
    m = oracle.ReplaySSMModel(params, anchor, L)
    for k in range(6):
        m.verify(drafts[k])
        m.commit([0] * len(drafts[k]))
    assert np.array_equal(m.anchor, anchor) and m.flushes == 0 and np.all(m.h() == 0)


def test_protocol_committed_stream_matches_plain_recurrence():
    """After any accept/reject pattern, anchor + committed records reproduce the
    plain recurrence over exactly the accepted tokens (rejected drafts never enter)."""
    params, anchor, drafts, acc, L = _protocol_case(12, steps=12)
    m = oracle.ReplaySSMModel(params, anchor, L)
    accepted = [[] for _ in range(len(anchor))]
    for k in range(len(drafts)):
        m.verify(drafts[k])
        m.commit(acc[k])
        for i in range(len(anchor)):
            for j in range(acc[k, i]):
                accepted[i].append(tuple(drafts[k][i][q][j] for q in range(4)))
    assert m.flushes > 0
    m.refresh(range(len(anchor)))
    for i in range(len(anchor)):
        rec = [np.stack([r[q] for r in accepted[i]]) for q in range(4)]
        _, fin = oracle.recurrence(rec[0], rec[1], params.A, rec[2], rec[3], params.D, params.dt_bias,
                                   init_state=anchor[i:i + 1])
        assert _relerr(m.anchor[i], fin[0]) < 1e-12


def test_protocol_drafts_equal_one_draft_verifies():
    """With committed records in place, the drafts of one verify give the outputs of one-draft
    verifies with each draft committed in turn (the same rows, the same outputs; no flush)."""
    params, anchor, drafts, _, L = _protocol_case(15, steps=2)
    S, T = len(anchor), drafts[0][0][0].shape[0]
    ma = oracle.ReplaySSMModel(params, anchor, L)
    mb = oracle.ReplaySSMModel(params, anchor, L)
    for m in (ma, mb):
        m.verify(drafts[0]); m.commit([3] * S)
    ya = ma.verify(drafts[1])
    for s in range(T):
        yb = mb.verify([tuple(f[s:s + 1] for f in dr) for dr in drafts[1]]); mb.commit([1] * S)
        assert _relerr(yb[:, 0], ya[:, s]) < 1e-12
    assert ma.flushes == 0 and mb.flushes == 0


def test_protocol_outputs_read_the_recast_copy():
    """After a refresh the outputs read a copy recast from the refreshed anchor: with no committed
    records left, the drafts' outputs are the recurrence over the drafts alone started from the bf16
    cast of the new anchor (both pieces pinned on their own above)."""
    params, anchor, drafts, acc, L = _protocol_case(14, steps=12)
    m = oracle.ReplaySSMModel(params, anchor, L)
    for k in range(len(drafts) - 1):
        m.verify(drafts[k])
        m.commit(acc[k])
    assert m.flushes > 0
    m.refresh(range(len(anchor)))
    nxt = drafts[-1]
    y = m.verify(nxt)
    for i in range(len(anchor)):
        x, dt, B, C = nxt[i]
        want, _ = oracle.recurrence(x, dt, params.A, B, C, params.D, params.dt_bias,
                                    init_state=oracle.bf16_round(m.anchor[i:i + 1]))
        assert _relerr(y[i], want) < 1e-12


def test_protocol_anchor_independent_of_read_precision():
    """Read-copy rounding never feeds the anchor (dual precision)."""
    params, anchor, drafts, acc, L = _protocol_case(13, steps=12)
    m1 = oracle.ReplaySSMModel(params, anchor, L)
    m2 = oracle.ReplaySSMModel(params, anchor, L, read_cast=lambda s: np.array(s, copy=True))  # unrounded
    y1 = y2 = None
    for k in range(len(drafts)):
        y1 = m1.verify(drafts[k]); m1.commit(acc[k])
        y2 = m2.verify(drafts[k]); m2.commit(acc[k])
    assert m1.flushes > 0
    assert np.array_equal(m1.anchor, m2.anchor)
    assert not np.array_equal(y1, y2)        # outputs do see the read precision


def test_bf16_round_matches_synth_rounding():
    rng = np.random.default_rng(14)
    v = rng.standard_normal(10000).astype(np.float32) * 7
    assert np.array_equal(oracle.bf16_round(v).astype(np.float32), synth.round_bf16(v))
    # ties go to even: 1 + 2^-8 lies halfway between bf16 neighbours 1 and 1 + 2^-7
    assert oracle.bf16_round(np.array([1.0 + 2.0 ** -8], np.float32))[0] == 1.0
    assert oracle.bf16_round(np.array([1.0 + 3 * 2.0 ** -8], np.float32))[0] == 1.0 + 2.0 ** -6


def test_bf16_round_matches_a_library_cast_over_the_whole_range():
    """The library's fp32 -> bf16 cast (PyTorch on the CPU, round-to-nearest-even) on magnitudes from
    the subnormals to past the largest finite bf16, exact ties and both signs."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(15)
    mant = rng.uniform(1.0, 2.0, 20000)
    expo = rng.integers(-133, 128, 20000)
    v = (mant * np.exp2(expo.astype(np.float64)) * rng.choice([-1.0, 1.0], 20000)).astype(np.float32)
    k = np.arange(128, dtype=np.float64)   # every halfway case of [1, 2) (spacing 2^-7) and [2, 4) (2^-6)
    ties = np.concatenate([1.0 + k * 2.0 ** -7 + 2.0 ** -8, 2.0 + k * 2.0 ** -6 + 2.0 ** -7]).astype(np.float32)
    edge = np.array([0.0, -0.0, 3.3895314e38, 3.3961776e38, np.finfo(np.float32).max, 2.0 ** -133, 2.0 ** -126],
                    np.float32)
    for a in (v, ties, -ties, edge):
        want = torch.from_numpy(a).to(torch.bfloat16).to(torch.float32).numpy()
        got = oracle.bf16_round(a).astype(np.float32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def _e4m3_table():
    """Every finite e4m3 value, decoded from the bit fields by the format's definition."""
    vals = []
    for code in range(256):
        sgn, ex, man = code >> 7, (code >> 3) & 0xF, code & 7
        if ex == 0xF and man == 7:
            continue                                   # the NaN codes
        v = (man / 8.0) * 2.0 ** -6 if ex == 0 else (1 + man / 8.0) * 2.0 ** (ex - 7)
        vals.append((-v if sgn else v, code))
    return vals


def test_e4m3_round_fixes_every_code_and_saturates():
    table = _e4m3_table()
    v = np.array([t[0] for t in table], dtype=np.float32)
    assert np.array_equal(oracle.e4m3_round(v), v)
    assert max(abs(t[0]) for t in table) == 448.0 and min(abs(t[0]) for t in table if t[0] != 0) == 2.0 ** -9
    assert np.array_equal(oracle.e4m3_round(np.array([1e6, -500.0, 449.0], np.float32)), np.array([448, -448, 448], np.float32))


def test_e4m3_round_matches_brute_force_nearest_even():
    table = [t for t in _e4m3_table() if t[0] >= 0]
    vals = np.array([t[0] for t in table])
    codes = np.array([t[1] for t in table])
    rng = np.random.Generator(np.random.PCG64(8))
    x = np.concatenate([rng.uniform(0, 448, 3000), 2.0 ** rng.uniform(-12, 9, 3000),
                        (vals[:-1] + vals[1:]) / 2])          # exact midpoints exercise the ties
    x = x.astype(np.float32).astype(np.float64)
    got = oracle.e4m3_round(x.astype(np.float32)).astype(np.float64)
    for xi, gi in zip(x, got):
        d = np.abs(vals - xi)
        best = np.nonzero(d == d.min())[0]
        want = vals[best[np.argmin(codes[best] & 1)]] if len(best) > 1 else vals[best[0]]   # tie: even code
        assert gi == want, (xi, gi, want)
    assert np.array_equal(oracle.e4m3_round(-x.astype(np.float32)), -oracle.e4m3_round(x.astype(np.float32)))


def test_fp8_row_scale_is_the_smallest_power_of_two_without_saturation():
    # hand-worked rows: amax = 448 -> s = 1; the next fp32 above 448 -> s = 2; 1.0 -> 2^-8
    # (256 <= 448 < 512); 0.21875 = 448 * 2^-11 exactly -> 2^-11; zero and tiny rows -> 2^-127
    above = float(np.nextafter(np.float32(448), np.float32(1e9)))
    got = oracle.fp8_row_scale_exponent(np.array([448.0, above, 1.0, 0.21875, 0.0, 2.0 ** -140]))
    assert list(got) == [0, 1, -8, -11, -127, -127]
    # brute force over random magnitudes: 448 * 2^(k-1) < amax <= 448 * 2^k
    rng = np.random.Generator(np.random.PCG64(3))
    amax = (rng.uniform(0.5, 1.0, 2000) * np.exp2(rng.integers(-100, 100, 2000))).astype(np.float32).astype(np.float64)
    k = oracle.fp8_row_scale_exponent(amax)
    assert np.all(amax <= 448.0 * np.exp2(k.astype(np.float64)))
    assert np.all(amax > 448.0 * np.exp2(k.astype(np.float64) - 1))


def test_fp8_rows_round_hand_worked_values():
    # row max 1.0 -> s = 2^-8: 0.3 * 256 = 76.8 lies in [64, 128) where e4m3 steps by 8 -> 80 -> 0.3125;
    # -0.5 * 256 = -128 is a code; 0.001 * 256 = 0.256 lies in [0.25, 0.5) (step 1/32) -> 0.25 -> 2^-10
    r = oracle.fp8_rows_round(np.array([[1.0, 0.3, -0.5, 0.001, 0.0]]))
    assert list(r[0]) == [1.0, 0.3125, -0.5, 2.0 ** -10, 0.0]
    # the next fp32 above 448 reads back as 448 (s = 2: 224.00002 rounds to the code 224)
    above = float(np.nextafter(np.float32(448), np.float32(1e9)))
    assert oracle.fp8_rows_round(np.array([[above, 1.0]]))[0, 0] == 448.0
    assert np.all(oracle.fp8_rows_round(np.zeros((2, 8))) == 0)


def test_fp8_rows_round_error_bound_and_exact_codes():
    rng = np.random.Generator(np.random.PCG64(9))
    a = rng.standard_normal((3, 4, 16, 128)) * np.exp(rng.uniform(-8, 8, (3, 4, 16, 1)))
    a[0, 0, 0] = 0.0
    r = oracle.fp8_rows_round(a)
    f = a.astype(np.float32).astype(np.float64)
    s = np.exp2(oracle.fp8_row_scale_exponent(np.abs(f).max(axis=-1, keepdims=True)).astype(np.float64))
    assert np.all(r[0, 0, 0] == 0)
    # e4m3 keeps 3 mantissa bits (half a quantum: 2^-4 relative) down to its subnormal step 2^-9
    assert np.all(np.abs(r - f) <= 2.0 ** -4 * np.abs(f) + 2.0 ** -10 * s)
    # every read value is a code times the row scale
    assert np.array_equal(oracle.e4m3_round((r / s).astype(np.float32)).astype(np.float64), r / s)


def _e2m1_table():
    """Every finite e2m1 value, decoded from the bit fields by the format's definition (bias 1;
    exponent field 0 is subnormal: 0.5 * mantissa)."""
    out = []
    for code in range(16):
        sgn = -1.0 if code & 8 else 1.0
        e, m = (code >> 1) & 3, code & 1
        v = 0.5 * m if e == 0 else (1 + 0.5 * m) * 2.0 ** (e - 1)
        out.append((sgn * v, code))
    return out


def test_e2m1_round_fixes_every_code_and_matches_brute_force():
    table = _e2m1_table()
    vals = np.array([t[0] for t in table], np.float32)
    assert sorted(set(np.abs(vals).tolist())) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert np.array_equal(oracle.e2m1_round(vals), vals)
    pos = [t for t in table if t[0] >= 0 and not (t[0] == 0 and t[1] == 8)]
    pv = np.array([t[0] for t in pos])
    pc = np.array([t[1] for t in pos])
    x = np.concatenate([np.linspace(0, 7.9, 4001), (pv[:-1] + pv[1:]) / 2])      # a grid plus every tie
    got = oracle.e2m1_round(x.astype(np.float32)).astype(np.float64)
    for xi, gi in zip(x, got):
        d = np.abs(pv - xi)
        best = np.nonzero(d == d.min())[0]
        want = min(6.0, pv[best[np.argmin(pc[best] & 1)]] if len(best) > 1 else pv[best[0]])  # tie: even mantissa
        if xi > 6.0:
            want = 6.0                                                                   # saturation
        assert gi == want, (xi, gi, want)
    assert np.array_equal(oracle.e2m1_round(-x.astype(np.float32)), -oracle.e2m1_round(x.astype(np.float32)))


def test_nvfp4_scales_and_hand_worked_values():
    # row scale: amax = 2688 -> k = 0; 6 -> -8 (2688 * 2^-9 = 5.25 < 6 <= 10.5); 1.0 -> -11; zero -> -127
    got = oracle.nvfp4_row_scale_exponent(np.array([2688.0, 6.0, 1.0, 0.0, float(np.nextafter(np.float32(2688), np.float32(1e9)))]))
    assert list(got) == [0, -8, -11, -127, 1]
    # block [1.0, 0.3, 0...] (row max 1.0): s = 2^-11; t = 2048; beta = e4m3(341.33) = 352 (step 32);
    # 1.0 -> 2048/352 = 5.82 -> e2m1 6 -> 6 * 352 / 2048 = 1.03125; 0.3 -> 1.745 -> 1.5 -> 0.2578125
    r, q, beta, k = oracle.nvfp4_rows_round(np.array([[1.0, 0.3] + [0.0] * 14]), parts=True)
    assert list(r[0, :3]) == [1.03125, 0.2578125, 0.0] and beta[0, 0] == 352 and k[0] == -11
    # a row whose values are e2m1 values with maximum 6 reads back exactly (s = 2^-8, beta = 256)
    e2 = np.array([6, -4, 3, 1.5, 0.5, 0, -6, 2, 1, -3, 4, 0.5, -1.5, 2, 6, -0.5] * 8, np.float64)[None]
    assert np.array_equal(oracle.nvfp4_rows_round(e2), e2)
    # a block far below its row's maximum: its beta underflows to 0 and it reads as zeros
    row = np.zeros((1, 32)); row[0, 0] = 1000.0; row[0, 16:] = 1e-6
    assert np.all(oracle.nvfp4_rows_round(row)[0, 16:] == 0)
    assert np.all(oracle.nvfp4_rows_round(np.zeros((2, 32))) == 0)


def test_nvfp4_values_are_codes_times_scales_within_bound():
    rng = np.random.Generator(np.random.PCG64(12))
    a = rng.standard_normal((3, 4, 16, 128)) * np.exp(rng.uniform(-8, 8, (3, 4, 16, 1)))
    r, q, beta, k = oracle.nvfp4_rows_round(a, parts=True)
    f = a.astype(np.float32).astype(np.float64)
    s = np.exp2(k.astype(np.float64))[..., None]
    qb = q.reshape(q.shape[:-1] + (8, 16)).astype(np.float64)
    assert np.array_equal(oracle.e2m1_round(q), q)                                   # codes are e2m1 values
    assert np.array_equal(oracle.e4m3_round(beta), beta)                             # block scales are e4m3
    assert np.array_equal((qb * beta[..., None]).reshape(f.shape) * s, r)
    # error: e2m1 rounding (half a step: 1/4 relative, 1/4 of beta*s absolute in the subnormal step)
    # plus the block-scale rounding that can push a block's maximum into saturation (2^-4 relative)
    fb = f.reshape(f.shape[:-1] + (8, 16))
    amax_b = np.abs(fb).max(axis=-1, keepdims=True)
    bs = (beta[..., None] * s[..., None])
    err = np.abs(r.reshape(fb.shape) - fb)
    assert np.all(err <= 0.25 * np.abs(fb) + 0.25 * bs + 2.0 ** -4 * amax_b * 1.01)


def _e2m1_nearest_even_f64(x):
    """Brute-force e2m1 rounding of fp64 values (no intermediate fp32 rounding): nearest magnitude of
    {0, 0.5, 1, 1.5, 2, 3, 4, 6}, ties to the even code, saturating at 6, sign kept."""
    pv = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    a = np.minimum(np.abs(np.asarray(x, np.float64)), 6.0)
    d = np.abs(a[..., None] - pv)
    dmin = d.min(axis=-1, keepdims=True)
    near = d == dmin
    # among equally near values take the one whose code is even (index parity = mantissa bit)
    even = near & ((np.arange(8) % 2) == 0)
    idx = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(near, axis=-1))
    return np.sign(x) * pv[idx]


def test_nvfp4_reciprocal_form_against_the_division_form():
    """The oracle's NVFP4 codes are e2m1(u * RN(1/beta)) with fp32 reciprocal and product; the plain
    definition of a block-scaled code is e2m1(u / beta).  RN(1/beta) and the fp32 product each add
    at most 2^-24 relative error, so |u * rcp - u / beta| < 2^-22.9 |u / beta|: the two forms can only
    differ where u / beta lies within that distance of a rounding midpoint (0.25, 0.75, 1.25, 1.75,
    2.5, 3.5, 5), and there by one e2m1 step.  Exact ties are where they do differ."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    step = {0.25: 0.5, 0.75: 0.5, 1.25: 0.5, 1.75: 0.5, 2.5: 1.0, 3.5: 1.0, 5.0: 2.0}
    # (1) exact ties: u = m * beta for every positive normal e4m3 beta in [2^-6, 448] and every midpoint
    betas = np.unique(oracle.e4m3_round(np.exp2(np.linspace(-6, 8.8, 4000)).astype(np.float32)))
    betas = betas[betas >= 2.0 ** -6]
    n_diff = 0
    for m in mids:
        u = (m * betas).astype(np.float32)                                   # exact: <= 7 significant bits
        assert np.array_equal(u.astype(np.float64), m * betas.astype(np.float64))
        rcp = (np.float32(1.0) / betas.astype(np.float32)).astype(np.float32)
        q_rcp = oracle.e2m1_round((u * rcp).astype(np.float32)).astype(np.float64)
        q_div = _e2m1_nearest_even_f64(u.astype(np.float64) / betas.astype(np.float64))
        diff = q_rcp != q_div
        n_diff += int(diff.sum())
        assert np.all(np.abs(q_rcp - q_div)[diff] == step[m])                # one step, never more
        assert np.all(q_div == _e2m1_nearest_even_f64(np.full(len(betas), m)))   # division: ties to even
    assert n_diff > 0                                                         # the readings do differ here
    # (2) random states: codes of the oracle's cast against the division form with the oracle's scales
    rng = np.random.Generator(np.random.PCG64(77))
    a = rng.standard_normal((64, 64, 128)) * np.exp(rng.uniform(-6, 6, (64, 64, 1)))
    r, q, beta, k = oracle.nvfp4_rows_round(a, parts=True)
    u = (a.astype(np.float32).astype(np.float64) / np.exp2(k.astype(np.float64))[..., None])
    ub = u.reshape(u.shape[:-1] + (8, 16))
    bb = beta.astype(np.float64)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bb > 0, ub / np.where(bb > 0, bb, 1.0), 0.0)
    q_div = np.where(bb > 0, _e2m1_nearest_even_f64(ratio), 0.0)
    qb = q.reshape(ub.shape).astype(np.float64)
    diff = qb != q_div
    near_mid = np.min(np.abs(np.abs(ratio)[..., None] - mids), axis=-1) <= 2.0 ** -22.9 * np.abs(ratio)
    assert np.all(near_mid[diff])                                             # only next to a midpoint
    assert np.all(np.abs(qb - q_div)[diff] <= 2.0)                            # by one step
    assert diff.sum() <= 1e-4 * diff.size                                     # and rarely


def test_philox4x32_10_known_answers():
    # the generator's published known-answer vectors (counter, key -> output)
    kat = [((0, 0, 0, 0), (0, 0), (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)),
           ((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF), (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)),
           ((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0),
            (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1))]
    for ctr, key, want in kat:
        assert tuple(int(x) for x in oracle.philox4x32_10(np.array(ctr, np.uint64), key)) == want
    # vectorised over leading axes
    c = np.array([k[0] for k in kat[:1]] * 3, np.uint64)
    assert np.array_equal(oracle.philox4x32_10(c, (0, 0)), np.array([kat[0][2]] * 3, np.uint32))


def test_sr_fp16_decisions():
    u = 2.0 ** -10
    # 1 + ulp/4 rounds up iff r < 2^30; on-grid values never move; the sign is kept
    assert oracle.sr_fp16(np.float32(1 + u / 4), np.uint32(2 ** 30 - 1)) == 1 + u
    assert oracle.sr_fp16(np.float32(1 + u / 4), np.uint32(2 ** 30)) == 1.0
    assert oracle.sr_fp16(np.float32(-(1 + u / 4)), np.uint32(0)) == -(1 + u)
    # in the subnormal range the spacing is 2^-24: 1.5 * 2^-24 rounds up iff r < 2^31
    assert oracle.sr_fp16(np.float32(1.5 * 2.0 ** -24), np.uint32(2 ** 31 - 1)) == 2.0 ** -23
    assert oracle.sr_fp16(np.float32(1.5 * 2.0 ** -24), np.uint32(2 ** 31)) == 2.0 ** -24
    # saturation at the fp16 maximum, zero stays zero
    assert oracle.sr_fp16(np.float32(70000.0), np.uint32(0)) == 65504.0
    assert oracle.sr_fp16(np.float32(0.0), np.uint32(0)) == 0.0
    rng = np.random.Generator(np.random.PCG64(5))
    v = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 15, 20000))).astype(np.float32)
    grid = v.astype(np.float16).astype(np.float32)
    for r in (0, 2 ** 31, 2 ** 32 - 1):
        assert np.array_equal(oracle.sr_fp16(grid, np.full(v.shape, r, np.uint32)), grid.astype(np.float64))
    # with r = 2^31 - 1 the rule rounds half-way cases up and everything else to nearest: it agrees
    # with numpy's fp16 conversion (nearest even) except at exact ties
    out = oracle.sr_fp16(v, np.full(v.shape, 2 ** 31 - 1, np.uint32))
    lo = oracle.sr_fp16(v, np.full(v.shape, 2 ** 32 - 1, np.uint32))
    hi = oracle.sr_fp16(v, np.zeros(v.shape, np.uint32))
    tie = np.abs(np.abs(v.astype(np.float64)) - np.abs(lo)) == np.abs(np.abs(hi) - np.abs(v.astype(np.float64)))
    ok = np.abs(v) < 65504
    assert np.array_equal(out[ok & ~tie], v.astype(np.float16).astype(np.float64)[ok & ~tie])


def test_sr_words_counter_layout():
    # element (h, d, n) of a slot takes word n % 4 of the generator at counter (nonce, slot, h*P + d, n // 4)
    w = oracle.sr_words((7, 9), 3, 5, 2, 4, 8)
    one = oracle.philox4x32_10(np.array([3, 5, 1 * 4 + 2, 1], np.uint64), (7, 9))
    assert np.array_equal(w[1, 2, 4:8], one)
    assert not np.array_equal(oracle.sr_words((7, 9), 4, 5, 2, 4, 8), w)   # a new nonce, new words


def test_sr_anchor_writes_take_their_own_slots_words():
    """A slot's stochastically rounded write (fp16 anchor or shared NVFP4 state) uses the words of its
    own counter: the same state written for two slots, or under two nonces, rounds differently,
    and the same (nonce, slot) reproduces its bits."""
    rng = np.random.Generator(np.random.PCG64(31))
    fin = rng.standard_normal((2, 4, 16)) * 3.0
    for write in (oracle.sr_fp16_anchor, oracle.nvfp4_sr_state):
        a = write(fin, (7, 9), 3, 5)
        assert np.array_equal(a, write(fin, (7, 9), 3, 5))
        assert not np.array_equal(a, write(fin, (7, 9), 3, 6))       # another slot
        assert not np.array_equal(a, write(fin, (7, 9), 4, 5))       # another nonce


def test_sr_fp16_is_unbiased():
    # averaged over an even grid of r, the rounded value equals the input to within the grid step
    v = np.float32(1 + 0.3 * 2.0 ** -10)
    rs = (np.arange(4096, dtype=np.uint64) * (2 ** 32 // 4096)).astype(np.uint32)
    mean = oracle.sr_fp16(np.full(4096, v, np.float32), rs).mean()
    assert abs(mean - float(v)) <= 2.0 ** -10 / 4096


def test_sr_e2m1_decisions():
    """Stochastic rounding onto the e2m1 grid, worked by hand: the spacing above lo is 0.5 below 2,
    1 below 4 and 2 below 6; |v| goes up iff r < 2^32 (|v| - lo) / step."""
    sr = lambda v, r: float(oracle.sr_e2m1(np.float32(v), np.uint32(r)))
    assert sr(0.75, 2 ** 31 - 1) == 1.0 and sr(0.75, 2 ** 31) == 0.5          # half-way in [0.5, 1]
    assert sr(5.0, 2 ** 31 - 1) == 6.0 and sr(5.0, 2 ** 31) == 4.0            # half-way in [4, 6]
    assert sr(-2.5, 0) == -3.0 and sr(-2.5, 2 ** 32 - 1) == -2.0               # sign kept
    # fp32(0.1) = 13421773 * 2^-27: (|v| - 0) / 0.5 * 2^32 = 13421773 * 64 = 858993472 exactly
    assert sr(0.1, 858993471) == 0.5 and sr(0.1, 858993472) == 0.0
    # 3.25 in [3, 4): a quarter of the way; 1.75 in [1.5, 2): half-way
    assert sr(3.25, 2 ** 30 - 1) == 4.0 and sr(3.25, 2 ** 30) == 3.0
    assert sr(1.75, 2 ** 31 - 1) == 2.0 and sr(1.75, 2 ** 31) == 1.5
    # saturation at 6 for any word
    for r in (0, 2 ** 31, 2 ** 32 - 1):
        assert sr(6.5, r) == 6.0 and sr(-100.0, r) == -6.0 and sr(5.99, 0) == 6.0
    # every grid value stays where it is for any word
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    grid = np.concatenate([grid, -grid[1:]])
    for r in (0, 1, 2 ** 31, 2 ** 32 - 1):
        assert np.array_equal(oracle.sr_e2m1(grid, np.full(grid.shape, r, np.uint32)), grid)


def test_sr_e2m1_is_round_to_nearest_at_mid_word_and_unbiased():
    rng = np.random.Generator(np.random.PCG64(13))
    v = rng.uniform(-6.5, 6.5, 20000).astype(np.float32)
    a = np.abs(v.astype(np.float64))
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    frac = (a - np.floor(a / step) * step) / step
    away = (np.abs(frac - 0.5) > 2.0 ** -20) | (a >= 6)
    # with r = 2^31 - 1 the rule goes up exactly when frac > 1/2 - 2^-32: round to nearest off ties
    got = oracle.sr_e2m1(v, np.full(v.shape, 2 ** 31 - 1, np.uint32))
    assert np.array_equal(got[away], oracle.e2m1_round(v)[away])
    # averaged over the 2^16 evenly spaced words k * 2^16, values on a step / 2^16 lattice come back
    # exactly (the count of words below frac * 2^32 is frac * 2^16)
    rs = (np.arange(2 ** 16, dtype=np.uint64) << np.uint64(16)).astype(np.uint32)
    for x in (0.3 - 0.3 % 2.0 ** -17, 2.0 + 0.7 - 0.7 % 2.0 ** -16, -(4.0 + 1.3 - 1.3 % 2.0 ** -15), 0.0):
        m = oracle.sr_e2m1(np.full(rs.shape, x, np.float32), rs).astype(np.float64).mean()
        assert m == x, (x, m)


def test_nvfp4_sr_cast_keeps_the_scales_and_brackets_each_value():
    """The stochastic NVFP4 cast has the round-to-nearest cast's row and block scales; each code is
    one of the two e2m1 neighbours of the scaled value; with every word 2^31 - 1 it is the
    round-to-nearest cast (ties aside); the words follow the anchor counter layout."""
    rng = np.random.Generator(np.random.PCG64(14))
    a = rng.standard_normal((2, 3, 8, 64)) * np.exp(rng.uniform(-6, 6, (2, 3, 8, 1)))
    words = rng.integers(0, 2 ** 32, a.shape, dtype=np.uint64).astype(np.uint32)
    r0, q0, b0, k0 = oracle.nvfp4_rows_round(a, parts=True)
    r1, q1, b1, k1 = oracle.nvfp4_rows_round(a, parts=True, words=words)
    assert np.array_equal(b0, b1) and np.array_equal(k0, k1)
    assert np.array_equal(oracle.e2m1_round(q1), q1)
    lo = oracle.nvfp4_rows_round(a, parts=True, words=np.full(a.shape, 2 ** 32 - 1, np.uint32))[1]
    hi = oracle.nvfp4_rows_round(a, parts=True, words=np.zeros(a.shape, np.uint32))[1]
    assert np.all((q1 == lo) | (q1 == hi)) and np.all(np.abs(hi) >= np.abs(lo))
    assert np.mean(q1 != q0) > 0.2                                                  # rounding did vary
    mid = oracle.nvfp4_rows_round(a, words=np.full(a.shape, 2 ** 31 - 1, np.uint32))
    assert np.mean(mid != r0) < 1e-3
    st = rng.standard_normal((2, 4, 32))
    got = oracle.nvfp4_sr_state(st, (3, 4), 11, 6)
    assert np.array_equal(got, oracle.nvfp4_rows_round(st, words=oracle.sr_words((3, 4), 11, 6, 2, 4, 32)))


def test_protocol_refresh_stores_the_rounded_anchor():
    """A model whose stored anchor is a rounding of the refreshed state (fp16 stochastic rounding,
    the shared NVFP4 state) stores rounding(refreshed state): with a rounding onto the grid of
    quarters, a refresh leaves the quarter rounding of the recurrence over the committed records from
    the previous stored anchor, every value a multiple of 1/4."""
    params, anchor, drafts, acc, L = _protocol_case(16, steps=6)
    q4 = lambda i, fin: np.round(np.asarray(fin, dtype=np.float64) * 4.0) / 4.0
    m = oracle.ReplaySSMModel(params, anchor, L, anchor_round=q4)
    for k in range(len(drafts)):
        m.verify(drafts[k]); m.commit(acc[k])
    which = [i for i in range(len(anchor)) if m.committed[i]]
    assert which
    before = {i: (m.anchor[i].copy(), [np.stack([r[f] for r in m.committed[i]]) for f in range(4)]) for i in which}
    m.refresh(which)
    for i in which:
        prev, (x, dt, B, C) = before[i]
        _, fin = oracle.recurrence(x, dt, params.A, B, C, params.D, params.dt_bias, init_state=prev[None])
        assert np.array_equal(m.anchor[i], q4(i, fin[0]))
        assert np.array_equal(m.anchor[i] * 4.0, np.round(m.anchor[i] * 4.0))


def test_protocol_shared_state_model():
    """A shared state: the read copy is the stored anchor itself after every refresh; an empty history
    (zero acceptance) never changes it; with an exact (identity) rounding the model is the fp32-anchor
    model with an fp64 read copy."""
    params, anchor, drafts, acc, L = _protocol_case(18, steps=12, N=32)
    key = (5, 6)
    nonce = {"v": 0}
    a0 = oracle.nvfp4_rows_round(anchor)
    m = oracle.ReplaySSMModel(params, a0, L, shared=True,
                              anchor_round=lambda i, fin: oracle.nvfp4_sr_state(fin, key, nonce["v"], i))
    m0 = oracle.ReplaySSMModel(params, a0, L, shared=True,
                               anchor_round=lambda i, fin: oracle.nvfp4_sr_state(fin, key, nonce["v"], i))
    for k in range(len(drafts)):
        nonce["v"] = 100 + k
        m.verify(drafts[k]); m.commit(acc[k])
        m0.verify(drafts[k]); m0.commit([0] * len(acc[k]))
        assert np.array_equal(m.read, m.anchor)
    assert m.flushes > 0 and m0.flushes == 0 and np.array_equal(m0.anchor, a0)
    ident = oracle.ReplaySSMModel(params, anchor, L, shared=True, anchor_round=lambda i, fin: fin)
    ref = oracle.ReplaySSMModel(params, anchor, L, read_cast=lambda x: np.asarray(x, dtype=np.float64))
    for k in range(len(drafts)):
        assert np.array_equal(ident.verify(drafts[k]), ref.verify(drafts[k]))
        ident.commit(acc[k]); ref.commit(acc[k])
    assert np.array_equal(ident.anchor, ref.anchor)


def test_protocol_anchor_independent_of_fp8_read_copy():
    """The fp32 anchor is the same whether outputs read a bf16, an FP8 or an NVFP4 copy."""
    params, anchor, drafts, acc, L = _protocol_case(17, steps=12, N=32)   # two 16-value blocks per row
    m1 = oracle.ReplaySSMModel(params, anchor, L)
    m2 = oracle.ReplaySSMModel(params, anchor, L, read_cast=oracle.fp8_rows_round)
    m3 = oracle.ReplaySSMModel(params, anchor, L, read_cast=oracle.nvfp4_rows_round)
    for k in range(len(drafts)):
        y1 = m1.verify(drafts[k]); m1.commit(acc[k])
        y2 = m2.verify(drafts[k]); m2.commit(acc[k])
        y3 = m3.verify(drafts[k]); m3.commit(acc[k])
    assert m1.flushes > 0 and np.array_equal(m1.anchor, m2.anchor) and np.array_equal(m1.anchor, m3.anchor)
    assert not np.array_equal(y1, y2) and not np.array_equal(y2, y3)


# ---- causal conv1d (exact-replay RFC, Evidence item 6: the conv's prefill and update paths) ----------
def test_silu_identities():
    z = np.linspace(-30, 30, 601)
    assert oracle.silu(np.array(0.0)) == 0.0
    assert np.allclose(oracle.silu(z) - oracle.silu(-z), z, rtol=0, atol=1e-12)     # sigmoid(z) + sigmoid(-z) = 1
    assert abs(oracle.silu(np.array(40.0)) - 40.0) < 1e-12
    assert abs(oracle.silu(np.array(1.0)) - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15


def test_conv1d_matches_numpy_convolve():
    rng = np.random.Generator(np.random.PCG64(41))
    for W in (2, 3, 4):
        T, C = 37, 5
        x = rng.standard_normal((T, C))
        w = rng.standard_normal((C, W))
        b = rng.standard_normal(C)
        init = rng.standard_normal((1, W - 1, C))
        y, fin = oracle.causal_conv1d(x, w, b, init_state=init, activation=False)
        u = np.concatenate([init[0], x])
        for c in range(C):
            want = np.convolve(u[:, c], w[c, ::-1], mode="valid") + b[c]
            assert np.allclose(y[:, c], want, rtol=1e-13, atol=1e-13)
        assert np.array_equal(fin[0], u[-(W - 1):])
        ya, _ = oracle.causal_conv1d(x, w, b, init_state=init, activation=True)
        assert np.allclose(ya, oracle.silu(y), rtol=1e-14, atol=1e-14)


def test_conv1d_identity_kernel_short_sequences_and_splits():
    rng = np.random.Generator(np.random.PCG64(42))
    W, C = 4, 3
    x = rng.standard_normal((9, C))
    eye = np.zeros((C, W)); eye[:, -1] = 1.0
    y, fin = oracle.causal_conv1d(x, eye, None, activation=False)
    assert np.array_equal(y, x) and np.array_equal(fin[0], x[-3:])
    # a sequence shorter than W - 1 keeps part of its initial state in the final state
    init = rng.standard_normal((1, W - 1, C))
    _, f1 = oracle.causal_conv1d(x[:1], eye, None, init_state=init)
    assert np.array_equal(f1[0], np.concatenate([init[0, 1:], x[:1]]))
    # splitting a sequence and carrying the state gives the single-shot result; packing is invariant
    w = rng.standard_normal((C, W)); b = rng.standard_normal(C)
    y0, f0 = oracle.causal_conv1d(x, w, b)
    ya, fa = oracle.causal_conv1d(x[:4], w, b)
    yb, fb = oracle.causal_conv1d(x[4:], w, b, init_state=fa)
    assert np.allclose(np.concatenate([ya, yb]), y0, rtol=1e-15, atol=1e-15) and np.array_equal(fb, f0)
    yp, fp = oracle.causal_conv1d(np.concatenate([x, x[:5]]), w, b, cu_seqlens=[0, 9, 14])
    assert np.array_equal(yp[:9], y0) and np.array_equal(yp[9:], oracle.causal_conv1d(x[:5], w, b)[0])
    assert np.array_equal(fp[0], f0[0])


# ---- gated delta rule (ReplaySSM notes, "Core equations": GDN residuals) ------------------------------
def _gdn_case(seed, T=7, d=None, bf16=False):
    d = d or synth.GdnDims(4, 2, 8, 6, 16)
    rng = np.random.Generator(np.random.PCG64(seed))
    toks = synth.make_gdn_tokens(rng, T, d, bf16)
    S0 = rng.standard_normal((d.nheads, d.dv, d.dk))
    return d, toks, S0


def test_golden_gdn_scalar_two_token():
    with open(os.path.join(HERE, "golden", "gdn_scalar_two_token.json")) as f:
        g = json.load(f)
    env = {"log": math.log, "exp": math.exp}
    inp = g["inputs"]
    T = len(inp["v"])
    col = lambda v: np.full((T, 1, 1), v, dtype=np.float64)
    o, S = oracle.gdn_recurrence(col(inp["q"]), col(inp["k"]), np.array(inp["v"]).reshape(T, 1, 1),
                                 np.full((T, 1), eval(inp["g"], env)), np.full((T, 1), inp["beta"]),
                                 np.full((1, 1, 1), inp["init_state"]))
    assert o[:, 0, 0] == pytest.approx([eval(e, env) for e in g["expected_o"]], rel=1e-14)
    assert S[0, 0, 0] == pytest.approx(eval(g["expected_final_state"], env), rel=1e-14)


def test_gdn_beta_zero_is_pure_decay():
    d, t, S0 = _gdn_case(61)
    o, S = oracle.gdn_recurrence(t.q, t.k, t.v, t.g, np.zeros_like(t.beta), S0)
    hg = np.arange(d.nheads) // (d.nheads // d.ngroups)
    gam = np.exp(np.cumsum(t.g.astype(np.float64), axis=0))              # [T, H]
    for s in range(t.g.shape[0]):
        want = gam[s][:, None] * np.einsum("hdn,hn->hd", S0, t.q[s][hg].astype(np.float64))
        assert np.allclose(o[s], want, rtol=1e-12, atol=1e-12)
    assert np.allclose(S, gam[-1][:, None, None] * S0, rtol=1e-12, atol=1e-12)


def test_gdn_delta_rule_writes_the_value_at_its_key():
    # no decay, beta = 1, unit keys: after token t the state maps k_t to v_t exactly
    d, t, S0 = _gdn_case(62)
    k = t.k.astype(np.float64)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    hg = np.arange(d.nheads) // (d.nheads // d.ngroups)
    for n in range(1, t.g.shape[0] + 1):
        _, S = oracle.gdn_recurrence(t.q[:n], k[:n], t.v[:n], np.zeros_like(t.g[:n]), np.ones_like(t.beta[:n]), S0)
        assert np.allclose(np.einsum("hdn,hn->hd", S, k[n - 1][hg]), t.v[n - 1], rtol=1e-12, atol=1e-12)


def test_gdn_triangular_solve_form():
    """The page's reassociation: with u from the triangular system
    u_j + sum_{i<j} beta_j gamma_{i+1:j} (k_i . k_j) u_i = beta_j (v_j - gamma_j S_ckpt k_j),
    S_h = gamma_h S_ckpt + sum_j gamma_{j+1:h} u_j k_j^T and o_s = S_s q_s in the same terms."""
    d, t, S0 = _gdn_case(63, T=9)
    o, Sfin = oracle.gdn_recurrence(t.q, t.k, t.v, t.g, t.beta, S0)
    T = t.g.shape[0]
    hg = np.arange(d.nheads) // (d.nheads // d.ngroups)
    for h in range(d.nheads):
        k = t.k[:, hg[h]].astype(np.float64); q = t.q[:, hg[h]].astype(np.float64)
        v = t.v[:, h].astype(np.float64); beta = t.beta[:, h].astype(np.float64)
        G = np.cumsum(t.g[:, h].astype(np.float64))
        gam = lambda a, b: np.exp(G[b] - (G[a - 1] if a > 0 else 0.0))   # prod_{i=a}^{b} alpha_i
        u = np.zeros((T, d.dv))
        for j in range(T):
            rhs = beta[j] * (v[j] - gam(0, j) * S0[h] @ k[j])
            for i in range(j):
                rhs -= beta[j] * gam(i + 1, j) * (k[i] @ k[j]) * u[i]
            u[j] = rhs
        S = gam(0, T - 1) * S0[h] + sum(gam(j + 1, T - 1) * np.outer(u[j], k[j]) if j + 1 <= T - 1
                                       else np.outer(u[j], k[j]) for j in range(T))
        assert np.allclose(S, Sfin[h], rtol=1e-11, atol=1e-11)
        for s in range(T):
            os_ = gam(0, s) * S0[h] @ q[s] + sum((gam(j + 1, s) if j < s else 1.0) * (k[j] @ q[s]) * u[j]
                                                 for j in range(s + 1))
            assert np.allclose(os_, o[s, h], rtol=1e-11, atol=1e-11)


def test_gdn_protocol_pins():
    """Zero acceptance keeps the anchor; the committed stream equals the plain recurrence from the
    anchor; the anchor does not depend on the read precision."""
    d = synth.GdnDims(4, 2, 8, 6, 5)
    rng = np.random.Generator(np.random.PCG64(64))
    S, T, K = 3, 3, 8
    anchor = rng.standard_normal((S, d.nheads, d.dv, d.dk))
    drafts = [[tuple(getattr(synth.make_gdn_tokens(rng, T, d, False), f) for f in ("q", "k", "v", "g", "beta"))
               for _ in range(S)] for _ in range(K)]
    acc = rng.integers(0, T + 1, size=(K, S))
    m0 = oracle.GdnReplayModel(anchor, d.window)
    for k in range(K):
        m0.verify(drafts[k]); m0.commit([0] * S)
    assert np.array_equal(m0.anchor, anchor) and m0.flushes == 0
    m1 = oracle.GdnReplayModel(anchor, d.window)
    m2 = oracle.GdnReplayModel(anchor, d.window, read_cast=lambda a: np.asarray(a, dtype=np.float64))
    stream = [[] for _ in range(S)]
    for k in range(K):
        y1 = m1.verify(drafts[k]); m1.commit(acc[k])
        y2 = m2.verify(drafts[k]); m2.commit(acc[k])
        for i in range(S):
            stream[i] += [tuple(f[j] for f in drafts[k][i]) for j in range(acc[k, i])]
    assert m1.flushes > 0 and np.array_equal(m1.anchor, m2.anchor) and not np.array_equal(y1, y2)
    for i in range(S):
        recs = tuple(np.stack([r[f] for r in stream[i]]) for f in range(5))
        _, want = oracle.gdn_recurrence(*recs, anchor[i])
        got = m2.anchor[i]
        rest = m2.committed[i]
        if rest:
            _, got = oracle.gdn_recurrence(*(np.stack([r[f] for r in rest]) for f in range(5)), got)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-12)


def test_gdn_protocol_drafts_and_recast_copy():
    """The drafts of one verify give the outputs of one-draft verifies with each committed in turn
    (the same rows, the same outputs); and a flushing verify's outputs read the copy recast from the
    folded anchor: the recurrence over the draft alone from the bf16 cast of the new anchor."""
    d = synth.GdnDims(4, 2, 8, 6, 5)
    rng = np.random.Generator(np.random.PCG64(65))
    S, T = 3, 3
    tok = lambda n: tuple(getattr(synth.make_gdn_tokens(rng, n, d, False), f) for f in ("q", "k", "v", "g", "beta"))
    anchor = rng.standard_normal((S, d.nheads, d.dv, d.dk))
    hist = [tok(2) for _ in range(S)]                       # two committed records per sequence
    drafts = [tok(T) for _ in range(S)]
    ma = oracle.GdnReplayModel(anchor, d.window)
    mb = oracle.GdnReplayModel(anchor, d.window)
    for m in (ma, mb):
        m.verify(hist); m.commit([2] * S)
    ya = ma.verify(drafts)
    for s in range(T):
        yb = mb.verify([tuple(f[s:s + 1] for f in dr) for dr in drafts]); mb.commit([1] * S)
        assert np.allclose(yb[:, 0], ya[:, s], rtol=1e-12, atol=1e-12)
    assert ma.flushes == 0 and mb.flushes == 0
    # mb now holds 5 = L records: the next one-draft verify flushes first
    nxt = [tok(1) for _ in range(S)]
    y = mb.verify(nxt)
    assert mb.flushes == S
    for i in range(S):
        want, _ = oracle.gdn_recurrence(*nxt[i], oracle.bf16_round(mb.anchor[i]))
        assert np.allclose(y[i], want, rtol=1e-12, atol=1e-12)
