"""fp64 CPU oracle for the Mamba2 SSD / exact-replay hot path.

TEST INFRASTRUCTURE ONLY: imported by the test suite, by the package smoke
check and by the bench's CPU-baseline leg, never by the product path.  It
shares no code with the CUDA library (only the seeded input generator in
``synth`` serves both).

Everything here reduces to the plain token-by-token recurrence in
``oracle.c`` (see its header):

    delta_t = softplus(dt_t + dt_bias),  S_t = exp(delta_t A) S_{t-1} + delta_t x_t B_t^T,
    y_t = S_t C_t + D x_t

The protocol models below (prefill, exact-replay decode, ReplaySSM verify and
commit) only decide WHICH tokens the recurrence runs over and from WHICH
starting state, following the exact-replay RFC (vLLM issue 55524, section 3
"Proposal") and the ReplaySSM reproduction notes ("Motivation and method",
"Core equations").

Every function is pinned to something other than itself in tests/test_oracle_pins.py: hand-worked
fixtures (tests/golden), closed forms, library routines (scipy's IIR filter, numpy's convolution,
PyTorch's bf16 cast), brute force over every code of a format, published known-answer vectors and
protocol invariants; tests/test_oracle_mutants.py and tests/test_oracle_py_mutants.py plant
plausible mistakes here and in oracle.c, each of which must fail a pin.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import List, Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
# The mutation test points this at a deliberately broken build of oracle.c.
_LIB_OVERRIDE = os.environ.get("ERS_ORACLE_LIB")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library next to it (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if _LIB_OVERRIDE:
                lib = ctypes.CDLL(_LIB_OVERRIDE)
            else:
                build()
                lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.oracle_ssm_recurrence.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int64)] + \
                [dp] * 9 + [ctypes.c_int]
            lib.oracle_ssm_recurrence.restype = ctypes.c_int
            lib.oracle_softplus.argtypes = [ctypes.c_double]
            lib.oracle_softplus.restype = ctypes.c_double
            _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def softplus(z: float) -> float:
    """fp64 softplus as the oracle recurrence evaluates it."""
    return float(_load().oracle_softplus(float(z)))


def recurrence(x, dt, A, B, C, D, dt_bias, cu_seqlens=None, init_state=None,
               nthreads: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """Run the recurrence over packed sequences.

    x [T,H,P], dt [T,H] (raw), A/D/dt_bias [H], B/C [T,G,N]; cu_seqlens [S+1]
    (default: one sequence of all T tokens); init_state [S,H,P,N] or None (zero).
    Returns (y [T,H,P], final_state [S,H,P,N]) in fp64.
    """
    x, dt, A, B, C, D, dt_bias = map(_f64, (x, dt, A, B, C, D, dt_bias))
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    if cu_seqlens is None:
        cu_seqlens = np.array([0, T], dtype=np.int64)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int64)
    S = cu.shape[0] - 1
    if cu[0] != 0 or cu[-1] != T or np.any(np.diff(cu) < 0):
        raise ValueError("bad cu_seqlens")
    state = np.zeros((S, H, P, N)) if init_state is None else np.array(init_state, dtype=np.float64, copy=True)
    if state.shape != (S, H, P, N):
        raise ValueError("init_state shape")
    state = np.ascontiguousarray(state)
    y = np.zeros((T, H, P))
    rc = _load().oracle_ssm_recurrence(
        S, H, G, P, N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), _ptr(x), _ptr(dt), _ptr(A),
        _ptr(B), _ptr(C), _ptr(D), _ptr(dt_bias), _ptr(state), _ptr(y),
        int(nthreads if nthreads is not None else default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_ssm_recurrence failed ({rc})")
    return y, state


def bf16_round(a: np.ndarray) -> np.ndarray:
    """Round to bf16 (round-to-nearest-even), through fp32 as the GPU anchor is
    stored in fp32.  Returned as fp64 values."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32)
    return r.view(np.float32).astype(np.float64)


E4M3_MAX = 448.0


def e4m3_round(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest FP8 e4m3 value (1 sign, 4 exponent bits with bias 7, 3
    mantissa bits, subnormals below 2^-6, no infinities), ties to even, magnitudes beyond 448
    saturated to 448.  Returned as fp32 values."""
    f = np.asarray(a, dtype=np.float32).astype(np.float64)
    mag = np.abs(f)
    _, e = np.frexp(mag)                          # mag = m * 2**e, m in [0.5, 1): floor(log2 mag) = e - 1
    ex = np.maximum(e - 1, -6)                    # subnormals share the quantum of the smallest binade
    quantum = np.ldexp(1.0, ex - 3)
    r = np.round(mag / quantum) * quantum         # numpy rounds halves to even
    r = np.minimum(r, E4M3_MAX)
    r = np.where(mag == 0, 0.0, r)
    return (np.sign(f) * r).astype(np.float32)


def fp8_row_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """k of an FP8 row scale s = 2**k: the smallest integer with amax <= 448 * 2**k (no code of the
    row saturates), at least -127 (so 1/s stays a finite fp32 power of two; all-zero and
    subnormal-max rows take -127).  With amax = m * 2**e, m in [0.5, 1) and 448 = 0.875 * 2**9,
    the condition reads m * 2**e <= 0.875 * 2**(9 + k)."""
    a = np.asarray(amax, dtype=np.float64)
    m, e = np.frexp(a)
    k = e.astype(np.int64) - 9 + (m > 0.875)
    tiny = a < 2.0 ** -126
    return np.where(tiny, -127, np.maximum(k, -127))


def fp8_rows_round(a: np.ndarray) -> np.ndarray:
    """FP8 read copy of an fp32 state with one power-of-two scale per row (the last axis is dstate):
    s = 2**fp8_row_scale_exponent(amax(|row|)), q = e4m3(v / s) (an exact scaling), read back as
    q * s (exact).  Input values are taken through fp32 as the GPU anchor is stored in fp32;
    returned as fp64."""
    f = np.ascontiguousarray(a, dtype=np.float32).astype(np.float64)
    k = fp8_row_scale_exponent(np.max(np.abs(f), axis=-1, keepdims=True))
    s = np.ldexp(1.0, k)
    q = e4m3_round(f / s).astype(np.float64)
    return q * s


E2M1_MAX = 6.0


def e2m1_round(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to the nearest FP4 e2m1 value (1 sign, 2 exponent bits with bias 1, 1
    mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6), ties to the even mantissa, magnitudes
    beyond 6 saturated to 6.  Returned as fp32 values."""
    f = np.asarray(a, dtype=np.float32).astype(np.float64)
    mag = np.abs(f)
    _, e = np.frexp(mag)                          # floor(log2 mag) = e - 1
    ex = np.maximum(e - 1, 0)                     # the subnormal 0.5 shares the quantum of [1, 2)
    quantum = np.ldexp(1.0, ex - 1)
    r = np.round(mag / quantum) * quantum         # halves to even: even multiples have mantissa 0
    r = np.minimum(r, E2M1_MAX)
    r = np.where(mag == 0, 0.0, r)
    return (np.sign(f) * r).astype(np.float32)


NVFP4_BLOCK = 16


def nvfp4_row_scale_exponent(amax: np.ndarray) -> np.ndarray:
    """k of an NVFP4 row scale s = 2**k: the smallest integer with amax <= 448 * 6 * 2**k (so no
    block scale saturates), at least -127.  448 * 6 = 2688 = 0.65625 * 2**12."""
    a = np.asarray(amax, dtype=np.float64)
    m, e = np.frexp(a)
    k = e.astype(np.int64) - 12 + (m > 0.65625)
    return np.where(a < 2.0 ** -126, -127, np.maximum(k, -127))


def sr_e2m1(v: np.ndarray, r: np.ndarray) -> np.ndarray:
    """Stochastic rounding of fp32 values to the e2m1 grid with one random 32-bit word r per value:
    with lo the largest e2m1 magnitude <= |v| and step the spacing above it (0.5 in [0, 2), 1 in
    [2, 4), 2 in [4, 6)), |v| rounds up to lo + step iff r < 2^32 (|v| - lo) / step, else down to lo;
    magnitudes at or above 6 give 6; the sign is kept.  Returned as fp32 values."""
    f = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(f)
    step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    lo = np.floor(a / step) * step
    frac = (a - lo) / step                                    # exact, in [0, 1)
    up = np.asarray(r, dtype=np.float64) < np.ldexp(frac, 32)
    out = np.where(a >= E2M1_MAX, E2M1_MAX, lo + up * step)
    return np.copysign(out, f).astype(np.float32)


def nvfp4_rows_round(a: np.ndarray, parts: bool = False, words: Optional[np.ndarray] = None):
    """NVFP4 read copy of an fp32 state (the last axis is dstate, a multiple of 16): FP4 e2m1 codes
    in blocks of 16 consecutive values, each block with an e4m3 scale beta, each row with a
    power-of-two scale s = 2**k (k from nvfp4_row_scale_exponent):
        beta = e4m3(t / 6) with t = amax(|block|) / s (exact) and an fp32 division,
        q    = e2m1((v / s) * rho), rho = 1 / beta (fp32 reciprocal, fp32 product); q = 0 if beta = 0,
        value = q * beta * s (exact).
    With words (uint32, the shape of a), q rounds stochastically instead (sr_e2m1 with one word per
    value); the scales are the same.  Input values are taken through fp32 as the GPU anchor is
    stored in fp32; returns fp64 values (and, with parts=True, also q, beta and k)."""
    f = np.ascontiguousarray(a, dtype=np.float32).astype(np.float64)
    N = f.shape[-1]
    k = nvfp4_row_scale_exponent(np.max(np.abs(f), axis=-1, keepdims=True))
    s = np.ldexp(1.0, k)
    fb = (f / s).reshape(f.shape[:-1] + (N // NVFP4_BLOCK, NVFP4_BLOCK))    # v / s, exact in fp64
    fb32 = fb.astype(np.float32)                                              # rounds only below fp32 normal range
    t = np.max(np.abs(fb32), axis=-1, keepdims=True).astype(np.float32)
    beta = e4m3_round(t / np.float32(6.0))
    with np.errstate(divide="ignore"):
        rho = np.where(beta > 0, np.float32(1.0) / np.where(beta > 0, beta, np.float32(1.0)), np.float32(0.0))
    y = (fb32 * rho.astype(np.float32)).astype(np.float32)
    if words is None:
        q = np.where(beta > 0, e2m1_round(y), np.float32(0.0))
    else:
        wb = np.asarray(words).reshape(y.shape)
        q = np.where(beta > 0, sr_e2m1(y, wb), np.float32(0.0))
    val = (q.astype(np.float64) * beta.astype(np.float64)).reshape(f.shape) * s
    if parts:
        return val, q.reshape(f.shape), beta[..., 0], k[..., 0]
    return val


# ---- counter-based random numbers and stochastic rounding of an fp16 anchor ---------------------------
# Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel random numbers: as easy as 1, 2, 3",
# SC 2011): a 4 x 32-bit counter and a 2 x 32-bit key; each of 10 rounds multiplies counter words 0
# and 2 by two constants (64-bit products), mixes the high halves with the other two words and the
# key, and the key advances by two Weyl constants between rounds.
PHILOX_M0, PHILOX_M1 = 0xD2511F53, 0xCD9E8D57
PHILOX_W0, PHILOX_W1 = 0x9E3779B9, 0xBB67AE85


def philox4x32_10(ctr: np.ndarray, key: Tuple[int, int]) -> np.ndarray:
    """ctr [..., 4] uint32 -> [..., 4] uint32 random words."""
    c = np.asarray(ctr, dtype=np.uint64) & 0xFFFFFFFF
    k0, k1 = np.uint64(key[0] & 0xFFFFFFFF), np.uint64(key[1] & 0xFFFFFFFF)
    m32 = np.uint64(0xFFFFFFFF)
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    for rnd in range(10):
        if rnd:
            k0 = (k0 + np.uint64(PHILOX_W0)) & m32
            k1 = (k1 + np.uint64(PHILOX_W1)) & m32
        p0 = c0 * np.uint64(PHILOX_M0)
        p1 = c2 * np.uint64(PHILOX_M1)
        hi0, lo0 = p0 >> np.uint64(32), p0 & m32
        hi1, lo1 = p1 >> np.uint64(32), p1 & m32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


FP16_MAX = 65504.0


def sr_fp16(v: np.ndarray, r: np.ndarray) -> np.ndarray:
    """Stochastic rounding of fp32 values to IEEE binary16 with one random 32-bit word r per value:
    with lo the fp16 value of |v| rounded toward zero and ulp the fp16 spacing there (2^-24 below
    2^-14), |v| rounds up to lo + ulp iff r < 2^32 (|v| - lo) / ulp, else down to lo; the sign is
    kept; magnitudes at or above 65504 give 65504.  Returned as fp64 values (all on the fp16 grid)."""
    f = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(f)
    _, e = np.frexp(a)                                        # a in [2^(e-1), 2^e)
    ue = np.maximum(e - 1, -14) - 10                          # log2 of the fp16 spacing at a
    t = np.ldexp(a, -ue)                                      # exact
    fl = np.floor(t)
    frac = t - fl                                             # exact, in [0, 1)
    up = np.asarray(r, dtype=np.float64) < np.ldexp(frac, 32)
    out = np.ldexp(fl + up, ue)
    out = np.where(a >= FP16_MAX, FP16_MAX, out)
    out = np.where(a == 0, 0.0, out)
    return np.copysign(out, f)


def sr_words(key: Tuple[int, int], nonce: int, slot: int, H: int, P: int, N: int) -> np.ndarray:
    """The random words of one slot's anchor write: element (h, d, n) takes word n % 4 of
    philox4x32_10(counter = (nonce, slot, h * P + d, n // 4), key).  Returns [H, P, N] uint32."""
    hd = np.arange(H * P, dtype=np.uint64)[:, None]
    jj = np.arange(N // 4, dtype=np.uint64)[None, :]
    ctr = np.stack(np.broadcast_arrays(np.uint64(nonce & 0xFFFFFFFF), np.uint64(slot & 0xFFFFFFFF), hd, jj), axis=-1)
    return philox4x32_10(ctr, key).reshape(H, P, N)


def sr_fp16_anchor(fin: np.ndarray, key: Tuple[int, int], nonce: int, slot: int) -> np.ndarray:
    """An fp16 anchor written by stochastic rounding of the refreshed state fin [H, P, N] (taken
    through fp32, as the GPU folds in fp32) with the slot's random words for this nonce."""
    H, P, N = fin.shape
    return sr_fp16(np.asarray(fin, dtype=np.float64).astype(np.float32), sr_words(key, nonce, slot, H, P, N))


def nvfp4_sr_state(fin: np.ndarray, key: Tuple[int, int], nonce: int, slot: int) -> np.ndarray:
    """A shared NVFP4 state written by a refresh: the NVFP4 cast of the refreshed state fin [H, P, N]
    (taken through fp32, as the GPU folds in fp32) with stochastically rounded codes, one word per
    value from the slot's random words for this nonce (the counter layout of the fp16 anchors)."""
    H, P, N = fin.shape
    return nvfp4_rows_round(np.asarray(fin, dtype=np.float64).astype(np.float32),
                            words=sr_words(key, nonce, slot, H, P, N))


# ---- causal depthwise conv1d with a conv state (exact-replay RFC, Evidence item 6) -------------------
def silu(a: np.ndarray) -> np.ndarray:
    """x * sigmoid(x) in fp64."""
    a = np.asarray(a, dtype=np.float64)
    return a / (1.0 + np.exp(-a))


def causal_conv1d(x: np.ndarray, weight: np.ndarray, bias: Optional[np.ndarray], cu_seqlens=None,
                  init_state: Optional[np.ndarray] = None, activation: bool = True):
    """Depthwise causal convolution over time, per packed sequence, in fp64:
        y[t, c] = act(bias[c] + sum_{k < W} weight[c, k] * u[t - W + 1 + k, c]),
    where u is the sequence's inputs preceded by its W - 1 earlier inputs (init_state[i], [W-1, C],
    oldest first; zeros when absent) and act is SiLU or the identity.  Returns (y [T, C], the final
    states [S, W-1, C]: the last W - 1 entries of u)."""
    x = _f64(x)
    w = _f64(weight)
    C, W = w.shape
    T = x.shape[0]
    cu = np.array([0, T] if cu_seqlens is None else cu_seqlens, dtype=np.int64)
    S = len(cu) - 1
    b = np.zeros(C) if bias is None else _f64(bias)
    y = np.zeros((T, C))
    fin = np.zeros((S, W - 1, C))
    for i in range(S):
        pre = np.zeros((W - 1, C)) if init_state is None else _f64(init_state[i])
        u = np.concatenate([pre, x[cu[i]:cu[i + 1]]])
        n = cu[i + 1] - cu[i]
        for t in range(n):
            acc = b.copy()
            for k in range(W):
                acc = acc + w[:, k] * u[t + k]
            y[cu[i] + t] = silu(acc) if activation else acc
        fin[i] = u[len(u) - (W - 1):]
    return y, fin


# ---- gated delta rule (GDN), the second layer family of the ReplaySSM notes ---------------------------
def gdn_recurrence(q, k, v, g, beta, state: np.ndarray):
    """Gated delta rule, token by token in fp64, for one sequence:
        a_t = exp(g_t),  u_t = beta_t (v_t - a_t S_{t-1} k_t),  S_t = a_t S_{t-1} + u_t k_t^T,
        o_t = S_t q_t,
    per value head h with key/query group h // (H / G).  q, k [T, G, dk]; v [T, H, dv]; g, beta
    [T, H]; state [H, dv, dk] (S maps keys to values).  Returns (o [T, H, dv], final state)."""
    S = np.array(state, dtype=np.float64, copy=True)
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    T, H = g.shape
    G = q.shape[1]
    hg = np.arange(H) // (H // G)
    out = np.zeros((T, H, S.shape[1]))
    for t in range(T):
        kt, qt = k[t][hg], q[t][hg]                       # [H, dk]
        a = np.exp(g[t])[:, None]
        Sk = np.einsum("hdn,hn->hd", S, kt)
        u = beta[t][:, None] * (v[t] - a * Sk)
        S = a[:, :, None] * S + u[:, :, None] * kt[:, None, :]
        out[t] = np.einsum("hdn,hn->hd", S, qt)
    return out, S


class GdnReplayModel:
    """ReplaySSM-style speculative decoding for a GDN layer (ReplaySSM notes, "Core equations" and
    "Data protocol and entry point"): per sequence an fp64 anchor, a read copy cast from it, and the
    committed records since the last refresh.  verify() flushes when h + T > L (folds the committed records
    into the anchor with the recurrence, recasts the read copy), then runs the recurrence from the
    READ COPY over committed records + drafts and returns the drafts' outputs; commit() appends the
    accepted drafts.  An empty history leaves the anchor unchanged."""

    def __init__(self, anchor: np.ndarray, L: int, read_cast=None):
        self.anchor = np.array(anchor, dtype=np.float64, copy=True)   # [S, H, dv, dk]
        self.read_cast = read_cast if read_cast is not None else bf16_round
        self.read = self.read_cast(self.anchor)
        self.L = L
        self.committed: List[list] = [[] for _ in range(self.anchor.shape[0])]
        self.flushes = 0

    def h(self) -> np.ndarray:
        return np.array([len(c) for c in self.committed], dtype=np.int32)

    @staticmethod
    def _stack(recs):
        return tuple(np.stack([r[f] for r in recs]) for f in range(5))

    def verify(self, drafts):
        """drafts[i] = (q [T,G,dk], k [T,G,dk], v [T,H,dv], g [T,H], beta [T,H]); returns [S, T, H, dv]."""
        T = drafts[0][0].shape[0]
        outs = []
        for i, dr in enumerate(drafts):
            if len(self.committed[i]) + T > self.L and self.committed[i]:   # flush (never an empty one)
                rec = self._stack(self.committed[i])
                _, fin = gdn_recurrence(*rec, self.anchor[i])
                self.anchor[i] = fin
                self.read[i] = self.read_cast(fin)
                self.committed[i] = []
                self.flushes += 1
            recs = self.committed[i]
            seq = tuple(np.concatenate([self._stack(recs)[f], dr[f]]) if recs else dr[f] for f in range(5))
            o, _ = gdn_recurrence(*seq, self.read[i])
            outs.append(o[len(recs):])
        self._pending = drafts
        return np.stack(outs)

    def commit(self, accepted):
        for i, a in enumerate(accepted):
            for j in range(int(a)):
                self.committed[i].append(tuple(self._pending[i][f][j] for f in range(5)))
        self._pending = None


class _Seq:
    __slots__ = ("x", "dt", "B", "C")

    def __init__(self, x, dt, B, C):
        self.x, self.dt, self.B, self.C = x, dt, B, C


def _pack(parts: Sequence[Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]]):
    lens = [p[0].shape[0] for p in parts]
    cu = np.zeros(len(parts) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lens)
    cat = [np.concatenate([p[i] for p in parts]) for i in range(4)]
    return cat, cu


class ReplaySSMModel:
    """ReplaySSM-style speculative decoding with a dual-precision anchor.

    Per sequence: an fp64 recurrence anchor, a bf16 read copy cast from it,
    and the committed input records since the last refresh (h of them).
    ``verify`` flushes when h + T > L (refresh the committed records into the
    anchor and recast the read copy), then returns the T draft outputs computed
    from the READ COPY over committed records + drafts 1..s.  ``commit`` appends
    the first ``accepted`` drafts to the committed records; rejected drafts
    never enter the recurrence.  (ReplaySSM reproduction notes, "Motivation and
    method" and "Core equations": outputs read the low-precision copy, refresh
    forms S from committed raw records and casts both copies from it.)
    """

    def __init__(self, params, anchor: np.ndarray, L: int, nthreads: Optional[int] = None, read_cast=None,
                 anchor_round=None, shared: bool = False):
        self.A, self.D, self.dt_bias = (_f64(params.A), _f64(params.D), _f64(params.dt_bias))
        self.anchor = np.array(anchor, dtype=np.float64, copy=True)  # [S,H,P,N]
        self.read_cast = read_cast if read_cast is not None else bf16_round
        # anchor_round(i, fin) -> the stored anchor of sequence i after a refresh (default: fin itself)
        self.anchor_round = anchor_round
        # shared: the stored anchor is also the read copy (one low-precision state; anchor_round
        # gives it, and the initial anchor must already be in that format)
        self.shared = shared
        self.read = self.anchor.copy() if shared else self.read_cast(self.anchor)
        self.L = L
        self.nthreads = nthreads
        S = anchor.shape[0]
        self.committed: List[List[Tuple[np.ndarray, ...]]] = [[] for _ in range(S)]
        self.flushes = 0

    def h(self) -> np.ndarray:
        return np.array([len(c) for c in self.committed], dtype=np.int32)

    def _records(self, i):
        c = self.committed[i]
        if not c:
            return None
        return tuple(np.stack([r[k] for r in c]) for k in range(4))

    def refresh(self, which: Sequence[int]):
        """Fold the committed records of the listed sequences into their anchors."""
        which = [i for i in which if self.committed[i]]
        if not which:
            return
        parts = [self._records(i) for i in which]
        (x, dt, B, C), cu = _pack(parts)
        _, fin = recurrence(x, dt, self.A, B, C, self.D, self.dt_bias, cu, self.anchor[which], self.nthreads)
        for k, i in enumerate(which):
            self.anchor[i] = fin[k] if self.anchor_round is None else self.anchor_round(i, fin[k])
            self.read[i] = self.anchor[i] if self.shared else self.read_cast(fin[k])
            self.committed[i] = []
        self.flushes += len(which)

    def verify(self, drafts: Sequence[Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]]) -> np.ndarray:
        """drafts[i] = (x [T,H,P], dt [T,H], B [T,G,N], C [T,G,N]).  Returns y [S,T,H,P]."""
        S = len(drafts)
        T = drafts[0][0].shape[0]
        flush = [i for i in range(S) if len(self.committed[i]) + T > self.L]
        self.refresh(flush)
        parts = []
        for i in range(S):
            rec = self._records(i)
            if rec is None:
                parts.append(drafts[i])
            else:
                parts.append(tuple(np.concatenate([rec[k], drafts[i][k]]) for k in range(4)))
        (x, dt, B, C), cu = _pack(parts)
        y, _ = recurrence(x, dt, self.A, B, C, self.D, self.dt_bias, cu, self.read, self.nthreads)
        H, P = x.shape[1], x.shape[2]
        out = np.zeros((S, T, H, P))
        for i in range(S):
            out[i] = y[cu[i + 1] - T:cu[i + 1]]
        self._pending = drafts
        return out

    def commit(self, accepted: Sequence[int]):
        for i, a in enumerate(accepted):
            if a < 0 or a > self._pending[i][0].shape[0]:
                raise ValueError("accepted out of range")
            for j in range(int(a)):
                self.committed[i].append(tuple(self._pending[i][k][j] for k in range(4)))
        self._pending = None
