"""Seeded synthetic inputs for the Mamba2 SSD / exact-replay workloads.

This module is shared by the fp64 oracle tests, the GPU parity tests and the
bench.  It draws random numbers and shapes them; it holds none of the method's
arithmetic (no softplus, no decay, no scan).

Value distributions follow the "realistic Mamba2 init" the exact-replay RFC
uses for its kernel evidence (vLLM issue 55524, section 2 "Evidence"):
  A[h]        = -U[1, 16]
  dt_raw      ~ N(0, 1)            (raw dt; the kernels apply softplus(dt + dt_bias))
  dt_bias[h]  = log(expm1(u)),  u ~ U[1e-3, 1e-1]  (so softplus(dt_bias) ~ U[1e-3, 1e-1])
  x, B, C, D  ~ N(0, 1)
x, B and C are rounded to bf16 (round-to-nearest-even) when a workload is bf16;
both the oracle and the GPU path consume the rounded values.

numpy's PCG64 generator is used because its stream is identical on x86_64 and
aarch64 hosts.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence, Tuple

import numpy as np

__all__ = [
    "Dims", "Params", "Tokens", "to_bf16_bits", "from_bf16_bits", "round_bf16",
    "make_params", "make_tokens", "WORKLOADS", "workload",
]


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (int16), round-to-nearest-even on the fp32 bits."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16).view(np.int16)


def from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (int16/uint16) -> float32 (exact)."""
    u = np.ascontiguousarray(b).view(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 value, returned as float32."""
    return from_bf16_bits(to_bf16_bits(a))


@dataclasses.dataclass(frozen=True)
class Dims:
    nheads: int      # H
    ngroups: int     # G
    headdim: int     # P
    dstate: int      # N
    chunk: int       # Q (chunk size; also the refresh period L in exact mode)


@dataclasses.dataclass
class Params:
    A: np.ndarray        # [H] float32, negative
    D: np.ndarray        # [H] float32
    dt_bias: np.ndarray  # [H] float32


@dataclasses.dataclass
class Tokens:
    """Token-major inputs.  x/B/C are float32 arrays holding bf16-representable
    values when ``bf16`` is true (their bf16 bit patterns are in *_bits)."""
    x: np.ndarray        # [T, H, P]
    dt: np.ndarray       # [T, H] raw dt (float32)
    B: np.ndarray        # [T, G, N]
    C: np.ndarray        # [T, G, N]
    bf16: bool

    @property
    def ntokens(self) -> int:
        return self.x.shape[0]

    def bits(self, name: str) -> np.ndarray:
        return to_bf16_bits(getattr(self, name))

    def slice(self, lo: int, hi: int) -> "Tokens":
        return Tokens(self.x[lo:hi], self.dt[lo:hi], self.B[lo:hi], self.C[lo:hi], self.bf16)

    @staticmethod
    def concat(parts: Sequence["Tokens"]) -> "Tokens":
        return Tokens(np.concatenate([p.x for p in parts]), np.concatenate([p.dt for p in parts]),
                      np.concatenate([p.B for p in parts]), np.concatenate([p.C for p in parts]),
                      parts[0].bf16)


def make_params(rng: np.random.Generator, H: int) -> Params:
    A = -rng.uniform(1.0, 16.0, size=H)
    u = rng.uniform(1e-3, 1e-1, size=H)
    dt_bias = np.log(np.expm1(u))
    D = rng.standard_normal(H)
    return Params(A.astype(np.float32), D.astype(np.float32), dt_bias.astype(np.float32))


def make_tokens(rng: np.random.Generator, T: int, dims: Dims, bf16: bool) -> Tokens:
    H, G, P, N = dims.nheads, dims.ngroups, dims.headdim, dims.dstate
    x = rng.standard_normal((T, H, P)).astype(np.float32)
    dt = rng.standard_normal((T, H)).astype(np.float32)
    B = rng.standard_normal((T, G, N)).astype(np.float32)
    C = rng.standard_normal((T, G, N)).astype(np.float32)
    if bf16:
        x, B, C = round_bf16(x), round_bf16(B), round_bf16(C)
    return Tokens(x, dt, B, C, bf16)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    bf16: bool
    seqlens: tuple = ()          # prefill workloads
    batch: int = 0               # decode / verify workloads
    steps: int = 0
    history_chunks: int = 0      # decode: full chunks of history before the partial chunk
    drafts: int = 0              # verify: draft tokens per step


WORKLOADS = {
    # 1 sequence, 64 tokens, 4 heads / 1 group, headdim 16, dstate 16, chunk 16, all fp32
    "tiny_fp32": Workload("tiny_fp32", Dims(4, 1, 16, 16, 16), False, seqlens=(64,)),
    # SSD prefill, batch 1, 2048 tokens, 32 heads / 1 group, headdim 64, dstate 128, chunk 256
    "prefill_2048_h32": Workload("prefill_2048_h32", Dims(32, 1, 64, 128, 256), True, seqlens=(2048,)),
    # varlen packed SSD prefill {2048, 777, 513, 1}, 64 heads / 8 groups
    "varlen_4seq_h64": Workload("varlen_4seq_h64", Dims(64, 8, 64, 128, 256), True, seqlens=(2048, 777, 513, 1)),
    # replay decode, 256 sequences, 64 heads / 8 groups, chunk = refresh period = 16, 64 steps
    "decode_b256_h64": Workload("decode_b256_h64", Dims(64, 8, 64, 128, 16), True, batch=256, steps=64,
                                history_chunks=2),
    # speculative verify, 512 sequences, 4 drafts, L = 16, 32 steps
    "verify_b512_t4": Workload("verify_b512_t4", Dims(64, 8, 64, 128, 16), True, batch=512, steps=32, drafts=4),
}


def workload(name: str) -> Workload:
    return WORKLOADS[name]


def prefill_inputs(w: Workload, seed: int = 0, seqlens: Optional[Sequence[int]] = None):
    """(params, tokens, cu_seqlens) for a packed varlen prefill workload."""
    rng = np.random.Generator(np.random.PCG64(seed))
    params = make_params(rng, w.dims.nheads)
    lens = tuple(seqlens) if seqlens is not None else w.seqlens
    toks = make_tokens(rng, int(sum(lens)), w.dims, w.bf16)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    return params, toks, cu


def decode_inputs(w: Workload, seed: int = 0, batch: Optional[int] = None, steps: Optional[int] = None):
    """Inputs for the replay-decode workload.

    Returns (params, history, p0, stream): history is a list (per sequence) of
    Tokens with history_chunks*Q + p0[i] entries (p0 ~ U{0..Q-1}); stream is a
    Tokens batch of shape [steps, batch, ...] flattened as steps*batch rows
    (row k*batch + i is sequence i's token at decode step k).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    S = batch if batch is not None else w.batch
    K = steps if steps is not None else w.steps
    Q = w.dims.chunk
    params = make_params(rng, w.dims.nheads)
    p0 = rng.integers(0, Q, size=S).astype(np.int32)
    hist = [make_tokens(rng, w.history_chunks * Q + int(p0[i]), w.dims, w.bf16) for i in range(S)]
    stream = make_tokens(rng, K * S, w.dims, w.bf16)
    return params, hist, p0, stream


def verify_inputs(w: Workload, seed: int = 0, batch: Optional[int] = None, steps: Optional[int] = None,
                  history: int = 32):
    """Inputs for the speculative-verify workload.

    Returns (params, hist, drafts, accepted): hist is Tokens with batch*history
    rows (sequence i owns rows [i*history, (i+1)*history)), prefilled to form
    the starting recurrence anchor; drafts is Tokens with steps*batch*T rows
    (row (k*batch + i)*T + j is draft j of sequence i at step k); accepted is an
    int32 [steps, batch] array with values ~ U{0..T}.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    S = batch if batch is not None else w.batch
    K = steps if steps is not None else w.steps
    T = w.drafts
    params = make_params(rng, w.dims.nheads)
    hist = make_tokens(rng, S * history, w.dims, w.bf16)
    drafts = make_tokens(rng, K * S * T, w.dims, w.bf16)
    accepted = rng.integers(0, T + 1, size=(K, S)).astype(np.int32)
    return params, hist, drafts, accepted


def exact_fold_inputs(seed: int, S: int, K: int, dims: Dims):
    """Inputs whose refresh folds are exact in fp32 (and fp64): A = 0 and dt_bias = 0, raw dt = 40
    (softplus passes large arguments through, so every step's weight is 40 and every decay 1), x in
    {k / 8 : |k| <= 16}, B in {k / 4 : |k| <= 8}, C and D ~ N(0, 1).  Every weighted product is then a
    multiple of 1/4 below 2^8, so a fold over at most 16 records adds less than 2^12 and the state
    stays exact in fp32 (24 bits) while its values are multiples of 2^-8 below 2^15: the initial state
    is N(0, 1) rounded to multiples of 2^-8.  Returns (params, stream [K*S rows], initial fp32 state
    [S, H, P, N])."""
    rng = np.random.Generator(np.random.PCG64(seed))
    H, G, P, N = dims.nheads, dims.ngroups, dims.headdim, dims.dstate
    params = Params(np.zeros(H, np.float32), rng.standard_normal(H).astype(np.float32), np.zeros(H, np.float32))
    T = K * S
    x = (rng.integers(-16, 17, (T, H, P)) / 8.0).astype(np.float32)
    dt = np.full((T, H), 40.0, np.float32)
    B = (rng.integers(-8, 9, (T, G, N)) / 4.0).astype(np.float32)
    C = round_bf16(rng.standard_normal((T, G, N)).astype(np.float32))
    state = (np.round(rng.standard_normal((S, H, P, N)) * 256.0) / 256.0).astype(np.float32)
    return params, Tokens(x, dt, B, C, True), state


def quant_probe_state(seed: int, shape: Tuple[int, ...]) -> np.ndarray:
    """fp32 states for read-copy quantisation checks: Gaussian rows with per-row magnitudes from
    2^-30 to 2^30, plus rows that stress the edge cases of a per-row scale: an all-zero row, a row
    with one large entry and the rest 2^-14 below it (codes in the subnormal range), a constant row,
    a row of alternating signs and a row with a single nonzero entry.  The last axis is dstate; the
    special rows sit in the first (sequence, head) and need at least 6 rows there."""
    rng = np.random.Generator(np.random.PCG64(seed))
    s = rng.standard_normal(shape).astype(np.float32)
    mag = np.exp2(rng.integers(-30, 31, size=shape[:-1] + (1,))).astype(np.float32)
    s *= mag
    first = s.reshape(-1, shape[-2], shape[-1])[0]
    N = shape[-1]
    first[0] = 0.0
    first[1] = rng.standard_normal(N).astype(np.float32) * np.float32(2.0 ** -14)
    first[1, 5] = 3.0
    first[2] = np.float32(0.7)
    first[3] = np.where(np.arange(N) % 2 == 0, 1.0, -1.0).astype(np.float32) * np.float32(1e-3)
    first[4] = 0.0
    first[4, N - 1] = -5e-20
    first[5] = rng.uniform(-448.0, 448.0, N).astype(np.float32)
    return s


# ---- gated delta rule (GDN) verify workload ---------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class GdnDims:
    nheads: int      # value heads H
    ngroups: int     # key/query heads G (head h uses group h // (H / G))
    dk: int
    dv: int
    window: int      # refresh window L


@dataclasses.dataclass
class GdnTokens:
    """q, k [T, G, dk] (unit L2 norm per group), v [T, H, dv], g [T, H] log-gates (< 0),
    beta [T, H] in (0, 1).  q, k, v are bf16-representable when bf16."""
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    g: np.ndarray
    beta: np.ndarray


GDN_VERIFY = dict(dims=GdnDims(32, 16, 128, 128, 16), batch=512, drafts=4, steps=32)


def make_gdn_tokens(rng: np.random.Generator, T: int, d: GdnDims, bf16: bool = True) -> GdnTokens:
    """Gated-delta-rule token inputs: q, k ~ N(0, 1) normalised to unit length per (token, group),
    v ~ N(0, 1), log-gate g = -softplus(N(0, 1)) * 0.1 (decay per token in ~[0.87, 1)), beta =
    sigmoid(N(0, 1)); q, k, v rounded to bf16 (RNE) when bf16."""
    q = rng.standard_normal((T, d.ngroups, d.dk))
    k = rng.standard_normal((T, d.ngroups, d.dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, d.nheads, d.dv))
    g = -np.log1p(np.exp(rng.standard_normal((T, d.nheads)))) * 0.1
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, d.nheads))))
    f32 = lambda a: a.astype(np.float32)
    if bf16:
        q, k, v = round_bf16(f32(q)), round_bf16(f32(k)), round_bf16(f32(v))
    return GdnTokens(f32(q), f32(k), f32(v), f32(g), f32(beta))


def gdn_verify_inputs(seed: int, batch: int, steps: int, dims: Optional[GdnDims] = None, drafts: int = 4):
    """(anchor [batch, H, dv, dk] fp32 ~ N(0, 0.1), drafts GdnTokens with steps*batch*T rows (row
    (k*batch + i)*T + j is draft j of sequence i at step k), accepted [steps, batch] ~ U{0..T})."""
    d = dims if dims is not None else GDN_VERIFY["dims"]
    rng = np.random.Generator(np.random.PCG64(seed))
    anchor = (rng.standard_normal((batch, d.nheads, d.dv, d.dk)) * 0.1).astype(np.float32)
    toks = make_gdn_tokens(rng, steps * batch * drafts, d)
    accepted = rng.integers(0, drafts + 1, size=(steps, batch)).astype(np.int32)
    return anchor, toks, accepted
