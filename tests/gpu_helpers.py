"""Shared helpers of the GPU parity tests (metrics and input plumbing; no method arithmetic)."""
import numpy as np
import torch

import synth
from synth import torch_io

# Parity tolerances: bf16 outputs mean|dy| <= 2e-3 mean|y|; fp32 states
# max|dS| <= 1e-5 max|S| per (sequence, head).  fp32-io outputs are held to 1e-5 as well.
OUT_TOL_BF16 = 2e-3
OUT_TOL_F32 = 1e-5
STATE_TOL = 1e-5


def dev():
    return torch.device("cuda:0")


def layer(params):
    import exact_replay_decode_gb300 as ers
    A, D, dtb = torch_io.params_to(params, dev())
    return ers.LayerParams(A, D, dtb)


# Sanity bound on single elements: within a unit (one sequence and head), max|dy| may not exceed
# this fraction of the unit's max|y|.  bf16 output rounding alone contributes at most 2^-8 of it
# (half an ulp of the largest binade); read copies with 4- or 8-bit codes get a looser bound, since
# one code the GPU's fp32 state and the oracle's fp64 state round to different sides moves an
# output by a fraction of a block's largest value.
MAX_REL_BF16 = 2.0 ** -6
MAX_REL_NARROW = 2.0 ** -3


def out_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.float().cpu().numpy().astype(np.float64)
    return float(np.abs(g - ref).mean() / np.abs(ref).mean())


def unit_errs(got, ref: np.ndarray, keep, cu=None):
    """Per-unit parity metrics.  A unit is one index of the `keep` axes (e.g. the head axis) within
    one packed sequence (rows cu[i]:cu[i+1] of axis 0 when cu is given).  Returns the arrays
    (mean|dy| / mean|y|, max|dy| / max|y|) over all units."""
    g = got.float().cpu().numpy().astype(np.float64) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    keep = tuple(a % g.ndim for a in (keep if isinstance(keep, (tuple, list)) else (keep,)))
    bounds = [(0, g.shape[0])] if cu is None else [(int(cu[i]), int(cu[i + 1])) for i in range(len(cu) - 1)]
    means, maxes = [], []
    for lo, hi in bounds:
        if hi <= lo:
            continue
        gs, rs = g[lo:hi], r[lo:hi]
        rest = [a for a in range(g.ndim) if a not in keep]
        gu = np.transpose(gs, keep + tuple(rest)).reshape(-1, int(np.prod([gs.shape[a] for a in rest])))
        ru = np.transpose(rs, keep + tuple(rest)).reshape(gu.shape)
        d = np.abs(gu - ru)
        means.append(d.mean(axis=1) / np.maximum(np.abs(ru).mean(axis=1), 1e-300))
        maxes.append(d.max(axis=1) / np.maximum(np.abs(ru).max(axis=1), 1e-300))
    return np.concatenate(means), np.concatenate(maxes)


def check_out(got, ref: np.ndarray, tol: float, keep, cu=None, max_rel=MAX_REL_BF16, what: str = "") -> float:
    """Asserts the output parity bar on the whole tensor AND on every unit (see unit_errs):
    mean|dy| <= tol * mean|y| for both, and max|dy| <= max_rel * max|y| per unit (max_rel None skips
    the element bound).  Returns the whole-tensor metric."""
    whole = out_err(got, ref) if isinstance(got, torch.Tensor) else \
        float(np.abs(np.asarray(got, np.float64) - ref).mean() / np.abs(ref).mean())
    assert whole <= tol, f"{what} whole-tensor mean|dy|/mean|y| = {whole:.3e} > {tol:.1e}"
    m, x = unit_errs(got, ref, keep, cu)
    w = int(np.argmax(m))
    assert m[w] <= tol, f"{what} unit {w}: mean|dy|/mean|y| = {m[w]:.3e} > {tol:.1e} (whole tensor {whole:.3e})"
    if max_rel is not None:
        w = int(np.argmax(x))
        assert x[w] <= max_rel, f"{what} unit {w}: max|dy|/max|y| = {x[w]:.3e} > {max_rel:.3e}"
    return whole


def state_err(got: torch.Tensor, ref: np.ndarray) -> float:
    """max over leading (seq, head) of max|dS| / max|S_ref|."""
    g = got.float().cpu().numpy().astype(np.float64)
    P, N = ref.shape[-2], ref.shape[-1]
    d = np.abs(g - ref).reshape(-1, P * N).max(axis=1)
    r = np.abs(ref).reshape(-1, P * N).max(axis=1)
    return float((d / np.maximum(r, 1e-30)).max())


def bits(t: torch.Tensor) -> torch.Tensor:
    return t.contiguous().view({2: torch.int16, 4: torch.int32}[t.element_size()])


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    return a.shape == b.shape and torch.equal(bits(a), bits(b))


def read_values(cache):
    """Inspection of a cache's read copy in the tests: its values as fp32 tensors (bf16 as is; FP8
    e4m3 code times the row scale; NVFP4 e2m1 code times block scale times row scale), or None
    without a read copy.  Decodes the stored bytes per the layouts include/ers.h documents."""
    if cache.read_copy is None:
        return None
    if cache.read_scale is None:
        return cache.read_copy.float()
    if cache.read_block_scale is None:
        return cache.read_copy.view(torch.float8_e4m3fn).float() * cache.read_scale.unsqueeze(-1)
    e2m1 = torch.tensor([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.0, -0.5, -1, -1.5, -2, -3, -4, -6],
                        dtype=torch.float32, device=cache.read_copy.device)
    c = cache.read_copy.long()
    q = torch.stack([e2m1[c & 15], e2m1[c >> 4]], dim=-1).flatten(-2)
    beta = cache.read_block_scale.view(torch.float8_e4m3fn).float().repeat_interleave(16, dim=-1)
    return q * beta * cache.read_scale.unsqueeze(-1)


def out_tol(tokens) -> float:
    return OUT_TOL_BF16 if tokens.bf16 else OUT_TOL_F32


def max_rel(tokens) -> float:
    """Element bound of check_out: bf16 outputs as MAX_REL_BF16; fp32 outputs 1e-4 of the unit's max."""
    return MAX_REL_BF16 if tokens.bf16 else 1e-4


class StepCheck:
    """Parity over a run of steps: each step's whole output tensor is held to `tol` when it arrives,
    and at the end every unit (the `keep` axes of one step's tensor, e.g. sequence and head) is held
    to check_out's bars over all steps together, so that a unit holds as many outputs as the run
    gives it rather than one noisy row."""

    def __init__(self, tol: float, keep, max_rel=MAX_REL_BF16, what: str = ""):
        self.tol, self.keep, self.max_rel, self.what = tol, tuple(keep), max_rel, what
        self.got, self.ref = [], []

    def step(self, got, ref, label=""):
        g = got.float().cpu().numpy().astype(np.float64)
        r = np.asarray(ref, np.float64)
        e = float(np.abs(g - r).mean() / np.abs(r).mean())
        assert e <= self.tol, f"{self.what} {label}: whole-step mean|dy|/mean|y| = {e:.3e} > {self.tol:.1e}"
        self.got.append(g)
        self.ref.append(r)

    def finish(self):
        return check_out(np.stack(self.got), np.stack(self.ref), self.tol, keep=tuple(k + 1 for k in self.keep),
                         max_rel=self.max_rel, what=self.what + " (all steps)")
