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


def out_err(got: torch.Tensor, ref: np.ndarray) -> float:
    g = got.float().cpu().numpy().astype(np.float64)
    return float(np.abs(g - ref).mean() / np.abs(ref).mean())


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


def out_tol(tokens) -> float:
    return OUT_TOL_BF16 if tokens.bf16 else OUT_TOL_F32
