"""Moves seeded synthetic inputs (numpy) onto a torch device.  Holds no method arithmetic."""
from __future__ import annotations

import numpy as np
import torch

from . import Params, Tokens, to_bf16_bits


def io_dtype(tokens: Tokens) -> torch.dtype:
    return torch.bfloat16 if tokens.bf16 else torch.float32


def _io(a: np.ndarray, bf16: bool, device) -> torch.Tensor:
    if bf16:
        return torch.from_numpy(np.ascontiguousarray(to_bf16_bits(a))).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def tokens_to(tokens: Tokens, device, lead=None):
    """(x, dt, B, C) on `device`; x/B/C in bf16 (bit-exact) or fp32.  `lead` reshapes the token axis."""
    x = _io(tokens.x, tokens.bf16, device)
    dt = torch.from_numpy(np.ascontiguousarray(tokens.dt, dtype=np.float32)).to(device)
    B = _io(tokens.B, tokens.bf16, device)
    C = _io(tokens.C, tokens.bf16, device)
    if lead is not None:
        x = x.reshape(*lead, *x.shape[1:])
        dt = dt.reshape(*lead, *dt.shape[1:])
        B = B.reshape(*lead, *B.shape[1:])
        C = C.reshape(*lead, *C.shape[1:])
    return x, dt, B, C


def params_to(params: Params, device):
    """(A, D, dt_bias) fp32 tensors on `device`."""
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)
    return f(params.A), f(params.D), f(params.dt_bias)
