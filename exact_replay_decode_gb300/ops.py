"""PyTorch-facing binding of the C ABI (include/ers.h).

Marshalling only: every step of the hot path runs in the CUDA library.  PyTorch provides device
memory, streams and shape/dtype checks; outputs and workspaces are allocated here with torch so
the library itself never allocates.
"""
from __future__ import annotations

import ctypes
import dataclasses
from typing import Optional, Sequence, Tuple, Union

import torch

from . import _abi

_IO = {torch.bfloat16: _abi.DTYPE_BF16, torch.float32: _abi.DTYPE_F32}


@dataclasses.dataclass
class LayerParams:
    """Per-head parameters, fp32 [H] on the device: A (< 0), D (skip) and dt_bias."""
    A: torch.Tensor
    D: torch.Tensor
    dt_bias: torch.Tensor

    def _c(self) -> _abi.Params:
        for t in (self.A, self.D, self.dt_bias):
            _need(t, torch.float32, "params")
        return _abi.Params(self.A.data_ptr(), self.D.data_ptr(), self.dt_bias.data_ptr())


def _need(t: torch.Tensor, dtype, name: str, shape: Optional[Sequence[int]] = None) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Status:
    """Device int32 status word the kernels report into; read() synchronises."""

    def __init__(self, device=None):
        self.t = torch.zeros(1, dtype=torch.int32, device=device or "cuda")

    def ptr(self) -> int:
        return self.t.data_ptr()

    def reset(self) -> None:
        self.t.zero_()

    def read(self) -> int:
        return int(self.t.item())

    def raise_if_error(self, where: str) -> None:
        code = self.read()
        if code != 0:
            raise _abi.ErsError(code, where)


def _finish(code: int, where: str, status: Optional[Status], check: bool) -> None:
    _abi.check(code, where)
    if check and status is not None:
        status.raise_if_error(where)


def _dims(H: int, G: int, P: int, N: int, Q: int, io: torch.dtype) -> _abi.Dims:
    if io not in _IO:
        raise TypeError(f"io dtype {io} not supported (bf16 or fp32)")
    return _abi.Dims(H, G, P, N, Q, _IO[io])


def _io_from(x: torch.Tensor) -> torch.dtype:
    if x.dtype not in _IO:
        raise TypeError(f"x dtype {x.dtype} not supported (bf16 or fp32)")
    return x.dtype


def _max_len(cu_seqlens: torch.Tensor, max_seqlen: Optional[int]) -> int:
    if max_seqlen is not None:
        return int(max_seqlen)
    lens = (cu_seqlens[1:] - cu_seqlens[:-1]).max() if cu_seqlens.numel() > 1 else torch.zeros(())
    return int(lens.item())


# ------------------------------------------------------------------------------------------------
def ssd_scan_fwd(x: torch.Tensor, dt: torch.Tensor, params: LayerParams, B: torch.Tensor, C: torch.Tensor,
                 chunk: int, cu_seqlens: Optional[torch.Tensor] = None, init_state: Optional[torch.Tensor] = None,
                 return_chunk_states: bool = False, max_seqlen: Optional[int] = None,
                 status: Optional[Status] = None, check: bool = True, stream=None,
                 out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None, workspace: Optional[torch.Tensor] = None):
    """Chunked SSD prefill over packed varlen sequences (ers_ssd_scan_fwd).

    x [T,H,P], dt [T,H] fp32 raw, B/C [T,G,N]; cu_seqlens int32 [S+1] (default: one sequence).
    Returns (y [T,H,P], final_state [S,H,P,N] fp32[, chunk_states [S,ceil(max_seqlen/Q),H,P,N]]).
    """
    io = _io_from(x)
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    dev = x.device
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    S = cu_seqlens.numel() - 1
    _need(x, io, "x", (T, H, P)); _need(dt, torch.float32, "dt", (T, H))
    _need(B, io, "B", (T, G, N)); _need(C, io, "C", (T, G, N)); _need(cu_seqlens, torch.int32, "cu_seqlens")
    if init_state is not None:
        _need(init_state, torch.float32, "init_state", (S, H, P, N))
    ms = _max_len(cu_seqlens, max_seqlen)
    dims = _dims(H, G, P, N, chunk, io)
    if out is None:
        y = torch.empty_like(x)
        fin = torch.empty(S, H, P, N, dtype=torch.float32, device=dev)
    else:
        y, fin = out
    cs = None
    if return_chunk_states:
        cs = torch.empty(S, (ms + chunk - 1) // chunk, H, P, N, dtype=torch.float32, device=dev)
    L = _abi.lib()
    wsz = L.ers_ssd_scan_fwd_workspace_size(ctypes.byref(dims), S, ms)
    if workspace is None or workspace.numel() < wsz:
        workspace = torch.empty(max(wsz, 1), dtype=torch.uint8, device=dev)
    st = status if status is not None else (Status(dev) if check else None)
    code = L.ers_ssd_scan_fwd(ctypes.byref(dims), ctypes.byref(params._c()), S, T, ms, cu_seqlens.data_ptr(),
                              x.data_ptr(), dt.data_ptr(), B.data_ptr(), C.data_ptr(), _ptr(init_state),
                              y.data_ptr(), fin.data_ptr(), _ptr(cs), workspace.data_ptr(), workspace.numel(),
                              _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_ssd_scan_fwd", st, check)
    return (y, fin, cs) if return_chunk_states else (y, fin)


def ssd_scan_fwd_static(x: torch.Tensor, dt: torch.Tensor, params: LayerParams, B: torch.Tensor, C: torch.Tensor,
                        chunk: int, cu_seqlens: Optional[torch.Tensor] = None,
                        init_state: Optional[torch.Tensor] = None, max_seqlen: Optional[int] = None,
                        status: Optional[Status] = None, check: bool = True, stream=None,
                        out: Optional[Tuple[torch.Tensor, torch.Tensor]] = None):
    """ssd_scan_fwd through ers_ssd_scan_fwd_static: the library's fixed device scratch
    (STATIC_SCRATCH_BYTES per device) instead of a workspace.  Raises ErsError (ERS_EWORKSPACE) when
    the call needs more scratch than that.  Calls that may overlap on one device race on the scratch."""
    io = _io_from(x)
    T, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    dev = x.device
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=dev)
    S = cu_seqlens.numel() - 1
    _need(x, io, "x", (T, H, P)); _need(dt, torch.float32, "dt", (T, H))
    _need(B, io, "B", (T, G, N)); _need(C, io, "C", (T, G, N)); _need(cu_seqlens, torch.int32, "cu_seqlens")
    if init_state is not None:
        _need(init_state, torch.float32, "init_state", (S, H, P, N))
    ms = _max_len(cu_seqlens, max_seqlen)
    dims = _dims(H, G, P, N, chunk, io)
    if out is None:
        y = torch.empty_like(x)
        fin = torch.empty(S, H, P, N, dtype=torch.float32, device=dev)
    else:
        y, fin = out
    st = status if status is not None else (Status(dev) if check else None)
    code = _abi.lib().ers_ssd_scan_fwd_static(
        ctypes.byref(dims), ctypes.byref(params._c()), S, T, ms, cu_seqlens.data_ptr(), x.data_ptr(),
        dt.data_ptr(), B.data_ptr(), C.data_ptr(), _ptr(init_state), y.data_ptr(), fin.data_ptr(), None,
        _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_ssd_scan_fwd_static", st, check)
    return y, fin


STATIC_SCRATCH_BYTES = 32 << 20


def selftest_bounded_wait(limit_ns: int, status: Status, stream=None) -> None:
    """ers_selftest_bounded_wait: two blocks whose waits (an mbarrier, a device flag) are never
    satisfied give up after limit_ns and report ERS_ETIMEOUT through `status`."""
    code = _abi.lib().ers_selftest_bounded_wait(int(limit_ns), _stream(stream), status.ptr())
    _finish(code, "ers_selftest_bounded_wait", None, False)


# ------------------------------------------------------------------------------------------------
class ReplayCache:
    """Per-slot exact-replay / ReplaySSM state: fp32 checkpoint (anchor), optional read copy,
    token-major partial-chunk buffers of (x, raw dt, B, C) and the per-slot position.

    read_dtype "bf16": read_copy [S,H,P,N] bf16.  read_dtype "fp8": read_copy [S,H,P,N] uint8 holding
    e4m3 codes and read_scale [S,H,P] fp32, one scale per state row (value = code * scale).
    read_dtype "nvfp4": read_copy [S,H,P,N/2] uint8 holding two e2m1 codes per byte (value n in the
    low nibble of byte n/2 when n is even), read_block_scale [S,H,P,N/16] e4m3 bytes (one per 16
    values) and read_scale [S,H,P] fp32 (value = code * block scale * row scale).

    anchor "fp32": state [S,H,P,N] fp32.  anchor "fp16_sr" (ReplaySSM only): state [S,H,P,N] fp16,
    written by stochastic rounding with random words keyed by sr_key and the attribute sr_nonce,
    which the caller sets to a fresh value before every call that may refresh anchors.  anchor
    "nvfp4_sr_shared" (ReplaySSM only, with an NVFP4 read copy): the read copy is the only state
    (state is None), rewritten at refresh with stochastically rounded codes; seed() casts an fp32
    state into it.

    paged=(page_rows, npages): the partial-chunk buffers are [npages, page_rows, ...] and
    buf_pages [S, chunk / page_rows] int32 maps each slot's logical pages to physical ones
    (initially slot s owns pages s * chunk / page_rows onward when npages allows, else page 0)."""

    def __init__(self, nslots: int, nheads: int, ngroups: int, headdim: int, dstate: int, chunk: int,
                 io_dtype: torch.dtype = torch.bfloat16, read_copy: bool = False, device="cuda",
                 read_dtype: str = "bf16", anchor: str = "fp32", sr_key: Tuple[int, int] = (0, 0),
                 paged: Optional[Tuple[int, int]] = None):
        if read_dtype not in ("bf16", "fp8", "nvfp4"):
            raise ValueError(f"read_dtype must be 'bf16', 'fp8' or 'nvfp4', got {read_dtype!r}")
        self.nslots, self.H, self.G, self.P, self.N, self.Q = nslots, nheads, ngroups, headdim, dstate, chunk
        if anchor not in ("fp32", "fp16_sr", "nvfp4_sr_shared"):
            raise ValueError(f"anchor must be 'fp32', 'fp16_sr' or 'nvfp4_sr_shared', got {anchor!r}")
        if anchor == "nvfp4_sr_shared" and not (read_copy and read_dtype == "nvfp4"):
            raise ValueError("anchor 'nvfp4_sr_shared' needs read_copy=True and read_dtype='nvfp4'")
        self.io = io_dtype
        self.read_dtype = read_dtype
        self.anchor = anchor
        self.sr_key = (int(sr_key[0]) & 0xFFFFFFFF, int(sr_key[1]) & 0xFFFFFFFF)
        self.sr_nonce = 0
        z = dict(device=device)
        shp = (nslots, nheads, headdim, dstate)
        self.state = None if anchor == "nvfp4_sr_shared" else \
            torch.zeros(*shp, dtype=torch.float16 if anchor == "fp16_sr" else torch.float32, **z)
        self.read_copy = None
        self.read_scale = None
        self.read_block_scale = None
        if read_copy:
            if read_dtype == "bf16":
                self.read_copy = torch.zeros(*shp, dtype=torch.bfloat16, **z)
            elif read_dtype == "fp8":
                self.read_copy = torch.zeros(*shp, dtype=torch.uint8, **z)
            else:
                if dstate % 16:
                    raise ValueError("an NVFP4 read copy needs dstate divisible by 16")
                self.read_copy = torch.zeros(nslots, nheads, headdim, dstate // 2, dtype=torch.uint8, **z)
                self.read_block_scale = torch.zeros(nslots, nheads, headdim, dstate // 16, dtype=torch.uint8, **z)
            if read_dtype != "bf16":
                self.read_scale = torch.zeros(nslots, nheads, headdim, dtype=torch.float32, **z)
        self.buf_pages = None
        self.page_rows = 0
        self.npages = 0
        lead = (nslots, chunk)
        if paged is not None:
            pr, npg = int(paged[0]), int(paged[1])
            if pr < 1 or chunk % pr or npg < 1:
                raise ValueError("paged=(page_rows, npages) needs page_rows dividing chunk and npages >= 1")
            self.page_rows, self.npages = pr, npg
            ppl = chunk // pr
            ids = torch.arange(nslots * ppl, dtype=torch.int32)
            self.buf_pages = torch.where(ids < npg, ids, torch.zeros_like(ids)).view(nslots, ppl).to(device)
            lead = (npg, pr)
        self.buf_x = torch.zeros(*lead, nheads, headdim, dtype=io_dtype, **z)
        self.buf_dt = torch.zeros(*lead, nheads, dtype=torch.float32, **z)
        self.buf_B = torch.zeros(*lead, ngroups, dstate, dtype=io_dtype, **z)
        self.buf_C = torch.zeros(*lead, ngroups, dstate, dtype=io_dtype, **z)
        self.pos = torch.zeros(nslots, dtype=torch.int32, **z)

    @property
    def dims(self) -> _abi.Dims:
        return _dims(self.H, self.G, self.P, self.N, self.Q, self.io)

    def _c(self) -> _abi.Cache:
        anc = {"fp32": _abi.ANCHOR_F32, "fp16_sr": _abi.ANCHOR_F16_SR,
               "nvfp4_sr_shared": _abi.ANCHOR_NVFP4_SHARED_SR}[self.anchor]
        return self._c_with(_ptr(self.state), anc)

    def _c_with(self, state_ptr, anchor_code) -> _abi.Cache:
        rd = {"bf16": _abi.READ_BF16, "fp8": _abi.READ_FP8_E4M3, "nvfp4": _abi.READ_NVFP4}[self.read_dtype]
        return _abi.Cache(state_ptr, _ptr(self.read_copy), self.buf_x.data_ptr(), self.buf_dt.data_ptr(),
                          self.buf_B.data_ptr(), self.buf_C.data_ptr(), self.pos.data_ptr(), self.nslots, rd,
                          _ptr(self.read_scale), _ptr(self.read_block_scale), anchor_code,
                          (ctypes.c_uint32 * 2)(*self.sr_key), int(self.sr_nonce) & 0xFFFFFFFF,
                          _ptr(self.buf_pages), self.page_rows, self.npages)

    def seed(self, state: torch.Tensor, params: "LayerParams", nseq: Optional[int] = None,
             slot: Optional[torch.Tensor] = None, stream=None) -> None:
        """Casts an fp32 state [nslots,H,P,N] into the shared NVFP4 state of the listed slots (all by
        default), rounding to nearest: the cast an fp32-anchor ReplaySSM refresh with an empty history
        writes into its NVFP4 copy (ers_refresh with that state and anchor code ERS_ANCHOR_F32).  The
        slots must have pos = 0."""
        if self.anchor != "nvfp4_sr_shared":
            raise ValueError("seed() is for the 'nvfp4_sr_shared' anchor")
        _need(state, torch.float32, "state", (self.nslots, self.H, self.P, self.N))
        S = self.nslots if nseq is None else nseq
        st = Status(self.pos.device)
        c = self._c_with(state.data_ptr(), _abi.ANCHOR_F32)
        code = _abi.lib().ers_refresh(ctypes.byref(self.dims), ctypes.byref(params._c()), ctypes.byref(c), S,
                                      _slot_arg(slot, S), _abi.FLAG_REPLAYSSM, self.Q + 1, _stream(stream),
                                      _ptr(st.t))
        _finish(code, "ers_refresh (seed)", st, True)

    def nbytes(self) -> int:
        ts = [self.buf_x, self.buf_dt, self.buf_B, self.buf_C, self.pos]
        ts += [t for t in (self.state, self.read_copy, self.read_scale, self.read_block_scale, self.buf_pages)
               if t is not None]
        return sum(t.numel() * t.element_size() for t in ts)


def _tok_checks(cache: ReplayCache, x, dt, B, C, lead: Tuple[int, ...]):
    _need(x, cache.io, "x", lead + (cache.H, cache.P)); _need(dt, torch.float32, "dt", lead + (cache.H,))
    _need(B, cache.io, "B", lead + (cache.G, cache.N)); _need(C, cache.io, "C", lead + (cache.G, cache.N))


def _slot_arg(slot: Optional[torch.Tensor], nseq: int):
    if slot is None:
        return None
    _need(slot, torch.int32, "slot", (nseq,))
    return slot.data_ptr()


def chunked_prefill(cache: ReplayCache, params: LayerParams, x, dt, B, C, cu_seqlens: Optional[torch.Tensor] = None,
                    slot: Optional[torch.Tensor] = None, max_seqlen: Optional[int] = None,
                    status: Optional[Status] = None, check: bool = True, stream=None,
                    workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Boundary-anchored (chunked) prefill into the cache (ers_chunked_prefill); returns y of the new tokens."""
    T = x.shape[0]
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=x.device)
    S = cu_seqlens.numel() - 1
    _tok_checks(cache, x, dt, B, C, (T,))
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    ms = _max_len(cu_seqlens, max_seqlen)
    y = torch.empty_like(x)
    L = _abi.lib()
    dims = cache.dims
    wsz = L.ers_chunked_prefill_workspace_size(ctypes.byref(dims), S, ms)
    if workspace is None or workspace.numel() < wsz:
        workspace = torch.empty(max(wsz, 1), dtype=torch.uint8, device=x.device)
    st = status if status is not None else (Status(x.device) if check else None)
    code = L.ers_chunked_prefill(ctypes.byref(dims), ctypes.byref(params._c()), ctypes.byref(cache._c()), S, T, ms,
                                 cu_seqlens.data_ptr(), _slot_arg(slot, S), x.data_ptr(), dt.data_ptr(),
                                 B.data_ptr(), C.data_ptr(), y.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                 _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_chunked_prefill", st, check)
    return y


def replay_decode(cache: ReplayCache, params: LayerParams, x, dt, B, C, slot: Optional[torch.Tensor] = None,
                  fuse_refresh: bool = True, replayssm: bool = False, status: Optional[Status] = None,
                  check: bool = True, stream=None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One exact-replay decode step per sequence (ers_replay_decode).  x [S,H,P], dt [S,H], B/C [S,G,N].

    fuse_refresh: exact mode refreshes a slot whose chunk fills in the same call; ReplaySSM mode
    applies the one-token flush rule first (a slot at h = L is flushed, then decodes as record 0)."""
    S = x.shape[0]
    _tok_checks(cache, x, dt, B, C, (S,))
    y = torch.empty_like(x) if out is None else out
    flags = (_abi.FLAG_REPLAYSSM if replayssm else 0) | (_abi.FLAG_FUSE_REFRESH if fuse_refresh else 0)
    st = status if status is not None else (Status(x.device) if check else None)
    code = _abi.lib().ers_replay_decode(ctypes.byref(cache.dims), ctypes.byref(params._c()), ctypes.byref(cache._c()),
                                        S, _slot_arg(slot, S), x.data_ptr(), dt.data_ptr(), B.data_ptr(),
                                        C.data_ptr(), flags, y.data_ptr(), _stream(stream),
                                        _ptr(st.t) if st else None)
    _finish(code, "ers_replay_decode", st, check)
    return y


def refresh(cache: ReplayCache, params: LayerParams, nseq: Optional[int] = None, slot: Optional[torch.Tensor] = None,
            replayssm: bool = False, drafts_T: int = 0, status: Optional[Status] = None, check: bool = True,
            stream=None) -> None:
    """Checkpoint refresh (ers_refresh): exact mode folds full chunks; ReplaySSM mode applies h + T > L."""
    S = cache.nslots if nseq is None else nseq
    st = status if status is not None else (Status(cache.pos.device) if check else None)
    code = _abi.lib().ers_refresh(ctypes.byref(cache.dims), ctypes.byref(params._c()), ctypes.byref(cache._c()), S,
                                  _slot_arg(slot, S), _abi.FLAG_REPLAYSSM if replayssm else 0, int(drafts_T),
                                  _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_refresh", st, check)


def spec_verify(cache: ReplayCache, params: LayerParams, x, dt, B, C, slot: Optional[torch.Tensor] = None,
                auto_flush: bool = True, status: Optional[Status] = None, check: bool = True, stream=None,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Output-only speculative verify of T drafts per sequence (ers_spec_verify).  x [S,T,H,P] ..."""
    S, T = x.shape[0], x.shape[1]
    _tok_checks(cache, x, dt, B, C, (S, T))
    y = torch.empty_like(x) if out is None else out
    st = status if status is not None else (Status(x.device) if check else None)
    code = _abi.lib().ers_spec_verify(ctypes.byref(cache.dims), ctypes.byref(params._c()), ctypes.byref(cache._c()),
                                      S, _slot_arg(slot, S), T, x.data_ptr(), dt.data_ptr(), B.data_ptr(),
                                      C.data_ptr(), _abi.FLAG_AUTO_FLUSH if auto_flush else 0, y.data_ptr(),
                                      _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_spec_verify", st, check)
    return y


def commit(cache: ReplayCache, accepted: torch.Tensor, T: int, slot: Optional[torch.Tensor] = None,
           auto_flush: bool = True, status: Optional[Status] = None, check: bool = True, stream=None) -> None:
    """Advance the committed pointer by the accepted draft count (ers_commit)."""
    S = accepted.numel()
    _need(accepted, torch.int32, "accepted", (S,))
    st = status if status is not None else (Status(accepted.device) if check else None)
    code = _abi.lib().ers_commit(ctypes.byref(cache.dims), ctypes.byref(cache._c()), S, _slot_arg(slot, S),
                                 accepted.data_ptr(), int(T), _abi.FLAG_AUTO_FLUSH if auto_flush else 0,
                                 _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_commit", st, check)


def _exact_ws(cache: ReplayCache, S: int, workspace: Optional[torch.Tensor], device) -> torch.Tensor:
    need = _abi.lib().ers_spec_verify_exact_workspace_size(ctypes.byref(cache.dims), S)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    return workspace


def spec_verify_exact(cache: ReplayCache, params: LayerParams, x, dt, B, C, slot: Optional[torch.Tensor] = None,
                      status: Optional[Status] = None, check: bool = True, stream=None,
                      out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Exact-mode speculative verify of T drafts per sequence that keeps the chunk grid
    (ers_spec_verify_exact): x [S,T,H,P], dt [S,T,H], B/C [S,T,G,N] -> y [S,T,H,P]; the cache is
    not changed."""
    S, T = x.shape[0], x.shape[1]
    _tok_checks(cache, x, dt, B, C, (S, T))
    y = torch.empty_like(x) if out is None else out
    ws = _exact_ws(cache, S, workspace, x.device)
    st = status if status is not None else (Status(x.device) if check else None)
    code = _abi.lib().ers_spec_verify_exact(ctypes.byref(cache.dims), ctypes.byref(params._c()),
                                            ctypes.byref(cache._c()), S, _slot_arg(slot, S), T, x.data_ptr(),
                                            dt.data_ptr(), B.data_ptr(), C.data_ptr(), y.data_ptr(), ws.data_ptr(),
                                            ws.numel(), _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_spec_verify_exact", st, check)
    return y


def commit_exact(cache: ReplayCache, params: LayerParams, accepted: torch.Tensor, x, dt, B, C,
                 slot: Optional[torch.Tensor] = None, status: Optional[Status] = None, check: bool = True,
                 stream=None, workspace: Optional[torch.Tensor] = None) -> None:
    """Commit the accepted drafts of an exact-mode verify (ers_commit_exact): the same x, dt, B, C."""
    S, T = x.shape[0], x.shape[1]
    _tok_checks(cache, x, dt, B, C, (S, T))
    _need(accepted, torch.int32, "accepted", (S,))
    ws = workspace if workspace is not None else torch.empty(max(256, 4 * S), dtype=torch.uint8, device=x.device)
    st = status if status is not None else (Status(x.device) if check else None)
    code = _abi.lib().ers_commit_exact(ctypes.byref(cache.dims), ctypes.byref(params._c()), ctypes.byref(cache._c()),
                                       S, _slot_arg(slot, S), accepted.data_ptr(), T, x.data_ptr(), dt.data_ptr(),
                                       B.data_ptr(), C.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream),
                                       _ptr(st.t) if st else None)
    _finish(code, "ers_commit_exact", st, check)


def ssu_update(state: torch.Tensor, params: LayerParams, x, dt, B, C, slot: Optional[torch.Tensor] = None,
               status: Optional[Status] = None, check: bool = True, stream=None,
               out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Per-token state-writeback update (ers_ssu_update); state [nslots,H,P,N] fp32 updated in place."""
    io = _io_from(x)
    S, H, P = x.shape
    G, N = B.shape[1], B.shape[2]
    nslots = state.shape[0]
    _need(state, torch.float32, "state", (nslots, H, P, N))
    _need(x, io, "x", (S, H, P)); _need(dt, torch.float32, "dt", (S, H))
    _need(B, io, "B", (S, G, N)); _need(C, io, "C", (S, G, N))
    y = torch.empty_like(x) if out is None else out
    dims = _dims(H, G, P, N, 1, io)
    st = status if status is not None else (Status(x.device) if check else None)
    code = _abi.lib().ers_ssu_update(ctypes.byref(dims), ctypes.byref(params._c()), state.data_ptr(), nslots, S,
                                     _slot_arg(slot, S), x.data_ptr(), dt.data_ptr(), B.data_ptr(), C.data_ptr(),
                                     y.data_ptr(), _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_ssu_update", st, check)
    return y


# ------------------------------------------------------------------------------------------------
def _conv_dims(C: int, W: int, io: torch.dtype, activation: bool) -> _abi.ConvDims:
    if io not in _IO:
        raise TypeError(f"io dtype {io} not supported (bf16 or fp32)")
    return _abi.ConvDims(C, W, _IO[io], _abi.CONV_SILU if activation else 0)


def _conv_params(weight: torch.Tensor, bias: Optional[torch.Tensor], io: torch.dtype):
    C, W = weight.shape
    _need(weight, io, "weight", (C, W))
    if bias is not None:
        _need(bias, io, "bias", (C,))
    return C, W


def conv1d_fwd(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor] = None,
               cu_seqlens: Optional[torch.Tensor] = None, conv_state: Optional[torch.Tensor] = None,
               slot: Optional[torch.Tensor] = None, read_state: bool = False, activation: bool = True,
               max_seqlen: Optional[int] = None, status: Optional[Status] = None, check: bool = True,
               stream=None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Causal depthwise conv1d over packed sequences (ers_conv1d_fwd).  x [T, C], weight [C, W],
    bias [C]; conv_state [nslots, W-1, C] (oldest input first) is read when read_state and, when
    given, receives each sequence's final state."""
    io = _io_from(x)
    T = x.shape[0]
    C, W = _conv_params(weight, bias, io)
    _need(x, io, "x", (T, C))
    if cu_seqlens is None:
        cu_seqlens = torch.tensor([0, T], dtype=torch.int32, device=x.device)
    _need(cu_seqlens, torch.int32, "cu_seqlens")
    S = cu_seqlens.numel() - 1
    nslots = 0
    if conv_state is not None:
        nslots = conv_state.shape[0]
        _need(conv_state, io, "conv_state", (nslots, W - 1, C))
    y = torch.empty_like(x) if out is None else out
    st = status if status is not None else (Status(x.device) if check else None)
    code = _abi.lib().ers_conv1d_fwd(ctypes.byref(_conv_dims(C, W, io, activation)), S, T,
                                     _max_len(cu_seqlens, max_seqlen), cu_seqlens.data_ptr(), x.data_ptr(),
                                     weight.data_ptr(), _ptr(bias), _ptr(conv_state), nslots, _slot_arg(slot, S),
                                     int(bool(read_state)), y.data_ptr(), _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_conv1d_fwd", st, check)
    return y


def conv1d_update(x: torch.Tensor, weight: torch.Tensor, bias: Optional[torch.Tensor], conv_state: torch.Tensor,
                  slot: Optional[torch.Tensor] = None, activation: bool = True, status: Optional[Status] = None,
                  check: bool = True, stream=None, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One conv1d step per sequence (ers_conv1d_update): x [S, C]; conv_state [nslots, W-1, C] is
    shifted by one and receives x."""
    io = _io_from(x)
    S = x.shape[0]
    C, W = _conv_params(weight, bias, io)
    _need(x, io, "x", (S, C))
    nslots = conv_state.shape[0]
    _need(conv_state, io, "conv_state", (nslots, W - 1, C))
    y = torch.empty_like(x) if out is None else out
    st = status if status is not None else (Status(x.device) if check else None)
    code = _abi.lib().ers_conv1d_update(ctypes.byref(_conv_dims(C, W, io, activation)), S, x.data_ptr(),
                                        weight.data_ptr(), _ptr(bias), conv_state.data_ptr(), nslots,
                                        _slot_arg(slot, S), y.data_ptr(), _stream(stream),
                                        _ptr(st.t) if st else None)
    _finish(code, "ers_conv1d_update", st, check)
    return y


# ------------------------------------------------------------------------------------------------
class GdnCache:
    """Per-slot ReplaySSM state of a gated-delta-rule layer: fp32 anchor [S,H,dv,dk], bf16 read copy,
    the committed records since the last refresh (k [S,L,G,dk], v [S,L,H,dv] in the io dtype; g, beta
    [S,L,H] and residuals u [S,L,H,dv] in fp32) and the committed count pos [S]."""

    def __init__(self, nslots: int, nheads: int, ngroups: int, dk: int = 128, dv: int = 128, window: int = 16,
                 io_dtype: torch.dtype = torch.bfloat16, device="cuda"):
        self.nslots, self.H, self.G, self.dk, self.dv, self.L = nslots, nheads, ngroups, dk, dv, window
        self.io = io_dtype
        z = dict(device=device)
        self.anchor = torch.zeros(nslots, nheads, dv, dk, dtype=torch.float32, **z)
        self.read_copy = torch.zeros(nslots, nheads, dv, dk, dtype=torch.bfloat16, **z)
        self.buf_k = torch.zeros(nslots, window, ngroups, dk, dtype=io_dtype, **z)
        self.buf_v = torch.zeros(nslots, window, nheads, dv, dtype=io_dtype, **z)
        self.buf_g = torch.zeros(nslots, window, nheads, dtype=torch.float32, **z)
        self.buf_beta = torch.zeros(nslots, window, nheads, dtype=torch.float32, **z)
        self.buf_u = torch.zeros(nslots, window, nheads, dv, dtype=torch.float32, **z)
        self.pos = torch.zeros(nslots, dtype=torch.int32, **z)

    @property
    def dims(self) -> _abi.GdnDims:
        if self.io not in _IO:
            raise TypeError(f"io dtype {self.io} not supported (bf16 or fp32)")
        return _abi.GdnDims(self.H, self.G, self.dk, self.dv, self.L, _IO[self.io])

    def _c(self) -> _abi.GdnCache:
        return _abi.GdnCache(self.anchor.data_ptr(), self.read_copy.data_ptr(), self.buf_k.data_ptr(),
                             self.buf_v.data_ptr(), self.buf_g.data_ptr(), self.buf_beta.data_ptr(),
                             self.buf_u.data_ptr(), self.pos.data_ptr(), self.nslots)


def gdn_verify(cache: GdnCache, q, k, v, g, beta, slot: Optional[torch.Tensor] = None, auto_flush: bool = True,
               status: Optional[Status] = None, check: bool = True, stream=None,
               out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Output-only verify of T drafts per sequence for a GDN layer (ers_gdn_verify).  q, k [S,T,G,dk],
    v [S,T,H,dv], g, beta [S,T,H]; returns o [S,T,H,dv]."""
    S, T = q.shape[0], q.shape[1]
    _need(q, cache.io, "q", (S, T, cache.G, cache.dk)); _need(k, cache.io, "k", (S, T, cache.G, cache.dk))
    _need(v, cache.io, "v", (S, T, cache.H, cache.dv))
    _need(g, torch.float32, "g", (S, T, cache.H)); _need(beta, torch.float32, "beta", (S, T, cache.H))
    o = torch.empty_like(v) if out is None else out
    st = status if status is not None else (Status(q.device) if check else None)
    code = _abi.lib().ers_gdn_verify(ctypes.byref(cache.dims), ctypes.byref(cache._c()), S, _slot_arg(slot, S), T,
                                     q.data_ptr(), k.data_ptr(), v.data_ptr(), g.data_ptr(), beta.data_ptr(),
                                     _abi.FLAG_AUTO_FLUSH if auto_flush else 0, o.data_ptr(), _stream(stream),
                                     _ptr(st.t) if st else None)
    _finish(code, "ers_gdn_verify", st, check)
    return o


def gdn_commit(cache: GdnCache, accepted: torch.Tensor, T: int, slot: Optional[torch.Tensor] = None,
               auto_flush: bool = True, status: Optional[Status] = None, check: bool = True, stream=None) -> None:
    """Advance the committed count by the accepted drafts (ers_gdn_commit)."""
    S = accepted.numel()
    _need(accepted, torch.int32, "accepted", (S,))
    st = status if status is not None else (Status(accepted.device) if check else None)
    code = _abi.lib().ers_gdn_commit(ctypes.byref(cache.dims), ctypes.byref(cache._c()), S, _slot_arg(slot, S),
                                     accepted.data_ptr(), int(T), _abi.FLAG_AUTO_FLUSH if auto_flush else 0,
                                     _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_gdn_commit", st, check)


def gdn_refresh(cache: GdnCache, drafts_T: int, nseq: Optional[int] = None, slot: Optional[torch.Tensor] = None,
                status: Optional[Status] = None, check: bool = True, stream=None) -> None:
    """Fold the committed records of slots with h + drafts_T > L into their anchors (ers_gdn_refresh)."""
    S = cache.nslots if nseq is None else nseq
    st = status if status is not None else (Status(cache.anchor.device) if check else None)
    code = _abi.lib().ers_gdn_refresh(ctypes.byref(cache.dims), ctypes.byref(cache._c()), S, _slot_arg(slot, S),
                                      int(drafts_T), _stream(stream), _ptr(st.t) if st else None)
    _finish(code, "ers_gdn_refresh", st, check)
