"""C-ABI library checks that need no GPU: it builds, loads, exports every function include/ers.h
declares, and rejects invalid calls during host validation (before any launch)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from exact_replay_decode_gb300 import build, _abi
    build.build()
    return _abi.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "ers.h")).read()
    return sorted(set(re.findall(r"^ERS_API [^(]*?\b(ers_\w+)\(", src, flags=re.M)))


def test_header_declares_expected_entry_points():
    names = _declared()
    for n in ("ers_ssd_scan_fwd", "ers_chunked_prefill", "ers_replay_decode", "ers_refresh", "ers_spec_verify",
              "ers_commit", "ers_ssu_update"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from exact_replay_decode_gb300 import _abi
    for n in _declared():
        assert hasattr(lib, n), n
    assert set(_declared()) == set(_abi.EXPORTS)


def test_status_strings(lib):
    from exact_replay_decode_gb300 import _abi
    for code in _abi.STATUS_NAMES:
        assert _abi.status_str(code)
    assert _abi.status_str(0) == "ok"
    assert lib.ers_version() >= 100


# Host-validation cases.  Each one fails a check that runs before any CUDA call, so no pointer is
# ever dereferenced; they are skipped on machines with a GPU so that a validation regression can
# never turn into a launch on fake pointers.
needs_no_gpu = pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host-only validation test")

FAKE = 1 << 20          # 16-byte aligned dummy address, never dereferenced
MISALIGNED = FAKE + 4


def _dims(**kw):
    from exact_replay_decode_gb300 import _abi
    d = dict(nheads=8, ngroups=2, headdim=64, dstate=128, chunk=16, io_dtype=_abi.DTYPE_BF16)
    d.update(kw)
    return _abi.Dims(**d)


def _prm(a=FAKE):
    from exact_replay_decode_gb300 import _abi
    return _abi.Params(a, FAKE, FAKE)


def _scan(lib, dims, prm, workspace=FAKE, wbytes=1 << 40, cu=FAKE):
    return lib.ers_ssd_scan_fwd(ctypes.byref(dims), ctypes.byref(prm), 1, 32, 32, cu, FAKE, FAKE, FAKE, FAKE,
                                None, FAKE, FAKE, None, workspace, wbytes, None, None)


@needs_no_gpu
def test_validation_rejects_bad_dims(lib):
    from exact_replay_decode_gb300 import _abi
    assert _scan(lib, _dims(io_dtype=7), _prm()) == 3                   # ERS_EDTYPE
    assert _scan(lib, _dims(ngroups=3), _prm()) == 2                    # nheads % ngroups
    assert _scan(lib, _dims(chunk=0), _prm()) == 2
    assert _scan(lib, _dims(chunk=257), _prm()) == 2
    assert _scan(lib, _dims(headdim=48), _prm()) == 2
    assert _scan(lib, _dims(dstate=96), _prm()) == 2


@needs_no_gpu
def test_validation_rejects_bad_pointers_and_workspace(lib):
    assert _scan(lib, _dims(), _prm(a=MISALIGNED)) == 4                 # ERS_EPTR
    assert _scan(lib, _dims(), _prm(a=0)) == 1                          # ERS_EINVAL (NULL)
    assert _scan(lib, _dims(), _prm(), cu=0) == 1
    assert _scan(lib, _dims(), _prm(), workspace=0) == 10               # ERS_EWORKSPACE
    assert _scan(lib, _dims(), _prm(), wbytes=16) == 10


@needs_no_gpu
def test_validation_rejects_bad_verify_and_commit_args(lib):
    from exact_replay_decode_gb300 import _abi
    d = _dims()
    c = _abi.Cache(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4)
    p = _prm()
    v = lambda T, flags=0: lib.ers_spec_verify(ctypes.byref(d), ctypes.byref(p), ctypes.byref(c), 4, None, T, FAKE,
                                               FAKE, FAKE, FAKE, flags, FAKE, None, None)
    assert v(0) == 1 and v(17) == 1 and v(4, flags=8) == 1
    nocopy = _abi.Cache(FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, 4)
    assert lib.ers_spec_verify(ctypes.byref(d), ctypes.byref(p), ctypes.byref(nocopy), 4, None, 4, FAKE, FAKE,
                               FAKE, FAKE, 0, FAKE, None, None) == 1    # read copy required
    assert lib.ers_commit(ctypes.byref(d), ctypes.byref(c), 4, None, FAKE, 0, 0, None, None) == 1
    assert lib.ers_commit(ctypes.byref(d), ctypes.byref(c), 5, None, FAKE, 4, 0, None, None) == 1  # nseq > nslots
    dec = lambda flags: lib.ers_replay_decode(ctypes.byref(d), ctypes.byref(p), ctypes.byref(c), 4, None, FAKE, FAKE,
                                              FAKE, FAKE, flags, FAKE, None, None)
    assert dec(64) == 1


@needs_no_gpu
def test_zero_sequences_is_a_noop(lib):
    d, p = _dims(), _prm()
    assert lib.ers_ssd_scan_fwd(ctypes.byref(d), ctypes.byref(p), 0, 0, 0, None, None, None, None, None, None,
                                None, None, None, None, 0, None, None) == 0


@needs_no_gpu
def test_empty_batches_are_noops_at_every_entry_point(lib):
    """Zero sequences: every per-sequence call checks its descriptors, returns ERS_OK and launches
    nothing (so the per-call pointers may be NULL); a negative count is ERS_EINVAL."""
    from exact_replay_decode_gb300 import _abi
    d, p = _dims(), _prm()
    c = _abi.Cache()
    c.state = c.read_copy = c.buf_x = c.buf_dt = c.buf_B = c.buf_C = c.pos = FAKE
    c.nslots = 4
    D, P, C = ctypes.byref(d), ctypes.byref(p), ctypes.byref(c)
    for n, want in ((0, 0), (-1, 1)):
        assert lib.ers_chunked_prefill(D, P, C, n, 0, 0, None, None, None, None, None, None, None, None, 0, None,
                                       None) == want
        for flags in (0, _abi.FLAG_FUSE_REFRESH, _abi.FLAG_REPLAYSSM | _abi.FLAG_FUSE_REFRESH):
            assert lib.ers_replay_decode(D, P, C, n, None, None, None, None, None, flags, None, None, None) == want
        assert lib.ers_refresh(D, P, C, n, None, _abi.FLAG_REPLAYSSM, 4, None, None) == want
        assert lib.ers_spec_verify(D, P, C, n, None, 4, None, None, None, None, _abi.FLAG_AUTO_FLUSH, None, None,
                                   None) == want
        assert lib.ers_commit(D, C, n, None, None, 4, _abi.FLAG_AUTO_FLUSH, None, None) == want
        assert lib.ers_spec_verify_exact(D, P, C, n, None, 4, None, None, None, None, None, None, 0, None,
                                         None) == want
        assert lib.ers_commit_exact(D, P, C, n, None, None, 4, None, None, None, None, None, 0, None, None) == want
        gd = _abi.GdnDims(8, 4, 128, 128, 16, _abi.DTYPE_BF16)
        gc = _abi.GdnCache(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4)
        GD, GC = ctypes.byref(gd), ctypes.byref(gc)
        assert lib.ers_gdn_verify(GD, GC, n, None, 4, None, None, None, None, None, _abi.FLAG_AUTO_FLUSH, None, None,
                                  None) == want
        assert lib.ers_gdn_commit(GD, GC, n, None, None, 4, _abi.FLAG_AUTO_FLUSH, None, None) == want
        assert lib.ers_gdn_refresh(GD, GC, n, None, 4, None, None) == want
        cd = _abi.ConvDims(64, 4, _abi.DTYPE_BF16, 1)
        assert lib.ers_conv1d_fwd(ctypes.byref(cd), n, 0, 0, None, None, None, None, None, 0, None, 0, None, None,
                                  None) == want
        assert lib.ers_conv1d_update(ctypes.byref(cd), n, None, None, None, None, 0, None, None, None, None) == want
        assert lib.ers_ssd_scan_fwd_static(D, P, n, 0, 0, None, None, None, None, None, None, None, None, None, None,
                                           None) == want   # no scratch lookup for an empty batch
    assert lib.ers_ssd_scan_fwd(D, P, -1, 0, 0, None, None, None, None, None, None, None, None, None, None, 0, None,
                                None) == 1


@needs_no_gpu
def test_validation_of_fp8_read_copies(lib):
    """FP8 / NVFP4 read copies: the dtype code is checked, the scales are required and aligned, and
    shapes the warp-per-head kernels do not cover (and NVFP4 outside ReplaySSM mode) return
    ERS_EUNSUPPORTED before any launch."""
    from exact_replay_decode_gb300 import _abi
    p = _prm()

    def cache(read_dtype=_abi.READ_FP8_E4M3, scale=FAKE, bscale=FAKE):
        return _abi.Cache(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, read_dtype, scale, bscale)

    def dec(d, c, flags=_abi.FLAG_REPLAYSSM):
        return lib.ers_replay_decode(ctypes.byref(d), ctypes.byref(p), ctypes.byref(c), 4, None, FAKE, FAKE, FAKE,
                                     FAKE, flags, FAKE, None, None)

    def ver(d, c):
        return lib.ers_spec_verify(ctypes.byref(d), ctypes.byref(p), ctypes.byref(c), 4, None, 4, FAKE, FAKE, FAKE,
                                   FAKE, 0, FAKE, None, None)

    def ref(d, c, flags=_abi.FLAG_REPLAYSSM):
        return lib.ers_refresh(ctypes.byref(d), ctypes.byref(p), ctypes.byref(c), 4, None, flags, 1, None, None)

    assert dec(_dims(), cache(read_dtype=3)) == 3                            # ERS_EDTYPE
    assert dec(_dims(), cache(read_dtype=_abi.READ_NVFP4, bscale=0)) == 1   # NVFP4 needs block scales
    assert dec(_dims(), cache(read_dtype=_abi.READ_NVFP4), flags=0) == 12   # NVFP4: ReplaySSM mode only
    assert ref(_dims(), cache(read_dtype=_abi.READ_NVFP4), flags=0) == 12
    assert dec(_dims(), cache(scale=0)) == 1                                 # scales required
    assert dec(_dims(), cache(scale=MISALIGNED)) == 4
    for d in (_dims(chunk=32), _dims(headdim=32, dstate=32), _dims(dstate=64)):
        assert dec(d, cache()) == 12                                         # ERS_EUNSUPPORTED
        assert ref(d, cache()) == 12
    assert ver(_dims(nheads=32, ngroups=2), cache()) == 12                   # 16 heads per group
    assert ver(_dims(chunk=32), cache()) == 12


@needs_no_gpu
def test_validation_of_fp16_sr_anchors(lib):
    """fp16 stochastic-rounding anchors: the dtype code is checked; exact-mode calls, fp32 io, a
    missing read copy and chunked prefill return ERS_EUNSUPPORTED before any launch."""
    from exact_replay_decode_gb300 import _abi
    p = _prm()

    def cache(anchor=_abi.ANCHOR_F16_SR, copy=FAKE):
        return _abi.Cache(FAKE, copy, FAKE, FAKE, FAKE, FAKE, FAKE, 4, _abi.READ_BF16, None, None, anchor)

    def dec(d, c, flags=_abi.FLAG_REPLAYSSM):
        return lib.ers_replay_decode(ctypes.byref(d), ctypes.byref(p), ctypes.byref(c), 4, None, FAKE, FAKE, FAKE,
                                     FAKE, flags, FAKE, None, None)

    assert dec(_dims(), cache(anchor=3)) == 3                                  # ERS_EDTYPE
    assert dec(_dims(), cache(), flags=0) == 12                                # exact mode
    assert dec(_dims(io_dtype=_abi.DTYPE_F32), cache()) == 12                  # fp32 io
    assert dec(_dims(chunk=32), cache()) == 12                                 # outside the warp-per-head shapes
    assert lib.ers_refresh(ctypes.byref(_dims()), ctypes.byref(p), ctypes.byref(cache(copy=0)), 4, None,
                           _abi.FLAG_REPLAYSSM, 1, None, None) == 12            # no read copy
    assert lib.ers_chunked_prefill(ctypes.byref(_dims()), ctypes.byref(p), ctypes.byref(cache()), 1, 16, 16, FAKE,
                                   None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None, None) == 12


@needs_no_gpu
def test_validation_of_shared_nvfp4_state(lib):
    """The shared NVFP4 state (anchor code 2): state may be NULL; it needs an NVFP4 read copy, bf16 io,
    ReplaySSM mode and the warp-per-head shapes, else ERS_EUNSUPPORTED before any launch; a NULL state
    is still an error for the other anchors."""
    from exact_replay_decode_gb300 import _abi
    p = _prm()

    def cache(anchor=_abi.ANCHOR_NVFP4_SHARED_SR, read_dtype=_abi.READ_NVFP4, state=0):
        return _abi.Cache(state, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, read_dtype, FAKE, FAKE, anchor)

    def dec(d, c, flags=_abi.FLAG_REPLAYSSM):
        return lib.ers_replay_decode(ctypes.byref(d), ctypes.byref(p), ctypes.byref(c), 4, None, FAKE, FAKE, FAKE,
                                     FAKE, flags, FAKE, None, None)

    assert dec(_dims(), cache(), flags=0) == 12                                # exact mode: no fp32 state
    assert dec(_dims(), cache(read_dtype=_abi.READ_BF16)) == 12                # the state is an NVFP4 copy
    assert dec(_dims(), cache(read_dtype=_abi.READ_FP8_E4M3)) == 12
    assert dec(_dims(io_dtype=_abi.DTYPE_F32), cache()) == 12                  # bf16 io only
    assert dec(_dims(chunk=32), cache()) == 12
    assert dec(_dims(), cache(anchor=_abi.ANCHOR_F32)) == 1                    # NULL state elsewhere
    assert dec(_dims(), cache(anchor=_abi.ANCHOR_F16_SR)) == 1
    assert lib.ers_chunked_prefill(ctypes.byref(_dims()), ctypes.byref(p), ctypes.byref(cache()), 1, 16, 16, FAKE,
                                   None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 40, None, None) == 12


def test_shared_state_cache_needs_an_nvfp4_copy():
    import exact_replay_decode_gb300 as ers
    with pytest.raises(ValueError):
        ers.ReplayCache(2, 8, 2, 64, 128, 16, read_copy=True, read_dtype="bf16", anchor="nvfp4_sr_shared",
                        device="cpu")
    with pytest.raises(ValueError):
        ers.ReplayCache(2, 8, 2, 64, 128, 16, read_copy=False, read_dtype="nvfp4", anchor="nvfp4_sr_shared",
                        device="cpu")
    c = ers.ReplayCache(2, 8, 2, 64, 128, 16, read_copy=True, read_dtype="nvfp4", anchor="nvfp4_sr_shared",
                        device="cpu")
    assert c.state is None and c.read_copy.shape == (2, 8, 64, 64) and c.read_block_scale.shape == (2, 8, 64, 8)


@needs_no_gpu
def test_validation_of_conv1d(lib):
    from exact_replay_decode_gb300 import _abi

    def fwd(C=64, W=4, io=_abi.DTYPE_BF16, flags=1, state=FAKE, read_state=1, nslots=4):
        d = _abi.ConvDims(C, W, io, flags)
        return lib.ers_conv1d_fwd(ctypes.byref(d), 2, 8, 4, FAKE, FAKE, FAKE, None, state, nslots, None, read_state,
                                  FAKE, None, None)

    assert fwd(C=63) == 2 and fwd(C=66) == 2 and fwd(W=5) == 2 and fwd(W=1) == 2   # ERS_ESHAPE
    assert fwd(io=9) == 3 and fwd(flags=2) == 1
    assert fwd(state=0) == 1                                        # reading a state needs one
    assert fwd(nslots=1) == 1                                       # 2 sequences, 1 slot, no indirection
    d = _abi.ConvDims(64, 4, _abi.DTYPE_BF16, 1)
    assert lib.ers_conv1d_update(ctypes.byref(d), 2, FAKE, FAKE, None, 0, 4, None, FAKE, None, None) == 1
    assert lib.ers_conv1d_update(ctypes.byref(d), 2, FAKE, MISALIGNED, None, FAKE, 4, None, FAKE, None, None) == 4
    assert lib.ers_conv1d_update(ctypes.byref(d), 0, None, None, None, None, 0, None, None, None, None) == 0


@needs_no_gpu
def test_validation_of_paged_buffers(lib):
    from exact_replay_decode_gb300 import _abi
    p = _prm()

    def dec(page_rows, npages, pages=FAKE, chunk=16):
        d = _dims(chunk=chunk)
        c = _abi.Cache(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, _abi.READ_BF16, None, None, 0, (0, 0), 0, pages,
                       page_rows, npages)
        return lib.ers_replay_decode(ctypes.byref(d), ctypes.byref(p), ctypes.byref(c), 4, None, FAKE, FAKE, FAKE,
                                     FAKE, _abi.FLAG_FUSE_REFRESH, FAKE, None, None)

    assert dec(0, 8) == 1 and dec(4, 0) == 1                       # page geometry
    assert dec(5, 8) == 2                                          # page_rows must divide the chunk
    assert dec(4, 8, pages=MISALIGNED) == 4


@needs_no_gpu
def test_validation_of_gdn_calls(lib):
    from exact_replay_decode_gb300 import _abi

    def ver(dk=128, L=16, T=4, io=_abi.DTYPE_BF16, H=8, G=4, flags=4):
        d = _abi.GdnDims(H, G, dk, 128, L, io)
        c = _abi.GdnCache(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4)
        return lib.ers_gdn_verify(ctypes.byref(d), ctypes.byref(c), 4, None, T, FAKE, FAKE, FAKE, FAKE, FAKE, flags,
                                  FAKE, None, None)

    assert ver(dk=64) == 2 and ver(L=33) == 2 and ver(T=9) == 2 and ver(H=6, G=4) == 2   # ERS_ESHAPE
    assert ver(io=5) == 3 and ver(T=0) == 1 and ver(L=2, T=3) == 1 and ver(flags=1) == 1


def test_bounded_wait_selftest_validation(lib):
    # host validation only: NULL status, zero and over-long limits are rejected before any launch
    assert lib.ers_selftest_bounded_wait(1000, None, None) == 1
    assert lib.ers_selftest_bounded_wait(0, None, ctypes.c_void_p(16)) == 1
    assert lib.ers_selftest_bounded_wait(20_000_000_000, None, ctypes.c_void_p(16)) == 1


def test_exact_speculation_validation(lib):
    from exact_replay_decode_gb300 import _abi
    d = _abi.Dims(8, 2, 64, 128, 16, _abi.DTYPE_BF16)
    assert lib.ers_spec_verify_exact_workspace_size(ctypes.byref(d), 4) > 4 * 8 * 64 * 128 * 4
    p16 = ctypes.c_void_p(16)
    prm = _abi.Params(p16, p16, p16)
    cache = _abi.Cache()
    cache.state = cache.buf_x = cache.buf_B = cache.buf_C = cache.buf_dt = cache.pos = 16
    cache.nslots = 4
    args = (4, None, 4, p16, p16, p16, p16)
    # T outside [1, Q], a missing workspace, a workspace too small: rejected before any launch
    assert lib.ers_spec_verify_exact(ctypes.byref(d), ctypes.byref(prm), ctypes.byref(cache), 4, None, 0, p16, p16,
                                     p16, p16, p16, p16, 1 << 30, None, None) == 1
    assert lib.ers_spec_verify_exact(ctypes.byref(d), ctypes.byref(prm), ctypes.byref(cache), *args, p16, None, 0,
                                     None, None) == 10
    assert lib.ers_spec_verify_exact(ctypes.byref(d), ctypes.byref(prm), ctypes.byref(cache), *args, p16, p16, 256,
                                     None, None) == 10
    assert lib.ers_commit_exact(ctypes.byref(d), ctypes.byref(prm), ctypes.byref(cache), 4, None, p16, 4, p16, p16,
                                p16, p16, p16, 8, None, None) == 10
    cache.anchor_dtype = 1   # fp16 anchors: exact mode keeps an fp32 checkpoint
    assert lib.ers_spec_verify_exact(ctypes.byref(d), ctypes.byref(prm), ctypes.byref(cache), *args, p16, p16,
                                     1 << 30, None, None) == 12


def test_missing_library_fails_loudly_and_the_package_has_no_fallback(monkeypatch):
    """Without the built library the binding raises instead of computing anything; no module of the
    package imports the oracle (the only CPU implementation of the method in the repository)."""
    from exact_replay_decode_gb300 import _abi
    monkeypatch.setattr(_abi, "LIB_PATH", os.path.join(ROOT, "_no_such_dir", "libers.so"))
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="is missing"):
        _abi.lib()
    pkg = os.path.join(ROOT, "exact_replay_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, flags=re.M), f
