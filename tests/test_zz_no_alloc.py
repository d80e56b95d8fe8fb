"""ers_ssd_scan_fwd_static: the chunked scan with the library's fixed device scratch instead of a
caller workspace.  Two calls in a row must match the workspace entry point (ers_ssd_scan_fwd) on the
same inputs within the parity tolerance (they run the same kernels, so in fact bit for bit), and a
call that needs more scratch than the fixed array must be rejected before any launch.  This file
is collected last so that it also runs after every other GPU test in the same process."""
import numpy as np
import pytest
import torch

import synth
from synth import torch_io
from gpu_helpers import OUT_TOL_BF16, OUT_TOL_F32, STATE_TOL, dev, layer, out_err, same_bits, state_err

pytestmark = pytest.mark.gpu


def _inputs(name, seed):
    w = synth.workload(name)
    params, toks, cu = synth.prefill_inputs(w, seed=seed)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    return w, layer(params), (x, dt, B, C), torch.from_numpy(cu).to(dev())


@pytest.mark.parametrize("name", ["prefill_2048_h32", "tiny_fp32"])
def test_static_scratch_scan_matches_workspace_scan_twice(name):
    import exact_replay_decode_gb300 as ers
    cases = [_inputs(name, seed) for seed in (0, 1)]
    # two calls in a row through the static scratch; the second reuses the scratch of the first
    got = [ers.ssd_scan_fwd_static(x, dt, prm, B, C, chunk=w.dims.chunk, cu_seqlens=cu)
           for w, prm, (x, dt, B, C), cu in cases]
    for (w, prm, (x, dt, B, C), cu), (y, fin) in zip(cases, got):
        y_ref, fin_ref = ers.ssd_scan_fwd(x, dt, prm, B, C, chunk=w.dims.chunk, cu_seqlens=cu)
        torch.cuda.synchronize()
        tol = OUT_TOL_BF16 if x.dtype == torch.bfloat16 else OUT_TOL_F32
        assert out_err(y, y_ref.float().cpu().numpy().astype(np.float64)) <= tol
        assert state_err(fin, fin_ref.cpu().numpy().astype(np.float64)) <= STATE_TOL
        assert same_bits(y, y_ref) and same_bits(fin, fin_ref)


def test_static_scratch_rejects_calls_beyond_its_size():
    import exact_replay_decode_gb300 as ers
    from exact_replay_decode_gb300 import _abi
    w, prm, (x, dt, B, C), cu = _inputs("varlen_4seq_h64", 0)   # needs 128 MiB of chunk-state scratch
    y = torch.full_like(x, 7.0)
    with pytest.raises(ers.ErsError) as e:
        ers.ssd_scan_fwd_static(x, dt, prm, B, C, chunk=w.dims.chunk, cu_seqlens=cu, out=(y, torch.empty(
            4, w.dims.nheads, w.dims.headdim, w.dims.dstate, device=dev())))
    assert e.value.code == 10   # ERS_EWORKSPACE
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())                                # nothing was launched
    assert np.isclose(ers.STATIC_SCRATCH_BYTES, 32 << 20)
    assert _abi.STATUS_NAMES[10] == "ERS_EWORKSPACE"
