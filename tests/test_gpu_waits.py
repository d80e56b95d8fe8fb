"""Bounded device waits run out without hanging the GPU: the library's wait routines (an mbarrier
phase and a device flag, the two kinds of wait its kernels use) give up after their limit, report
ERS_ETIMEOUT through the status word, and leave the context usable."""
import time

import pytest
import torch

import synth
from synth import torch_io
from gpu_helpers import dev, layer, same_bits

pytestmark = pytest.mark.gpu


def test_bounded_waits_time_out_and_the_context_stays_usable():
    import exact_replay_decode_gb300 as ers
    w = synth.workload("prefill_2048_h32")
    params, toks, _ = synth.prefill_inputs(w, seed=9, seqlens=(300,))
    prm = layer(params)
    x, dt, B, C = torch_io.tokens_to(toks, dev())
    y0, f0 = ers.ssd_scan_fwd(x, dt, prm, B, C, chunk=256)
    st = ers.Status(dev())
    t0 = time.perf_counter()
    ers.selftest_bounded_wait(2_000_000, st)          # 2 ms: nothing ever completes either wait
    torch.cuda.synchronize()
    assert st.read() == 9                              # ERS_ETIMEOUT
    assert time.perf_counter() - t0 < 5.0
    y1, f1 = ers.ssd_scan_fwd(x, dt, prm, B, C, chunk=256)   # the context still runs the scan, same bits
    assert same_bits(y0, y1) and same_bits(f0, f1)
    with pytest.raises(ers.ErsError):
        ers.selftest_bounded_wait(0, st)               # a zero limit is rejected on the host
