"""Causal depthwise conv1d with a conv state on the GPU (exact-replay RFC, §2 Evidence item 6: the
conv's prefill and decode-update paths agree bit for bit; bf16 operands promoted to fp32).  Parity
with the oracle; token-by-token updates and state-carrying chunked prefill equal a single-shot
prefill bit for bit; varlen, short sequences, widths 2-4, bf16 and fp32, slot indirection."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import MAX_REL_BF16, OUT_TOL_BF16, OUT_TOL_F32, check_out, dev, same_bits

pytestmark = pytest.mark.gpu


def _ers():
    import exact_replay_decode_gb300 as ers
    return ers


def _inputs(seed, T, C, W, S_state, io):
    rng = np.random.Generator(np.random.PCG64(seed))
    cast = (lambda a: torch.from_numpy(a.astype(np.float32)).to(io).to(dev()))   # rounded on the host
    x = cast(rng.standard_normal((T, C)))
    w = cast(rng.standard_normal((C, W)) * 0.5)
    b = cast(rng.standard_normal(C) * 0.1)
    st = cast(rng.standard_normal((S_state, W - 1, C)))
    return x, w, b, st


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
def test_conv1d_prefill_matches_oracle(W, io):
    ers = _ers()
    lens = [100, 1, 3, 257, 64, 0, 130]
    C = 520                                           # two channel blocks, the second partial
    T = sum(lens)
    x, w, b, st = _inputs(W * 10 + (io == torch.float32), T, C, W, len(lens), io)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev())
    for read_state in (False, True):
        state = st.clone()
        y = ers.conv1d_fwd(x, w, b, cu, conv_state=state, read_state=read_state)
        y_o, fin_o = oracle.causal_conv1d(_np(x), _np(w), _np(b), cu.cpu().numpy(),
                                          init_state=_np(st) if read_state else None)
        tol = OUT_TOL_BF16 if io == torch.bfloat16 else OUT_TOL_F32
        mr = MAX_REL_BF16 if io == torch.bfloat16 else 1e-4
        check_out(y, y_o, tol, keep=(), cu=cu.cpu().numpy(), max_rel=mr, what="conv1d prefill")   # per sequence
        assert np.array_equal(_np(state), fin_o)       # final states are copies of inputs
    y_lin = ers.conv1d_fwd(x, w, None, cu, activation=False)
    y_o, _ = oracle.causal_conv1d(_np(x), _np(w), None, cu.cpu().numpy(), activation=False)
    check_out(y_lin, y_o, OUT_TOL_BF16 if io == torch.bfloat16 else OUT_TOL_F32, keep=(), cu=cu.cpu().numpy(),
              max_rel=MAX_REL_BF16 if io == torch.bfloat16 else 1e-4, what="conv1d, no activation")


@pytest.mark.parametrize("io", [torch.bfloat16, torch.float32])
def test_conv1d_update_and_chunked_prefill_equal_single_shot(io):
    ers = _ers()
    S, n, C, W = 6, 40, 6144, 4
    x, w, b, st = _inputs(7, S * n, C, W, S, io)
    cu = torch.arange(0, S * n + 1, n, dtype=torch.int32, device=dev())
    ref_state = st.clone()
    y_ss = ers.conv1d_fwd(x, w, b, cu, conv_state=ref_state, read_state=True)
    # token-by-token updates from the same initial states
    state = st.clone()
    xs = x.view(S, n, C)
    ys = torch.stack([ers.conv1d_update(xs[:, t].contiguous(), w, b, state) for t in range(n)], dim=1)
    assert same_bits(ys.reshape(S * n, C), y_ss) and same_bits(state, ref_state)
    # chunked prefill: splits at 1, 17 and the rest, carrying the state
    state = st.clone()
    parts = []
    for a, z in ((0, 1), (1, 18), (18, n)):
        xc = xs[:, a:z].reshape(S * (z - a), C).contiguous()
        cuc = torch.arange(0, S * (z - a) + 1, z - a, dtype=torch.int32, device=dev())
        parts.append(ers.conv1d_fwd(xc, w, b, cuc, conv_state=state, read_state=True).view(S, z - a, C))
    assert same_bits(torch.cat(parts, dim=1).reshape(S * n, C), y_ss) and same_bits(state, ref_state)


def test_conv1d_decode_workload_and_slots():
    """256 sequences x 6144 channels (x, B and C of the decode workload), width 4, slot indirection;
    sampled rows against the oracle; a slot out of range is reported."""
    ers = _ers()
    S, C, W, nslots = 256, 6144, 4, 300
    x, w, b, st = _inputs(8, S, C, W, nslots, torch.bfloat16)
    slot = torch.from_numpy(np.random.Generator(np.random.PCG64(9)).permutation(nslots)[:S].astype(np.int32)).to(dev())
    state = st.clone()
    y = ers.conv1d_update(x, w, b, state, slot=slot)
    sl = slot.long().cpu().numpy()
    for i in (0, 1, 100, 255):
        y_o, fin_o = oracle.causal_conv1d(_np(x[i:i + 1]), _np(w), _np(b), init_state=_np(st[sl[i]])[None])
        check_out(y[i:i + 1], y_o, OUT_TOL_BF16, keep=(), what=f"conv1d update row {i}")
        assert np.array_equal(_np(state[sl[i]]), fin_o[0])
    untouched = np.setdiff1d(np.arange(nslots), sl)
    assert same_bits(state[torch.from_numpy(untouched).to(dev())], st[torch.from_numpy(untouched).to(dev())])
    bad = slot.clone()
    bad[3] = nslots
    stat = ers.Status(dev())
    ers.conv1d_update(x, w, b, state.clone(), slot=bad, status=stat, check=False)
    assert stat.read() == 8                                 # ERS_ESLOT
