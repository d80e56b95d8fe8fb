"""The parity metric of the GPU tests (tests/gpu_helpers.py) on planted mistakes, on the CPU: a
wrong row or a wrong short sequence that the whole-tensor mean would absorb is caught per
(sequence, head), and a single wrong element is caught by the element bound."""
import numpy as np
import pytest

from gpu_helpers import MAX_REL_BF16, check_out, unit_errs

import synth


def _bf16_like(rng, shape):
    ref = rng.standard_normal(shape)
    return ref, synth.round_bf16(ref.astype(np.float32)).astype(np.float64)   # output rounding only


def test_bf16_rounding_alone_passes_every_unit():
    rng = np.random.Generator(np.random.PCG64(1))
    ref, got = _bf16_like(rng, (3339, 8, 64))
    cu = np.array([0, 2048, 2825, 3338, 3339])
    check_out(got, ref, 2e-3, keep=1, cu=cu)
    m, x = unit_errs(got, ref, 1, cu)
    assert m.shape == (4 * 8,) and m.max() < 2e-3 and x.max() <= 2.0 ** -8   # half an ulp of the top binade


def test_one_token_sequence_wrong_is_caught_per_unit_not_by_the_whole():
    rng = np.random.Generator(np.random.PCG64(2))
    ref, got = _bf16_like(rng, (3339, 8, 64))
    cu = np.array([0, 2048, 2825, 3338, 3339])
    got[3338, 5] = -got[3338, 5]                       # the one-token sequence, one head: sign flipped
    whole = np.abs(got - ref).mean() / np.abs(ref).mean()
    assert whole < 2e-3                                # the whole-tensor metric misses it
    with pytest.raises(AssertionError, match="unit"):
        check_out(got, ref, 2e-3, keep=1, cu=cu)


def test_single_wrong_element_is_caught_by_the_element_bound():
    rng = np.random.Generator(np.random.PCG64(3))
    ref, got = _bf16_like(rng, (64, 16, 8, 64))       # [S, K, H, P]
    got[10, 2, 3, 7] += 0.05 * np.abs(ref[10, :, 3]).max()
    m, _ = unit_errs(got, ref, (0, 2))
    assert m.max() < 2e-3                              # the per-unit mean misses a single element
    with pytest.raises(AssertionError, match="max"):
        check_out(got, ref, 2e-3, keep=(0, 2), max_rel=MAX_REL_BF16)


def test_units_follow_the_kept_axes():
    rng = np.random.Generator(np.random.PCG64(4))
    ref, got = _bf16_like(rng, (5, 7, 3, 16))
    got[4, :, 1] *= 1.01                                # sequence 4, head 1 over every draft
    m, _ = unit_errs(got, ref, (0, 2))
    assert m.shape == (15,) and int(np.argmax(m)) == 4 * 3 + 1
