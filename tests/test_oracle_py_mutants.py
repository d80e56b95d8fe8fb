"""The pins must reject a broken oracle: the Python-side definitions (gated delta rule, its protocol
model, stochastic rounding onto the e2m1 grid, the fp16 stochastic rounding, the bf16, e4m3 and e2m1
roundings and the FP8 / NVFP4 row scales, the causal conv1d and SiLU, the Philox generator and the counter layout of the random words, and the ReplaySSM protocol model's
outputs, commit and recast).

Each case plants one plausible mistake in a scratch copy of oracle/__init__.py (never in the
committed file), lays out a scratch tree with that copy, the committed synth package and the pin
suite, and runs the pins there in a subprocess (against the committed, already built C recurrence).
Every mutant must fail at least one pin.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "__init__.py")

MUTANTS = {
    "gdn_delta_sign": ("u = beta[t][:, None] * (v[t] - a * Sk)", "u = beta[t][:, None] * (v[t] + a * Sk)"),
    "gdn_missing_beta": ("u = beta[t][:, None] * (v[t] - a * Sk)", "u = v[t] - a * Sk"),
    "gdn_state_not_decayed": ("S = a[:, :, None] * S + u[:, :, None] * kt[:, None, :]",
                              "S = S + u[:, :, None] * kt[:, None, :]"),
    "gdn_output_before_update": (
        "        S = a[:, :, None] * S + u[:, :, None] * kt[:, None, :]\n"
        "        out[t] = np.einsum(\"hdn,hn->hd\", S, qt)",
        "        out[t] = np.einsum(\"hdn,hn->hd\", S, qt)\n"
        "        S = a[:, :, None] * S + u[:, :, None] * kt[:, None, :]"),
    "gdn_key_for_query": ("out[t] = np.einsum(\"hdn,hn->hd\", S, qt)", "out[t] = np.einsum(\"hdn,hn->hd\", S, kt)"),
    "gdn_group_index_mod": ("hg = np.arange(H) // (H // G)", "hg = np.arange(H) % G"),
    "gdn_flush_one_early": ("if len(self.committed[i]) + T > self.L and self.committed[i]:",
                            "if len(self.committed[i]) + T >= self.L and self.committed[i]:"),
    "mamba_flush_one_early": ("flush = [i for i in range(S) if len(self.committed[i]) + T > self.L]",
                              "flush = [i for i in range(S) if len(self.committed[i]) + T >= self.L]"),
    "sr_e2m1_inclusive_threshold": (
        "frac = (a - lo) / step                                    # exact, in [0, 1)\n"
        "    up = np.asarray(r, dtype=np.float64) < np.ldexp(frac, 32)",
        "frac = (a - lo) / step                                    # exact, in [0, 1)\n"
        "    up = np.asarray(r, dtype=np.float64) <= np.ldexp(frac, 32)"),
    "sr_e2m1_step_of_one_below_two": ("step = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))",
                                      "step = np.where(a < 2.0, 1.0, np.where(a < 4.0, 1.0, 2.0))"),
    "sr_fp16_spacing_off_by_one": ("ue = np.maximum(e - 1, -14) - 10", "ue = np.maximum(e - 1, -14) - 11"),
    "bf16_truncates": ("r = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32)",
                       "r = ((u >> 16) << 16).astype(np.uint32)"),
    "bf16_ties_away_from_zero": ("r = (((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16).astype(np.uint32)",
                                 "r = (((u + 0x8000) >> 16) << 16).astype(np.uint32)"),
    "e4m3_subnormal_quantum": ("ex = np.maximum(e - 1, -6)", "ex = np.maximum(e - 1, -7)"),
    "e4m3_no_saturation": ("r = np.minimum(r, E4M3_MAX)", "r = np.minimum(r, 480.0)"),
    "fp8_scale_boundary": ("k = e.astype(np.int64) - 9 + (m > 0.875)", "k = e.astype(np.int64) - 9 + (m >= 0.875)"),
    "e2m1_subnormal_quantum": ("ex = np.maximum(e - 1, 0)", "ex = np.maximum(e - 1, -1)"),
    "nvfp4_scale_boundary": ("k = e.astype(np.int64) - 12 + (m > 0.65625)",
                             "k = e.astype(np.int64) - 12 + (m >= 0.65625)"),
    "conv_taps_reversed": ("acc = acc + w[:, k] * u[t + k]",
                          "acc = acc + w[:, W - 1 - k] * u[t + k]"),
    "conv_bias_dropped": ("            acc = b.copy()\n",
                         "            acc = np.zeros_like(b)\n"),
    "conv_state_not_prepended": ("pre = np.zeros((W - 1, C)) if init_state is None else _f64(init_state[i])",
                                "pre = np.zeros((W - 1, C))"),
    "conv_final_state_off_by_one": ("fin[i] = u[len(u) - (W - 1):]",
                                   "fin[i] = u[len(u) - W:len(u) - 1]"),
    "silu_sign": ("return a / (1.0 + np.exp(-a))",
                 "return a / (1.0 + np.exp(a))"),
    "philox_nine_rounds": ("    for rnd in range(10):\n        if rnd:\n            k0 = (k0 + np.uint64(PHILOX_W0)) & m32",
                          "    for rnd in range(9):\n        if rnd:\n            k0 = (k0 + np.uint64(PHILOX_W0)) & m32"),
    "philox_key_not_bumped": ("            k1 = (k1 + np.uint64(PHILOX_W1)) & m32\n",
                             "            k1 = k1\n"),
    "sr_words_nonce_and_slot_swapped": ("np.uint64(nonce & 0xFFFFFFFF), np.uint64(slot & 0xFFFFFFFF), hd, jj)",
                                       "np.uint64(slot & 0xFFFFFFFF), np.uint64(nonce & 0xFFFFFFFF), hd, jj)"),
    "sr_fp16_no_saturation": ("out = np.where(a >= FP16_MAX, FP16_MAX, out)",
                             "out = out"),
    "replayssm_outputs_from_anchor": (
        "y, _ = recurrence(x, dt, self.A, B, C, self.D, self.dt_bias, cu, self.read, self.nthreads)",
        "y, _ = recurrence(x, dt, self.A, B, C, self.D, self.dt_bias, cu, self.anchor, self.nthreads)"),
    "replayssm_commit_keeps_rejected": (
        "            for j in range(int(a)):\n                self.committed[i].append(tuple(self._pending[i][k][j] for k in range(4)))",
        "            for j in range(self._pending[i][0].shape[0]):\n                self.committed[i].append(tuple(self._pending[i][k][j] for k in range(4)))"),
    "replayssm_refresh_keeps_stale_copy": (
        "            self.read[i] = self.anchor[i] if self.shared else self.read_cast(fin[k])\n",
        "            self.read[i] = self.anchor[i] if self.shared else self.read[i]\n"),
    "gdn_outputs_from_anchor": (
        "o, _ = gdn_recurrence(*seq, self.read[i])",
        "o, _ = gdn_recurrence(*seq, self.anchor[i])"),
    "gdn_refresh_keeps_stale_copy": (
        "                self.read[i] = self.read_cast(fin)\n",
        ""),
    "gdn_commit_keeps_rejected": (
        "            for j in range(int(a)):\n                self.committed[i].append(tuple(self._pending[i][f][j] for f in range(5)))",
        "            for j in range(self._pending[i][0].shape[0]):\n                self.committed[i].append(tuple(self._pending[i][f][j] for f in range(5)))"),
    "gdn_outputs_of_committed_rows": (
        "outs.append(o[len(recs):])",
        "outs.append(o[:o.shape[0] - len(recs)])"),
    "replayssm_outputs_of_committed_rows": (
        "            out[i] = y[cu[i + 1] - T:cu[i + 1]]",
        "            out[i] = y[cu[i]:cu[i] + T]"),
    "replayssm_flush_on_h_plus_T_only_when_full": (
        "flush = [i for i in range(S) if len(self.committed[i]) + T > self.L]",
        "flush = [i for i in range(S) if len(self.committed[i]) >= self.L]"),
    "nvfp4_block_scale_over_four": (
        "beta = e4m3_round(t / np.float32(6.0))",
        "beta = e4m3_round(t / np.float32(4.0))"),
    "nvfp4_block_of_eight": (
        "fb = (f / s).reshape(f.shape[:-1] + (N // NVFP4_BLOCK, NVFP4_BLOCK))",
        "fb = (f / s).reshape(f.shape[:-1] + (N // 8, 8))"),
    "nvfp4_row_scale_not_applied": (
        "val = (q.astype(np.float64) * beta.astype(np.float64)).reshape(f.shape) * s",
        "val = (q.astype(np.float64) * beta.astype(np.float64)).reshape(f.shape)"),
    "replayssm_anchor_round_ignored": (
        "            self.anchor[i] = fin[k] if self.anchor_round is None else self.anchor_round(i, fin[k])\n",
        "            self.anchor[i] = fin[k]\n"),
    "replayssm_shared_copy_recast": (
        "            self.read[i] = self.anchor[i] if self.shared else self.read_cast(fin[k])\n",
        "            self.read[i] = self.read_cast(fin[k])\n"),
    "sr_e2m1_sign_dropped": (
        "    return np.copysign(out, f).astype(np.float32)\n",
        "    return out.astype(np.float32)\n"),
    "sr_e2m1_no_saturation": (
        "out = np.where(a >= E2M1_MAX, E2M1_MAX, lo + up * step)",
        "out = lo + up * step"),
    "sr_fp16_sign_dropped": (
        "    return np.copysign(out, f)\n",
        "    return out\n"),
    "fp8_rows_scale_not_applied": (
        "    q = e4m3_round(f / s).astype(np.float64)\n    return q * s\n",
        "    q = e4m3_round(f / s).astype(np.float64)\n    return q\n"),
    "sr_fp16_words_from_other_slot": (
        "return sr_fp16(np.asarray(fin, dtype=np.float64).astype(np.float32), sr_words(key, nonce, slot, H, P, N))",
        "return sr_fp16(np.asarray(fin, dtype=np.float64).astype(np.float32), sr_words(key, nonce, 0, H, P, N))"),
    "nvfp4_sr_words_from_other_slot": ("words=sr_words(key, nonce, slot, H, P, N))", "words=sr_words(key, nonce, 0, H, P, N))"),
    "conv_window_crosses_sequences": (
        "pre = np.zeros((W - 1, C)) if init_state is None else _f64(init_state[i])",
        "pre = (np.zeros((W - 1, C)) if cu[i] < W - 1 else x[cu[i] - (W - 1):cu[i]]) if init_state is None else _f64(init_state[i])"),
    "e4m3_sign_dropped": (
        "    return (np.sign(f) * r).astype(np.float32)\n\n\ndef fp8_row_scale_exponent",
        "    return r.astype(np.float32)\n\n\ndef fp8_row_scale_exponent"),
    "e2m1_sign_dropped": (
        "    return (np.sign(f) * r).astype(np.float32)\n\n\nNVFP4_BLOCK",
        "    return r.astype(np.float32)\n\n\nNVFP4_BLOCK"),
    "fp8_tiny_rows_not_floored": (
        "    return np.where(tiny, -127, np.maximum(k, -127))",
        "    return np.maximum(k, -127)"),
    "replayssm_verify_skips_flush": (
        "        flush = [i for i in range(S) if len(self.committed[i]) + T > self.L]\n        self.refresh(flush)\n",
        "        flush = [i for i in range(S) if len(self.committed[i]) + T > self.L]\n"),
}


def _oracle_lib():
    """The committed C oracle, built if it is missing or stale."""
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import oracle
    return oracle._LIB_OVERRIDE or oracle.build()


def _run_mutant(name, root, lib):
    """Runs the pin suite against the oracle with mutant `name` planted, in a scratch tree under root
    (lib: the built C oracle); returns (exit code, output)."""
    before, after = MUTANTS[name]
    src = open(SRC).read()
    if src.count(before) != 1:
        return None, "mutation site no longer present (once) in oracle/__init__.py"
    (root / "oracle").mkdir()
    (root / "oracle" / "__init__.py").write_text(src.replace(before, after))
    shutil.copy(os.path.join(ROOT, "oracle", "oracle.c"), root / "oracle" / "oracle.c")
    shutil.copytree(os.path.join(ROOT, "synth"), root / "synth", ignore=shutil.ignore_patterns("__pycache__"))
    (root / "tests").mkdir()
    for f in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), root / "tests" / f)
    golden = os.path.join(ROOT, "tests", "golden")
    if os.path.isdir(golden):
        shutil.copytree(golden, root / "tests" / "golden")
    env = dict(os.environ, ERS_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        str(root / "tests" / "test_oracle_pins.py")],
                       cwd=str(root), env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.fixture(scope="module")
def mutant_runs(tmp_path_factory):
    """Every mutant's pin run, run side by side (each is a separate process on a scratch tree)."""
    lib = _oracle_lib()
    assert os.path.exists(lib), "the C oracle is built on import"
    names = sorted(MUTANTS)
    roots = {n: tmp_path_factory.mktemp(n) for n in names}   # made here: the threads only run processes
    with ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        runs = ex.map(lambda n: _run_mutant(n, roots[n], lib), names)
        return dict(zip(names, runs))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_python_mutant(name, mutant_runs):
    code, out = mutant_runs[name]
    assert code is not None, out
    assert "passed" in out or "failed" in out, out
    assert code != 0, f"mutant {name} passed every pin:\n{out}"
