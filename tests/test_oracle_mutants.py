"""The oracle pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, a wrong index, a transposed operand), builds it on the CPU
and runs the pin suite against it; the suite must fail for every mutant.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ref_attn.c")
PIN_FILES = [os.path.join(ROOT, "tests", f)
             for f in ("test_oracle_pins.py", "test_oracle_window_pins.py", "test_oracle_blocks_pins.py",
                       "test_oracle_decode_pins.py", "test_oracle_fp8_pins.py")]

MUTANTS = {
    "scores_without_tau": ("p[j] = tau * dot(q, K + j * d, d);", "p[j] = dot(q, K + j * d, d);"),
    "causal_mask_reversed": ("if (vs->causal && j > i + vs->offset) return 0;",
                             "if (vs->causal && j < i + vs->offset) return 0;"),
    "causal_mask_strict": ("if (vs->causal && j > i + vs->offset) return 0;",
                           "if (vs->causal && j >= i + vs->offset && i > 0) return 0;"),
    "decode_offset_sign": ("if (vs->causal && j > i + vs->offset) return 0;",
                           "if (vs->causal && j > i - vs->offset) return 0;"),
    "decode_offset_ignored": ("if (vs->causal && j > i + vs->offset) return 0;",
                              "if (vs->causal && j > i) return 0;"),
    "window_off_by_one": ("if (vs->window > 0 && j <= i - vs->window) return 0;",
                          "if (vs->window > 0 && j < i - vs->window) return 0;"),
    "window_ignored": ("if (vs->window > 0 && j <= i - vs->window) return 0;",
                       "if (vs->window > 0 && j <= i - 2 * vs->window) return 0;"),
    "blocks_transposed": ("(i / vs->blk) * vs->nkb + j / vs->blk]", "(j / vs->blk) * vs->nkb + i / vs->blk]"),
    "blocks_ignored": ("if (vs->blocks && !vs->blocks[", "if (0 && !vs->blocks["),
    "blocks_one_head": ("vs->blocks[bh * vs->head_stride + ", "vs->blocks[0 * vs->head_stride + "),
    "blocks_edge_off_by_one": ("(i / vs->blk) * vs->nkb + j / vs->blk]", "((i + 1) / vs->blk) * vs->nkb + j / vs->blk]"),
    "empty_row_not_guarded": ("    if (seen == 0) {", "    if (seen < 0) {"),
    "e4m3_bias_off_by_one": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal_scale": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_mantissa_width": ("ldexp(1.0 + (double)m / 8.0,", "ldexp(1.0 + (double)m / 16.0,"),
    "lse_without_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "no_normalisation": ("for (int64_t j = 0; j < N; ++j) p[j] /= l;", ""),
    "output_wrong_value_row": ("const double* v = V + j * d;", "const double* v = V + (N - 1 - j) * d;"),
    "dq_without_tau": ("for (int64_t k = 0; k < d; ++k) g[k] *= tau;", ""),
    "dq_uses_queries": ("g[k] += w * Kh[j * d + k];", "g[k] += w * Qh[j * d + k];"),
    "dk_uses_keys": ("gk[k] += ws * Qh[i * d + k];", "gk[k] += ws * Kh[i * d + k];"),
    "dk_transposed_ds": ("double ws = dS[i * N + j], wp = P[i * N + j];",
                         "double ws = dS[j * N + i], wp = P[i * N + j];"),
    "dv_transposed_p": ("double ws = dS[i * N + j], wp = P[i * N + j];",
                        "double ws = dS[i * N + j], wp = P[j * N + i];"),
    "ds_sign_flipped": ("dSi[j] = Pi[j] * (dSi[j] - Di);", "dSi[j] = Pi[j] * (dSi[j] + Di);"),
    "ds_drops_D": ("dSi[j] = Pi[j] * (dSi[j] - Di);", "dSi[j] = Pi[j] * dSi[j];"),
    "dp_uses_values_of_query": ("dot(dOh + i * d, Vh + j * d, d)", "dot(dOh + i * d, Vh + i * d, d)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor not found: {old}"
    mutated = src.replace(old, new, 1)
    cfile = tmp_path / "ref_attn_mutant.c"
    cfile.write_text(mutated)
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-o", str(lib), str(cfile), "-lm"])
    env = dict(os.environ, FA_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] + PIN_FILES,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"


def test_unmutated_copy_passes(tmp_path):
    lib = tmp_path / "libcopy.so"
    shutil.copy(SRC, tmp_path / "ref_attn_copy.c")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-o", str(lib), str(tmp_path / "ref_attn_copy.c"), "-lm"])
    env = dict(os.environ, FA_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] + PIN_FILES,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
