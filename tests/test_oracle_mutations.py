"""The oracle's pins must catch plausible mistakes (no GPU).

Each case copies oracle/mfa_oracle.c into a temporary package, plants one
mistake (a dropped term, a wrong sign, a wrong index, a swapped operand, a
wrong constant), rebuilds it and runs tests/test_oracle.py against the mutant.
The run must fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "scale_dropped": ("s[j] = scale * dot;", "s[j] = dot;"),
    "max_instead_min": ("if (s[j] > m) m = s[j];", "if (s[j] < m) m = s[j];"),
    "lse_without_max": ("*lse_out = m + log(z);", "*lse_out = log(z);"),
    "not_normalised": ("out_row[i] /= z;", "out_row[i] /= 1.0;"),
    "page_row_reversed": ("slot[j] = (int64_t)page * page_size + j % page_size;",
                          "slot[j] = (int64_t)page * page_size + (page_size - 1 - j % page_size);"),
    "k_used_as_v": ("out_row[i] += p * cache_value(v_cache, v_scale",
                    "out_row[i] += p * cache_value(k_cache, k_scale"),
    "head_index_dropped": ("const uint16_t* qrow = q + ((int64_t)b * H + h) * D;",
                           "const uint16_t* qrow = q + ((int64_t)b * H + 0) * D;"),
    "e4m3_bias": ("mag = ldexp(1.0 + (double)m / 8.0, e - 7);",
                  "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    "e4m3_truncates": ("double r = nearbyint(a / quantum);", "double r = floor(a / quantum);"),
    "quant_wrong_max": ("float s = (amax > 0.0f) ? amax / 448.0f : 1.0f;",
                        "float s = (amax > 0.0f) ? amax / 240.0f : 1.0f;"),
    "append_no_increment": ("seq_lens[b] = (int32_t)(start + n_new);",
                            "seq_lens[b] = (int32_t)(start);"),
    "e2m1_nibble_order": ("oracle_e2m1_to_f64((i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15))",
                          "oracle_e2m1_to_f64((i & 1) ? (uint8_t)(byte & 15) : (uint8_t)(byte >> 4))"),
    "e2m1_bias": ("ldexp(1.0 + 0.5 * m, e - 1);", "ldexp(1.0 + 0.5 * m, e - 2);"),
    "e2m1_quant_wrong_max": ("? amax / 6.0f : 1.0f;", "? amax / 4.0f : 1.0f;"),
    "e2m1_ties_to_odd": ("(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)"),
}


def _run_pins(tmp_path, source):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "mfa_oracle.c").write_text(source)
    shutil.copy(os.path.join(ROOT, "oracle", "__init__.py"), pkg / "__init__.py")
    env = dict(os.environ, PYTHONPATH=f"{tmp_path}{os.pathsep}{ROOT}",
               MFA_ORACLE_EXPECT_DIR=str(pkg))
    return subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         os.path.join(ROOT, "tests", "test_oracle.py"), os.path.join(ROOT, "tests", "test_oracle_fp4.py")],
        env=env, cwd=str(tmp_path), capture_output=True, text=True, timeout=600)


def test_unmutated_copy_passes(tmp_path):
    """Control: the harness itself runs the pins green on an unchanged copy."""
    r = _run_pins(tmp_path, open(os.path.join(ROOT, "oracle", "mfa_oracle.c")).read())
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    src = open(os.path.join(ROOT, "oracle", "mfa_oracle.c")).read()
    before, after = MUTANTS[name]
    assert src.count(before) == 1, "mutation anchor not found in the oracle source"
    r = _run_pins(tmp_path, src.replace(before, after))
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
