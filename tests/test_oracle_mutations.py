"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutant is compiled from a modified copy of ``oracle/attn_ref.c`` in a
temporary directory, on the CPU, and the pin suites ``tests/test_oracle.py``,
``tests/test_oracle_fp8.py`` and ``tests/test_oracle_qlen.py`` must fail (or
crash) against it.  The committed oracle is never modified.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTANTS = {
    "kv head taken as h % G": ("const int g = h / group;", "const int g = h % group;"),
    "scale dropped": ("s[i] = scale * dot;", "s[i] = dot;"),
    "exponent sign flipped": ("s[i] = exp(s[i] - mx);", "s[i] = exp(mx - s[i]);"),
    "page slot and page index swapped": (
        "row = ((int64_t)phys * w->page + t % w->page) * w->hkv + g;",
        "row = ((int64_t)phys * w->page + t / w->page) * w->hkv + g;"),
    "K read in place of V": ("const uint8_t *vrow = kv_row(vw, b, t0 + i, g);",
                             "const uint8_t *vrow = kv_row(kw, b, t0 + i, g);"),
    "ln Z dropped from LSE": ("*lse = mx + log(z);", "*lse = mx;"),
    "merge weight not normalised": ("const double w = exp(lse_parts[i] - g);",
                                    "const double w = exp(lse_parts[i] - lse_max);"),
    "online correction inverted": ("exp(m - m_new);", "exp(m_new - m);"),
    "query row indexed by kv head": ("const uint16_t *qrow = q + (((int64_t)b * q_len + i_tok) * hq + h) * d;",
                                     "const uint16_t *qrow = q + (((int64_t)b * q_len + i_tok) * hq + g) * d;"),
    "causal end off by one": ("int end = L - q_len + i_tok + 1;", "int end = L - q_len + i_tok;"),
    "new tokens see the whole cache": ("int end = L - q_len + i_tok + 1;", "int end = L;"),
    "query rows of a request not strided by q_len": (
        "const uint16_t *qrow = q + (((int64_t)b * q_len + i_tok) * hq + h) * d;",
        "const uint16_t *qrow = q + (((int64_t)b + i_tok) * hq + h) * d;"),
    "token and head of a query row swapped": ("const int i_tok = r / hq, h = r % hq;",
                                              "const int i_tok = r % q_len, h = r / q_len;"),
    "last token dropped": ("const int n = t1 - t0;", "const int n = t1 - t0 - (t1 - t0 > 1);"),
    "fp16 exponent bias off by one": ("v = ldexp((double)(m + 1024), e - 25);", "v = ldexp((double)(m + 1024), e - 24);"),
    "fp16 subnormals flushed": ("v = ldexp((double)m, -24);", "v = 0.0;"),
    "e4m3 exponent bias off by one": ("v = ldexp((double)(m + 8), e - 10);",
                                      "v = ldexp((double)(m + 8), e - 9);"),
    "e4m3 subnormals flushed": ("v = ldexp((double)m, -9);", "v = 0.0;"),
    "e4m3 top exponent taken as NaN": ("else if (e == 15 && m == 7)", "else if (e == 15)"),
    "e5m2 decoded as e4m3": ("        return e5m2_to_f64(row[j]);", "        return e4m3_to_f64(row[j]);"),
    "e5m2 exponent bias off by one": ("v = ldexp((double)(m + 4), e - 17);",
                                      "v = ldexp((double)(m + 4), e - 16);"),
    "k_scale applied to V": ("o[j] += p * (v_scale * kv_elem(vrow, j, kvtype));",
                             "o[j] += p * (k_scale * kv_elem(vrow, j, kvtype));"),
    "k_scale dropped": ("(k_scale * kv_elem(krow, j, kvtype))", "(kv_elem(krow, j, kvtype))"),
    "FP8 row stride taken as 2 bytes": ("return w->base + row * w->d * w->esize;",
                                        "return w->base + row * w->d * 2;"),
}


@pytest.mark.parametrize("name", list(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(os.path.join(ROOT, "oracle", "attn_ref.c")).read()
    assert src.count(before) == 1, "mutation anchor not found"
    for sub in ("oracle", "tests", "fd_synth"):
        shutil.copytree(os.path.join(ROOT, sub), tmp_path / sub,
                        ignore=shutil.ignore_patterns("*.so", "__pycache__", "test_oracle_mutations.py"))
    (tmp_path / "oracle" / "attn_ref.c").write_text(src.replace(before, after))
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle.py",
                        "tests/test_oracle_fp8.py", "tests/test_oracle_qlen.py", "-q", "-x",
                        "-p", "no:cacheprovider"],
                       cwd=tmp_path, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant '{name}' passed every pin:\n{r.stdout[-2000:]}"
