"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutant is compiled from a modified copy of ``oracle/attn_ref.c`` in a
temporary directory, on the CPU, and the pin suite ``tests/test_oracle.py``
must fail (or crash) against it.  The committed oracle is never modified.
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
    "K read in place of V": ("const uint16_t *vrow = kv_row(vw, b, t0 + i, g);",
                             "const uint16_t *vrow = kv_row(kw, b, t0 + i, g);"),
    "ln Z dropped from LSE": ("*lse = mx + log(z);", "*lse = mx;"),
    "merge weight not normalised": ("const double w = exp(lse_parts[i] - g);",
                                    "const double w = exp(lse_parts[i] - lse_max);"),
    "online correction inverted": ("exp(m - m_new);", "exp(m_new - m);"),
    "query row indexed by kv head": ("const uint16_t *qrow = q + ((int64_t)b * hq + h) * d;",
                                     "const uint16_t *qrow = q + ((int64_t)b * hq + g) * d;"),
    "last token dropped": ("const int n = t1 - t0;", "const int n = t1 - t0 - (t1 - t0 > 1);"),
    "fp16 exponent bias off by one": ("v = ldexp((double)(m + 1024), e - 25);", "v = ldexp((double)(m + 1024), e - 24);"),
    "fp16 subnormals flushed": ("v = ldexp((double)m, -24);", "v = 0.0;"),
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
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle.py", "-q", "-x",
                        "-p", "no:cacheprovider"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0, f"mutant '{name}' passed every pin:\n{r.stdout[-2000:]}"
