"""Build libfd.so (the CUDA library behind include/fd.h) in-tree for sm_103a.

Usage: ``python -m decode_attention_decoding_gb300.build`` or call :func:`build`.
Each translation unit is compiled by its own nvcc process, in parallel, then
linked into ``decode_attention_decoding_gb300/libfd.so``.  ``fd_split_inst.cu``
is compiled once per split-kernel variant (layout x K/V element type x head_dim),
each with its own defines.  Objects go to ``decode_attention_decoding_gb300/_build/``.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfd.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


SPLIT_INST = "fd_split_inst.cu"
KV_NAMES = ("bf16", "f16", "e4m3", "e5m2")
SPLIT_VARIANTS = [(paged, kv, d) for paged in (0, 1) for kv in range(4) for d in (64, 128, 256)]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _units():
    """(source, object name, extra defines) for every translation unit."""
    units = []
    for src in _sources():
        stem = os.path.basename(src)[:-3]
        if os.path.basename(src) == SPLIT_INST:
            for paged, kv, d in SPLIT_VARIANTS:
                defs = [f"-DFD_INST_PAGED={'true' if paged else 'false'}", f"-DFD_INST_KV={kv}",
                        f"-DFD_INST_D={d}"]
                units.append((src, f"{stem}_{'paged' if paged else 'contig'}_{KV_NAMES[kv]}_d{d}", defs))
        else:
            units.append((src, stem, []))
    return units


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link libfd.so if any source changed; returns its path."""
    if not force and up_to_date():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    flags = NVCC_FLAGS + list(extra_flags) + (["-Xptxas", "-v"] if verbose else [])

    def compile_one(unit):
        src, stem, defs = unit
        obj = os.path.join(BUILD, stem + ".o")
        cmd = [nvcc] + flags + defs + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, _units()))
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
