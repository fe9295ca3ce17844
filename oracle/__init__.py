"""CPU oracle for single-query decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product library never
loads it, and it shares no code with the CUDA path: the arithmetic lives in
``attn_ref.c`` (plain fp64 C), this file only marshals arrays.

Functions (each cites its passage in ``attn_ref.c``):

* :func:`attend` -- O and natural-log LSE by the full-softmax definition,
  contiguous or paged, optionally for a sample of (b, h) query rows or for a
  token range (a split's partial result).
* :func:`lse_merge` -- the LSE merge of split partials.
* :func:`online_blocks` -- the online-softmax recurrence, block by block.

Every function is pinned by ``tests/test_oracle.py`` to closed forms, the
pages' worked example and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_D = ctypes.c_double


def build(force: bool = False) -> str:
    """Compile attn_ref.c into liboracle.so next to it (plain gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared",
                               "-fno-fast-math", "-ffp-contract=off",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.oracle_attend.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _D, _I,
                                          _I, _D, _D, _I, _P, _I, _P, _P, _P]
            lib.oracle_attend.restype = _I
            lib.oracle_lse_merge.argtypes = [_P, _P, _I, _I, _P, _P]
            lib.oracle_lse_merge.restype = None
            lib.oracle_online_blocks.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P, _P]
            lib.oracle_online_blocks.restype = _I
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


_KV_CODES = {"bf16": 0, "f16": 1, "e4m3": 2, "e5m2": 3}


def attend_raw(q, k, v, seq_lens, num_q_heads, num_kv_heads, scale, *,
               page_size=0, block_table=None, items=None, threads=1, dtype="bf16",
               kv_dtype=None, k_scale=1.0, v_scale=1.0):
    """Oracle attention on raw arrays.

    q: uint16 bf16 (or fp16, dtype='f16') bits [B, Hq, D], or [B, q_len, Hq, D] for several
    new query tokens per request (new token i sees tokens 0 .. L - q_len + i);
    k, v: [B, S_max, Hkv, D] (contiguous)
    or [num_pages, P, Hkv, D] (paged, with block_table int32 [B, max_blocks]), uint16 bits of
    q's type, or (kv_dtype 'e4m3' / 'e5m2') uint8 FP8 codes dequantised by k_scale / v_scale.
    items: int32 [n, 4] rows (b, r, t0, t1) with query row r = i * Hq + h, t1 < 0
    meaning "to the row's causal end" (L_b when q_len = 1); default is every
    row over its whole visible length.  Returns (o [n, D], lse [n]) in fp64;
    with items=None they are reshaped like q ([B, Hq, D] / [B, q_len, Hq, D])
    and [B, Hq] / [B, q_len, Hq].
    """
    lib = _load()
    kv_dtype = kv_dtype or dtype
    kvcode = _KV_CODES[kv_dtype]
    kv_np = np.uint8 if kvcode >= 2 else np.uint16
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=kv_np)
    v = np.ascontiguousarray(v, dtype=kv_np)
    lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    if q.ndim == 4:
        B, q_len, hq, d = q.shape
    else:
        (B, hq, d), q_len = q.shape, 1
    if page_size:
        table = np.ascontiguousarray(block_table, dtype=np.int32)
        s_max, max_blocks, num_pages = 0, table.shape[1], k.shape[0]
        cap = max_blocks * page_size
    else:
        table, s_max, max_blocks, num_pages = None, k.shape[1], 0, 0
        cap = s_max
    full = items is None
    if full:
        bb, hh = np.meshgrid(np.arange(B), np.arange(q_len * hq), indexing="ij")
        items = np.stack([bb.ravel(), hh.ravel(), np.zeros(bb.size), -np.ones(bb.size)], 1)
    items = np.ascontiguousarray(items, dtype=np.int32).reshape(-1, 4)
    n = items.shape[0]
    o = np.zeros((n, d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    maxlen = int(lens.max()) if lens.size else 0
    maxlen = max(1, min(maxlen, cap) if cap else maxlen)

    def run(lo, hi):
        scratch = np.empty(maxlen, dtype=np.float64)
        rc = lib.oracle_attend(_ptr(q), _ptr(k), _ptr(v), _ptr(lens), B, hq, num_kv_heads, d,
                               s_max, page_size, _ptr(table), max_blocks, num_pages,
                               float(scale), 1 if dtype == "f16" else 0, kvcode, float(k_scale),
                               float(v_scale), q_len, _ptr(items[lo:hi]), hi - lo,
                               _ptr(scratch),
                               _ptr(o[lo:hi]), _ptr(lse[lo:hi]))
        if rc != 0:
            raise ValueError("oracle_attend: invalid arguments (bad page, head or length)")

    threads = max(1, int(threads))
    if threads == 1 or n < 2:
        run(0, n)
    else:
        bounds = np.linspace(0, n, min(n, 4 * threads) + 1).astype(int)
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(lambda i: run(bounds[i], bounds[i + 1]), range(len(bounds) - 1)))
    if full:
        if q.ndim == 4:
            return o.reshape(B, q_len, hq, d), lse.reshape(B, q_len, hq)
        return o.reshape(B, hq, d), lse.reshape(B, hq)
    return o, lse


def attend(w, items=None, threads=1):
    """Oracle attention for a workload object (see ``fd_synth.Workload``)."""
    return attend_raw(w.q, w.k, w.v, w.seq_lens, w.num_q_heads, w.num_kv_heads, w.scale,
                      page_size=w.page_size, block_table=w.block_table, items=items,
                      threads=threads, dtype=getattr(w, "dtype", "bf16"),
                      kv_dtype=getattr(w, "kv_dtype", None), k_scale=getattr(w, "k_scale", 1.0),
                      v_scale=getattr(w, "v_scale", 1.0))


def lse_merge(o_parts, lse_parts):
    """Merge normalised partials o_parts [n, d] with natural-log lse_parts [n]."""
    lib = _load()
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, d = o_parts.shape
    o = np.zeros(d, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    lib.oracle_lse_merge(_ptr(o_parts), _ptr(lse_parts), n, d, _ptr(o), _ptr(lse))
    return o, float(lse[0])


def online_blocks(scores, values, block):
    """Online softmax of one score row, `block` scores at a time.

    values: [n] or [n, dv] (dv <= 64).  Returns (m [nb], l [nb], O [nb, dv],
    final [dv]) where O is the unnormalised running output after each block.
    """
    lib = _load()
    s = np.ascontiguousarray(scores, dtype=np.float64)
    val = np.asarray(values, dtype=np.float64)
    if val.ndim == 1:
        val = val[:, None]
    val = np.ascontiguousarray(val)
    n, dv = val.shape
    nb_max = (n + block - 1) // block
    m = np.zeros(nb_max)
    l = np.zeros(nb_max)
    O = np.zeros((nb_max, dv))
    fin = np.zeros(dv)
    nb = lib.oracle_online_blocks(_ptr(s), _ptr(val), n, dv, block, _ptr(m), _ptr(l), _ptr(O),
                                  _ptr(fin))
    if nb < 0:
        raise ValueError("online_blocks: dv > 64 or block <= 0")
    return m[:nb], l[:nb], O[:nb], fin
