"""Split-KV ("Flash-Decoding") single-query decode attention for GB300.

A thin ctypes binding over ``libfd.so`` (the C ABI of ``include/fd.h``).  The
functions carry the C names and only marshal arguments: every step of the
computation runs in the library's CUDA kernels.  PyTorch supplies device
memory and the current stream.  There is no CPU fallback: if the library is
missing, the first call raises ImportError.

Build the library first with ``python -m decode_attention_decoding_gb300.build``
(or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

__all__ = [
    "FdError", "fd_workspace_size", "fd_workspace_init", "fd_decode", "fd_decode_paged",
    "fd_get_device_error", "fd_status_string", "fd_version", "make_workspace", "library_path",
    "FD_OK", "FD_ERR_INVALID_ARG", "FD_ERR_UNSUPPORTED", "FD_ERR_WORKSPACE_TOO_SMALL",
    "FD_ERR_CUDA", "FD_ERR_TIMEOUT", "FD_ERR_DEVICE_INPUT", "FD_FLAG_TEST_STARVE_FIRST_TILE",
    "FD_FLAG_CUDA_CORES", "FD_FLAG_NO_4D_BOXES", "FD_FLAG_NO_HEAD_FUSION", "FD_FLAG_NO_GATHER",
    "FD_FLAG_FUSE_HEADS", "FD_FLAG_NO_PREFETCH", "FD_FLAG_TMEM_SCORES", "FD_FLAG_NO_TMEM_SCORES", "FD_KV_AS_Q", "FD_KV_FP8_E4M3", "FD_KV_FP8_E5M2",
    "fd_decode_noalloc", "fd_decode_partial", "fd_decode_paged_partial", "fd_merge_partials",
    "KV_END",
]

FD_OK, FD_ERR_INVALID_ARG, FD_ERR_UNSUPPORTED, FD_ERR_WORKSPACE_TOO_SMALL = 0, 1, 2, 3
FD_ERR_CUDA, FD_ERR_TIMEOUT, FD_ERR_DEVICE_INPUT = 4, 5, 6
FD_FLAG_TEST_STARVE_FIRST_TILE = 0x1
FD_FLAG_CUDA_CORES = 0x2
FD_FLAG_NO_4D_BOXES = 0x4
FD_FLAG_NO_HEAD_FUSION = 0x8
FD_FLAG_NO_GATHER = 0x20
FD_FLAG_FUSE_HEADS = 0x10
FD_FLAG_NO_PREFETCH = 0x40
FD_FLAG_TMEM_SCORES = 0x80
FD_FLAG_NO_TMEM_SCORES = 0x100
FD_KV_AS_Q, FD_KV_FP8_E4M3, FD_KV_FP8_E5M2 = 0, 1, 2
KV_END = 2 ** 31 - 1   # kv_end of a range that runs to the end of every request

_P, _I, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class FdOptions(ctypes.Structure):
    _fields_ = [("num_ctas", ctypes.c_int), ("flags", ctypes.c_uint),
                ("wait_timeout_ns", ctypes.c_ulonglong),
                ("split_start_event", ctypes.c_void_p), ("split_end_event", ctypes.c_void_p),
                ("dtype", ctypes.c_int), ("kv_dtype", ctypes.c_int), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("q_len", ctypes.c_int)]


def library_path() -> str:
    return _build.LIB


def _load():
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m decode_attention_decoding_gb300.build`")
    lib = ctypes.CDLL(path)
    lib.fd_workspace_size.argtypes = [_I, _I, _I, _I, _I, _I]
    lib.fd_workspace_size.restype = _SZ
    lib.fd_workspace_size_q.argtypes = [_I, _I, _I, _I, _I, _I, _I]
    lib.fd_workspace_size_q.restype = _SZ
    lib.fd_workspace_init.argtypes = [_P, _SZ, _P]
    lib.fd_workspace_init.restype = _I
    lib.fd_decode.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _SZ,
                              ctypes.POINTER(FdOptions), _P]
    lib.fd_decode.restype = _I
    lib.fd_decode_paged.argtypes = [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                                    _P, _SZ, ctypes.POINTER(FdOptions), _P]
    lib.fd_decode_paged.restype = _I
    lib.fd_decode_partial.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P, _SZ,
                                      ctypes.POINTER(FdOptions), _P]
    lib.fd_decode_partial.restype = _I
    lib.fd_decode_paged_partial.argtypes = [_P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                                            _P, _P, _P, _SZ, ctypes.POINTER(FdOptions), _P]
    lib.fd_decode_paged_partial.restype = _I
    lib.fd_merge_partials.argtypes = [_P, _P, _I, _I, _I, _P, _P, _P]
    lib.fd_merge_partials.restype = _I
    lib.fd_decode_noalloc.argtypes = [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P, _P, _P, _P]
    lib.fd_decode_noalloc.restype = _I
    lib.fd_get_device_error.argtypes = [_P, _P]
    lib.fd_get_device_error.restype = _I
    lib.fd_status_string.argtypes = [_I]
    lib.fd_status_string.restype = ctypes.c_char_p
    lib.fd_version.argtypes = []
    lib.fd_version.restype = _I
    return lib


class _Lazy:
    """Loads libfd.so on first use; raises ImportError if it has not been built."""
    _lib = None

    def __getattr__(self, name):
        if _Lazy._lib is None:
            _Lazy._lib = _load()
        return getattr(_Lazy._lib, name)


_lib = _Lazy()


class FdError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fd_status_string(status)}")


def fd_status_string(status: int) -> str:
    return _lib.fd_status_string(int(status)).decode()


def fd_version() -> int:
    return _lib.fd_version()


def fd_workspace_size(batch, num_q_heads, num_kv_heads, head_dim=128, max_kv_len=0, page_size=0,
                      q_len=1) -> int:
    return int(_lib.fd_workspace_size_q(batch, num_q_heads, num_kv_heads, head_dim, max_kv_len, page_size,
                                        q_len))


def _stream_ptr(stream, device=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def fd_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    st = _lib.fd_workspace_init(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream_ptr(stream, workspace.device))
    if st != FD_OK:
        raise FdError(st, "fd_workspace_init")


def make_workspace(batch, num_q_heads, num_kv_heads, head_dim=128, max_kv_len=0, page_size=0,
                   device="cuda", q_len=1) -> torch.Tensor:
    """Allocate (with torch) and initialise a workspace for this shape."""
    n = fd_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_kv_len, page_size, q_len)
    if n == 0:
        raise FdError(FD_ERR_INVALID_ARG, "fd_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    fd_workspace_init(ws)
    return ws


def _bits(t, name):
    if t.dtype not in (torch.bfloat16, torch.float16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must be bf16 or fp16 (or its 16-bit pattern), got {t.dtype}")
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


_FP8_TORCH = {getattr(torch, n): c for n, c in (("float8_e4m3fn", 1), ("float8_e5m2", 2))
              if hasattr(torch, n)}
_KV_NAMES = {"e4m3": FD_KV_FP8_E4M3, "e5m2": FD_KV_FP8_E5M2}


def _kv_code(k, v, kv_dtype):
    """FD_KV_* for the cache tensors: FP8 from their torch float8 type or, for
    uint8 / int8 codes, from kv_dtype ('e4m3' / 'e5m2'); else the type of q."""
    for t, name in ((k, "k"), (v, "v")):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if kv_dtype is not None:
        code = _KV_NAMES[kv_dtype]
        if k.element_size() != 1 or v.element_size() != 1:
            raise TypeError("an FP8 cache holds one byte per element")
        return code
    if k.dtype in _FP8_TORCH:
        if v.dtype != k.dtype:
            raise TypeError("k and v must have the same FP8 type")
        return _FP8_TORCH[k.dtype]
    _bits(k, "k"); _bits(v, "v")
    return FD_KV_AS_Q


def _i32(t, name):
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise TypeError(f"{name} must be contiguous int32")
    return t


FD_DTYPE_BF16, FD_DTYPE_F16 = 0, 1


def _dtype_code(t, dtype):
    if dtype is not None:
        return {"bf16": FD_DTYPE_BF16, "f16": FD_DTYPE_F16}[dtype]
    return FD_DTYPE_F16 if t.dtype == torch.float16 else FD_DTYPE_BF16


def _options(num_ctas, flags, wait_timeout_ns, split_events, dtype_code=FD_DTYPE_BF16,
             kv_code=FD_KV_AS_Q, k_scale=1.0, v_scale=1.0, q_len=1):
    ev0 = ev1 = None
    if split_events is not None:
        for e in split_events:
            if not e.cuda_event:
                raise ValueError("split_events must be created (recorded once) before use")
        ev0 = ctypes.c_void_p(split_events[0].cuda_event)
        ev1 = ctypes.c_void_p(split_events[1].cuda_event)
    return FdOptions(int(num_ctas), int(flags), int(wait_timeout_ns), ev0, ev1, int(dtype_code),
                     int(kv_code), float(k_scale), float(v_scale), int(q_len))


def _q_shape(q):
    """(B, q_len, Hq, D) of q: [B, Hq, D] (one new token) or [B, q_len, Hq, D]."""
    if q.dim() == 4:
        return tuple(q.shape)
    B, hq, d = q.shape
    return B, 1, hq, d


def _outputs(q, out, lse):
    shape_o, shape_l = tuple(q.shape), tuple(q.shape[:-1])
    if out is None:
        out = torch.empty(shape_o, dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty(shape_l, dtype=torch.float32, device=q.device)
    if out.dtype != torch.float32 or not out.is_contiguous() or tuple(out.shape) != shape_o:
        raise ValueError(f"out must be contiguous fp32 {list(shape_o)}")
    if lse is not False and (lse.dtype != torch.float32 or not lse.is_contiguous()
                             or tuple(lse.shape) != shape_l):
        raise ValueError(f"lse must be contiguous fp32 {list(shape_l)}")
    return out, lse


def fd_decode(q, k, v, seq_lens=None, seq_lens_host=None, scale=None, out=None, lse=None,
              workspace=None, num_ctas=0, flags=0, wait_timeout_ns=0, split_events=None,
              stream=None, check=True, dtype=None, kv_dtype=None, k_scale=1.0, v_scale=1.0):
    """Decode attention over a contiguous KV cache (see fd_decode in include/fd.h).

    q [B, Hq, D] bf16 or fp16 (``dtype`` 'bf16'/'f16' overrides the tensor's
    own type, e.g. for int16 views), or [B, q_len, Hq, D] for q_len new tokens
    per request (token i sees cache positions 0 .. L - q_len + i; out and lse
    then carry the q_len axis too); k/v [B, S_max, Hkv, D] of q's type, or an
    FP8 cache: torch float8_e4m3fn / float8_e5m2 tensors, or uint8 codes with
    ``kv_dtype`` 'e4m3' / 'e5m2', dequantised by ``k_scale`` / ``v_scale``.
    seq_lens int32 [B] on the device (None = every request has S_max tokens);
    seq_lens_host an optional CPU int32 copy used for host-side validation
    (and to size the launch).  Pass ``lse=False`` to skip the LSE output.
    Returns (out, lse).
    """
    _bits(q, "q")
    kv_code = _kv_code(k, v, kv_dtype)
    B, q_len, hq, d = _q_shape(q)
    _, s_max, hkv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out, lse = _outputs(q, out, lse)
    if workspace is None:
        workspace = make_workspace(B, hq, hkv, d, s_max, 0, q.device, q_len=q_len)
    opts = _options(num_ctas, flags, wait_timeout_ns, split_events, _dtype_code(q, dtype), kv_code,
                    k_scale, v_scale, q_len)
    lh = None
    if seq_lens_host is not None:
        lh = seq_lens_host.to(torch.int32).contiguous().cpu()
    st = _lib.fd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(_i32(seq_lens, "seq_lens")), _ptr(lh),
                        B, hq, hkv, d, s_max, float(scale), _ptr(out),
                        None if lse is False else _ptr(lse), _ptr(workspace),
                        workspace.numel(), ctypes.byref(opts), _stream_ptr(stream, q.device))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode")
    return out, (None if lse is False else lse)


def fd_decode_paged(q, k_pages, v_pages, block_table, seq_lens, seq_lens_host=None, scale=None,
                    out=None, lse=None, workspace=None, num_ctas=0, flags=0, wait_timeout_ns=0,
                    split_events=None, stream=None, check=True, dtype=None, kv_dtype=None,
                    k_scale=1.0, v_scale=1.0):
    """Decode attention over a paged KV cache (see fd_decode_paged in include/fd.h).

    k_pages/v_pages [num_pages, P, Hkv, D] of q's type or an FP8 cache (as for
    fd_decode); block_table int32 [B, max_blocks]; seq_lens int32 [B] on the device.
    """
    _bits(q, "q")
    kv_code = _kv_code(k_pages, v_pages, kv_dtype)
    _i32(block_table, "block_table"); _i32(seq_lens, "seq_lens")
    B, q_len, hq, d = _q_shape(q)
    num_pages, page, hkv, _ = k_pages.shape
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out, lse = _outputs(q, out, lse)
    if workspace is None:
        workspace = make_workspace(B, hq, hkv, d, max_blocks * page, page, q.device, q_len=q_len)
    opts = _options(num_ctas, flags, wait_timeout_ns, split_events, _dtype_code(q, dtype), kv_code,
                    k_scale, v_scale, q_len)
    lh = None
    if seq_lens_host is not None:
        lh = seq_lens_host.to(torch.int32).contiguous().cpu()
    st = _lib.fd_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), max_blocks,
                              _ptr(seq_lens), _ptr(lh), B, hq, hkv, d, page, num_pages, float(scale),
                              _ptr(out), None if lse is False else _ptr(lse), _ptr(workspace),
                              workspace.numel(), ctypes.byref(opts), _stream_ptr(stream, q.device))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode_paged")
    return out, (None if lse is False else lse)


def fd_decode_partial(q, k, v, seq_lens, kv_begin, kv_end=KV_END, seq_lens_host=None, scale=None,
                      out=None, lse=None, workspace=None, num_ctas=0, flags=0, wait_timeout_ns=0,
                      split_events=None, stream=None, check=True, dtype=None, kv_dtype=None, k_scale=1.0,
                      v_scale=1.0):
    """Attention over cache positions [kv_begin, min(L_b, kv_end)) of every
    request (see fd_decode_partial in include/fd.h): k/v [B, S, Hkv, D] hold
    the range (row t' = position kv_begin + t'); seq_lens are the whole
    lengths.  Returns (out, lse): the output normalised over the range and its
    natural-log LSE (-inf where the range holds no visible position)."""
    _bits(q, "q")
    kv_code = _kv_code(k, v, kv_dtype)
    B, q_len, hq, d = _q_shape(q)
    _, s_max, hkv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out, lse = _outputs(q, out, lse)
    if lse is False:
        raise ValueError("a partial result needs its LSE")
    if workspace is None:
        workspace = make_workspace(B, hq, hkv, d, s_max, 0, q.device, q_len=q_len)
    opts = _options(num_ctas, flags, wait_timeout_ns, split_events, _dtype_code(q, dtype), kv_code,
                    k_scale, v_scale, q_len)
    lh = None if seq_lens_host is None else seq_lens_host.to(torch.int32).contiguous().cpu()
    st = _lib.fd_decode_partial(_ptr(q), _ptr(k), _ptr(v), _ptr(_i32(seq_lens, "seq_lens")), _ptr(lh),
                                B, hq, hkv, d, s_max, int(kv_begin), int(kv_end), float(scale), _ptr(out),
                                _ptr(lse), _ptr(workspace), workspace.numel(), ctypes.byref(opts),
                                _stream_ptr(stream, q.device))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode_partial")
    return out, lse


def fd_decode_paged_partial(q, k_pages, v_pages, block_table, seq_lens, kv_begin, kv_end=KV_END,
                            seq_lens_host=None, scale=None, out=None, lse=None, workspace=None, num_ctas=0,
                            flags=0, wait_timeout_ns=0, split_events=None, stream=None, check=True, dtype=None,
                            kv_dtype=None, k_scale=1.0, v_scale=1.0):
    """fd_decode_partial over a paged cache: block_table maps the range's own
    tokens (token t' = position kv_begin + t'); see include/fd.h."""
    _bits(q, "q")
    kv_code = _kv_code(k_pages, v_pages, kv_dtype)
    _i32(block_table, "block_table"); _i32(seq_lens, "seq_lens")
    B, q_len, hq, d = _q_shape(q)
    num_pages, page, hkv, _ = k_pages.shape
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out, lse = _outputs(q, out, lse)
    if lse is False:
        raise ValueError("a partial result needs its LSE")
    if workspace is None:
        workspace = make_workspace(B, hq, hkv, d, max_blocks * page, page, q.device, q_len=q_len)
    opts = _options(num_ctas, flags, wait_timeout_ns, split_events, _dtype_code(q, dtype), kv_code,
                    k_scale, v_scale, q_len)
    lh = None if seq_lens_host is None else seq_lens_host.to(torch.int32).contiguous().cpu()
    st = _lib.fd_decode_paged_partial(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table), max_blocks,
                                      _ptr(seq_lens), _ptr(lh), B, hq, hkv, d, page, num_pages, int(kv_begin),
                                      int(kv_end), float(scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                      workspace.numel(), ctypes.byref(opts), _stream_ptr(stream, q.device))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode_paged_partial")
    return out, lse


def fd_merge_partials(o_parts, lse_parts, out=None, lse=None, stream=None, check=True):
    """Merge n partial sets (see fd_merge_partials in include/fd.h).

    o_parts fp32 [n, *rows_shape, D] and lse_parts fp32 [n, *rows_shape] on
    the device (e.g. every rank's fd_decode_partial result, stacked in rank
    order); returns (out [*rows_shape, D], lse [*rows_shape])."""
    for t, name in ((o_parts, "o_parts"), (lse_parts, "lse_parts")):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
    n, d = o_parts.shape[0], o_parts.shape[-1]
    rows_shape = tuple(o_parts.shape[1:-1])
    if tuple(lse_parts.shape) != (n,) + rows_shape:
        raise ValueError(f"lse_parts must be {[n] + list(rows_shape)}")
    rows = 1
    for x in rows_shape:
        rows *= x
    if out is None:
        out = torch.empty(rows_shape + (d,), dtype=torch.float32, device=o_parts.device)
    if lse is None:
        lse = torch.empty(rows_shape, dtype=torch.float32, device=o_parts.device)
    st = _lib.fd_merge_partials(_ptr(o_parts), _ptr(lse_parts), n, rows, d, _ptr(out),
                                None if lse is False else _ptr(lse), _stream_ptr(stream, o_parts.device))
    if check and st != FD_OK:
        raise FdError(st, "fd_merge_partials")
    return out, (None if lse is False else lse)


def fd_decode_noalloc(q, k, v, seq_lens, o, lse=None, device_status=None, scale=None, stream=None,
                      check=True):
    """fd_decode without a workspace (see fd_decode_noalloc in include/fd.h).

    For callers that cannot allocate device memory where they run attention:
    the scratch is a fixed array inside the library, and the caller passes
    only inputs and preallocated outputs (o fp32 [B, Hq, D], optional lse fp32
    [B, Hq] and device_status uint32/int32 [1]).  Returns the C status.
    """
    B, hq, d = q.shape
    _, s_max, hkv, _ = k.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    st = _lib.fd_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), B, hq, hkv, d, s_max,
                                float(scale), _ptr(o), _ptr(lse), _ptr(device_status),
                                _stream_ptr(stream, q.device))
    if check and st != FD_OK:
        raise FdError(st, "fd_decode_noalloc")
    return st


def fd_get_device_error(workspace, stream=None) -> int:
    """Read and clear the workspace's sticky device-error word (synchronises the stream)."""
    return int(_lib.fd_get_device_error(_ptr(workspace), _stream_ptr(stream, workspace.device)))
