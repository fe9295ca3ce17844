"""fd_decode_noalloc: the entry point for callers that cannot allocate device
memory where they run attention (it keeps its scratch in a fixed array inside
the library instead of a caller workspace).

Called through the C ABI with ctypes, twice in a row on different inputs, and
compared with fd_decode on the same inputs within the GPU tests' tolerance.
This file is collected last so that a stop-at-first-failure run has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import fd_synth as syn
from gpu_util import LSE_ATOL, O_ATOL, O_RTOL, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from decode_attention_decoding_gb300 import build
    lib = ctypes.CDLL(build.build())
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.fd_decode_noalloc.argtypes = [P, P, P, P, I, I, I, I, I, ctypes.c_float, P, P, P, P]
    lib.fd_decode_noalloc.restype = I
    return lib


def call_noalloc(lib, d, w, o, lse, status):
    B, hq, D = w.q.shape
    return lib.fd_decode_noalloc(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
                                 d["seq_lens"].data_ptr(), B, hq, w.num_kv_heads, D, w.k.shape[1],
                                 ctypes.c_float(w.scale), o.data_ptr(), lse.data_ptr(), status.data_ptr(),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def assert_close(o, lse, ro, rl):
    o, lse, ro, rl = (x.cpu().numpy().astype(np.float64) for x in (o, lse, ro, rl))
    assert np.all(np.abs(o - ro) <= O_ATOL + O_RTOL * np.abs(ro))
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse)) and np.all(lse[~fin] == rl[~fin])
    assert np.all(np.abs(lse[fin] - rl[fin]) <= LSE_ATOL)


def test_noalloc_matches_fd_decode_on_two_calls_in_a_row(lib):
    import decode_attention_decoding_gb300 as fd
    cases = [syn.make_contiguous(700, 4, 16, 4, 128, 1500, [1500, 3, 0, 777]),
             syn.make_contiguous(701, 4, 16, 4, 128, 1500, [64, 1499, 1000, 1])]
    o = torch.full((4, 16, 128), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((4, 16), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for w in cases:                       # consecutive calls share the fixed scratch
        d = to_device(w)
        assert call_noalloc(lib, d, w, o, lse, status) == fd.FD_OK
        ro, rl = fd.fd_decode(d["q"], d["k"], d["v"], d["seq_lens"], scale=w.scale)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert_close(o, lse, ro, rl)


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    import decode_attention_decoding_gb300 as fd
    w = syn.make_contiguous(702, 1, 8, 1, 128, 64, [64])
    d = to_device(w)
    o = torch.empty((1, 8, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((1, 8), dtype=torch.float32, device="cuda")
    st = lib.fd_decode_noalloc(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), None,
                               4096, 64, 8, 128, 64, ctypes.c_float(0.1), o.data_ptr(), lse.data_ptr(),
                               None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == fd.FD_ERR_WORKSPACE_TOO_SMALL
