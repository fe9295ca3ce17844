"""fd_decode_noalloc: the entry point for callers that cannot allocate device
memory where they run attention (it keeps its scratch in a fixed array inside
the library instead of a caller workspace).

Called through the C ABI with ctypes, twice in a row on different inputs, and
compared with the fp64 oracle within the GPU tests' tolerance, for each group
size it serves (CUDA-core consumers for MHA, tensor-core consumers for GQA).
This file is collected last so that a stop-at-first-failure run has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import fd_synth as syn
import oracle
from gpu_util import check, to_device

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


@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(lib, group):
    import decode_attention_decoding_gb300 as fd
    oracle.build()
    hkv = 4
    cases = [syn.make_contiguous(700 + group, 4, hkv * group, hkv, 128, 1500, [1500, 3, 0, 777]),
             syn.make_contiguous(710 + group, 4, hkv * group, hkv, 128, 1500, [64, 1499, 1000, 1])]
    o = torch.full((4, hkv * group, 128), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((4, hkv * group), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for w in cases:                       # consecutive calls share the fixed scratch
        d = to_device(w)
        assert call_noalloc(lib, d, w, o, lse, status) == fd.FD_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ro, rl = oracle.attend(w, threads=8)
        check(o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl,
              f"noalloc G={group}")


def test_noalloc_large_batch_two_calls_in_a_row(lib):
    """Batches over 32 take the merge path that reads the tile prefix back
    from the fixed array; two calls with different lengths share it."""
    import decode_attention_decoding_gb300 as fd
    oracle.build()
    B, hkv, group = 40, 2, 4
    lens_a = syn.randint(720, B, 0, 900).astype(np.int32)
    lens_b = syn.randint(721, B, 0, 900).astype(np.int32)
    cases = [syn.make_contiguous(720, B, hkv * group, hkv, 128, 900, lens_a),
             syn.make_contiguous(721, B, hkv * group, hkv, 128, 900, lens_b)]
    o = torch.full((B, hkv * group, 128), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, hkv * group), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    for w in cases:
        d = to_device(w)
        assert call_noalloc(lib, d, w, o, lse, status) == fd.FD_OK
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        ro, rl = oracle.attend(w, threads=8)
        check(o.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), ro, rl,
              "noalloc B=40")


def test_noalloc_reports_a_device_length_above_capacity(lib):
    """A device length above s_max is clamped to s_max and reported in the
    status word (FD_DEVICE_STATUS_BAD_LENGTH); the next good call reports 0."""
    import decode_attention_decoding_gb300 as fd
    oracle.build()
    w = syn.make_contiguous(722, 3, 8, 2, 128, 200, [200, 50, 7])
    d = to_device(w)
    o = torch.empty((3, 8, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((3, 8), dtype=torch.float32, device="cuda")
    status = torch.zeros((1,), dtype=torch.int32, device="cuda")
    d["seq_lens"] = torch.tensor([200, 50, 201], dtype=torch.int32, device="cuda")   # 201 > s_max
    assert call_noalloc(lib, d, w, o, lse, status) == fd.FD_OK
    torch.cuda.synchronize()
    assert int(status.item()) & 0x2    # FD_DEVICE_STATUS_BAD_LENGTH
    ro, rl = oracle.attend(w, items=np.array([[0, h, 0, -1] for h in range(8)], dtype=np.int32), threads=4)
    check(o[0].cpu().numpy().astype(np.float64), lse[0].cpu().numpy().astype(np.float64), ro, rl,
          "noalloc, the request with a valid length")
    d["seq_lens"] = torch.from_numpy(w.seq_lens).cuda()
    assert call_noalloc(lib, d, w, o, lse, status) == fd.FD_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0


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
