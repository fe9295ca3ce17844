"""The C ABI on the host: exported symbols, argument checks, schedule invariants.

None of these calls reaches the GPU: every case fails validation before the
first CUDA call, or exercises pure host functions.
"""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fd.h")


@pytest.fixture(scope="module")
def lib():
    from decode_attention_decoding_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


@pytest.fixture(scope="module")
def fd():
    import decode_attention_decoding_gb300 as fd
    return fd


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fd_[a-z_]+)\s*\(", text)))


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert {"fd_workspace_size", "fd_decode", "fd_decode_paged"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", os.path.join(ROOT, "decode_attention_decoding_gb300", "libfd.so")],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (fd_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        getattr(lib, n)


def test_status_strings_and_version(fd):
    for st in range(7):
        assert fd.fd_status_string(st).startswith("FD_")
    assert fd.fd_status_string(99) == "FD_ERR_UNKNOWN"
    assert fd.fd_version() >= 10000


def test_workspace_size_is_host_only_and_rejects_bad_shapes(fd):
    assert fd.fd_workspace_size(1, 32, 32, 128, 4096, 0) > 0
    assert fd.fd_workspace_size(1, 32, 5, 128, 4096, 0) == 0
    assert fd.fd_workspace_size(-1, 32, 8, 128, 4096, 0) == 0
    # independent of the lengths, growing with batch
    assert fd.fd_workspace_size(4, 32, 8, 128, 10, 0) == fd.fd_workspace_size(4, 32, 8, 128, 10 ** 6, 16)
    assert fd.fd_workspace_size(8, 32, 8, 128, 10, 0) > fd.fd_workspace_size(4, 32, 8, 128, 10, 0)
    # room for one fp32 partial (G rows of D outputs + G LSEs) per slot
    for B, hq, hkv in ((1, 32, 32), (64, 32, 8), (1, 64, 8)):
        slots = B * hkv + 1024
        assert fd.fd_workspace_size(B, hq, hkv, 128, 1, 0) >= slots * (hq // hkv) * 129 * 4
    # q_len new tokens: G x q_len partial rows per slot
    assert fd.fd_workspace_size(4, 8, 2, 128, 1, 0, q_len=2) >= (4 * 2 + 1024) * 8 * 129 * 4
    assert fd.fd_workspace_size(4, 8, 2, 128, 1, 0, q_len=1) == fd.fd_workspace_size(4, 8, 2, 128, 1, 0)
    # 16 columns (GQA-8 with two new tokens), and paired heads of 64 dims with 2 x 16 slots
    assert fd.fd_workspace_size(4, 16, 2, 128, 1, 0, q_len=2) >= (4 * 2 + 1024) * 16 * 129 * 4
    assert fd.fd_workspace_size(4, 32, 4, 64, 1, 0, q_len=2) >= (4 * 2 + 1024) * 32 * 65 * 4
    assert fd.fd_workspace_size(4, 16, 2, 128, 1, 0, q_len=3) == 0


ALIGNED = 1 << 20          # fake, 256-byte aligned device addresses (never dereferenced)


def call_decode(lib, **over):
    a = dict(q=ALIGNED, k=ALIGNED, v=ALIGNED, sl=None, slh=None, B=2, hq=8, hkv=2, d=128, smax=64,
             scale=0.1, o=ALIGNED, lse=ALIGNED, ws=ALIGNED, wsb=1 << 30, opts=None, stream=None)
    a.update(over)
    f = lib.fd_decode
    f.restype = ctypes.c_int
    return f(ctypes.c_void_p(a["q"]), ctypes.c_void_p(a["k"]), ctypes.c_void_p(a["v"]), a["sl"], a["slh"],
             a["B"], a["hq"], a["hkv"], a["d"], a["smax"], ctypes.c_float(a["scale"]),
             ctypes.c_void_p(a["o"]), ctypes.c_void_p(a["lse"]), ctypes.c_void_p(a["ws"]),
             ctypes.c_size_t(a["wsb"]), a["opts"], a["stream"])


def test_decode_argument_checks(lib, fd):
    E = fd
    assert call_decode(lib, q=0) == E.FD_ERR_INVALID_ARG
    assert call_decode(lib, o=0) == E.FD_ERR_INVALID_ARG
    assert call_decode(lib, ws=0) == E.FD_ERR_INVALID_ARG
    assert call_decode(lib, hq=6, hkv=4) == E.FD_ERR_INVALID_ARG
    assert call_decode(lib, q=ALIGNED + 8) == E.FD_ERR_INVALID_ARG
    assert call_decode(lib, k=ALIGNED + 2) == E.FD_ERR_INVALID_ARG
    assert call_decode(lib, ws=ALIGNED + 16) == E.FD_ERR_INVALID_ARG
    assert call_decode(lib, smax=-1) == E.FD_ERR_INVALID_ARG
    for d in (32, 96, 192, 512):
        assert call_decode(lib, d=d) == E.FD_ERR_UNSUPPORTED
    for d in (64, 128, 256):   # accepted head dims reach the workspace check
        assert call_decode(lib, d=d, wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    assert call_decode(lib, hq=6, hkv=2, wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL   # group 3: padded to 4
    assert call_decode(lib, hq=32, hkv=2, wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL   # group 16
    assert call_decode(lib, hq=64, hkv=2) == E.FD_ERR_UNSUPPORTED      # group 32
    # several new tokens: group x q_len query columns must fit 16
    for g, ql, ok in ((4, 2, True), (1, 8, True), (2, 3, True), (4, 3, True), (8, 2, True), (1, 9, True),
                      (1, 16, True), (16, 1, True), (8, 3, False), (1, 17, False), (16, 2, False)):
        opts = fd.FdOptions(0, 0, 0, None, None, 0, 0, 0.0, 0.0, ql)
        st = call_decode(lib, hq=2 * g, hkv=2, opts=ctypes.byref(opts), wsb=1024)
        assert st == (E.FD_ERR_WORKSPACE_TOO_SMALL if ok else E.FD_ERR_UNSUPPORTED), (g, ql)
    # over 8 columns run on the tensor-core consumers only: rejected on the
    # host with FD_FLAG_CUDA_CORES, and for an FP8 head of 64 dims that cannot
    # pair (odd Hkv, or FD_FLAG_NO_HEAD_FUSION)
    for g, ql, flags, kv, d, hkv, ok in ((8, 2, 0x2, 0, 128, 2, False), (8, 1, 0x2, 0, 128, 2, True),
                                         (4, 3, 0x2, 0, 128, 2, False), (8, 2, 0, 1, 64, 2, True),
                                         (8, 2, 0, 1, 64, 3, False), (8, 2, 0x8, 2, 64, 2, False),
                                         (8, 2, 0x8, 1, 128, 2, True), (8, 2, 0x8, 0, 64, 2, True)):
        opts = fd.FdOptions(0, flags, 0, None, None, 0, kv, 0.0, 0.0, ql)
        st = call_decode(lib, hq=hkv * g, hkv=hkv, d=d, opts=ctypes.byref(opts), wsb=1024)
        assert st == (E.FD_ERR_WORKSPACE_TOO_SMALL if ok else E.FD_ERR_UNSUPPORTED), (g, ql, flags, kv, d)
    opts = fd.FdOptions(0, 0, 0, None, None, 0, 0, 0.0, 0.0, -1)
    assert call_decode(lib, opts=ctypes.byref(opts)) == E.FD_ERR_INVALID_ARG
    assert call_decode(lib, B=5000) == E.FD_ERR_UNSUPPORTED
    assert call_decode(lib, wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    lens = (ctypes.c_int32 * 2)(10, 65)
    assert call_decode(lib, slh=lens) == E.FD_ERR_INVALID_ARG
    lens = (ctypes.c_int32 * 2)(10, -1)
    assert call_decode(lib, slh=lens) == E.FD_ERR_INVALID_ARG
    opts = fd.FdOptions(2000, 0, 0, None, None)
    assert call_decode(lib, opts=ctypes.byref(opts)) == E.FD_ERR_INVALID_ARG
    # FP8 cache options: type code and scales are checked on the host
    for kv, ks, vs in ((3, 0.0, 0.0), (-1, 0.0, 0.0), (1, -1.0, 1.0), (2, 1.0, float("nan")),
                       (1, float("inf"), 1.0)):
        opts = fd.FdOptions(0, 0, 0, None, None, 0, kv, ks, vs)
        assert call_decode(lib, opts=ctypes.byref(opts)) == E.FD_ERR_INVALID_ARG, (kv, ks, vs)
    for kv in (1, 2):   # valid FP8 options reach the workspace check
        opts = fd.FdOptions(0, 0, 0, None, None, 0, kv, 0.5, 2.0)
        assert call_decode(lib, opts=ctypes.byref(opts), wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    assert call_decode(lib, B=0) == E.FD_OK                           # nothing to do, no CUDA call


def call_paged(lib, **over):
    a = dict(q=ALIGNED, k=ALIGNED, v=ALIGNED, table=ALIGNED, mb=4, sl=ALIGNED, slh=None, B=2, hq=8,
             hkv=2, d=128, page=16, npages=8, scale=0.1, o=ALIGNED, lse=ALIGNED, ws=ALIGNED,
             wsb=1 << 30, opts=None)
    a.update(over)
    f = lib.fd_decode_paged
    f.restype = ctypes.c_int
    return f(ctypes.c_void_p(a["q"]), ctypes.c_void_p(a["k"]), ctypes.c_void_p(a["v"]),
             ctypes.c_void_p(a["table"]), a["mb"], ctypes.c_void_p(a["sl"]), a["slh"], a["B"], a["hq"],
             a["hkv"], a["d"], a["page"], a["npages"], ctypes.c_float(a["scale"]), ctypes.c_void_p(a["o"]),
             ctypes.c_void_p(a["lse"]), ctypes.c_void_p(a["ws"]), ctypes.c_size_t(a["wsb"]), a["opts"], None)


def test_paged_argument_checks(lib, fd):
    E = fd
    assert call_paged(lib, table=0) == E.FD_ERR_INVALID_ARG
    assert call_paged(lib, sl=0) == E.FD_ERR_INVALID_ARG
    assert call_paged(lib, mb=0) == E.FD_ERR_INVALID_ARG
    assert call_paged(lib, npages=0) == E.FD_ERR_INVALID_ARG
    assert call_paged(lib, page=0) == E.FD_ERR_INVALID_ARG
    assert call_paged(lib, page=24) == E.FD_ERR_UNSUPPORTED
    # one-token FP8 pages of head_dim 64 are 64-byte TMA boxes: below the 128-byte alignment
    fp8 = fd.FdOptions(0, 0, 0, None, None, 0, 1, 1.0, 1.0)
    assert call_paged(lib, page=1, d=64, opts=ctypes.byref(fp8)) == E.FD_ERR_UNSUPPORTED
    assert call_paged(lib, page=2, d=64, opts=ctypes.byref(fp8), wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    assert call_paged(lib, page=1, d=64, wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL   # bf16: 128 bytes
    assert call_paged(lib, page=96) == E.FD_ERR_UNSUPPORTED
    # over 8 columns need the tensor-core consumers (any page size; pages under 8
    # tokens are copied with cp.async), which a 64-dim FP8 head reaches only by
    # pairing kv heads, and pairing needs pages of at least 8 tokens
    many = fd.FdOptions(0, 0, 0, None, None, 0, 0, 0.0, 0.0, 2)
    assert call_paged(lib, page=4, hq=16, opts=ctypes.byref(many), wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    assert call_paged(lib, page=8, hq=16, opts=ctypes.byref(many), wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    many_cc = fd.FdOptions(0, 0x2, 0, None, None, 0, 0, 0.0, 0.0, 2)
    assert call_paged(lib, page=8, hq=16, opts=ctypes.byref(many_cc)) == E.FD_ERR_UNSUPPORTED
    many_fp8 = fd.FdOptions(0, 0, 0, None, None, 0, 1, 0.0, 0.0, 2)
    assert call_paged(lib, page=4, hq=16, d=64, opts=ctypes.byref(many_fp8)) == E.FD_ERR_UNSUPPORTED
    assert call_paged(lib, page=8, hq=16, d=64, opts=ctypes.byref(many_fp8), wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    lens = (ctypes.c_int32 * 2)(64, 65)                     # capacity 4 pages * 16
    assert call_paged(lib, slh=lens) == E.FD_ERR_INVALID_ARG
    assert call_paged(lib, wsb=100) == E.FD_ERR_WORKSPACE_TOO_SMALL
    for ok_page in (1, 2, 8, 16, 32, 64, 128, 256):
        assert call_paged(lib, page=ok_page, B=0) == E.FD_OK


def call_partial(lib, **over):
    a = dict(q=ALIGNED, k=ALIGNED, v=ALIGNED, sl=None, slh=None, B=2, hq=8, hkv=2, d=128, smax=64, t0=0,
             t1=2 ** 31 - 1, scale=0.1, o=ALIGNED, lse=ALIGNED, ws=ALIGNED, wsb=1 << 30, opts=None)
    a.update(over)
    f = lib.fd_decode_partial
    f.restype = ctypes.c_int
    return f(ctypes.c_void_p(a["q"]), ctypes.c_void_p(a["k"]), ctypes.c_void_p(a["v"]), a["sl"], a["slh"],
             a["B"], a["hq"], a["hkv"], a["d"], a["smax"], a["t0"], a["t1"], ctypes.c_float(a["scale"]),
             ctypes.c_void_p(a["o"]), ctypes.c_void_p(a["lse"]), ctypes.c_void_p(a["ws"]),
             ctypes.c_size_t(a["wsb"]), a["opts"], None)


def call_paged_partial(lib, **over):
    a = dict(q=ALIGNED, k=ALIGNED, v=ALIGNED, table=ALIGNED, mb=4, sl=ALIGNED, slh=None, B=2, hq=8,
             hkv=2, d=128, page=16, npages=8, t0=0, t1=2 ** 31 - 1, scale=0.1, o=ALIGNED, lse=ALIGNED,
             ws=ALIGNED, wsb=1 << 30, opts=None)
    a.update(over)
    f = lib.fd_decode_paged_partial
    f.restype = ctypes.c_int
    return f(ctypes.c_void_p(a["q"]), ctypes.c_void_p(a["k"]), ctypes.c_void_p(a["v"]),
             ctypes.c_void_p(a["table"]), a["mb"], ctypes.c_void_p(a["sl"]), a["slh"], a["B"], a["hq"],
             a["hkv"], a["d"], a["page"], a["npages"], a["t0"], a["t1"], ctypes.c_float(a["scale"]),
             ctypes.c_void_p(a["o"]), ctypes.c_void_p(a["lse"]), ctypes.c_void_p(a["ws"]),
             ctypes.c_size_t(a["wsb"]), a["opts"], None)


def test_partial_argument_checks(lib, fd):
    """The range entry points check the range and the host lengths against the
    range's own capacity (n_b = min(L_b, kv_end) - kv_begin <= s_max)."""
    E = fd
    assert call_partial(lib, lse=0) == E.FD_ERR_INVALID_ARG          # a partial needs its LSE
    assert call_partial(lib, t0=-1) == E.FD_ERR_INVALID_ARG
    assert call_partial(lib, t0=10, t1=9) == E.FD_ERR_INVALID_ARG
    assert call_partial(lib, t0=2 ** 31 - 64) == E.FD_ERR_INVALID_ARG  # kv_begin + s_max past int32
    assert call_partial(lib, t0=10, t1=10, wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL   # empty range: valid
    assert call_partial(lib, d=96) == E.FD_ERR_UNSUPPORTED
    # capacity is the range's: s_max 64 holds positions kv_begin .. kv_begin + 63
    lens = (ctypes.c_int32 * 2)(74, 5)
    assert call_partial(lib, slh=lens, t0=10, wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    lens = (ctypes.c_int32 * 2)(75, 5)
    assert call_partial(lib, slh=lens, t0=10) == E.FD_ERR_INVALID_ARG
    lens = (ctypes.c_int32 * 2)(1000, 5)                             # clipped by kv_end
    assert call_partial(lib, slh=lens, t0=10, t1=70, wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    lens = (ctypes.c_int32 * 2)(-1, 5)
    assert call_partial(lib, slh=lens, t0=10) == E.FD_ERR_INVALID_ARG
    assert call_partial(lib, B=0) == E.FD_OK
    assert call_paged_partial(lib, lse=0) == E.FD_ERR_INVALID_ARG
    assert call_paged_partial(lib, sl=0) == E.FD_ERR_INVALID_ARG
    assert call_paged_partial(lib, t0=5, t1=4) == E.FD_ERR_INVALID_ARG
    assert call_paged_partial(lib, page=24) == E.FD_ERR_UNSUPPORTED
    lens = (ctypes.c_int32 * 2)(64 + 100, 0)                         # 4 pages of 16 from position 100
    assert call_paged_partial(lib, slh=lens, t0=100, wsb=1024) == E.FD_ERR_WORKSPACE_TOO_SMALL
    lens = (ctypes.c_int32 * 2)(65 + 100, 0)
    assert call_paged_partial(lib, slh=lens, t0=100) == E.FD_ERR_INVALID_ARG
    assert call_paged_partial(lib, B=0) == E.FD_OK


def test_merge_partials_argument_checks(lib, fd):
    E = fd
    f = lib.fd_merge_partials
    f.restype = ctypes.c_int

    def call(op=ALIGNED, lp=ALIGNED, n=2, rows=4, d=128, o=ALIGNED, lse=ALIGNED):
        return f(ctypes.c_void_p(op), ctypes.c_void_p(lp), n, rows, d, ctypes.c_void_p(o), ctypes.c_void_p(lse),
                 None)

    assert call(op=0) == E.FD_ERR_INVALID_ARG
    assert call(lp=0) == E.FD_ERR_INVALID_ARG
    assert call(o=0) == E.FD_ERR_INVALID_ARG
    assert call(n=0) == E.FD_ERR_INVALID_ARG
    assert call(rows=-1) == E.FD_ERR_INVALID_ARG
    assert call(op=ALIGNED + 4) == E.FD_ERR_INVALID_ARG
    assert call(o=ALIGNED + 8) == E.FD_ERR_INVALID_ARG
    assert call(lp=ALIGNED + 2) == E.FD_ERR_INVALID_ARG
    for d in (32, 96, 512):
        assert call(d=d) == E.FD_ERR_UNSUPPORTED
    for d in (64, 128, 256):
        assert call(d=d, rows=0) == E.FD_OK       # nothing to merge: no launch
    assert call(rows=0, lse=0) == E.FD_OK


# ---------------------------------------------------------------------------
# The split schedule (fd_sched.h), through a small g++-compiled shim
# ---------------------------------------------------------------------------

@pytest.fixture(scope="module")
def sched(tmp_path_factory):
    d = tmp_path_factory.mktemp("shim")
    so = str(d / "libshim.so")
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-shared", "-fPIC",
                           "-I" + os.path.join(ROOT, "decode_attention_decoding_gb300", "csrc"),
                           os.path.join(ROOT, "tests", "sched_shim.cpp"), "-o", so])
    s = ctypes.CDLL(so)
    s.shim_schedule_cta_of_tile.restype = ctypes.c_int
    s.shim_request_of_tile.restype = ctypes.c_int
    s.shim_slots.restype = ctypes.c_int
    return s


def make_plan(lens, hkv, tt=64):
    """The Schedule's two arrays for these lengths: tile prefix and non-empty requests."""
    ntiles = (np.asarray(lens, dtype=np.int64) + tt - 1) // tt
    prefix = np.concatenate([[0], np.cumsum(ntiles * hkv)]).astype(np.int32)
    nonempty = np.concatenate([[0], np.cumsum(ntiles > 0)]).astype(np.int32)
    return ntiles, prefix, nonempty


def ranges(sched, prefix, nonempty, hkv, w, P):
    B = len(prefix) - 1
    pre = (ctypes.c_int * len(prefix))(*prefix.tolist())
    ne = (ctypes.c_int * len(nonempty))(*nonempty.tolist())
    out = []
    b, e = ctypes.c_int(), ctypes.c_int()
    for c in range(P):
        sched.shim_schedule_range(pre, ne, B, hkv, w, P, c, ctypes.byref(b), ctypes.byref(e))
        out.append((b.value, e.value))
    return out, pre, ne


def brute_positions(ntiles, hkv, w):
    """Cost position of every tile, tile by tile: +1 per tile, +w at each segment start."""
    pos, x = [], 0
    for n in ntiles:
        for _h in range(hkv):
            for j in range(int(n)):
                x += w if j == 0 else 0
                pos.append(x)
                x += 1
    return pos, x


@pytest.mark.parametrize("w", [0, 1, 2, 5])
def test_schedule_partitions_tiles_by_cost(sched, w):
    """Contiguous runs covering every tile once; the owner of a tile agrees
    with the runs and with the tile's cost position (+1 per tile, +w at each
    segment start); w = 0 gives runs of equal length."""
    rng = np.random.default_rng(11 + w)
    for trial in range(40):
        B = int(rng.integers(1, 40))
        hkv = int(rng.choice([1, 2, 8]))
        lens = rng.integers(0, 3000, B)
        lens[rng.random(B) < 0.2] = 0
        ntiles, prefix, nonempty = make_plan(lens, hkv)
        T = int(prefix[-1])
        P = int(rng.integers(1, 300))
        r, pre, ne = ranges(sched, prefix, nonempty, hkv, w, P)
        assert r[0][0] == 0 and r[-1][1] == T
        for (b0, e0), (b1, _) in zip(r, r[1:]):
            assert e0 == b1 and b0 <= e0
        pos, C = brute_positions(ntiles, hkv, w)
        assert C == T + w * hkv * int((ntiles > 0).sum())
        Pe = min(P, C)   # CTAs that take tiles
        for c, (b0, e0) in enumerate(r):
            if c >= Pe:
                assert b0 == e0 == T
            for t in range(b0, e0):
                assert c * C <= pos[t] * Pe < (c + 1) * C
        # the CTAs of a segment are consecutive and each owns some of its tiles
        owners = {}
        for c, (b0, e0) in enumerate(r):
            for t in range(b0, e0):
                b = int(np.searchsorted(prefix, t, side="right") - 1)
                owners.setdefault((b, (t - prefix[b]) // ntiles[b]), set()).add(c)
        for cs in owners.values():
            assert cs == set(range(min(cs), max(cs) + 1))
        for t in sorted(set([0, T - 1, T // 2, *range(0, T, max(1, T // 97))])):
            if 0 <= t < T:
                c = sched.shim_schedule_cta_of_tile(pre, ne, len(lens), hkv, w, P, t)
                assert r[c][0] <= t < r[c][1]
        if w == 0 and T:
            sizes = [e - b for b, e in r]
            assert max(sizes) - min(sizes) <= 1


def test_partial_slots_are_unique_and_bounded(sched):
    rng = np.random.default_rng(3)
    tt = sched.shim_tile_tokens()
    for trial in range(30):
        B = int(rng.integers(1, 40))
        hkv = int(rng.choice([1, 2, 8]))
        lens = rng.integers(0, 3000, B)
        lens[rng.random(B) < 0.2] = 0
        ntiles, prefix, nonempty = make_plan(lens, hkv, tt)
        P = int(rng.integers(1, 300))
        for w in (0, 2):
            r, pre, ne = ranges(sched, prefix, nonempty, hkv, w, P)
            seen = set()
            for c, (b0, e0) in enumerate(r):
                segs = set()
                for t in range(b0, e0):
                    b = sched.shim_request_of_tile(pre, B, t)
                    assert prefix[b] <= t < prefix[b + 1]
                    h = (t - prefix[b]) // ntiles[b]
                    segs.add(b * hkv + h)
                for u in segs:
                    slot = u + c
                    assert slot not in seen
                    seen.add(slot)
                    assert slot < sched.shim_slots(B, hkv)


def test_c_caller_compiles_links_and_sees_the_documented_checks(lib, tmp_path):
    """A C11 program (tests/c_abi_check.c) includes the header, links libfd.so
    and calls the host-side entry points: the boundary is usable from C."""
    import shutil
    import subprocess
    from decode_attention_decoding_gb300 import build
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    libdir = os.path.dirname(build.LIB)
    exe = str(tmp_path / "c_abi_check")
    r = subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(root, "include"), os.path.join(root, "tests", "c_abi_check.c"),
                        "-L", libdir, "-lfd", "-Wl,-rpath," + libdir, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C ABI checks passed" in r.stdout
