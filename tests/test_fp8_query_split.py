"""The split of a 16-bit query into FP8 parts that the tcgen05 score path
multiplies against an FP8 key tile: with x = q 2^-sh (the column's largest
|x| in [128, 256)), part 0 = FP8(x) and part k+1 = FP8(R r_k) of the scaled
remainder (R = 16 for E4M3, 8 for E5M2), the parts reproduce every bf16
query exactly with 2 (E4M3) or 3 (E5M2) parts and every fp16 query with 3 or
4, for elements within 2^13 of the column's largest; smaller elements are
off by under 2^-21 of the largest.  Host arithmetic only (torch's float8
casts round to nearest even, as the kernel's cvt does); no GPU."""
import numpy as np
import pytest
import torch

PARTS = {("e4m3", "bf16"): 2, ("e4m3", "f16"): 3, ("e5m2", "bf16"): 3, ("e5m2", "f16"): 4}
RADIX = {"e4m3": 16.0, "e5m2": 8.0}
F8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
F16 = {"bf16": torch.bfloat16, "f16": torch.float16}


def split(x, fmt, n):
    """The parts of fp32 x (already scaled), as fp64 values."""
    parts, v = [], torch.from_numpy(x.astype(np.float32))
    for _ in range(n):
        p = v.to(F8[fmt]).to(torch.float32)
        parts.append(p.double().numpy())
        v = (v - p) * RADIX[fmt]   # exact in fp32
    return parts


def column_scale(q):
    """2^-sh with the column's largest |q 2^-sh| in [128, 256)."""
    amax = np.abs(q).max()
    e = int(np.floor(np.log2(amax)))
    return 2.0 ** -(e - 7)


@pytest.mark.parametrize("fmt,qtype", sorted(PARTS))
def test_split_reproduces_the_query(fmt, qtype):
    rng = np.random.default_rng(7)
    n = PARTS[(fmt, qtype)]
    for trial in range(200):
        # a query row of 128 dims: N(0, 1) scaled by a random power of two,
        # with a spread of element magnitudes
        lo, hi = (-12, 12) if qtype == "bf16" else (-6, 7)   # fp16: stay under its 65504
        raw = rng.standard_normal(128) * 2.0 ** rng.integers(lo, hi) * 2.0 ** rng.integers(-4, 5, 128)
        q = torch.from_numpy(raw).to(F16[qtype]).double().numpy()
        if not np.any(q):
            continue
        s = column_scale(q)
        x = q * s
        assert 128 <= np.abs(x).max() < 256
        parts = split(x, fmt, n)
        back = sum(p * RADIX[fmt] ** -k for k, p in enumerate(parts))
        big = np.abs(x) >= np.abs(x).max() * 2.0 ** -13
        assert np.array_equal(back[big], x[big]), (trial, np.abs(back - x)[big].max())
        assert np.abs(back - x).max() <= np.abs(x).max() * 2.0 ** -21


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_one_part_fewer_is_not_enough(fmt):
    """The part counts are the smallest that work: one part fewer leaves some
    bf16 value inexact (a planted shortfall the test above would catch)."""
    rng = np.random.default_rng(11)
    n = PARTS[(fmt, "bf16")] - 1
    raw = rng.standard_normal(4096)
    q = torch.from_numpy(raw).to(torch.bfloat16).double().numpy()
    x = q * column_scale(q)
    back = sum(p * RADIX[fmt] ** -k for k, p in enumerate(split(x, fmt, n)))
    big = np.abs(x) >= np.abs(x).max() * 2.0 ** -13
    assert not np.array_equal(back[big], x[big])
