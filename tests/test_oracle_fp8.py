"""Pins for the oracle's FP8 KV cache (OCP E4M3 / E5M2 codes with per-tensor
dequantisation scales).  No GPU, no CUDA library.

The decoders are checked code by code against PyTorch's own float8 types (a
library routine independent of the C oracle); the attention over an FP8
cache against the already-pinned 16-bit path on exactly re-encoded values,
against multi-precision brute force, and against closed forms.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import fd_synth as syn
import oracle

mpmath = pytest.importorskip("mpmath")

TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
FMTS = ["e4m3", "e5m2"]


def decode(codes, fmt):
    """FP8 codes -> fp64 through PyTorch's float8 dtype."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(TORCH_FP8[fmt]).to(torch.float64).numpy()


def fp8_workload(q, k8, v8, lens, hq, hkv, scale, fmt, k_scale=1.0, v_scale=1.0, dtype="bf16"):
    return syn.Workload("fp8", q, k8, v8, np.asarray(lens, np.int32), hq, hkv, q.shape[-1], scale,
                        dtype=dtype, kv_dtype=fmt, k_scale=k_scale, v_scale=v_scale)


@pytest.mark.parametrize("fmt", FMTS)
def test_every_value_code_decodes_as_the_format_defines(fmt):
    """L = 1 gives O = v_scale * V_0 exactly: a 256-dim V row holding every
    code reads back as PyTorch decodes it (NaN codes as NaN, E5M2 infinities
    as infinities)."""
    d = 256
    codes = np.arange(256, dtype=np.uint8)
    q = syn.normal_bf16(1, (1, 1, d))
    k8 = np.zeros((1, 1, 1, d), np.uint8)
    v8 = codes.reshape(1, 1, 1, d)
    w = fp8_workload(q, k8, v8, [1], 1, 1, 0.1, fmt, v_scale=1.0)
    o, lse = oracle.attend(w)
    ref = decode(codes, fmt)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isnan(o[0, 0]), np.isnan(ref))
    assert np.array_equal(o[0, 0][~np.isnan(ref)], ref[~np.isnan(ref)])
    assert lse[0, 0] == 0.0          # a zero key row gives score 0
    # landmarks of the formats, written out
    if fmt == "e4m3":
        assert (ref[0x38], ref[0x7E], ref[0x01], ref[0x08], ref[0xB8]) == (1.0, 448.0, 2 ** -9, 2 ** -6, -1.0)
        assert fin.sum() == 254      # only S.1111.111 is NaN, no infinities
    else:
        assert (ref[0x3C], ref[0x7B], ref[0x01], ref[0x04]) == (1.0, 57344.0, 2 ** -16, 2 ** -14)
        assert np.isinf(ref[0x7C]) and np.isinf(ref[0xFC]) and fin.sum() == 248


@pytest.mark.parametrize("fmt", FMTS)
def test_every_key_code_decodes_as_the_format_defines(fmt):
    """One-hot queries read single K elements: with L = 1 the LSE is the
    score scale * k_scale * K_0[j] for query head j."""
    d = hq = 256
    codes = np.arange(256, dtype=np.uint8)
    # non-finite codes would make every 0 * K_j product NaN; the V test covers them
    codes[~np.isfinite(decode(codes, fmt))] = 0
    q = syn.f64_to_bf16_bits(np.eye(d)).reshape(1, hq, d)
    k8 = codes.reshape(1, 1, 1, d)
    v8 = np.zeros((1, 1, 1, d), np.uint8)
    k_scale = 2.0 ** -3
    w = fp8_workload(q, k8, v8, [1], hq, 1, 0.5, fmt, k_scale=k_scale)
    _, lse = oracle.attend(w)
    assert np.array_equal(lse[0], 0.5 * k_scale * decode(codes, fmt))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("layout", ["contig", "paged"])
def test_fp8_equals_16_bit_path_on_exactly_reencoded_values(fmt, layout):
    """With power-of-two scales every dequantised value is a bf16 value, so the
    FP8 cache and its bf16 re-encoding give bitwise identical results."""
    lens = [1, 17, 70, 0, 129]
    k_scale, v_scale = 2.0 ** -4, 2.0 ** -2
    w8 = syn.make_contiguous(301, len(lens), 8, 2, 128, 129, lens, kv_dtype=fmt,
                             k_scale=k_scale, v_scale=v_scale)
    kb = syn.f64_to_bf16_bits(decode(w8.k, fmt) * k_scale)
    vb = syn.f64_to_bf16_bits(decode(w8.v, fmt) * v_scale)
    w16 = dataclasses.replace(w8, k=kb, v=vb, kv_dtype=None, k_scale=1.0, v_scale=1.0)
    if layout == "paged":
        w8, w16 = paged(w8, 16, 5), paged(w16, 16, 5)
    o8, l8 = oracle.attend(w8)
    o16, l16 = oracle.attend(w16)
    assert np.array_equal(o8, o16) and np.array_equal(l8, l16)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("L", [1, 5, 64, 65])
def test_fp8_brute_force_with_arbitrary_scales(fmt, L):
    """Non-power-of-two scales: against 40-digit brute force on the decoded,
    scaled values (k_scale enters the scores only, v_scale the output only)."""
    k_scale, v_scale = syn.fp32(0.0371), syn.fp32(1.7)
    w = syn.make_contiguous(310 + L, 1, 2, 1, 128, L, [L], kv_dtype=fmt, k_scale=k_scale,
                            v_scale=v_scale)
    o, lse = oracle.attend(w)
    K = decode(w.k[0, :L, 0], fmt) * k_scale
    V = decode(w.v[0, :L, 0], fmt) * v_scale
    for h in range(2):
        ro, rl = mp_attention(syn.bf16_bits_to_f64(w.q[0, h]), K, V, w.scale)
        np.testing.assert_allclose(o[0, h], ro, rtol=1e-12, atol=1e-14)
        assert lse[0, h] == pytest.approx(rl, rel=1e-13, abs=1e-13)


@pytest.mark.parametrize("fmt", FMTS)
def test_identical_fp8_keys_give_scaled_mean_of_values(fmt):
    L, d = 37, 64
    q = syn.normal_bf16(2, (1, 1, d))
    row = syn.f64_to_fp8_bits(np.linspace(-3, 3, d), fmt)
    k8 = np.broadcast_to(row, (1, L, 1, d)).copy()
    v8 = syn.normal_fp8(3, (1, L, 1, d), fmt, 0.25)
    w = fp8_workload(q, k8, v8, [L], 1, 1, 0.125, fmt, k_scale=0.5, v_scale=0.25)
    o, lse = oracle.attend(w)
    mean = decode(v8[0, :, 0], fmt).mean(axis=0) * 0.25
    np.testing.assert_allclose(o[0, 0], mean, rtol=1e-13, atol=1e-15)
    s = 0.125 * math.fsum(syn.bf16_bits_to_f64(q[0, 0]) * 0.5 * decode(row, fmt))
    assert lse[0, 0] == pytest.approx(s + math.log(L), rel=1e-13)


@pytest.mark.parametrize("fmt", FMTS)
def test_fp8_paged_equals_contiguous_and_skips_poison(fmt):
    lens = [3, 64, 0, 200]
    w = syn.make_contiguous(320, len(lens), 4, 2, 128, 200, lens, kv_dtype=fmt, k_scale=0.05,
                            v_scale=0.3)
    o, lse = oracle.attend(w)
    op, lp = oracle.attend(paged(w, 8, 2, poison=True))
    assert np.array_equal(o, op) and np.array_equal(lse, lp)


def test_fp16_query_with_fp8_cache():
    """q's element type and the cache's are independent."""
    L = 9
    w = syn.make_contiguous(330, 1, 2, 1, 128, L, [L], dtype="f16", kv_dtype="e4m3", k_scale=0.1,
                            v_scale=0.2)
    o, lse = oracle.attend(w)
    K = decode(w.k[0, :L, 0], "e4m3") * w.k_scale
    V = decode(w.v[0, :L, 0], "e4m3") * w.v_scale
    for h in range(2):
        ro, rl = mp_attention(syn.f16_bits_to_f64(w.q[0, h]), K, V, w.scale)
        np.testing.assert_allclose(o[0, h], ro, rtol=1e-12, atol=1e-14)
        assert lse[0, h] == pytest.approx(rl, rel=1e-13, abs=1e-13)


# ---------------------------------------------------------------------------

def mp_attention(qrow, K, V, scale):
    """One query row in 40-digit arithmetic on fp64 inputs."""
    mp = mpmath.mp
    mp.dps = 40
    qs = [mp.mpf(float(x)) for x in qrow]
    s = [mp.mpf(scale) * mp.fsum(a * mp.mpf(float(b)) for a, b in zip(qs, krow)) for krow in K]
    m = max(s)
    e = [mp.e ** (x - m) for x in s]
    z = mp.fsum(e)
    o = [mp.fsum(ei * mp.mpf(float(vr[j])) for ei, vr in zip(e, V)) / z for j in range(len(qrow))]
    return np.array([float(x) for x in o]), float(m + mp.log(z))


def paged(w, page, perm_seed, poison=False):
    """The workload's cache in shuffled pages; unused slots hold NaN codes when poisoned."""
    B, S, hkv, d = w.k.shape
    lens = w.seq_lens
    used = sum((int(L) + page - 1) // page for L in lens)
    n_pages = used + 3
    perm = syn.permutation(perm_seed, n_pages)
    table = syn.build_block_table(lens, page, max(1, (S + page - 1) // page), perm)
    fp8 = w.kv_dtype in ("e4m3", "e5m2")
    fill = (np.uint8(0x7F) if fp8 else syn.BF16_NAN) if poison else 0
    kp = np.full((n_pages, page, hkv, d), fill, w.k.dtype)
    vp = np.full((n_pages, page, hkv, d), fill, w.v.dtype)
    for b in range(B):
        for t in range(int(lens[b])):
            kp[table[b, t // page], t % page] = w.k[b, t]
            vp[table[b, t // page], t % page] = w.v[b, t]
    return dataclasses.replace(w, k=kp, v=vp, page_size=page, block_table=table)
