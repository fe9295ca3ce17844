"""FP8 KV caches (OCP E4M3 / E5M2 codes with per-tensor dequantisation
scales): the CUDA library against the fp64 oracle on the same codes, on both
consumer paths, both layouts, fused heads, extreme query magnitudes and an
exact gather probe."""
import dataclasses

import numpy as np
import pytest
import torch

import fd_synth as syn
import oracle
from gpu_util import check, contig_to_paged, run, small_page_twin_flags

pytestmark = pytest.mark.gpu

CUDA_CORES = 0x2
NO_FUSION = 0x8
FUSE = 0x10
FMTS = ["e4m3", "e5m2"]
RAGGED = [1000, 1, 0, 63, 64, 65, 129, 700]
SCALES = (0.0371, 1.7)          # k_scale, v_scale (not powers of two)


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_attention_decoding_gb300 import build
    build.build()
    oracle.build()


def decode(codes, fmt):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2).to(torch.float64).numpy()


@pytest.mark.parametrize("flags", [0, CUDA_CORES])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("fmt", FMTS)
def test_contiguous_vs_oracle(fmt, d, group, flags):
    hkv = 2
    w = syn.make_contiguous(1600 + d + group, len(RAGGED), hkv * group, hkv, d, 1024, RAGGED,
                            kv_dtype=fmt, k_scale=SCALES[0], v_scale=SCALES[1])
    ro, rl = oracle.attend(w, threads=8)
    for ctas in (0, 7):
        o, l = run(w, num_ctas=ctas, flags=flags)
        check(o, l, ro, rl, f"{fmt} d={d} G={group} flags={flags} ctas={ctas}")


@pytest.mark.parametrize("page", [2, 8, 16, 64])
@pytest.mark.parametrize("group", [1, 4])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("fmt", FMTS)
def test_paged_vs_oracle_and_contiguous(fmt, d, group, page):
    w = syn.make_contiguous(1700 + d + page, len(RAGGED), 2 * group, 2, d, 1024, RAGGED, kv_dtype=fmt,
                            k_scale=SCALES[0], v_scale=SCALES[1])
    wp = contig_to_paged(w, page, perm_seed=page + d, poison=True)
    flags = small_page_twin_flags(w) if page < 8 else 0
    ro, rl = oracle.attend(wp, threads=8)
    for ctas in (0, 5):
        op, lp = run(wp, num_ctas=ctas)
        check(op, lp, ro, rl, f"{fmt} d={d} P={page} G={group} ctas={ctas}")
        oc, lc = run(w, num_ctas=ctas, flags=flags)
        assert np.array_equal(op, oc) and np.array_equal(lp, lc)


# (64, 1, 4) and (64, 2, 4) fuse four 64-code heads into one shared 256-byte row;
# the others pair two heads (one per warp of a pair), (128, 8, 2) included
@pytest.mark.parametrize("d,group,hkv", [(64, 1, 4), (64, 2, 4), (128, 1, 4), (128, 4, 2), (64, 4, 2),
                                         (128, 8, 2)])
@pytest.mark.parametrize("fmt", FMTS)
def test_fused_heads(fmt, d, group, hkv):
    w = syn.make_contiguous(1800 + d + group, len(RAGGED), hkv * group, hkv, d, 1024, RAGGED,
                            kv_dtype=fmt, k_scale=SCALES[0], v_scale=SCALES[1])
    ro, rl = oracle.attend(w, threads=8)
    for flags in (FUSE, NO_FUSION):
        out = torch.full((w.batch, w.num_q_heads, d), float("nan"), device="cuda")
        o, l = run(w, num_ctas=7, flags=flags, out=out)
        assert not np.isnan(o).any()
        check(o, l, ro, rl, f"{fmt} d={d} G={group} flags={flags}")


@pytest.mark.parametrize("qexp", [-40, -20, 20, 60])
@pytest.mark.parametrize("fmt", FMTS)
def test_query_magnitude_far_outside_fp16(fmt, qexp):
    """The tensor-core path converts q to fp16 after a per-head power-of-two
    scaling; queries 2^qexp times larger (bf16-exact) with the scale divided
    by the same power give the same attention."""
    w = syn.make_contiguous(1900, len(RAGGED), 8, 2, 128, 1024, RAGGED, kv_dtype=fmt,
                            k_scale=SCALES[0], v_scale=SCALES[1])
    ro, rl = oracle.attend(w, threads=8)
    big = dataclasses.replace(w, q=syn.scale_bf16_bits(w.q, 2.0 ** qexp),
                              scale=float(np.float32(w.scale * 2.0 ** -qexp)))
    for flags in (0, CUDA_CORES):
        o, l = run(big, num_ctas=7, flags=flags)
        check(o, l, ro, rl, f"{fmt} q x 2^{qexp} flags={flags}")


@pytest.mark.parametrize("fmt", FMTS)
def test_fp16_query(fmt):
    w = syn.make_contiguous(1950, len(RAGGED), 8, 2, 128, 1024, RAGGED, dtype="f16", kv_dtype=fmt,
                            k_scale=SCALES[0], v_scale=SCALES[1])
    ro, rl = oracle.attend(w, threads=8)
    for flags in (0, CUDA_CORES):
        o, l = run(w, num_ctas=7, flags=flags)
        check(o, l, ro, rl, f"{fmt} f16 q flags={flags}")


@pytest.mark.parametrize("flags", [0, CUDA_CORES])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("fmt", FMTS)
def test_bit_exact_gather(fmt, d, flags):
    """q = +-1, K[t*] = 16 q (exact in both formats), so t*'s score leads by
    more than 110 natural units; V rows hold the token's base-8 digits (exact)
    and the output must be exactly v_scale * V[t*]."""
    L, group, hkv, v_scale = 2000, 4, 2, 0.5
    w = syn.make_contiguous(1990 + d, 1, hkv * group, hkv, d, L, [L], kv_dtype=fmt, k_scale=1.0,
                            v_scale=v_scale)
    signs = np.where(syn.normal_bf16(7, (hkv, d)).view(np.int16) < 0, -1.0, 1.0)
    w.q[0] = np.repeat(syn.f64_to_bf16_bits(signs), group, axis=0)
    t = np.arange(L)
    for t_star in (0, 63, 64, 1023, L - 1):
        k, v = w.k.copy(), w.v.copy()
        for g in range(hkv):
            k[0, t_star, g] = syn.f64_to_fp8_bits(16.0 * signs[g], fmt)
            for j in range(4):
                v[0, :, g, j] = syn.f64_to_fp8_bits(((t >> (3 * j)) & 7).astype(np.float64), fmt)
        wt = dataclasses.replace(w, k=k, v=v)
        s = w.scale * decode(k[0, :, :], fmt) @ signs.T       # [L, hkv, hkv]
        for g in range(hkv):
            sg = s[:, g, g]
            assert sg[t_star] - np.delete(sg, t_star).max() > 110, "probe margin too small"
        o, _ = run(wt, num_ctas=7, flags=flags)
        for h in range(hkv * group):
            g = h // group
            assert np.array_equal(o[0, h], v_scale * decode(v[0, t_star, g], fmt)), (t_star, h)
            assert sum(int(o[0, h, j] / v_scale) << (3 * j) for j in range(4)) == t_star


def test_one_token_fp8_pages_of_head_dim_64_are_rejected_before_launch():
    """64-byte page boxes would miss the 128-byte TMA alignment: the host refuses them."""
    import decode_attention_decoding_gb300 as fd
    w = syn.make_contiguous(2000, 2, 4, 2, 64, 64, [10, 64], kv_dtype="e4m3")
    wp = contig_to_paged(w, 1, perm_seed=1)
    with pytest.raises(fd.FdError) as e:
        run(wp)
    assert e.value.status == fd.FD_ERR_UNSUPPORTED
    w128 = syn.make_contiguous(2001, 2, 4, 2, 128, 64, [10, 64], kv_dtype="e4m3")
    wp = contig_to_paged(w128, 1, perm_seed=1)
    ro, rl = oracle.attend(wp)
    o, l = run(wp)
    check(o, l, ro, rl, "e4m3 d=128 P=1")
