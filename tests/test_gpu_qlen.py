"""Several new query tokens per request (q_len > 1) under the causal mask:
new token i of a request with cache length L sees positions 0 .. L - q_len + i.
The CUDA library against the fp64 oracle on both consumer paths, both layouts,
fused heads and FP8 caches, plus an exact causal gather probe."""
import dataclasses

import numpy as np
import pytest
import torch

import fd_synth as syn
import oracle
from gpu_util import check, contig_to_paged, run, small_page_twin_flags

pytestmark = pytest.mark.gpu

CUDA_CORES = 0x2
FUSE = 0x10
NO_FUSION = 0x8
# lengths include requests shorter than q_len (rows that see no position)
LENS = [1000, 1, 0, 2, 63, 64, 65, 129, 700]


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_attention_decoding_gb300 import build
    build.build()
    oracle.build()


@pytest.mark.parametrize("flags", [0, CUDA_CORES])
@pytest.mark.parametrize("group,q_len", [(1, 2), (1, 3), (1, 8), (2, 2), (2, 4), (4, 2), (3, 2), (1, 5)])
def test_contiguous_vs_oracle(group, q_len, flags):
    hkv = 2
    w = syn.make_contiguous(2100 + 10 * group + q_len, len(LENS), hkv * group, hkv, 128, 1024, LENS,
                            q_len=q_len)
    ro, rl = oracle.attend(w, threads=8)
    for ctas in (0, 7):
        out = torch.full(w.q.shape, float("nan"), device="cuda")
        o, l = run(w, num_ctas=ctas, flags=flags, out=out)
        assert o.shape == ro.shape and not np.isnan(o).any()
        check(o, l, ro, rl, f"G={group} q_len={q_len} flags={flags} ctas={ctas}")


# over 8 query columns per kv head: two n8 tiles on the tensor-core consumers
# (GQA-8 with two new tokens, MHA with up to 16, GQA-16 with one, padded counts)
@pytest.mark.parametrize("d,group,q_len", [(128, 8, 2), (128, 1, 16), (128, 1, 9), (128, 4, 3), (128, 16, 1),
                                           (64, 8, 2), (64, 1, 16), (256, 8, 2), (256, 1, 12)])
def test_sixteen_columns(d, group, q_len):
    w = syn.make_contiguous(2150 + d + 10 * group + q_len, len(LENS), 2 * group, 2, d, 1024, LENS, q_len=q_len)
    ro, rl = oracle.attend(w, threads=8)
    for flags, ctas in ((0, 0), (0, 7), (NO_FUSION, 7), (FUSE, 7)):
        out = torch.full(w.q.shape, float("nan"), device="cuda")
        o, l = run(w, num_ctas=ctas, flags=flags, out=out)
        assert not np.isnan(o).any()
        check(o, l, ro, rl, f"d={d} G={group} q_len={q_len} flags={flags} ctas={ctas}")


# pages of 1 and 4 tokens: rows copied with cp.async into the tensor-core tiles
@pytest.mark.parametrize("page", [1, 4, 8, 16, 128])
def test_sixteen_columns_paged(page):
    w = syn.make_contiguous(2170 + page, len(LENS), 16, 2, 128, 1024, LENS, q_len=2)
    wp = contig_to_paged(w, page, perm_seed=page, poison=True)
    ro, rl = oracle.attend(wp, threads=8)
    for ctas in (0, 5):
        op, lp = run(wp, num_ctas=ctas)
        check(op, lp, ro, rl, f"P={page} G=8 q_len=2 ctas={ctas}")
        oc, lc = run(w, num_ctas=ctas)
        assert np.array_equal(op, oc) and np.array_equal(lp, lc)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("d", [64, 128])
def test_sixteen_columns_fp8(fmt, d):
    """FP8 heads of 64 dims are paired so their rows reach 128 bytes."""
    w = syn.make_contiguous(2180 + d, len(LENS), 16, 2, d, 1024, LENS, q_len=2, kv_dtype=fmt, k_scale=0.05,
                            v_scale=0.7)
    ro, rl = oracle.attend(w, threads=8)
    for flags in ((0, FUSE) if d == 64 else (0, NO_FUSION, FUSE)):
        o, l = run(w, num_ctas=7, flags=flags)
        check(o, l, ro, rl, f"{fmt} d={d} G=8 q_len=2 flags={flags}")


def test_sixteen_columns_need_tensor_cores():
    import decode_attention_decoding_gb300 as fd
    w = syn.make_contiguous(2190, 2, 16, 2, 128, 64, [10, 64], q_len=2)
    with pytest.raises(fd.FdError) as e:
        run(w, flags=CUDA_CORES)
    assert e.value.status == fd.FD_ERR_UNSUPPORTED


@pytest.mark.parametrize("d", [64, 256])
@pytest.mark.parametrize("group,q_len", [(1, 4), (4, 2)])
def test_head_dims(d, group, q_len):
    w = syn.make_contiguous(2200 + d + q_len, len(LENS), 2 * group, 2, d, 1024, LENS, q_len=q_len)
    ro, rl = oracle.attend(w, threads=8)
    for flags in (0, CUDA_CORES):
        o, l = run(w, num_ctas=7, flags=flags)
        check(o, l, ro, rl, f"d={d} G={group} q_len={q_len} flags={flags}")


@pytest.mark.parametrize("page", [4, 16, 64])
@pytest.mark.parametrize("group,q_len", [(1, 4), (2, 2)])
def test_paged_vs_oracle_and_contiguous(group, q_len, page):
    w = syn.make_contiguous(2300 + page + q_len, len(LENS), 2 * group, 2, 128, 1024, LENS, q_len=q_len)
    wp = contig_to_paged(w, page, perm_seed=page, poison=True)
    flags = small_page_twin_flags(w) if page < 8 else 0
    ro, rl = oracle.attend(wp, threads=8)
    for ctas in (0, 5):
        op, lp = run(wp, num_ctas=ctas)
        check(op, lp, ro, rl, f"P={page} G={group} q_len={q_len}")
        oc, lc = run(w, num_ctas=ctas, flags=flags)
        assert np.array_equal(op, oc) and np.array_equal(lp, lc)


@pytest.mark.parametrize("d,group,q_len,hkv", [(64, 1, 2, 4), (128, 2, 2, 2), (128, 1, 4, 2), (64, 2, 2, 2)])
def test_fused_heads(d, group, q_len, hkv):
    w = syn.make_contiguous(2400 + d + q_len, len(LENS), hkv * group, hkv, d, 1024, LENS, q_len=q_len)
    ro, rl = oracle.attend(w, threads=8)
    for flags in (FUSE, NO_FUSION):
        out = torch.full(w.q.shape, float("nan"), device="cuda")
        o, l = run(w, num_ctas=7, flags=flags, out=out)
        assert not np.isnan(o).any()
        check(o, l, ro, rl, f"d={d} G={group} q_len={q_len} flags={flags}")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_cache(fmt):
    w = syn.make_contiguous(2500, len(LENS), 4, 2, 128, 1024, LENS, q_len=3, kv_dtype=fmt, k_scale=0.05,
                            v_scale=0.7)
    ro, rl = oracle.attend(w, threads=8)
    for flags in (0, CUDA_CORES, FUSE):
        o, l = run(w, num_ctas=7, flags=flags)
        check(o, l, ro, rl, f"{fmt} q_len=3 flags={flags}")


@pytest.mark.parametrize("flags", [0, CUDA_CORES])
@pytest.mark.parametrize("group,q_len", [(1, 8), (2, 4), (4, 2), (8, 2), (1, 16), (4, 3)])
def test_causal_gather_probe(group, q_len, flags):
    """Key at position L - q_len + j is 2^(4+j) q (q = +-1): every new token's
    largest visible score is its own position by more than 110 natural
    units, and V rows encode their position, so new token i must return
    exactly V[L - q_len + i]; seeing a later position would return another."""
    if flags == CUDA_CORES and group * q_len > 8:
        pytest.skip("over 8 columns run on the tensor-core consumers only")
    L, hkv, d = 1500, 2, 128
    w = syn.make_contiguous(2600 + group, 1, hkv * group, hkv, d, L, [L], q_len=q_len)
    signs = np.where(syn.normal_bf16(9, (hkv, d)).view(np.int16) < 0, -1.0, 1.0)
    qrow = np.repeat(syn.f64_to_bf16_bits(signs), group, axis=0)      # [Hq, D]
    w.q[0] = np.broadcast_to(qrow, (q_len,) + qrow.shape)
    t = np.arange(L)
    for g in range(hkv):
        for j in range(q_len):
            w.k[0, L - q_len + j, g] = syn.f64_to_bf16_bits(2.0 ** (4 + j) * signs[g])
        w.v[0, :, g, 0] = syn.f64_to_bf16_bits((t >> 8).astype(np.float64))
        w.v[0, :, g, 1] = syn.f64_to_bf16_bits((t & 255).astype(np.float64))
    K = syn.bf16_bits_to_f64(w.k[0])
    for g in range(hkv):
        s = w.scale * K[:, g] @ signs[g]
        for i in range(q_len):
            vis = s[:L - q_len + i + 1]
            assert vis[-1] - np.max(vis[:-1]) > 110, "probe margin too small"
    o, l = run(w, num_ctas=7, flags=flags)
    for i in range(q_len):
        for h in range(hkv * group):
            pos = L - q_len + i
            assert np.array_equal(o[0, i, h], syn.bf16_bits_to_f64(w.v[0, pos, h // group])), (i, h)
            assert o[0, i, h, 0] * 256 + o[0, i, h, 1] == pos
