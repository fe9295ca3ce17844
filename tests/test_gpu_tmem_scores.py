"""Scores on the tcgen05 tensor cores (FD_FLAG_TMEM_SCORES): FP8 caches (E4M3
and E5M2) with paired kv heads of 128 dims, the score MMAs reading the FP8 K
tile and the query split into two to four parts of the same format from
shared memory into tensor memory.  The
CUDA library against the fp64 oracle: contiguous and paged (poisoned)
layouts (pages under 64 tokens keep the warp MMAs), ragged lengths, every
column count the path takes, several new tokens (causal), fp16 queries,
extreme query magnitudes, split counts, and the full-size workloads."""
import dataclasses

import numpy as np
import pytest
import torch

import fd_synth as syn
import oracle
from gpu_util import check, contig_to_paged, run

pytestmark = pytest.mark.gpu

FUSE = 0x10
TMEM = 0x80
NO_TMEM = 0x100
RAGGED = [1000, 1, 0, 63, 64, 65, 129, 700, 2049]
FMTS = ["e4m3", "e5m2"]
SCALES = (0.0371, 1.7)          # k_scale, v_scale (not powers of two)


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_attention_decoding_gb300 import build
    build.build()
    oracle.build()


def workload(seed, group, hkv=2, q_len=1, dtype="bf16", lens=RAGGED, s_max=2112, fmt="e4m3"):
    return syn.make_contiguous(seed, len(lens), hkv * group, hkv, 128, s_max, lens, dtype=dtype, kv_dtype=fmt,
                               k_scale=SCALES[0], v_scale=SCALES[1], q_len=q_len)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("hkv", [2, 4])
def test_contiguous_vs_oracle(group, hkv, fmt):
    w = workload(2100 + 10 * group + hkv, group, hkv, fmt=fmt)
    ro, rl = oracle.attend(w, threads=8)
    for ctas in (0, 1, 7, 40):
        o, l = run(w, num_ctas=ctas, flags=FUSE | TMEM)
        check(o, l, ro, rl, f"TMEM scores {fmt} G={group} hkv={hkv} ctas={ctas}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_default_choice(group, fmt):
    """Paired E4M3 heads take the tcgen05 scores by default for up to 4
    columns per kv head (on calls of at least 24 paired tiles per CTA: here
    two CTAs) and the warp MMAs above: the default launch equals the forced
    one bit for bit and differs from the other (the scores come from another
    unit, summed in another order); all match the oracle."""
    w = workload(2150 + group, group, fmt=fmt)
    ro, rl = oracle.attend(w, threads=8)
    runs = {name: run(w, num_ctas=2, flags=FUSE | f) for name, f in (("default", 0), ("tmem", TMEM),
                                                                      ("warp", NO_TMEM))}
    for name, (o, l) in runs.items():
        check(o, l, ro, rl, f"G={group} {name}")
    same, other = ("tmem", "warp") if group <= 4 else ("warp", "tmem")
    assert np.array_equal(runs["default"][0], runs[same][0]) and np.array_equal(runs["default"][1], runs[same][1])
    assert not np.array_equal(runs["default"][0], runs[other][0])
    # a shorter call (7 CTAs, under 24 paired tiles each): the warp MMAs by default
    o, l = run(w, num_ctas=7, flags=FUSE)
    assert np.array_equal(o, run(w, num_ctas=7, flags=FUSE | NO_TMEM)[0])
    # both flags: the warp MMAs
    o, l = run(w, num_ctas=2, flags=FUSE | TMEM | NO_TMEM)
    assert np.array_equal(o, runs["warp"][0]) and np.array_equal(l, runs["warp"][1])


@pytest.mark.parametrize("fmt", FMTS)
def test_bit_exact_gather(fmt):
    """q = +-1 and K[t*] = 16 q (exact in E4M3 and in the query parts), so t*'s
    score leads by more than 110 natural units; V rows hold the token's
    base-8 digits (exact) and the output must be exactly v_scale * V[t*]."""
    L, group, hkv, v_scale = 2000, 4, 2, 0.5
    w = syn.make_contiguous(2160, 1, hkv * group, hkv, 128, L, [L], kv_dtype=fmt, k_scale=1.0,
                            v_scale=v_scale)
    signs = np.where(syn.normal_bf16(7, (hkv, 128)).view(np.int16) < 0, -1.0, 1.0)
    w.q[0] = np.repeat(syn.f64_to_bf16_bits(signs), group, axis=0)
    t = np.arange(L)
    for t_star in (0, 63, 64, 1023, L - 1):
        k, v = w.k.copy(), w.v.copy()
        for g in range(hkv):
            k[0, t_star, g] = syn.f64_to_fp8_bits(16.0 * signs[g], fmt)
            for j in range(4):
                v[0, :, g, j] = syn.f64_to_fp8_bits(((t >> (3 * j)) & 7).astype(np.float64), fmt)
        wt = dataclasses.replace(w, k=k, v=v)
        f8 = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
        kf = torch.from_numpy(np.ascontiguousarray(k[0])).view(f8).to(torch.float64).numpy()
        s = w.scale * kf @ signs.T       # [L, hkv, hkv]
        for g in range(hkv):
            sg = s[:, g, g]
            assert sg[t_star] - np.delete(sg, t_star).max() > 110, "probe margin too small"
        o, _ = run(wt, num_ctas=7, flags=FUSE | TMEM)
        vf = torch.from_numpy(np.ascontiguousarray(v[0, t_star])).view(f8).to(torch.float64)
        for h in range(hkv * group):
            g = h // group
            assert np.array_equal(o[0, h], v_scale * vf[g].numpy()), (t_star, h)
            assert sum(int(o[0, h, j] / v_scale) << (3 * j) for j in range(4)) == t_star


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("page", [8, 16, 64, 128, 256])
@pytest.mark.parametrize("group", [4, 8])
def test_paged_vs_oracle(page, group, fmt):
    w = workload(2200 + page + group, group, fmt=fmt)
    wp = contig_to_paged(w, page, perm_seed=page + group, poison=True)
    ro, rl = oracle.attend(wp, threads=8)
    for ctas in (0, 5):
        o, l = run(wp, num_ctas=ctas, flags=FUSE | TMEM)
        check(o, l, ro, rl, f"TMEM scores P={page} G={group} ctas={ctas}")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("group,q_len", [(1, 2), (2, 4), (4, 2), (1, 8)])
def test_several_new_tokens(group, q_len, fmt):
    w = workload(2300 + 10 * group + q_len, group, q_len=q_len, fmt=fmt)
    ro, rl = oracle.attend(w, threads=8)
    for ctas in (0, 7):
        o, l = run(w, num_ctas=ctas, flags=FUSE | TMEM)
        check(o, l, ro, rl, f"TMEM scores G={group} q_len={q_len} ctas={ctas}")


@pytest.mark.parametrize("fmt", FMTS)
def test_fp16_query(fmt):
    w = workload(2400, 4, dtype="f16", fmt=fmt)
    ro, rl = oracle.attend(w, threads=8)
    o, l = run(w, num_ctas=7, flags=FUSE | TMEM)
    check(o, l, ro, rl, f"TMEM scores {fmt}, fp16 q")


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("qexp", [-40, -20, 20, 60])
def test_query_magnitude(qexp, fmt):
    """Queries 2^qexp times larger (bf16-exact) with the scale divided by the
    same power give the same attention: the per-column power-of-two scaling
    of the E4M3 query parts follows the query's range."""
    w = workload(2500, 4, fmt=fmt)
    ro, rl = oracle.attend(w, threads=8)
    big = dataclasses.replace(w, q=syn.scale_bf16_bits(w.q, 2.0 ** qexp),
                              scale=float(np.float32(w.scale * 2.0 ** -qexp)))
    o, l = run(big, num_ctas=7, flags=FUSE | TMEM)
    check(o, l, ro, rl, f"TMEM scores, q x 2^{qexp}")


@pytest.mark.parametrize("fmt", FMTS)
def test_query_with_small_elements(fmt):
    """Query rows whose elements span 2^-20 .. 2^7 of the row's largest (the
    small ones fall below the E4M3 parts' exact range) still match the oracle."""
    w = workload(2550, 4, fmt=fmt)
    q = syn.bf16_bits_to_f64(w.q)
    expo = np.arange(q.shape[-1]) % 28 - 20
    q = np.sign(q) * np.maximum(np.abs(q), 0.5) * 2.0 ** expo
    w = dataclasses.replace(w, q=syn.f64_to_bf16_bits(q), scale=float(np.float32(w.scale * 2.0 ** -7)))
    ro, rl = oracle.attend(w, threads=8)
    o, l = run(w, num_ctas=7, flags=FUSE | TMEM)
    check(o, l, ro, rl, "TMEM scores, wide query range")


@pytest.mark.parametrize("config_id,fmt", [(2, "e4m3"), (3, "e4m3"), (4, "e4m3"), (5, "e4m3"), (2, "e5m2"),
                                           (5, "e5m2")])
def test_full_size_workloads(config_id, fmt):
    """The E4M3 benchmark workloads at full size, every query row, with the
    tcgen05 scores wherever they apply (workload 4's 16-token pages keep the
    warp MMAs; its default-flag run is in the full-size configuration tests)."""
    w = syn.make_config(config_id, kv_dtype=fmt)
    ro, rl = oracle.attend(w, threads=16)
    o, l = run(w, flags=TMEM)
    stats = check(o, l, ro, rl, f"config {config_id} {fmt} TMEM scores")
    print(f"config {config_id} kv={fmt} TMEM scores: max|dO|={stats[0]:.3g} max rel(|r|>=1e-2)={stats[1]:.3g} "
          f"max|dLSE|={stats[2]:.3g}")
