"""Head dimensions 64 and 256 (besides 128): the CUDA library against the
fp64 oracle on both consumer paths and both KV layouts, the two tensor-map
box layouts against each other, and the bit-exact gather probe.

A head_dim of 64 gives 128-byte rows (one swizzled part, 8 lanes per row on
CUDA cores); 256 gives 512-byte rows (four swizzled parts, one row per warp
step on CUDA cores, 16 k-steps per tensor-core score)."""
import numpy as np
import pytest

import fd_synth as syn
import oracle
from gpu_util import check, contig_to_paged, run, small_page_twin_flags

pytestmark = pytest.mark.gpu

CUDA_CORES = 0x2      # FD_FLAG_CUDA_CORES
NO_4D = 0x4           # FD_FLAG_NO_4D_BOXES: one TMA box per 64-dim part
RAGGED = [1000, 1, 0, 63, 64, 65, 129, 700]


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_attention_decoding_gb300 import build
    build.build()
    oracle.build()


@pytest.mark.parametrize("flags", [0, CUDA_CORES])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("d", [64, 256])
def test_contiguous_vs_oracle(d, group, flags):
    hkv = 2
    w = syn.make_contiguous(900 + d + group, len(RAGGED), hkv * group, hkv, d, 1024, RAGGED)
    ro, rl = oracle.attend(w, threads=8)
    for ctas in (0, 7):
        o, l = run(w, num_ctas=ctas, flags=flags)
        check(o, l, ro, rl, f"d={d} G={group} flags={flags} ctas={ctas}")


@pytest.mark.parametrize("page", [1, 8, 16, 128])
@pytest.mark.parametrize("group", [1, 4])
@pytest.mark.parametrize("d", [64, 256])
def test_paged_vs_oracle_and_contiguous(d, page, group):
    w = syn.make_contiguous(950 + d + page, len(RAGGED), 2 * group, 2, d, 1024, RAGGED)
    wp = contig_to_paged(w, page, perm_seed=page + d, poison=True)
    # pages under 8 tokens take unfused consumers (tensor cores for GQA)
    flags = small_page_twin_flags(w) if page < 8 else 0
    ro, rl = oracle.attend(wp, threads=8)
    for ctas in (0, 5):
        op, lp = run(wp, num_ctas=ctas)
        check(op, lp, ro, rl, f"d={d} paged P={page} G={group} ctas={ctas}")
        # same logical data, tiles and consumers: bitwise identical to the contiguous call
        oc, lc = run(w, num_ctas=ctas, flags=flags)
        assert np.array_equal(op, oc) and np.array_equal(lp, lc)


@pytest.mark.parametrize("page", [0, 8, 32])
@pytest.mark.parametrize("d", [64, 256])
def test_tensor_core_box_layouts_agree(d, page):
    """4-D boxes (every 64-dim part in one box) and 3-D boxes (one per part)
    fill the same swizzled tile, so the results are bitwise identical."""
    w = syn.make_contiguous(970 + d, len(RAGGED), 8, 2, d, 1024, RAGGED)
    if page:
        w = contig_to_paged(w, page, perm_seed=d + page, poison=True)
    a = run(w, num_ctas=11)
    b = run(w, num_ctas=11, flags=NO_4D)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    ro, rl = oracle.attend(w, threads=8)
    check(a[0], a[1], ro, rl, f"d={d} P={page}")


@pytest.mark.parametrize("d", [64, 256])
def test_long_request_many_splits(d):
    """One long request split over many CTAs, next to short ones."""
    lens = [9000, 3, 4097]
    w = syn.make_contiguous(990 + d, len(lens), 16, 2, d, 9000, lens)
    ro, rl = oracle.attend(w, threads=8)
    for flags in (0, CUDA_CORES):
        for ctas in (0, 37):
            o, l = run(w, num_ctas=ctas, flags=flags)
            check(o, l, ro, rl, f"d={d} long flags={flags} ctas={ctas}")


@pytest.mark.parametrize("d", [64, 256])
def test_f16_inputs(d):
    w = syn.make_contiguous(995 + d, len(RAGGED), 8, 2, d, 1024, RAGGED, dtype="f16")
    ro, rl = oracle.attend(w, threads=8)
    for flags in (0, CUDA_CORES):
        o, l = run(w, num_ctas=7, flags=flags)
        check(o, l, ro, rl, f"f16 d={d} flags={flags}")


@pytest.mark.parametrize("flags", [0, CUDA_CORES])
@pytest.mark.parametrize("d", [64, 256])
def test_bit_exact_gather(d, flags):
    """One key aligned with q and scaled far above the rest selects its value
    row; the output must equal that row exactly (it encodes the token).

    Exactness needs every other weight, and every other split's merge weight,
    to vanish in fp32: a score margin above 110 natural units (e^-110 is
    below the smallest fp32 subnormal).  The margin grows as
    factor |q|^2 / sqrt(d), so head_dim 64 takes a 32x key (|q|^2 ~ 64)."""
    L, group, hkv = 2000, 4, 2
    factor = 32.0 if d == 64 else 16.0
    for t_star in (0, 63, 64, 1023, L - 1):
        w = syn.make_contiguous(999, 1, hkv * group, hkv, d, L, [L])
        qg = syn.bf16_bits_to_f64(w.q[0, ::group])
        w.q[0] = np.repeat(w.q[0, ::group], group, axis=0)
        for g in range(hkv):
            w.k[0, t_star, g] = syn.f64_to_bf16_bits(factor * qg[g])
            t = np.arange(L)
            w.v[0, :, g, 0] = syn.f64_to_bf16_bits((t >> 8).astype(np.float64))
            w.v[0, :, g, d - 1] = syn.f64_to_bf16_bits((t & 255).astype(np.float64))
        K = syn.bf16_bits_to_f64(w.k[0])
        s = w.scale * np.einsum("tgd,gd->tg", K, qg)
        assert np.all(s[t_star] - np.delete(s, t_star, axis=0).max(axis=0) > 110), "probe margin too small"
        o, _ = run(w, num_ctas=7, flags=flags)
        for h in range(hkv * group):
            expect = syn.bf16_bits_to_f64(w.v[0, t_star, h // group])
            assert np.array_equal(o[0, h], expect), (d, t_star, h)
            assert o[0, h, 0] * 256 + o[0, h, d - 1] == t_star
