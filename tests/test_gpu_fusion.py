"""Fused kv heads: F adjacent kv heads read as one row of F * head_dim dims
(the same bytes).  Two heads are paired (each warp of a pair takes one head);
four share one tensor-core tile with zeros for the other heads' dims (the
FP8 tests cover that launch).  The fused launch must give what the unfused
one gives: each query head attends to its own kv head only, and writes only
its own head_dim outputs."""
import numpy as np
import pytest
import torch

import fd_synth as syn
import oracle
from gpu_util import check, contig_to_paged, run, to_device

pytestmark = pytest.mark.gpu

CUDA_CORES = 0x2
NO_FUSION = 0x8       # FD_FLAG_NO_HEAD_FUSION
FUSE = 0x10           # FD_FLAG_FUSE_HEADS: fuse whenever the shape allows it
RAGGED = [1000, 1, 0, 63, 64, 65, 129, 700]


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_attention_decoding_gb300 import build
    build.build()
    oracle.build()


# (head_dim, group, hkv): the launch the library picks is in the comment
SHAPES = [(64, 1, 4),    # paired heads (two 64-dim heads per 256-byte row)
          (64, 2, 4),    # paired
          (64, 4, 2),    # paired
          (64, 2, 6),    # paired
          (128, 1, 4),   # paired: 256 dims per row
          (128, 2, 2),   # paired
          (128, 4, 2),   # paired
          (128, 8, 2),   # paired: 8 query heads per warp, 16 per launch head
          (64, 1, 3)]    # no fusion: odd Hkv


@pytest.mark.parametrize("d,group,hkv", SHAPES)
def test_fused_and_unfused_match_the_oracle(d, group, hkv):
    w = syn.make_contiguous(1100 + d + 10 * group + hkv, len(RAGGED), hkv * group, hkv, d, 1024, RAGGED)
    ro, rl = oracle.attend(w, threads=8)
    dev = to_device(w)
    for flags in (0, FUSE, NO_FUSION):
        for ctas in (0, 7):
            # NaN-filled outputs: every element must be written exactly by its own head
            out = torch.full((w.batch, w.num_q_heads, d), float("nan"), device="cuda")
            lse = torch.full((w.batch, w.num_q_heads), float("nan"), device="cuda")
            o, l = run(w, dev, num_ctas=ctas, flags=flags, out=out, lse=lse)
            assert not np.isnan(o).any() and not np.isnan(l).any()
            check(o, l, ro, rl, f"d={d} G={group} Hkv={hkv} flags={flags} ctas={ctas}")


@pytest.mark.parametrize("page", [8, 16, 64])
@pytest.mark.parametrize("d,group,hkv", [(64, 1, 4), (128, 4, 2), (128, 1, 2)])
def test_fused_paged_matches_oracle_and_contiguous(d, group, hkv, page):
    w = syn.make_contiguous(1200 + page + d, len(RAGGED), hkv * group, hkv, d, 1024, RAGGED)
    wp = contig_to_paged(w, page, perm_seed=page + group, poison=True)
    ro, rl = oracle.attend(wp, threads=8)
    for ctas in (0, 5):
        op, lp = run(wp, num_ctas=ctas, flags=FUSE)
        check(op, lp, ro, rl, f"d={d} G={group} P={page} ctas={ctas}")
        oc, lc = run(w, num_ctas=ctas, flags=FUSE)
        assert np.array_equal(op, oc) and np.array_equal(lp, lc)


@pytest.mark.parametrize("d,group,hkv", [(64, 1, 4), (64, 2, 4), (128, 2, 2), (128, 4, 2), (128, 8, 2),
                                         (64, 8, 4)])
def test_fused_heads_never_mix(d, group, hkv):
    """Each kv head gets its own dominating token; a query head that saw
    another head's keys or values would pick the wrong token."""
    L = 1500
    stars = [7 + 301 * g for g in range(hkv)]
    w = syn.make_contiguous(1300 + d, 1, hkv * group, hkv, d, L, [L])
    qg = syn.bf16_bits_to_f64(w.q[0, ::group])
    w.q[0] = np.repeat(w.q[0, ::group], group, axis=0)
    factor = 32.0 if d == 64 else 16.0
    t = np.arange(L)
    for g in range(hkv):
        w.k[0, stars[g], g] = syn.f64_to_bf16_bits(factor * qg[g])
        w.v[0, :, g, 0] = syn.f64_to_bf16_bits((t >> 8).astype(np.float64))
        w.v[0, :, g, d - 1] = syn.f64_to_bf16_bits((t & 255).astype(np.float64))
    K = syn.bf16_bits_to_f64(w.k[0])
    s = w.scale * np.einsum("tgd,gd->tg", K, qg)
    for g in range(hkv):
        assert s[stars[g], g] - np.delete(s[:, g], stars[g]).max() > 110, "probe margin too small"
    for ctas in (0, 7):
        o, _ = run(w, num_ctas=ctas, flags=FUSE)
        for h in range(hkv * group):
            g = h // group
            assert np.array_equal(o[0, h], syn.bf16_bits_to_f64(w.v[0, stars[g], g])), (ctas, h)
            assert o[0, h, 0] * 256 + o[0, h, d - 1] == stars[g]


def test_fused_f16_inputs():
    w = syn.make_contiguous(1400, len(RAGGED), 8, 4, 128, 1024, RAGGED, dtype="f16")
    ro, rl = oracle.attend(w, threads=8)
    for flags in (FUSE, NO_FUSION):
        o, l = run(w, num_ctas=7, flags=flags)
        check(o, l, ro, rl, f"f16 flags={flags}")


@pytest.mark.parametrize("d,page", [(64, 0), (128, 16), (64, 16)])
def test_default_fuses_long_calls_with_short_rows(d, page):
    """The default picks fusion for a long call with short rows; the result
    equals the forced-fusion launch bit for bit and matches the oracle."""
    lens = [6000, 4000, 5000, 3000]
    w = syn.make_contiguous(1500 + d + page, len(lens), 8, 4, d, 6000, lens)
    if page:
        w = contig_to_paged(w, page, perm_seed=page)
    ro, rl = oracle.attend(w, threads=8)
    o, l = run(w, num_ctas=8)          # (sum of tiles) x Hkv / 8 CTAs >= 24 per CTA
    of, lf = run(w, num_ctas=8, flags=FUSE)
    assert np.array_equal(o, of) and np.array_equal(l, lf)
    check(o, l, ro, rl, f"d={d} P={page} default")
