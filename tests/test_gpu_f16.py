"""fp16 inputs (the other element type the first page's tensor-map helper
accepts): the CUDA library against the fp64 oracle on the same fp16 bits,
on both consumer paths and both KV layouts, plus the bit-exact gather probe."""
import numpy as np
import pytest

import fd_synth as syn
import oracle
from gpu_util import check, contig_to_paged, run, small_page_twin_flags

pytestmark = pytest.mark.gpu

CUDA_CORES = 0x2
RAGGED = [1000, 1, 0, 63, 64, 65, 129, 700]


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_attention_decoding_gb300 import build
    build.build()
    oracle.build()


@pytest.mark.parametrize("flags", [0, CUDA_CORES])
@pytest.mark.parametrize("group", [1, 2, 4, 8])
def test_f16_contiguous_vs_oracle(group, flags):
    hkv = 2
    w = syn.make_contiguous(800 + group, len(RAGGED), hkv * group, hkv, 128, 1024, RAGGED, dtype="f16")
    for ctas in (0, 7):
        o, l = run(w, num_ctas=ctas, flags=flags)
        ro, rl = oracle.attend(w, threads=8)
        check(o, l, ro, rl, f"f16 G={group} flags={flags} ctas={ctas}")


@pytest.mark.parametrize("page", [4, 16, 64])
@pytest.mark.parametrize("group", [1, 4])
def test_f16_paged_vs_oracle_and_contiguous(page, group):
    w = syn.make_contiguous(820 + page, len(RAGGED), 2 * group, 2, 128, 1024, RAGGED, dtype="f16")
    wp = contig_to_paged(w, page, perm_seed=page, poison=True)
    # pages under 8 tokens take unfused consumers (tensor cores for GQA)
    flags = small_page_twin_flags(w) if page < 8 else 0
    op, lp = run(wp, num_ctas=5)
    ro, rl = oracle.attend(wp, threads=8)
    check(op, lp, ro, rl, f"f16 paged P={page} G={group}")
    oc, lc = run(w, num_ctas=5, flags=flags)
    assert np.array_equal(op, oc) and np.array_equal(lp, lc)


@pytest.mark.parametrize("flags", [0, CUDA_CORES])
def test_f16_bit_exact_gather(flags):
    L, group, hkv, d = 2000, 4, 2, 128
    for t_star in (0, 63, 64, 1023, L - 1):
        w = syn.make_contiguous(840, 1, hkv * group, hkv, d, L, [L], dtype="f16")
        qg = syn.f16_bits_to_f64(w.q[0, ::group])
        w.q[0] = np.repeat(w.q[0, ::group], group, axis=0)
        for g in range(hkv):
            w.k[0, t_star, g] = syn.f64_to_f16_bits(16.0 * qg[g])
            t = np.arange(L)
            w.v[0, :, g, 0] = syn.f64_to_f16_bits((t >> 8).astype(np.float64))
            w.v[0, :, g, 1] = syn.f64_to_f16_bits((t & 255).astype(np.float64))
        o, _ = run(w, num_ctas=7, flags=flags)
        for h in range(hkv * group):
            expect = syn.f16_bits_to_f64(w.v[0, t_star, h // group])
            assert np.array_equal(o[0, h], expect), (t_star, h)
