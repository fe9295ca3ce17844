"""The seeded input generator: exact bf16 rounding, the SplitMix64 stream, shuffles."""
from fractions import Fraction

import numpy as np
import pytest

import fd_synth as syn

MASK = (1 << 64) - 1


def splitmix64_sequential(seed, n):
    """The published SplitMix64 `next()` loop, in plain Python integers."""
    x, out = seed & MASK, []
    for _ in range(n):
        x = (x + 0x9E3779B97F4A7C15) & MASK
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK
        out.append(z ^ (z >> 31))
    return out


def test_splitmix_counter_form_matches_sequential():
    for seed in (0, 1, 0xFD000011, MASK):
        ref = splitmix64_sequential(seed, 50)
        assert [int(x) for x in syn.splitmix64(seed, 50)] == ref
        assert [int(x) for x in syn.splitmix64(seed, 10, offset=40)] == ref[40:]


def bf16_round_exact(x: float) -> float:
    """Nearest bf16 (8 significant bits), ties to even, by exact rational arithmetic."""
    if x == 0:
        return 0.0
    f = Fraction(x)
    sign = -1 if f < 0 else 1
    f = abs(f)
    e = 0
    while f >= 2:
        f /= 2; e += 1
    while f < 1:
        f *= 2; e -= 1
    scaled = f * 128                      # 1.xxxxxxx -> 8-bit integer part
    lo = int(scaled)
    rem = scaled - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * float(Fraction(lo, 128) * Fraction(2) ** e)


def test_bf16_rounding_is_nearest_even_from_fp64():
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-30, 30, 2000),
                         [1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 1 + 2 ** -8 + 2 ** -40,
                          255.5, 256.5, 2.0 ** -126, 3.0e38, 0.0]])
    got = syn.bf16_bits_to_f64(syn.f64_to_bf16_bits(xs))
    ref = np.array([bf16_round_exact(float(x)) for x in xs])
    assert np.array_equal(got, ref)
    # a value just above a tie must round up even though fp32 would have rounded it to the tie
    assert syn.bf16_bits_to_f64(syn.f64_to_bf16_bits(np.array([1 + 2 ** -8 + 2 ** -40])))[0] == 1 + 2 ** -7


def test_bf16_rejects_subnormal_and_nonfinite():
    for bad in (1e-40, np.inf, np.nan):
        with pytest.raises(ValueError):
            syn.f64_to_bf16_bits(np.array([bad]))


def test_normals_are_deterministic_and_standard():
    a = syn.normal_bf16(123, (1 << 20,))
    b = syn.normal_bf16(123, (1 << 20,))
    assert np.array_equal(a, b)
    x = syn.bf16_bits_to_f64(a)
    assert abs(x.mean()) < 5e-3 and abs(x.std() - 1) < 5e-3
    # chunked generation equals one-shot generation
    part = syn.normal_bf16(123, (1000,))
    assert np.array_equal(part, a[:1000])
    assert not np.array_equal(a, syn.normal_bf16(124, (1 << 20,)))


def test_shuffles_and_lengths():
    p = syn.permutation(7, 5000)
    assert sorted(p.tolist()) == list(range(5000))
    assert not np.array_equal(p, np.arange(5000))
    c = syn.choose(5, 262144, 2621)
    assert len(set(c.tolist())) == 2621 and c.min() >= 0 and c.max() < 262144
    for cid, lo, hi in ((3, 512, 8192), (4, 1, 16384)):
        L = syn.config_lens(cid)
        assert L.min() >= lo and L.max() <= hi
    assert syn.config_lens(3).shape == (16,) and syn.config_lens(4).shape == (64,)


def test_block_table_assigns_each_page_once():
    lens = syn.config_lens(4)
    need = [(int(L) + 15) // 16 for L in lens]
    perm = syn.permutation(syn.seed_for(4, syn.TENSOR_PERM), sum(need))
    t = syn.build_block_table(lens, 16, 1024, perm)
    used = np.concatenate([t[b, :n] for b, n in enumerate(need)])
    assert sorted(used.tolist()) == list(range(sum(need)))
    assert all(np.all(t[b, n:] == -1) for b, n in enumerate(need))


def test_default_scale_is_fp32_inverse_sqrt():
    assert syn.default_scale(128) == float(np.float32(1) / np.sqrt(np.float32(128)))


def f16_round_exact(x: float) -> float:
    """Nearest IEEE fp16 (11 significant bits, subnormal quantum 2^-24), ties to even."""
    if x == 0:
        return 0.0
    f = abs(Fraction(x))
    sign = -1 if x < 0 else 1
    e = 0
    while f >= 2:
        f /= 2; e += 1
    while f < 1:
        f *= 2; e -= 1
    if e < -14:
        q = abs(Fraction(x)) / Fraction(2) ** -24
        lo = int(q); rem = q - lo
        if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2):
            lo += 1
        return sign * float(lo * Fraction(2) ** -24)
    scaled = f * 1024
    lo = int(scaled); rem = scaled - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2):
        lo += 1
    return sign * float(Fraction(lo, 1024) * Fraction(2) ** e)


def test_f16_rounding_is_nearest_even_from_fp64():
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-8, 4, 3000),
                         [1 + 2 ** -11, 1 + 3 * 2 ** -11, 1 + 2 ** -11 + 2 ** -40, 2 ** -25, 3 * 2 ** -26,
                          1.5 * 2 ** -24, 65504.0, 0.0]])
    got = syn.f16_bits_to_f64(syn.f64_to_f16_bits(xs))
    ref = np.array([f16_round_exact(float(x)) for x in xs])
    assert np.array_equal(got, ref)
    with pytest.raises(ValueError):
        syn.f64_to_f16_bits(np.array([70000.0]))


# ---------------------------------------------------------------------------
# FP8 codes (OCP E4M3 / E5M2)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("fmt,tdt,vmax", [("e4m3", "float8_e4m3fn", 448.0), ("e5m2", "float8_e5m2", 57344.0)])
def test_fp8_rounding_matches_torch_and_saturates(fmt, tdt, vmax):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    # fp32-exact inputs: torch converts through fp32, so only those are rounded once there
    x = (rng.standard_normal(100000) * 10 ** rng.uniform(-5, 3, 100000)).astype(np.float32)
    x = np.concatenate([x, np.linspace(-vmax, vmax, 20001, dtype=np.float32)]).astype(np.float64)
    x = x[np.abs(x) <= vmax]
    ref = torch.from_numpy(x).to(getattr(torch, tdt)).view(torch.uint8).numpy()
    assert np.array_equal(syn.f64_to_fp8_bits(x, fmt), ref)
    top = syn.f64_to_fp8_bits(np.array([vmax * 1.2, -1e30, vmax]), fmt)
    assert top[0] == top[2] and top[1] == (top[0] | 0x80)   # saturate, never NaN or inf


def test_fp8_single_rounding_at_halfway_points():
    """x just above a halfway point rounds up (a detour through fp32 would round to even)."""
    assert syn.f64_to_fp8_bits(np.array([84.00000000000006]), "e4m3")[0] == 0x6B   # 88 = 1.375 * 2^6
    assert syn.f64_to_fp8_bits(np.array([84.0]), "e4m3")[0] == 0x6A                # 80 (even fraction)
    assert syn.f64_to_fp8_bits(np.array([4.500000088419607]), "e5m2")[0] == 0x45   # 5


def test_fp8_workload_is_seeded_and_scaled():
    w = syn.make_contiguous(5, 2, 4, 2, 64, 16, [16, 3], kv_dtype="e4m3", k_scale=0.05, v_scale=0.5)
    w2 = syn.make_contiguous(5, 2, 4, 2, 64, 16, [16, 3], kv_dtype="e4m3", k_scale=0.05, v_scale=0.5)
    assert w.k.dtype == np.uint8 and np.array_equal(w.k, w2.k) and np.array_equal(w.v, w2.v)
    assert w.k_scale == float(np.float32(0.05)) and w.kv_bytes() == 19 * 2 * 64 * 2
    # codes are x / scale: with k_scale 0.05, |code value| ~ 20 |x|
    assert 5 < np.median(np.abs(w.k.view(np.int8).astype(np.int64) & 0x7F)) < 127


@pytest.mark.parametrize("page", [1, 2, 8, 64])
def test_repage_keeps_every_logical_row(page):
    """repage moves K/V rows between layouts without changing any (request,
    position) row; page entries are distinct and the rest of the table is -1."""
    w = syn.make_contiguous(41, 3, 4, 2, 64, 200, [200, 5, 0])
    p = syn.repage(syn.repage(w, 4, perm_seed=1), page, perm_seed=2)
    for b, L in enumerate(w.seq_lens):
        for t in range(int(L)):
            e = p.block_table[b, t // page]
            assert np.array_equal(p.k[e, t % page], w.k[b, t]) and np.array_equal(p.v[e, t % page], w.v[b, t])
        assert np.all(p.block_table[b, (int(L) + page - 1) // page:] == -1)
    used = p.block_table[p.block_table >= 0]
    assert len(set(used.tolist())) == len(used)
