"""Pins for the CPU oracle (no GPU, no CUDA library involved).

Each test checks the oracle against something other than itself: the values
printed on the handbook page's worked example, closed forms, invariants of
softmax attention, or brute force in multi-precision arithmetic.  A plausible
slip in the oracle (a dropped scale, a wrong sign in an exponent, a head or
page index taken the wrong way round, K and V swapped) fails at least one.
"""
import math

import numpy as np
import pytest

import fd_synth as syn
import oracle
from conftest import read_golden

mpmath = pytest.importorskip("mpmath")


def bf(x):
    return syn.f64_to_bf16_bits(np.asarray(x, dtype=np.float64))


def wide(bits):
    return syn.bf16_bits_to_f64(bits)


def contig(q, k, v, lens, hq, hkv, scale):
    return syn.Workload("t", q, k, v, np.asarray(lens, np.int32), hq, hkv, q.shape[-1], scale)


def rand_bits(seed, shape, mult=1.0):
    x = syn._normal_chunk(seed, 0, int(np.prod(shape))).reshape(shape) * mult
    return bf(x)


# ---------------------------------------------------------------------------
# The handbook's worked example (exercise 1 of the FlashAttention page)
# ---------------------------------------------------------------------------

def test_worked_example_online_recurrence():
    g = read_golden("online_softmax_worked_example.txt")
    s = g["scores_block1"] + g["scores_block2"]
    v = g["values_block1"] + g["values_block2"]
    m, l, O, fin = oracle.online_blocks(s, v, 2)
    rel = 5e-4
    assert m.tolist() == [g["block1_m"][0], g["block2_m"][0]]
    assert l[0] == pytest.approx(g["block1_l"][0], rel=rel)
    assert O[0, 0] == pytest.approx(g["block1_O"][0], rel=rel)
    assert l[1] == pytest.approx(g["block2_l"][0], rel=rel)
    assert O[1, 0] == pytest.approx(g["block2_O"][0], rel=rel)
    assert fin[0] == pytest.approx(g["final"][0], rel=rel)
    # the page's direct check: weights proportional to e^s
    w = [math.exp(x) for x in s]
    assert w == pytest.approx(g["direct_weights"], rel=rel)
    assert sum(w) == pytest.approx(g["direct_weight_sum"][0], rel=rel)


def _worked_example_workload():
    """Scores [1,3,2,5] and V column 0 = [10,20,30,40] as an attention problem (scale 1)."""
    d = 128
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 1.0
    k = np.zeros((1, 4, 1, d)); k[0, :, 0, 0] = [1, 3, 2, 5]
    v = np.zeros((1, 4, 1, d)); v[0, :, 0, 0] = [10, 20, 30, 40]
    return contig(bf(q), bf(k), bf(v), [4], 1, 1, 1.0)


def test_worked_example_as_attention_and_split_merge():
    g = read_golden("online_softmax_worked_example.txt")
    w = _worked_example_workload()
    o, lse = oracle.attend(w)
    e = [math.exp(x) for x in (1, 3, 2, 5)]
    exact_o = math.fsum(a * b for a, b in zip(e, (10, 20, 30, 40))) / math.fsum(e)
    assert o[0, 0, 0] == pytest.approx(exact_o, rel=1e-14)
    assert o[0, 0, 0] == pytest.approx(g["final"][0], rel=5e-4)
    assert lse[0, 0] == pytest.approx(math.log(math.fsum(e)), rel=1e-14)
    assert np.all(o[0, 0, 1:] == 0.0)
    # two splits of two tokens: partials are the per-block results, normalised
    items = np.array([[0, 0, 0, 2], [0, 0, 2, 4]])
    po, pl = oracle.attend(w, items=items)
    assert po[0, 0] == pytest.approx(g["block1_O"][0] / g["block1_l"][0], rel=5e-4)
    assert pl[0] == pytest.approx(3 + math.log(g["block1_l"][0]), rel=1e-4)
    assert pl[1] == pytest.approx(5 + math.log(math.exp(-3) + 1), rel=1e-14)
    mo, ml = oracle.lse_merge(po, pl)
    assert mo[0] == pytest.approx(exact_o, rel=1e-14)
    assert ml == pytest.approx(lse[0, 0], rel=1e-14)


# ---------------------------------------------------------------------------
# Closed forms
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("paged", [False, True])
def test_single_token_gives_v0_and_its_score(paged):
    d, hq, hkv, B = 128, 4, 2, 3
    q = rand_bits(11, (B, hq, d))
    k = rand_bits(12, (B, 1, hkv, d), 3.0)
    v = rand_bits(13, (B, 1, hkv, d))
    scale = syn.default_scale(d)
    w = contig(q, k, v, [1] * B, hq, hkv, scale)
    if paged:
        w = to_paged(w, 4, perm_seed=5)
    o, lse = oracle.attend(w)
    for b in range(B):
        for h in range(hq):
            g = h // (hq // hkv)
            assert np.array_equal(o[b, h], wide(v[b, 0, g]))
            s = scale * math.fsum(wide(q[b, h]) * wide(k[b, 0, g]))
            assert lse[b, h] == pytest.approx(s, rel=1e-13, abs=1e-13)


def test_identical_keys_give_mean_of_values():
    d, L = 128, 37
    q = rand_bits(21, (1, 1, d))
    krow = rand_bits(22, (d,))
    k = np.broadcast_to(krow, (1, L, 1, d)).copy()
    v = rand_bits(23, (1, L, 1, d))
    scale = 0.3
    o, lse = oracle.attend(contig(q, k, v, [L], 1, 1, scale))
    mean = np.array([math.fsum(col) / L for col in wide(v[0, :, 0]).T])
    np.testing.assert_allclose(o[0, 0], mean, rtol=1e-13, atol=1e-14)
    s = scale * math.fsum(wide(q[0, 0]) * wide(krow))
    assert lse[0, 0] == pytest.approx(s + math.log(L), rel=1e-13)


def test_identical_values_give_that_row():
    d, L = 128, 500
    q = rand_bits(31, (1, 2, d))
    k = rand_bits(32, (1, L, 1, d), 4.0)
    vrow = rand_bits(33, (d,))
    v = np.broadcast_to(vrow, (1, L, 1, d)).copy()
    o, _ = oracle.attend(contig(q, k, v, [L], 2, 1, syn.default_scale(d)))
    for h in range(2):
        np.testing.assert_allclose(o[0, h], wide(vrow), rtol=1e-13, atol=1e-15)


def test_one_hot_values_recover_softmax_weights():
    from scipy.special import softmax
    d, L = 128, 100
    c = 2.0
    a = wide(rand_bits(41, (L,), 2.0))          # bf16-exact key magnitudes
    q = np.zeros((1, 1, d)); q[0, 0, 0] = c
    k = np.zeros((1, L, 1, d)); k[0, :, 0, 0] = a
    v = np.zeros((1, L, 1, d)); v[0, np.arange(L), 0, np.arange(L)] = 1.0
    scale = 0.125
    o, lse = oracle.attend(contig(bf(q), bf(k), bf(v), [L], 1, 1, scale))
    ref = softmax(scale * c * a)
    np.testing.assert_allclose(o[0, 0, :L], ref, rtol=1e-13, atol=1e-16)
    assert np.all(o[0, 0, L:] == 0)
    from scipy.special import logsumexp
    assert lse[0, 0] == pytest.approx(logsumexp(scale * c * a), rel=1e-14)


def test_scale_enters_the_scores():
    d = 128
    q = np.zeros((1, 1, d)); q[0, 0, 3] = 2.0
    k = np.zeros((1, 2, 1, d)); k[0, 0, 0, 3] = 1.0; k[0, 1, 0, 3] = -1.0
    v = np.zeros((1, 2, 1, d)); v[0, 0, 0, 0] = 1.0; v[0, 1, 0, 0] = -1.0
    for scale in (1.0, 0.5, 0.088388347648318):
        o, lse = oracle.attend(contig(bf(q), bf(k), bf(v), [2], 1, 1, scale))
        x = 2.0 * scale
        assert o[0, 0, 0] == pytest.approx(math.tanh(x), rel=1e-14)
        assert lse[0, 0] == pytest.approx(math.log(math.exp(x) + math.exp(-x)), rel=1e-14)


def test_gqa_mapping_consecutive_heads_share_kv_head():
    d, L, hq, hkv = 128, 9, 8, 2
    group = hq // hkv
    q = rand_bits(51, (1, hq, d))
    k = rand_bits(52, (1, L, hkv, d))
    v = np.zeros((1, L, hkv, d))
    for g in range(hkv):
        v[0, :, g, :] = g + 1.0
    o, _ = oracle.attend(contig(q, k, bf(v), [L], hq, hkv, 0.1))
    for h in range(hq):
        assert np.all(o[0, h] == pytest.approx(h // group + 1.0, rel=1e-14))


# ---------------------------------------------------------------------------
# Empty inputs and the merge
# ---------------------------------------------------------------------------

def test_zero_length_and_empty_ranges():
    d = 128
    q = rand_bits(61, (2, 2, d))
    k = rand_bits(62, (2, 5, 1, d))
    v = rand_bits(63, (2, 5, 1, d))
    o, lse = oracle.attend(contig(q, k, v, [0, 5], 2, 1, 0.1))
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))
    po, pl = oracle.attend(contig(q, k, v, [0, 5], 2, 1, 0.1), items=[[1, 0, 3, 3]])
    assert np.all(po == 0) and np.isneginf(pl[0])


def test_merge_of_any_split_equals_full_and_skips_empty():
    d, L = 128, 1000
    w = syn.make_contiguous(91, 1, 2, 1, d, L, [L])
    o, lse = oracle.attend(w)
    rng = np.random.default_rng(0)
    for trial in range(5):
        cuts = np.sort(rng.choice(np.arange(1, L), size=rng.integers(1, 12), replace=False))
        edges = [0, *cuts.tolist(), L]
        items = [[0, 1, a, b] for a, b in zip(edges[:-1], edges[1:])]
        items.insert(1, [0, 1, 7, 7])                       # an empty split
        po, pl = oracle.attend(w, items=np.array(items))
        mo, ml = oracle.lse_merge(po, pl)
        np.testing.assert_allclose(mo, o[0, 1], rtol=1e-12, atol=1e-14)
        assert ml == pytest.approx(lse[0, 1], rel=1e-13)
    mo, ml = oracle.lse_merge(np.ones((2, 3)), np.array([-np.inf, -np.inf]))
    assert np.all(mo == 0) and ml == -np.inf


# ---------------------------------------------------------------------------
# Paged layout
# ---------------------------------------------------------------------------

def to_paged(w, page, perm_seed, extra_pages=3, poison=False):
    """Copy a contiguous workload into shuffled pages (unused slots NaN if poison)."""
    B, S, hkv, d = w.k.shape
    lens = w.seq_lens
    used = sum((int(L) + page - 1) // page for L in lens)
    n_pages = used + extra_pages
    perm = syn.permutation(perm_seed, n_pages)
    max_blocks = max(1, (S + page - 1) // page)
    table = syn.build_block_table(lens, page, max_blocks, perm)
    fill = syn.BF16_NAN if poison else np.uint16(0)
    kp = np.full((n_pages, page, hkv, d), fill, np.uint16)
    vp = np.full((n_pages, page, hkv, d), fill, np.uint16)
    for b in range(B):
        for t in range(int(lens[b])):
            pg = table[b, t // page]
            kp[pg, t % page] = w.k[b, t]
            vp[pg, t % page] = w.v[b, t]
    return syn.Workload(w.name + "_paged", w.q, kp, vp, lens.copy(), w.num_q_heads, w.num_kv_heads,
                        d, w.scale, page_size=page, block_table=table)


@pytest.mark.parametrize("page", [1, 16, 64])
def test_permuted_pages_equal_contiguous_bitwise(page):
    lens = [1, 17, 300, 0, 129]
    w = syn.make_contiguous(71, len(lens), 4, 2, 128, 300, lens)
    o, lse = oracle.attend(w)
    op, lp = oracle.attend(to_paged(w, page, perm_seed=page))
    assert np.array_equal(o, op)
    assert np.array_equal(lse, lp)


def test_positions_past_length_and_unused_pages_are_never_read():
    lens = [5, 64, 65, 200]
    w = syn.make_contiguous(72, len(lens), 2, 1, 128, 200, lens)
    o, lse = oracle.attend(w)
    wp = syn.Workload(w.name, w.q, w.k.copy(), w.v.copy(), w.seq_lens, 2, 1, 128, w.scale)
    for b, L in enumerate(lens):
        wp.k[b, L:] = syn.BF16_NAN
        wp.v[b, L:] = syn.BF16_NAN
    o2, l2 = oracle.attend(wp)
    assert np.array_equal(o, o2) and np.array_equal(lse, l2)
    o3, l3 = oracle.attend(to_paged(w, 16, perm_seed=9, poison=True))
    assert np.all(np.isfinite(o3)) and np.array_equal(o, o3) and np.array_equal(lse, l3)


def test_bad_page_is_rejected():
    w = to_paged(syn.make_contiguous(73, 1, 1, 1, 128, 40, [40]), 16, perm_seed=1)
    w.block_table[0, 1] = w.num_pages + 5
    with pytest.raises(ValueError):
        oracle.attend(w)


# ---------------------------------------------------------------------------
# Brute force in multi-precision
# ---------------------------------------------------------------------------

def mp_attention(qrow, K, V, scale):
    """Attention of one query row in 40-digit arithmetic (bf16 products are exact)."""
    mp = mpmath.mp
    mp.dps = 40
    qs = [mp.mpf(float(x)) for x in qrow]
    s = [mp.mpf(scale) * mp.fsum(a * mp.mpf(float(b)) for a, b in zip(qs, krow)) for krow in K]
    m = max(s)
    e = [mp.e ** (x - m) for x in s]
    z = mp.fsum(e)
    o = [mp.fsum(ei * mp.mpf(float(vr[j])) for ei, vr in zip(e, V)) / z for j in range(len(qrow))]
    return np.array([float(x) for x in o]), float(m + mp.log(z))


@pytest.mark.parametrize("L", [1, 2, 17, 63, 64, 65])
def test_brute_force_tails(L):
    d = 128
    w = syn.make_contiguous(80 + L, 1, 2, 1, d, L, [L])
    o, lse = oracle.attend(w)
    for h in range(2):
        ro, rl = mp_attention(wide(w.q[0, h]), wide(w.k[0, :L, 0]), wide(w.v[0, :L, 0]), w.scale)
        np.testing.assert_allclose(o[0, h], ro, rtol=1e-12, atol=1e-14)
        assert lse[0, h] == pytest.approx(rl, rel=1e-13, abs=1e-13)


def test_brute_force_long_row_fsum():
    d, L = 128, 1000
    w = syn.make_contiguous(99, 1, 1, 1, d, L, [L])
    o, lse = oracle.attend(w)
    qd = wide(w.q[0, 0]); K = wide(w.k[0, :, 0]); V = wide(w.v[0, :, 0])
    s = [w.scale * math.fsum(qd * K[t]) for t in range(L)]
    m = max(s)
    e = [math.exp(x - m) for x in s]
    z = math.fsum(e)
    ref = np.array([math.fsum(e[t] * V[t, j] for t in range(L)) / z for j in range(d)])
    np.testing.assert_allclose(o[0, 0], ref, rtol=1e-11, atol=1e-13)
    assert lse[0, 0] == pytest.approx(m + math.log(z), rel=1e-13)


@pytest.mark.parametrize("factor", [8.0, 32.0])
def test_softmax_stress_scaled_keys(factor):
    d, L = 128, 150
    w = syn.make_contiguous(100 + int(factor), 1, 2, 1, d, L, [L])
    toks = syn.choose(5, L, 3)
    syn.scale_keys(w, toks, factor)
    o, lse = oracle.attend(w)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    for h in range(2):
        ro, rl = mp_attention(wide(w.q[0, h]), wide(w.k[0, :, 0]), wide(w.v[0, :, 0]), w.scale)
        np.testing.assert_allclose(o[0, h], ro, rtol=1e-12, atol=1e-14)
        assert lse[0, h] == pytest.approx(rl, rel=1e-13)


# ---------------------------------------------------------------------------
# fp16 inputs (the first page's tensor-map helper takes fp16 as well as bf16)
# ---------------------------------------------------------------------------

def f16(x):
    return syn.f64_to_f16_bits(np.asarray(x, dtype=np.float64))


def test_f16_single_token_gives_v0_exactly_including_subnormals():
    d = 128
    q = f16(np.linspace(-1, 1, d).reshape(1, 1, d))
    k = f16(np.linspace(2, -2, d).reshape(1, 1, 1, d))
    vals = np.concatenate([[2 ** -24, 3 * 2 ** -24, -(2 ** -20), 6.1e-5, 65504.0, -2.5],
                           np.linspace(-3, 3, d - 6)])
    v = f16(vals.reshape(1, 1, 1, d))
    w = syn.Workload("f16", q, k, v, np.array([1], np.int32), 1, 1, d, 0.25, dtype="f16")
    o, lse = oracle.attend(w)
    # reference widening by numpy's float16 (independent of the C oracle)
    assert np.array_equal(o[0, 0], v.view(np.float16).astype(np.float64)[0, 0, 0])
    s = 0.25 * math.fsum(q.view(np.float16).astype(np.float64)[0, 0] * k.view(np.float16).astype(np.float64)[0, 0, 0])
    assert lse[0, 0] == pytest.approx(s, rel=1e-14, abs=1e-15)


@pytest.mark.parametrize("L", [17, 65])
def test_f16_brute_force(L):
    w = syn.make_contiguous(120 + L, 1, 2, 1, 128, L, [L], dtype="f16")
    o, lse = oracle.attend(w)
    wd = lambda a: syn.f16_bits_to_f64(a)
    for h in range(2):
        ro, rl = mp_attention(wd(w.q[0, h]), wd(w.k[0, :L, 0]), wd(w.v[0, :L, 0]), w.scale)
        np.testing.assert_allclose(o[0, h], ro, rtol=1e-12, atol=1e-14)
        assert lse[0, h] == pytest.approx(rl, rel=1e-13, abs=1e-13)


def test_f16_paged_equals_contiguous():
    lens = [1, 40, 0, 129]
    w = syn.make_contiguous(131, len(lens), 4, 2, 128, 200, lens, dtype="f16")
    o, lse = oracle.attend(w)
    wp = to_paged(w, 16, perm_seed=4)
    wp.dtype = "f16"
    op, lp = oracle.attend(wp)
    assert np.array_equal(o, op) and np.array_equal(lse, lp)
