"""Pins for the oracle's several-new-tokens decode (q_len > 1) under the
causal mask: the cache of length L holds the q_len new tokens, and new token
i sees positions 0 .. L - q_len + i.  No GPU, no CUDA library."""
import dataclasses

import numpy as np
import pytest

import fd_synth as syn
import oracle

mpmath = pytest.importorskip("mpmath")

LENS = [1, 2, 5, 64, 65, 130, 0]


def rows_visible(L, q_len, i):
    return max(0, L - q_len + i + 1)


# up to 16 new tokens: the most query columns per kv head the library takes
@pytest.mark.parametrize("q_len", [2, 3, 8, 16])
def test_each_row_is_brute_force_over_its_visible_prefix(q_len):
    hq, hkv, d = 4, 2, 64
    w = syn.make_contiguous(400 + q_len, len(LENS), hq, hkv, d, 130, LENS, q_len=q_len)
    o, lse = oracle.attend(w)
    assert o.shape == (len(LENS), q_len, hq, d) and lse.shape == (len(LENS), q_len, hq)
    K, V = syn.bf16_bits_to_f64(w.k), syn.bf16_bits_to_f64(w.v)
    for b, L in enumerate(LENS):
        for i in range(q_len):
            n = rows_visible(L, q_len, i)
            for h in range(hq):
                g = h // (hq // hkv)
                if n == 0:
                    assert np.all(o[b, i, h] == 0) and lse[b, i, h] == -np.inf
                    continue
                ro, rl = mp_attention(syn.bf16_bits_to_f64(w.q[b, i, h]), K[b, :n, g], V[b, :n, g], w.scale)
                np.testing.assert_allclose(o[b, i, h], ro, rtol=1e-12, atol=1e-14)
                assert lse[b, i, h] == pytest.approx(rl, rel=1e-13, abs=1e-13)


def test_single_new_token_as_4d_query_equals_the_3d_call():
    w3 = syn.make_contiguous(410, len(LENS), 8, 2, 128, 130, LENS)
    w4 = dataclasses.replace(w3, q=w3.q[:, None])
    o3, l3 = oracle.attend(w3)
    o4, l4 = oracle.attend(w4)
    assert np.array_equal(o3, o4[:, 0]) and np.array_equal(l3, l4[:, 0])


def test_last_new_token_sees_the_whole_cache_and_earlier_ones_do_not_see_later_tokens():
    q_len, L = 4, 100
    w = syn.make_contiguous(420, 1, 2, 1, 128, L, [L], q_len=q_len)
    o, lse = oracle.attend(w)
    # the last new token is ordinary single-query decode over the whole cache
    last = dataclasses.replace(w, q=w.q[:, q_len - 1])
    ol, ll = oracle.attend(last)
    assert np.array_equal(o[:, q_len - 1], ol) and np.array_equal(lse[:, q_len - 1], ll)
    # changing the cache at position L - 1 moves only the rows that see it
    w2 = dataclasses.replace(w, k=w.k.copy(), v=w.v.copy())
    w2.k[0, L - 1] = syn.scale_bf16_bits(w2.k[0, L - 1], 4.0)
    w2.v[0, L - 1] = syn.scale_bf16_bits(w2.v[0, L - 1], 4.0)
    o2, l2 = oracle.attend(w2)
    assert np.array_equal(o[0, :q_len - 1], o2[0, :q_len - 1])
    assert np.array_equal(lse[0, :q_len - 1], l2[0, :q_len - 1])
    assert not np.array_equal(o[0, q_len - 1], o2[0, q_len - 1])


def test_paged_equals_contiguous_with_several_new_tokens():
    q_len = 3
    w = syn.make_contiguous(430, len(LENS), 4, 2, 128, 130, LENS, q_len=q_len)
    o, lse = oracle.attend(w)
    from test_oracle_fp8 import paged
    op, lp = oracle.attend(paged(w, 16, 3, poison=True))
    assert np.array_equal(o, op) and np.array_equal(lse, lp)


def test_split_ranges_merge_to_the_causal_row():
    """A row's split partials over [0, m) and [m, end) merge to the full row."""
    q_len, L = 5, 90
    w = syn.make_contiguous(440, 1, 2, 1, 128, L, [L], q_len=q_len)
    o, lse = oracle.attend(w)
    for i in range(q_len):
        r = i * 2 + 1                     # token i, head 1
        end = L - q_len + i + 1
        items = np.array([[0, r, 0, 40], [0, r, 40, -1]], np.int32)
        po, pl = oracle.attend(w, items=items)
        mo, ml = oracle.lse_merge(po, pl)
        np.testing.assert_allclose(mo, o[0, i, 1], rtol=1e-13, atol=1e-15)
        assert ml == pytest.approx(lse[0, i, 1], rel=1e-14)
        assert end > 40


def mp_attention(qrow, K, V, scale):
    mp = mpmath.mp
    mp.dps = 40
    qs = [mp.mpf(float(x)) for x in qrow]
    s = [mp.mpf(scale) * mp.fsum(a * mp.mpf(float(b)) for a, b in zip(qs, krow)) for krow in K]
    m = max(s)
    e = [mp.e ** (x - m) for x in s]
    z = mp.fsum(e)
    o = [mp.fsum(ei * mp.mpf(float(vr[j])) for ei, vr in zip(e, V)) / z for j in range(len(qrow))]
    return np.array([float(x) for x in o]), float(m + mp.log(z))
