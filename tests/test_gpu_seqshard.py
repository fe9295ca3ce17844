"""Sequence sharding on one GPU: every range's partial (fd_decode_partial /
fd_decode_paged_partial, through the C ABI binding) against the oracle's
attention over the same positions, and fd_merge_partials of the ranges'
partials against the oracle's whole-cache result.  The ranks of a sharded
run are emulated one after another on the device; nothing waits on another
launch.  Also the merge call alone against the oracle's LSE merge, with empty
sets (LSE = -inf), rows that no set saw, and more sets than a warp has lanes."""
import dataclasses

import numpy as np
import pytest
import torch

import fd_synth as syn
import oracle
from gpu_util import check, contig_to_paged, to_device

pytestmark = pytest.mark.gpu

BIG = 2 ** 31 - 1


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_attention_decoding_gb300 import build
    build.build()
    oracle.build()


def oracle_range(w, t0, t1):
    B, rows = w.batch, w.q_len * w.num_q_heads
    items = np.array([[b, r, t0, t1] for b in range(B) for r in range(rows)], dtype=np.int32)
    o, l = oracle.attend(w, items=items, threads=8)
    return o.reshape(B, rows, -1), l.reshape(B, rows)


def shard(w, t0, t1):
    """The positions [t0, t1) of every request as their own contiguous cache
    (rows t' = position t0 + t'), with the range's token counts."""
    S = w.k.shape[1]
    e = min(t1, S)
    cap = max(e - t0, 1)
    k = np.zeros((w.batch, cap) + w.k.shape[2:], w.k.dtype)
    v = np.zeros_like(k)
    k[:, :e - t0] = w.k[:, t0:e]
    v[:, :e - t0] = w.v[:, t0:e]
    n = np.clip(np.minimum(w.seq_lens.astype(np.int64), t1) - t0, 0, None).astype(np.int32)
    return dataclasses.replace(w, k=k, v=v, seq_lens=n)


def run_partial(w, ws_local, t0, t1, page=0, flags=0):
    import decode_attention_decoding_gb300 as fd
    kw = {}
    if getattr(w, "kv_dtype", None) in ("e4m3", "e5m2"):
        kw = dict(kv_dtype=w.kv_dtype, k_scale=w.k_scale, v_scale=w.v_scale)
    lens = torch.from_numpy(w.seq_lens.astype(np.int32)).cuda()   # whole lengths
    lens_h = torch.from_numpy(w.seq_lens.astype(np.int32))
    if page:
        wp = contig_to_paged(ws_local, page, perm_seed=t0 + 7)
        d = to_device(wp)
        o, l = fd.fd_decode_paged_partial(d["q"], d["k"], d["v"], d["block_table"], lens, t0, t1,
                                          seq_lens_host=lens_h, scale=w.scale, flags=flags, **kw)
    else:
        d = to_device(ws_local)
        o, l = fd.fd_decode_partial(d["q"], d["k"], d["v"], lens, t0, t1, seq_lens_host=lens_h,
                                    scale=w.scale, flags=flags, **kw)
    return o, l


CASES = [
    # (name, hq, hkv, head_dim, q_len, page, kv, cuts)
    ("gqa4", 8, 2, 128, 1, 0, None, [0, 512, 1100, BIG]),
    ("mha", 4, 4, 128, 1, 0, None, [0, 700, BIG]),
    ("gqa4_q2", 8, 2, 128, 2, 0, None, [0, 1000, 1499, BIG]),
    ("gqa8_paged16", 16, 2, 128, 1, 16, None, [0, 333, 1200, BIG]),
    ("gqa4_paged1", 8, 2, 128, 1, 1, None, [0, 640, BIG]),
    ("gqa4_d64_paged64", 8, 2, 64, 1, 64, None, [0, 256, BIG]),
    ("gqa4_e4m3", 8, 2, 128, 1, 0, "e4m3", [0, 900, BIG]),
]


@pytest.mark.parametrize("name,hq,hkv,d,q_len,page,kv,cuts", CASES, ids=[c[0] for c in CASES])
def test_partials_and_merge_match_the_oracle(name, hq, hkv, d, q_len, page, kv, cuts):
    import decode_attention_decoding_gb300 as fd
    lens = [1500, 3, 0, 777, 1000]
    sc = 0.125 if kv else 1.0   # FP8 dequantisation scales (16-bit caches take none)
    w = syn.make_contiguous(980 + len(name), len(lens), hq, hkv, d, 1500, lens, kv_dtype=kv,
                            k_scale=sc, v_scale=sc, q_len=q_len)
    B, rows = w.batch, q_len * hq
    o_parts, l_parts = [], []
    for t0, t1 in zip(cuts[:-1], cuts[1:]):
        o, l = run_partial(w, shard(w, t0, t1), t0, t1, page=page)
        torch.cuda.synchronize()
        ro, rl = oracle_range(w, t0, t1)
        got_o = o.reshape(B, rows, d).cpu().numpy().astype(np.float64)
        got_l = l.reshape(B, rows).cpu().numpy().astype(np.float64)
        check(got_o, got_l, ro, rl, f"{name} range [{t0}, {t1})")
        o_parts.append(o.reshape(B, rows, d))
        l_parts.append(l.reshape(B, rows))
    om, lm = fd.fd_merge_partials(torch.stack(o_parts), torch.stack(l_parts))
    torch.cuda.synchronize()
    ro, rl = oracle.attend(w, threads=8)
    check(om.cpu().numpy().astype(np.float64), lm.cpu().numpy().astype(np.float64),
          ro.reshape(B, rows, d), rl.reshape(B, rows), f"{name} merged")


def test_whole_range_equals_fd_decode_bitwise():
    """A range [0, end) of the whole cache takes the same launch as fd_decode."""
    import decode_attention_decoding_gb300 as fd
    w = syn.make_contiguous(990, 3, 8, 2, 128, 900, [900, 64, 1])
    d = to_device(w)
    lens_h = torch.from_numpy(w.seq_lens)
    o1, l1 = fd.fd_decode(d["q"], d["k"], d["v"], d["seq_lens"], seq_lens_host=lens_h, scale=w.scale)
    o2, l2 = fd.fd_decode_partial(d["q"], d["k"], d["v"], d["seq_lens"], 0, BIG, seq_lens_host=lens_h,
                                  scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("n,d", [(1, 128), (2, 64), (5, 256), (40, 128)])
def test_merge_partials_alone(n, d):
    import decode_attention_decoding_gb300 as fd
    rng = np.random.default_rng(n * 1000 + d)
    rows = 37
    o_parts = rng.standard_normal((n, rows, d)).astype(np.float32)
    l_parts = (rng.standard_normal((n, rows)) * 20).astype(np.float32)
    l_parts[rng.random((n, rows)) < 0.3] = -np.inf     # empty sets
    l_parts[:, 5] = -np.inf                             # a row that no set saw
    o_parts[np.isneginf(l_parts)] = np.nan              # never read
    om, lm = fd.fd_merge_partials(torch.from_numpy(o_parts).cuda(), torch.from_numpy(l_parts).cuda())
    torch.cuda.synchronize()
    got_o, got_l = om.cpu().numpy().astype(np.float64), lm.cpu().numpy().astype(np.float64)
    for r in range(rows):
        keep = np.isfinite(l_parts[:, r])
        if keep.any():
            ro, rl = oracle.lse_merge(o_parts[keep, r].astype(np.float64), l_parts[keep, r].astype(np.float64))
        else:
            ro, rl = np.zeros(d), -np.inf
        assert np.all(np.abs(got_o[r] - ro) <= 1e-5 + 1e-5 * np.abs(ro)), r
        assert (np.isneginf(got_l[r]) and np.isneginf(rl)) or abs(got_l[r] - rl) <= 1e-5, r
    assert np.all(got_o[5] == 0) and np.isneginf(got_l[5])
