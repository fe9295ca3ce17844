"""The merge inside the split kernel (FD_FLAG_FUSED_MERGE) against the merge
kernel (the default) and the fp64 oracle: split counts up to grids far
larger than the CTAs resident at once, empty requests, several new tokens,
paged caches, token ranges, repeated calls on one workspace (the segment
counters reset themselves), and one workspace shared by launches of
different shapes (fused and unfused heads)."""
import numpy as np
import pytest
import torch

import fd_synth as syn
import oracle
from gpu_util import check, contig_to_paged, run, to_device

pytestmark = pytest.mark.gpu

FUSED = 0x200
FUSE = 0x10
NO_FUSION = 0x8
RAGGED = [1000, 0, 1, 63, 64, 65, 129, 700, 0, 2049]


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_attention_decoding_gb300 import build
    build.build()
    oracle.build()


@pytest.mark.parametrize("ctas", [0, 1, 7, 40, 300, 1024])
@pytest.mark.parametrize("group,d", [(1, 128), (4, 128), (8, 64), (2, 256)])
def test_fused_matches_separate_and_oracle(group, d, ctas):
    w = syn.make_contiguous(3100 + 10 * group + d, len(RAGGED), 2 * group, 2, d, 2112, RAGGED)
    ro, rl = oracle.attend(w, threads=8)
    o, l = run(w, num_ctas=ctas, flags=FUSED)
    check(o, l, ro, rl, f"fused merge G={group} d={d} ctas={ctas}")
    os_, ls = run(w, num_ctas=ctas)
    check(os_, ls, ro, rl, f"merge kernel G={group} d={d} ctas={ctas}")
    # the empty requests' rows come from the split kernel alone
    for b in np.flatnonzero(np.asarray(RAGGED) == 0):
        assert np.all(o[b] == 0) and np.all(np.isneginf(l[b]))


@pytest.mark.parametrize("flags", [0, FUSE, 0x2])
def test_paged_and_several_new_tokens(flags):
    w = syn.make_contiguous(3200 + flags, len(RAGGED), 8, 2, 128, 2112, RAGGED, q_len=2)
    wp = contig_to_paged(w, 16, perm_seed=3, poison=True)
    ro, rl = oracle.attend(wp, threads=8)
    for ctas in (0, 9, 500):
        o, l = run(wp, num_ctas=ctas, flags=flags | FUSED)
        check(o, l, ro, rl, f"paged q_len=2 flags={flags} ctas={ctas}")


def test_repeated_calls_on_one_workspace_are_identical():
    """The counters return to zero after every call: a sequence of calls on
    one workspace gives the same bits each time."""
    import decode_attention_decoding_gb300 as fd
    w = syn.make_contiguous(3300, len(RAGGED), 8, 2, 128, 2112, RAGGED)
    dev = to_device(w)
    ws = fd.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, 128, 2112)
    outs = []
    for _ in range(4):
        o, l = run(w, dev, num_ctas=11, flags=FUSED, workspace=ws)
        outs.append((o, l))
    for o, l in outs[1:]:
        assert np.array_equal(o, outs[0][0]) and np.array_equal(l, outs[0][1])
    assert fd.fd_get_device_error(ws) == fd.FD_OK
    ro, rl = oracle.attend(w, threads=8)
    check(outs[0][0], outs[0][1], ro, rl, "repeated")


def test_one_workspace_across_launch_shapes():
    """Fused-head and unfused launches lay their partials out differently; the
    counters sit at the same place for every shape, so alternating them on
    one workspace stays correct."""
    import decode_attention_decoding_gb300 as fd
    lens = [3000, 2500, 0, 4000]
    w = syn.make_contiguous(3400, len(lens), 8, 4, 64, 4096, lens)
    dev = to_device(w)
    ws = fd.make_workspace(w.batch, w.num_q_heads, w.num_kv_heads, 64, 4096)
    ro, rl = oracle.attend(w, threads=8)
    for flags in (FUSE, NO_FUSION, FUSE, NO_FUSION, 0):
        o, l = run(w, dev, num_ctas=13, flags=flags | FUSED, workspace=ws)
        check(o, l, ro, rl, f"shared workspace flags={flags}")
    assert fd.fd_get_device_error(ws) == fd.FD_OK


def test_token_ranges():
    """Partial calls over token ranges merge inside the split kernel too."""
    import decode_attention_decoding_gb300 as fd
    w = syn.make_contiguous(3500, len(RAGGED), 8, 2, 128, 2112, RAGGED)
    dev = to_device(w)
    lens_h = torch.from_numpy(w.seq_lens.astype(np.int32))
    rows = w.num_q_heads
    for t0, t1 in ((0, 700), (700, 2112), (64, 65)):
        o, l = fd.fd_decode_partial(dev["q"], dev["k"][:, t0:].contiguous(), dev["v"][:, t0:].contiguous(),
                                    dev["seq_lens"], t0, t1, seq_lens_host=lens_h, scale=w.scale, num_ctas=17,
                                    flags=FUSED)
        items = np.array([[b, r, t0, t1] for b in range(w.batch) for r in range(rows)], dtype=np.int32)
        ro, rl = oracle.attend(w, items=items, threads=8)
        check(o.cpu().numpy().astype(np.float64).reshape(w.batch * rows, -1),
              l.cpu().numpy().astype(np.float64).reshape(-1), ro.reshape(w.batch * rows, -1), rl.reshape(-1),
              f"range [{t0}, {t1})")


def test_grid_of_many_waves():
    """1024 CTAs with tiles, several times the CTAs resident at once: segments
    whose CTAs run in different waves still merge (no CTA waits for another)."""
    lens = [20000, 17000, 1, 19999]
    w = syn.make_contiguous(3600, len(lens), 16, 4, 128, 20000, lens)
    ro, rl = oracle.attend(w, threads=16)
    for flags in (FUSED, 0):
        o, l = run(w, num_ctas=1024, flags=flags)
        check(o, l, ro, rl, f"1024 CTAs flags={flags}")
