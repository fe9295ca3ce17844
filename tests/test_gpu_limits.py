"""The library at the edges of what it accepts: the largest batch, the
largest CTA count (several waves of persistent CTAs), and the thresholds
inside the merge (batches of up to 32 take the segment geometry from the
lengths, larger ones from the workspace; segments split up to 16 ways are
merged in one load round trip, more ways through shared memory)."""
import numpy as np
import pytest

import fd_synth as syn
import oracle
from gpu_util import check, contig_to_paged, run, sample_items

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from decode_attention_decoding_gb300 import build
    build.build()
    oracle.build()


def sampled_check(w, o, l, n, seed, what):
    items = sample_items(w, n, seed)
    ro, rl = oracle.attend(w, items=items, threads=8)
    rows = items[:, 0], items[:, 1]
    check(o[rows], l[rows], ro, rl, what)


@pytest.mark.parametrize("flags", [0, 0x2])
def test_largest_batch(flags):
    """4096 requests (the limit), lengths 0..300 with empty ones among them."""
    B = 4096
    lens = syn.randint(77, B, 0, 300).astype(np.int32)
    lens[::97] = 0
    w = syn.make_contiguous(3000, B, 8, 2, 128, 300, lens)
    o, l = run(w, flags=flags)
    sampled_check(w, o, l, 400, 1, f"B=4096 flags={flags}")
    empty = np.nonzero(lens == 0)[0]
    assert np.all(o[empty] == 0) and np.all(l[empty] == -np.inf)


@pytest.mark.parametrize("page", [0, 16])
def test_largest_cta_count(page):
    """1024 persistent CTAs: more than fit at once, so they run in waves."""
    lens = [5000, 1, 3000, 0, 777, 4096]
    w = syn.make_contiguous(3010, len(lens), 8, 2, 128, 5000, lens)
    if page:
        w = contig_to_paged(w, page, perm_seed=3)
    ro, rl = oracle.attend(w, threads=8)
    o, l = run(w, num_ctas=1024)
    check(o, l, ro, rl, f"1024 CTAs P={page}")


@pytest.mark.parametrize("batch", [31, 32, 33, 64])
def test_merge_geometry_threshold(batch):
    """Batches of up to 32 derive the merge geometry from the lengths, larger
    ones read the workspace prefix; both must agree with the oracle."""
    lens = syn.randint(90 + batch, batch, 0, 1500).astype(np.int32)
    w = syn.make_contiguous(3020 + batch, batch, 8, 2, 128, 1500, lens)
    ro, rl = oracle.attend(w, threads=8)
    for ctas in (0, 37):
        o, l = run(w, num_ctas=ctas)
        check(o, l, ro, rl, f"B={batch} ctas={ctas}")


@pytest.mark.parametrize("ctas,flags", [(12, 0), (16, 0), (17, 0), (152, 0), (500, 0x2)])
def test_segment_split_many_ways(ctas, flags):
    """One long segment split over `ctas` CTAs: up to 16 partials take the
    one-round-trip merge, more the staged one."""
    L = 70000
    w = syn.make_contiguous(3030, 1, 1, 1, 128, L, [L])
    ro, rl = oracle.attend(w)
    o, l = run(w, num_ctas=ctas, flags=flags)
    check(o, l, ro, rl, f"split {ctas} ways")


def test_no_length_array_means_full_length():
    """seq_lens = NULL: every request spans s_max (the merge derives its
    geometry from the capacity then)."""
    import torch
    import decode_attention_decoding_gb300 as fd
    from gpu_util import to_device
    S = 3000
    w = syn.make_contiguous(3040, 3, 8, 2, 128, S, [S, S, S])
    ro, rl = oracle.attend(w, threads=8)
    dev = to_device(w)
    for ctas in (0, 7):
        o, l = fd.fd_decode(dev["q"], dev["k"], dev["v"], None, scale=w.scale, num_ctas=ctas)
        torch.cuda.synchronize()
        check(o.cpu().numpy().astype(np.float64), l.cpu().numpy().astype(np.float64), ro, rl,
              f"no lengths ctas={ctas}")
