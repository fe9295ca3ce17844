"""Sequence sharding on CPU ranks (gloo, world size 2 and 3): each rank holds
one range of cache positions and its oracle partial (output normalised over
the range, natural-log LSE); the library's exchange step stacks every rank's
partial in rank order, and the LSE merge of the stacked partials equals the
oracle's whole-cache result.  Covers several new tokens under the causal mask
(a rank whose range some query rows cannot see) and a request shorter than
the first rank's range (empty partials on the other ranks)."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BIG = 2 ** 31 - 1


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload(q_len):
    sys.path.insert(0, ROOT)
    import fd_synth as syn
    # request 3: with two new tokens, token 0 sees positions up to 199 and
    # token 1 up to 200, so the range starting at 200 holds one visible
    # position for token 1 and none for token 0
    return syn.make_contiguous(960 + q_len, 4, 8, 2, 64, 300, [300, 5, 170, 201], q_len=q_len)


def _ranges(world):
    cuts = {2: [0, 128, BIG], 3: [0, 100, 200, BIG]}[world]
    return list(zip(cuts[:-1], cuts[1:]))


def _partial(w, t0, t1):
    """The oracle's partial for every query row over positions [t0, t1)."""
    import oracle
    B, rows = w.batch, w.q_len * w.num_q_heads
    items = np.array([[b, r, t0, t1] for b in range(B) for r in range(rows)], dtype=np.int32)
    o, l = oracle.attend(w, items=items)
    return o.reshape(B, rows, -1), l.reshape(B, rows)


def _worker(rank, world, port, q_len, queue):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from decode_attention_decoding_gb300.seqshard import all_gather_partials
        w = _workload(q_len)
        t0, t1 = _ranges(world)[rank]
        o, l = _partial(w, t0, t1)
        o_all, l_all = all_gather_partials(torch.from_numpy(o), torch.from_numpy(l))
        queue.put((rank, o_all.numpy(), l_all.numpy(), o, l))
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("world,q_len", [(2, 1), (3, 1), (3, 2)])
def test_sharded_partials_exchange_and_merge_to_the_whole_cache(world, q_len):
    import oracle
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q_len, queue)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted((queue.get(timeout=240) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    own = [(o, l) for _, _, _, o, l in got]
    w = _workload(q_len)
    ref_o, ref_l = oracle.attend(w)
    B, rows = w.batch, w.q_len * w.num_q_heads
    ref_o, ref_l = ref_o.reshape(B, rows, -1), ref_l.reshape(B, rows)
    for rank, o_all, l_all, _, _ in got:
        assert o_all.shape == (world, B, rows, w.head_dim) and l_all.shape == (world, B, rows)
        for r in range(world):   # rank order, bit for bit
            assert np.array_equal(o_all[r], own[r][0]) and np.array_equal(l_all[r], own[r][1])
        for b in range(B):
            for i in range(rows):
                o, l = oracle.lse_merge(o_all[:, b, i], l_all[:, b, i])
                assert np.allclose(o, ref_o[b, i], rtol=1e-12, atol=1e-12), (rank, b, i)
                assert l == pytest.approx(ref_l[b, i], rel=1e-13, abs=1e-13)
    # the short request (5 tokens) sits in the first range alone
    assert np.all(np.isneginf(np.stack([l for _, l in own[1:]])[:, 1]))
    if world == 3 and q_len == 2:   # request 3 on the last rank: token 0 sees nothing, token 1 one position
        hq = w.num_q_heads
        assert np.all(np.isneginf(own[2][1][3, :hq])) and np.all(np.isfinite(own[2][1][3, hq:]))
