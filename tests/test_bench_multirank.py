"""The benchmark's multi-rank path on CPU (gloo, world size 2): the timed value
is the slowest rank's, every rank agrees on it, and the whole-job throughput
counts every rank's replica; the reference arm prints on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = [1.5, 4.0][rank]
    got = bench.max_over_ranks(ms, dist, "cpu")
    tbs = bench.whole_job_tbs(10 ** 9, world, got)
    dist.barrier()
    q.put((rank, got, tbs))
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [4.0, 4.0]
    for _, _, tbs in res:
        assert tbs == pytest.approx(2 * 1e9 / 4e-3 / 1e12)


def test_partial_count_matches_schedule_brute_force():
    """bench.partial_count mirrors the split schedule: tiles in contiguous runs
    of equal cost (+1 per tile, +w at each segment start), one partial per
    (CTA, segment) for segments split over several CTAs."""
    sys.path.insert(0, ROOT)
    import bench
    import numpy as np
    rng = np.random.default_rng(5)
    for _ in range(40):
        B = int(rng.integers(1, 20)); hkv = int(rng.choice([1, 2, 8])); P = int(rng.integers(1, 200))
        w = int(rng.choice([0, 1, 2]))
        lens = rng.integers(0, 5000, B)
        nt = (lens + 63) // 64
        owner, pos, x = [], [], 0
        for b in range(B):
            for h in range(hkv):
                for j in range(int(nt[b])):
                    x += w if j == 0 else 0
                    owner.append((b, h))
                    pos.append(x)
                    x += 1
        C = x
        Pe = min(P, C)   # CTAs that take tiles
        counts = {}
        for seg, p in zip(owner, pos):
            counts.setdefault(seg, set()).add(p * Pe // C)
        for cs in counts.values():   # a segment's CTAs are consecutive
            assert cs == set(range(min(cs), max(cs) + 1))
        expect = sum(len(cs) for cs in counts.values() if len(cs) > 1)
        assert bench.partial_count(lens, hkv, P, w) == expect


def test_reference_arm_rank1_prints_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_oracle_sample_bytes_count_each_kv_row_once():
    """The CPU baseline's bytes follow the GPU's algorithmic count: every
    (request, kv head) unit's K+V rows once, not once per query row of a GQA
    group, plus its q rows, O rows and LSEs."""
    sys.path.insert(0, ROOT)
    import bench
    import fd_synth as syn
    w = syn.make_contiguous(950, 3, 8, 2, 64, 100, [100, 7, 50])
    items, by, n = bench.oracle_units(w, 10 ** 6)
    assert n == 3 * 2 and items.shape == (3 * 8, 4)
    bc = bench.byte_counts(w, 152)
    assert by == bc["kv"] + bc["q"] + bc["out"]
    items, by, n = bench.oracle_units(w, 1)   # request 0, kv head 0: its four query rows
    assert n == 1 and sorted(items[:, 1].tolist()) == [0, 1, 2, 3]
    assert by == 100 * 64 * 2 * 2 + 4 * (64 * 2 + 64 * 4 + 4)
