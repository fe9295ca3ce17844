"""The five benchmark workloads at full size, in the launch configuration the
benchmark times (planner defaults), checked against the oracle on every query
row, elementwise."""
import os

import numpy as np
import pytest

import fd_synth as syn
import oracle
from gpu_util import check, repage, run

THREADS = os.cpu_count() or 1

pytestmark = pytest.mark.gpu


_CACHE = {}


def workload(config_id, kv=None):
    key = (config_id, kv)
    if key not in _CACHE:
        _CACHE.clear()
        _CACHE[key] = syn.make_config(config_id, kv_dtype=kv)
    return _CACHE[key]


# flags 2 = FD_FLAG_CUDA_CORES: the GQA workloads are checked on both consumer paths;
# kv: the benchmark's FP8 variants of the workloads (bench.py --kv)
@pytest.mark.parametrize("config_id,flags,kv", [(1, 0, None), (2, 0, None), (3, 0, None), (3, 2, None),
                                                (4, 0, None), (4, 2, None), (5, 0, None), (5, 2, None),
                                                (2, 0, "e4m3"), (3, 0, "e5m2"), (4, 0, "e4m3"),
                                                (5, 0, "e4m3"), (5, 2, "e4m3")])
def test_full_size_config_sampled(config_id, flags, kv):
    from decode_attention_decoding_gb300 import build
    build.build()
    w = workload(config_id, kv)
    o, l = run(w, flags=flags)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    ro, rl = oracle.attend(w, threads=THREADS)
    stats = check(o, l, ro, rl, f"config {config_id} kv={kv}")
    print(f"config {config_id} flags={flags} kv={kv}: max|dO|={stats[0]:.3g} max rel(|r|>=1e-2)={stats[1]:.3g} "
          f"max|dLSE|={stats[2]:.3g}")


# Small pages at full size: workload 4 on one-token pages (tensor cores with
# cp.async rows; CUDA cores with gathered rows), workload 5 on four-token pages,
# workload 2 (MHA) on two-token pages (gathered rows).
@pytest.mark.parametrize("config_id,page,flags", [(4, 1, 0), (4, 1, 2), (5, 4, 0), (2, 2, 0)])
def test_full_size_config_small_pages_sampled(config_id, page, flags):
    from decode_attention_decoding_gb300 import build
    build.build()
    w = repage(workload(config_id), page, perm_seed=100 + page)
    o, l = run(w, flags=flags)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    ro, rl = oracle.attend(w, threads=THREADS)
    stats = check(o, l, ro, rl, f"config {config_id} P={page} flags={flags}")
    print(f"config {config_id} P={page} flags={flags}: max|dO|={stats[0]:.3g} max rel={stats[1]:.3g} "
          f"max|dLSE|={stats[2]:.3g}")
