"""The five benchmark workloads at full size, in the launch configuration the
benchmark times (planner defaults), checked against the oracle on a sample of
query rows (every row the oracle computes is compared elementwise)."""
import numpy as np
import pytest

import fd_synth as syn
import oracle
from gpu_util import check, run, sample_items

pytestmark = pytest.mark.gpu


_CACHE = {}


def workload(config_id):
    if config_id not in _CACHE:
        _CACHE.clear()
        _CACHE[config_id] = syn.make_config(config_id)
    return _CACHE[config_id]


# flags 2 = FD_FLAG_CUDA_CORES: the GQA workloads are checked on both consumer paths
@pytest.mark.parametrize("config_id,flags", [(1, 0), (2, 0), (3, 0), (3, 2), (4, 0), (4, 2), (5, 0), (5, 2)])
def test_full_size_config_sampled(config_id, flags):
    from decode_attention_decoding_gb300 import build
    build.build()
    w = workload(config_id)
    o, l = run(w, flags=flags)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    items = sample_items(w, 24, seed=config_id)
    if config_id == 1:          # small enough for every row
        items = None
    ro, rl = oracle.attend(w, items=items, threads=16)
    if items is None:
        stats = check(o, l, ro, rl, f"config {config_id}")
    else:
        b, h = items[:, 0], items[:, 1]
        stats = check(o[b, h], l[b, h], ro, rl, f"config {config_id}")
    print(f"config {config_id} flags={flags}: max|dO|={stats[0]:.3g} max rel(|r|>=1e-2)={stats[1]:.3g} "
          f"max|dLSE|={stats[2]:.3g}")
