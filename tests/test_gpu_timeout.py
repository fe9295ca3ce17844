"""Failure detection without a GPU fault: a wait that can never complete runs
out after a short limit, the kernel returns, the host reads FD_ERR_TIMEOUT,
and the context stays usable."""
import numpy as np
import pytest

import fd_synth as syn
import oracle
from gpu_util import check, run, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("paged", [False, True])
def test_starved_wait_times_out_and_context_survives(paged):
    import decode_attention_decoding_gb300 as fd
    from gpu_util import contig_to_paged
    w = syn.make_contiguous(600, 2, 8, 2, 128, 2000, [2000, 777])
    if paged:
        w = contig_to_paged(w, 16, perm_seed=3)
    d = to_device(w)
    ws = fd.make_workspace(2, 8, 2, 128, 2000, 16 if paged else 0)
    kw = dict(scale=w.scale, workspace=ws, num_ctas=4, flags=fd.FD_FLAG_TEST_STARVE_FIRST_TILE,
              wait_timeout_ns=50_000_000)
    if paged:
        fd.fd_decode_paged(d["q"], d["k"], d["v"], d["block_table"], d["seq_lens"], **kw)
    else:
        fd.fd_decode(d["q"], d["k"], d["v"], d["seq_lens"], **kw)
    assert fd.fd_get_device_error(ws) == fd.FD_ERR_TIMEOUT
    # the same workspace and context still give correct results afterwards
    o, l = run(w, d, workspace=ws)
    ro, rl = oracle.attend(w)
    check(o, l, ro, rl, "after timeout")
    assert fd.fd_get_device_error(ws) == fd.FD_OK
