"""Failure detection without a GPU fault: a wait that can never complete runs
out after a short limit, the kernel returns, the host reads FD_ERR_TIMEOUT,
and the context stays usable."""
import numpy as np
import pytest

import fd_synth as syn
import oracle
from gpu_util import check, run, to_device

pytestmark = pytest.mark.gpu


# page 0: contiguous (TMA); 16: page boxes (TMA); 4: rows copied with cp.async
# on the tensor-core consumers; 1 with one query head per kv head: gathered rows
@pytest.mark.parametrize("page,group", [(0, 4), (16, 4), (4, 4), (1, 1)])
def test_starved_wait_times_out_and_context_survives(page, group):
    import decode_attention_decoding_gb300 as fd
    from gpu_util import contig_to_paged
    paged = page > 0
    w = syn.make_contiguous(600, 2, 2 * group, 2, 128, 2000, [2000, 777])
    if paged:
        w = contig_to_paged(w, page, perm_seed=3)
    d = to_device(w)
    ws = fd.make_workspace(2, 2 * group, 2, 128, 2000, page)
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


def test_starved_wait_on_the_tmem_score_path():
    """The tcgen05 score kernel (E4M3, paired heads): the producer, the score
    issuer and the consumers all give up on the starved first tile, every
    warp reaches the kernel's last barrier and the tensor memory is freed;
    the host reads FD_ERR_TIMEOUT and later calls on the same context and
    workspace are correct."""
    import decode_attention_decoding_gb300 as fd
    w = syn.make_contiguous(601, 2, 8, 2, 128, 2000, [2000, 777], kv_dtype="e4m3", k_scale=0.05, v_scale=0.5)
    d = to_device(w)
    ws = fd.make_workspace(2, 8, 2, 128, 2000)
    flags = fd.FD_FLAG_FUSE_HEADS | fd.FD_FLAG_TMEM_SCORES
    fp8 = dict(kv_dtype="e4m3", k_scale=w.k_scale, v_scale=w.v_scale)
    fd.fd_decode(d["q"], d["k"], d["v"], d["seq_lens"], scale=w.scale, workspace=ws, num_ctas=4,
                 flags=flags | fd.FD_FLAG_TEST_STARVE_FIRST_TILE, wait_timeout_ns=50_000_000, **fp8)
    assert fd.fd_get_device_error(ws) == fd.FD_ERR_TIMEOUT
    o, l = run(w, d, workspace=ws, num_ctas=4, flags=flags)
    ro, rl = oracle.attend(w)
    check(o, l, ro, rl, "TMEM scores after timeout")
    assert fd.fd_get_device_error(ws) == fd.FD_OK
