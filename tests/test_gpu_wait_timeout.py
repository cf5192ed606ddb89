"""Failure detection of the warp-specialised kernels, on the GPU without a fault.

Every internal wait of the tensor-core kernels is bounded.  Here the bound is set far
below the time a wait normally takes (100 SM cycles: a TMA load or an MMA takes longer),
so the first wait that is not already satisfied gives up: the kernel records where, every
other wait of its CTA returns at once, the copies in flight are drained, tensor memory is
freed and the launch returns.  The host then reads SBA_ERR_TIMEOUT with the location, and
a launch with the default bound on the same context passes parity against the oracle.
Nothing here hangs or faults: every wait, including the drain, is bounded.
"""

import numpy as np
import pytest
import torch

import oracle
from selected_block_attention_gb300 import workloads
from tests._parity import assert_attention_close, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sba():
    import __graft_entry__

    __graft_entry__.build()
    import selected_block_attention_gb300 as m

    yield m
    m.set_wait_timeout_cycles(0)


def _blocksparse(sba, w):
    m = w.mask
    bnd = sba.sparse_mask_bounds(m.q_positions, m.q_segment_ids, m.kv_positions, m.kv_segment_ids,
                                 128, 128, causal=True, window_left=m.window_left,
                                 window_right=m.window_right)
    out, lse = sba.blocksparse_attn_fwd(w.q, w.k, w.v, m.q_positions, m.q_segment_ids,
                                        m.kv_positions, m.kv_segment_ids, *bnd, 128, 128,
                                        causal=True, window_left=m.window_left,
                                        window_right=m.window_right)
    return out, lse


def _nsa(sba, w):
    return sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts, w.block_size,
                              causal=True)


def test_wait_limit_setting(sba):
    default = sba.get_wait_timeout_cycles()
    assert default == 4_000_000_000
    sba.set_wait_timeout_cycles(12345)
    assert sba.get_wait_timeout_cycles() == 12345
    sba.set_wait_timeout_cycles(0)
    assert sba.get_wait_timeout_cycles() == default
    with pytest.raises(sba.SBAError):
        sba.set_wait_timeout_cycles(-1)


@pytest.mark.parametrize("kernel", ["blocksparse_attn", "nsa_select"])
def test_timeout_is_reported_and_the_next_launch_is_exact(sba, kernel):
    if kernel == "blocksparse_attn":
        w = workloads.blocksparse(device=DEV, B=1, T=2048, Hq=4, Hkv=2, D=128, mean_doc=600,
                                  pad_tail=30, window=(512, 0), seed=321)
        run = lambda: _blocksparse(sba, w)
    else:
        w = workloads.nsa_prefill(device=DEV, B=1, T=2048, Hq=16, Hkv=1, D=128, seed=322)
        run = lambda: _nsa(sba, w)
    sba.check_error()  # nothing pending from earlier tests
    sba.set_wait_timeout_cycles(100)
    try:
        run()
        with pytest.raises(sba.SBAError) as e:
            sba.check_error()
    finally:
        sba.set_wait_timeout_cycles(0)
    assert e.value.code == -4, str(e.value)
    assert f"[{kernel} role" in str(e.value), str(e.value)
    # the error word was cleared by the read; the context is usable and exact again
    out, lse = run()
    sba.check_error()
    if kernel == "blocksparse_attn":
        m = w.mask
        host = [t.cpu().numpy() for t in (m.q_positions, m.q_segment_ids, m.kv_positions,
                                          m.kv_segment_ids)]
        rb = oracle.sparse_mask_bounds(*host, 128, 128, causal=True, window_left=m.window_left,
                                       window_right=m.window_right)
        rows = [(0, t) for t in range(0, 2048, 13)]
        ref, ref_lse = oracle.blocksparse_attention(
            to_np(w.q), to_np(w.k), to_np(w.v), *host, rb[0], rb[1], 128, 128, causal=True,
            window_left=m.window_left, window_right=m.window_right, rows=rows)
    else:
        rows = [(0, t) for t in range(0, 2048, 13)]
        ref, ref_lse = oracle.nsa_select_attention(
            to_np(w.q), to_np(w.k), to_np(w.v), w.block_indices.cpu().numpy(),
            w.block_counts.cpu().numpy(), w.block_size, rows=rows)
    idx = tuple(np.array(rows).T)
    assert_attention_close(to_np(out)[idx], ref[idx], to_np(lse)[idx], ref_lse[idx],
                           what=f"{kernel} after a timeout")
