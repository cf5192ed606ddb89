"""GPU test of sba_ragged_decode_fwd_noalloc, the decode entry point for callers that
cannot allocate device memory when they call the library (device memory owned by
another allocator, plugin interfaces that only receive input and output buffers, loops
that must avoid the synchronisation of cudaMalloc/cudaFree).  It keeps the split
partials in a fixed array inside the library instead of a caller workspace.

This file is collected last so that a run stopping at the first failure has already run
every other test.  It must pass alone in a fresh process and after the other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

from selected_block_attention_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sba():
    import __graft_entry__

    __graft_entry__.build()
    import selected_block_attention_gb300 as m

    return m


def _kwargs(w):
    return dict(window_left=w.window_left, window_right=w.window_right,
                logits_soft_cap=w.logits_soft_cap, sink_bias=w.sink_bias)


def test_noalloc_matches_workspace_entry_point_twice(sba):
    """Two calls in a row through the C ABI (different rows, so the second call
    overwrites the shared partials of the first), each against the entry point that
    takes a caller workspace."""
    for seed, ends in ((900, [1, 17, 4096, 5000, 9000, 12000, 3, 700]),
                       (901, [12000, 1, 2, 8191, 64, 640, 6400, 11999])):
        w = workloads.decode(device=DEV, B=len(ends), Hq=32, Hkv=8, S=12000, window=(4096, 0),
                             cap=50.0, num_sinks=4, ends=ends, seed=seed)
        ref, ref_lse = sba.ragged_decode_fwd(w.q, w.k, w.v, w.sequence_start, w.sequence_end,
                                             **_kwargs(w))
        out = torch.full_like(w.q, float("nan"))
        lse = torch.full((w.q.shape[0], w.q.shape[1]), float("nan"), device=DEV)
        got, got_lse = sba.ragged_decode_fwd_noalloc(w.q, w.k, w.v, w.sequence_start,
                                                     w.sequence_end, out=out, lse=lse,
                                                     **_kwargs(w))
        sba.check_error()
        assert got.data_ptr() == out.data_ptr()
        # same kernels, same split count, same inputs: the results must be identical
        # (a loose tolerance could hide partials left in the shared array by the
        # previous call)
        assert torch.equal(got, ref), f"noalloc seed {seed}: output differs"
        assert torch.equal(got_lse, ref_lse), f"noalloc seed {seed}: LSE differs"


def test_noalloc_full_decode_workload(sba):
    """The B=64, S=32768, window (4096, 0) decode workload fits the built-in scratch."""
    w = workloads.decode(device=DEV)
    ref, ref_lse = sba.ragged_decode_fwd(w.q, w.k, w.v, w.sequence_start, w.sequence_end,
                                         **_kwargs(w))
    got, got_lse = sba.ragged_decode_fwd_noalloc(w.q, w.k, w.v, w.sequence_start,
                                                 w.sequence_end, **_kwargs(w))
    sba.check_error()
    assert torch.equal(got, ref) and torch.equal(got_lse, ref_lse), "noalloc full: differs"


def test_noalloc_rejects_sizes_beyond_the_scratch(sba):
    """No left window over a long cache needs more partials than the array holds."""
    lib = sba.load_library()
    need = lib.sba_ragged_decode_workspace_size(64, 32, 1 << 20, 128, -1)
    assert need > (16 << 20)
    q = torch.zeros((64, 32, 128), dtype=torch.bfloat16, device=DEV)
    kv = torch.zeros((64, 16, 8, 128), dtype=torch.bfloat16, device=DEV)  # never read
    se = torch.zeros(64, dtype=torch.int32, device=DEV)
    out = torch.empty_like(q)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.sba_ragged_decode_fwd_noalloc(
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kv.data_ptr()),
        ctypes.c_void_p(kv.data_ptr()), ctypes.c_void_p(se.data_ptr()),
        ctypes.c_void_p(se.data_ptr()), 64, 32, 8, 1 << 20, 128, 0.0, -1, -1, 0.0, None, 0, 0,
        ctypes.c_void_p(out.data_ptr()), None, stream)
    assert rc == -1
    assert b"16777216" in lib.sba_last_error()
