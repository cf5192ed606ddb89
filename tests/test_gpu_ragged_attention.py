"""GPU parity: ragged multi-query attention (split-KV + combine) vs the fp64 oracle."""

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

    return m


def _gpu(sba, w):
    out, lse = sba.ragged_flash_attention_fwd(
        w.q, w.k, w.v, w.sequence_start, w.sequence_end, window_left=w.window_left,
        window_right=w.window_right, logits_soft_cap=w.logits_soft_cap, sink_bias=w.sink_bias)
    sba.check_error()
    return out, lse


def _compare(sba, w, rows=None, what=""):
    """rows: None (every (b, i)) or a list of (b, i) pairs."""
    out, lse = _gpu(sba, w)
    B, Q = w.q.shape[:2]
    pairs = [(b, i) for b in range(B) for i in range(Q)] if rows is None else list(rows)
    bs = sorted({b for b, _ in pairs})
    remap = {b: j for j, b in enumerate(bs)}
    ref, ref_lse = oracle.ragged_flash_attention(
        to_np(w.q)[bs], w.k[bs].float().cpu().numpy(), w.v[bs].float().cpu().numpy(),
        w.sequence_start.cpu().numpy()[bs], w.sequence_end.cpu().numpy()[bs],
        window_left=w.window_left, window_right=w.window_right,
        logits_soft_cap=w.logits_soft_cap,
        sink_bias=None if w.sink_bias is None else w.sink_bias.cpu().numpy(),
        rows=[(remap[b], i) for b, i in pairs])
    got, got_lse = to_np(out), to_np(lse)
    g = np.stack([got[b, i] for b, i in pairs])
    gl = np.stack([got_lse[b, i] for b, i in pairs])
    r = np.stack([ref[remap[b], i] for b, i in pairs])
    rl = np.stack([ref_lse[remap[b], i] for b, i in pairs])
    return assert_attention_close(g, r, gl, rl, what=what)


@pytest.mark.parametrize("Q,Hq,Hkv", [(1, 8, 2), (2, 8, 2), (4, 8, 2), (3, 12, 1), (5, 16, 1),
                                      (37, 6, 2), (64, 2, 2), (9, 4, 4)])
def test_query_and_group_shapes(sba, Q, Hq, Hkv):
    """Row tiles of 16 (query, head) pairs: one tile, tiles straddling queries, a ragged
    last tile, one query per tile (G = 16), the page's Hkv = Hq case."""
    ends = [1, Q, Q + 15, 300, 513, 1200, 1999, 2048]
    w = workloads.ragged_attention(device=DEV, B=len(ends), Q=Q, Hq=Hq, Hkv=Hkv, S=2048,
                                   window=(300, 0), cap=50.0, num_sinks=4, ends=ends,
                                   seed=500 + Q)
    _compare(sba, w, what=f"mq Q={Q} Hq={Hq} Hkv={Hkv}")


@pytest.mark.parametrize("window,cap,sinks", [((-1, -1), 0.0, 0), ((-1, 0), 0.0, 0),
                                              ((100, 3), 2.0, 3), ((0, 0), 0.0, 4),
                                              ((511, 0), 0.0, 16), ((40, -1), 50.0, 2),
                                              ((-1, 7), 5.0, 0)])
def test_window_cap_sink_mix(sba, window, cap, sinks):
    """Both window sides (a look-ahead right window included), soft caps, 0-16 sinks;
    several splits per row (no window over a 3000-key cache)."""
    ends = [3, 40, 512, 513, 1024, 1500, 2999, 3000]
    w = workloads.ragged_attention(device=DEV, B=len(ends), Q=6, Hq=8, Hkv=2, S=3000,
                                   window=window, cap=cap, num_sinks=sinks, ends=ends, seed=510)
    _compare(sba, w, what=f"mq {window} {cap} {sinks}")


def test_ragged_starts_empty_rows_and_queries_before_start(sba):
    """start > 0; end <= start (all queries empty); more queries than the range holds
    (queries left of start see only in-range sinks); a shared [num_sinks] bias."""
    ends = [10, 100, 700, 700, 5, 20]
    starts = [0, 2, 600, 0, 5, 1]
    w = workloads.ragged_attention(device=DEV, B=6, Q=8, Hq=8, Hkv=4, S=800, window=(64, 0),
                                   cap=0.0, num_sinks=4, ends=ends, starts=starts, seed=511)
    w.sink_bias = w.sink_bias[0].contiguous()
    _compare(sba, w, what="mq starts / empty")
    _, lse = _gpu(sba, w)
    assert torch.isneginf(lse[4]).all()          # end == start
    # row 2: range [600, 700), queries at 692..699 see their windows only (no sinks in range)
    assert torch.isfinite(lse[2]).all()


def test_sinks_seen_from_queries_left_of_the_range(sba):
    """Q = 8 over a 3-token range [1, 4) with right window 0: queries 0..3 sit at
    -4..-1 (nothing in their window) but sinks 1..3 are in range, so they are not empty."""
    w = workloads.ragged_attention(device=DEV, B=1, Q=8, Hq=4, Hkv=2, S=64, window=(2, 0),
                                   cap=0.0, num_sinks=4, ends=[4], starts=[1], seed=512)
    _compare(sba, w, what="mq sinks left of range")
    _, lse = _gpu(sba, w)
    assert torch.isfinite(lse).all()


def test_sinks_right_of_a_tile_window(sba):
    """G = 16: every row tile is one query.  With end = 12 and window (2, 0) the tile of
    query 0 (position 4) has window [2, 5) while sinks run to 9: sinks on both sides of
    the tile's window."""
    w = workloads.ragged_attention(device=DEV, B=2, Q=8, Hq=16, Hkv=1, S=64, window=(2, 0),
                                   cap=0.0, num_sinks=10, ends=[12, 64], seed=516)
    _compare(sba, w, what="mq sinks right of window")


def test_single_query_matches_decode(sba):
    """Q = 1 is the decode operation: both entry points agree with each other."""
    w = workloads.ragged_attention(device=DEV, B=8, Q=1, Hq=16, Hkv=4, S=2048, window=(500, 0),
                                   cap=50.0, num_sinks=4, seed=513)
    out, lse = _gpu(sba, w)
    dout, dlse = sba.ragged_decode_fwd(w.q[:, 0].contiguous(), w.k, w.v, w.sequence_start,
                                       w.sequence_end, window_left=500, window_right=0,
                                       logits_soft_cap=50.0, sink_bias=w.sink_bias)
    sba.check_error()
    assert_attention_close(to_np(out[:, 0]), to_np(dout), to_np(lse[:, 0]), to_np(dlse),
                           what="Q=1 vs decode")


def test_spec_decode_full_size_sampled(sba):
    """B=64 rows verifying Q=4 tokens each against an S=32768 cache, Hq=32, Hkv=8,
    window (4096, 0), cap 50, 4 per-head sinks, in the benchmark's launch
    configuration; sampled rows against the oracle."""
    w = workloads.ragged_attention(device=DEV)
    ends = w.sequence_end.cpu().numpy()
    bs = [0, 1, int(np.argmin(ends)), int(np.argmax(ends)), 17, 33, 50, 63]
    rows = [(b, i) for b in bs for i in range(4)]
    _compare(sba, w, rows=rows, what="mq spec-decode full sampled")


def test_chunked_prefill_sampled(sba):
    """B=4 rows appending a 512-token chunk to an S=16384 cache (Hq=32, Hkv=8, window
    (-1, 0): causal over the whole prefix); sampled queries against the oracle."""
    w = workloads.ragged_attention(device=DEV, B=4, Q=512, S=16384, window=(-1, 0), cap=0.0,
                                   num_sinks=0, seed=514)
    rows = [(b, i) for b in range(4) for i in (0, 1, 255, 256, 510, 511)]
    _compare(sba, w, rows=rows, what="mq chunked prefill sampled")


def test_workspace_contract(sba):
    w = workloads.ragged_attention(device=DEV, B=2, Q=3, Hq=8, Hkv=2, S=256, window=(32, 0),
                                   seed=515)
    need = sba.ragged_flash_attention_workspace_size(2, 3, 8, 256, 128, 32, 0)
    short = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(sba.SBAError):
        sba.ragged_flash_attention_fwd(w.q, w.k, w.v, w.sequence_start, w.sequence_end,
                                       window_left=32, window_right=0, workspace=short)


@pytest.mark.parametrize("Q,Hq,Hkv,S,window", [
    (128, 4, 2, 1000, (-1, 0)),      # exactly one query block, causal prefix
    (200, 4, 2, 1000, (300, 0)),     # partial last query block, left window
    (300, 3, 1, 777, (-1, -1)),      # odd G (a head slot of its own), no window, S % 128 != 0
    (256, 2, 2, 900, (100, 20)),     # G = 1 (the page's Hkv = Hq), look-ahead right window
    (160, 8, 2, 640, (0, 0)),        # one key per query
])
def test_long_chunks_on_the_block_pipeline(sba, Q, Hq, Hkv, S, window):
    """Q >= 128 without cap or sinks runs on the tensor-memory block pipeline: every
    (query, head) row against the oracle, with ragged starts / ends, an empty row and a
    row whose first queries sit left of its range."""
    ends = [S, S - 37, Q // 2, 600 % S + 1]
    starts = [0, 5, 0, 600 % S + 1]          # the last row is empty (end == start)
    w = workloads.ragged_attention(device=DEV, B=4, Q=Q, Hq=Hq, Hkv=Hkv, S=S, window=window,
                                   cap=0.0, num_sinks=0, ends=ends, starts=starts,
                                   seed=520 + Q)
    _compare(sba, w, what=f"mq block pipeline Q={Q} Hq={Hq} Hkv={Hkv} S={S} {window}")
    _, lse = _gpu(sba, w)
    assert torch.isneginf(lse[3]).all()



@pytest.mark.parametrize("B,equal", [(5, True), (40, False)])
def test_block_pipeline_row_order(sba, B, equal):
    """The block pipeline hands rows out longest first when there are at most 32 of them
    (ties by index) and in index order otherwise: rows of equal lengths, and more than 32
    rows of mixed lengths, against the oracle."""
    Q, S = 128, 512
    rng = np.random.default_rng(530 + B)
    ends = [S] * B if equal else [int(x) for x in rng.integers(Q, S + 1, size=B)]
    w = workloads.ragged_attention(device=DEV, B=B, Q=Q, Hq=4, Hkv=2, S=S, window=(-1, 0),
                                   cap=0.0, num_sinks=0, ends=ends, seed=530 + B)
    _compare(sba, w, what=f"mq block pipeline row order B={B} equal={equal}")