"""GPU parity: ragged decode (split-KV + combine) vs the fp64 oracle."""

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


def _run(sba, w, rows=None, starts=None):
    if starts is not None:
        w.sequence_start = torch.as_tensor(starts, dtype=torch.int32, device=DEV)
    out, lse = sba.ragged_decode_fwd(w.q, w.k, w.v, w.sequence_start, w.sequence_end,
                                     window_left=w.window_left, window_right=w.window_right,
                                     logits_soft_cap=w.logits_soft_cap, sink_bias=w.sink_bias)
    sba.check_error()
    rows_l = list(range(w.q.shape[0])) if rows is None else list(rows)
    k = w.k[rows_l].double().cpu().numpy()
    v = w.v[rows_l].double().cpu().numpy()
    ref, ref_lse = oracle.ragged_decode_attention(
        to_np(w.q)[rows_l], k, v, w.sequence_start.cpu().numpy()[rows_l],
        w.sequence_end.cpu().numpy()[rows_l], window_left=w.window_left,
        window_right=w.window_right, logits_soft_cap=w.logits_soft_cap,
        sink_bias=None if w.sink_bias is None else w.sink_bias.cpu().numpy())
    return to_np(out)[rows_l], ref, to_np(lse)[rows_l], ref_lse


@pytest.mark.parametrize("G", [1, 4, 8, 16])
def test_small_group_sizes(sba, G):
    ends = [1, 15, 16, 17, 600, 2000, 2047, 2048]
    w = workloads.decode(device=DEV, B=len(ends), Hq=2 * G, Hkv=2, S=2048, window=(300, 0),
                         cap=50.0, num_sinks=4, ends=ends, seed=300 + G)
    assert_attention_close(*_run(sba, w), what=f"decode G={G}")


@pytest.mark.parametrize("window,cap,sinks", [((-1, -1), 0.0, 0), ((100, 0), 0.0, 0),
                                              ((100, 0), 2.0, 3), ((-1, -1), 50.0, 16),
                                              ((511, 0), 0.0, 1), ((0, 0), 0.0, 4)])
def test_small_feature_mix(sba, window, cap, sinks):
    ends = [1, 3, 40, 512, 513, 1024, 1500, 3000]
    w = workloads.decode(device=DEV, B=len(ends), Hq=8, Hkv=2, S=3000, window=window, cap=cap,
                         num_sinks=sinks, ends=ends, seed=400)
    assert_attention_close(*_run(sba, w), what=f"decode {window} {cap} {sinks}")


def test_shared_sink_bias_and_starts(sba):
    ends = [10, 100, 700, 700, 5]
    w = workloads.decode(device=DEV, B=5, Hq=8, Hkv=4, S=800, window=(64, 0), cap=0.0,
                         num_sinks=4, ends=ends, seed=401)
    w.sink_bias = w.sink_bias[0].contiguous()  # [num_sinks], shared by every head
    got, ref, gl, rl = _run(sba, w, starts=[0, 2, 600, 0, 5])
    assert np.isneginf(rl[4]).all()   # end <= start: empty row
    assert_attention_close(got, ref, gl, rl, what="shared sinks, starts")


def test_full_size_sampled(sba):
    """B=64, S=32768 cache, window (4096, 0), cap 50, 4 per-head sinks, in the
    benchmark's launch configuration; 8 sampled rows against the oracle."""
    w = workloads.decode(device=DEV)
    ends = w.sequence_end.cpu().numpy()
    rows = [0, 1, int(np.argmin(ends)), int(np.argmax(ends)), 17, 33, 50, 63]
    assert_attention_close(*_run(sba, w, rows=rows), what="decode full sampled")


def test_workspace_contract(sba):
    w = workloads.decode(device=DEV, B=2, Hq=8, Hkv=2, S=256, window=(-1, -1), cap=0.0,
                         num_sinks=0, ends=[256, 17], seed=402)
    need = sba.ragged_decode_workspace_size(2, 8, 256, 128, -1)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device=DEV)
    with pytest.raises(sba.SBAError):
        sba.ragged_decode_fwd(w.q, w.k, w.v, w.sequence_start, w.sequence_end, workspace=small)


def test_long_rows_beyond_the_parallel_combine(sba):
    """No window over a 200,000-key cache: 196 splits of 1,024 keys per row, more than
    the combining CTA stages in shared memory, so it merges them one at a time; a short
    row in the same launch uses the staged path."""
    ends = [200_000, 3_000]
    w = workloads.decode(device=DEV, B=2, Hq=8, Hkv=2, S=200_000, window=(-1, -1), cap=0.0,
                         num_sinks=2, ends=ends, seed=403)
    assert_attention_close(*_run(sba, w), what="decode long rows")


@pytest.mark.parametrize("cap,sinks", [(0.0, 0), (50.0, 4)])
def test_unowned_cache_slots_do_not_leak(sba, cap, sinks):
    """Cache slots outside a row's [start, end) belong to nobody (never written, here
    NaN).  Keys there are masked out of the softmax, and their values must not reach the
    output either: rows shorter than one 64-key stage, ranges that start mid-cache, ends
    just past a stage boundary, and a cache of fewer than 64 slots per row."""
    for S, ends, starts in [(700, [1, 5, 63, 64, 65, 129, 700, 300], [0, 3, 0, 10, 60, 100, 650, 0]),
                            (40, [1, 17, 40, 39], [0, 2, 30, 0])]:
        w = workloads.decode(device=DEV, B=len(ends), Hq=8, Hkv=2, S=S, window=(100, 0),
                             cap=cap, num_sinks=sinks, ends=ends, seed=404)
        w.sequence_start = torch.as_tensor(starts, dtype=torch.int32, device=DEV)
        for b, (st, en) in enumerate(zip(starts, ends)):
            for t in (w.k, w.v):
                t[b, :st] = float("nan")
                t[b, en:] = float("nan")
        got, ref, gl, rl = _run(sba, w)
        assert np.isfinite(got).all(), f"S={S}: NaN from unowned cache slots"
        assert_attention_close(got, ref, gl, rl, what=f"unowned slots S={S} cap={cap} sinks={sinks}")
