"""GPU parity: SparseMask bounds + block-sparse attention vs the fp64 oracle."""

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


def _run(sba, w, kv_block=128, rows=None, heads=None, softmax_scale=None):
    """Bounds from the oracle on the host arrays feed the oracle's attention, so the
    reference key set never comes from the CUDA path; the GPU bounds (which the GPU
    attention consumes) must equal them bit for bit."""
    m = w.mask
    np_ = lambda t: t.cpu().numpy()
    ref_bounds = oracle.sparse_mask_bounds(
        np_(m.q_positions), np_(m.q_segment_ids), np_(m.kv_positions), np_(m.kv_segment_ids),
        m.q_blocksize, kv_block, causal=m.causal, window_left=m.window_left,
        window_right=m.window_right, padding_segment_id=m.padding_segment_id)
    bounds = sba.sparse_mask_bounds(m.q_positions, m.q_segment_ids, m.kv_positions,
                                    m.kv_segment_ids, m.q_blocksize, kv_block, causal=m.causal,
                                    window_left=m.window_left, window_right=m.window_right,
                                    padding_segment_id=m.padding_segment_id)
    out, lse = sba.blocksparse_attn_fwd(w.q, w.k, w.v, m.q_positions, m.q_segment_ids,
                                        m.kv_positions, m.kv_segment_ids, *bounds, m.q_blocksize,
                                        kv_block, causal=m.causal, window_left=m.window_left,
                                        window_right=m.window_right,
                                        padding_segment_id=m.padding_segment_id,
                                        softmax_scale=softmax_scale)
    sba.check_error()
    for name, g, r in zip(("lower", "upper", "lower_full", "upper_full"), bounds, ref_bounds):
        assert np.array_equal(np_(g), r), f"GPU {name} bounds differ from the oracle's"
    ref, ref_lse = oracle.blocksparse_attention(
        to_np(w.q), to_np(w.k), to_np(w.v), np_(m.q_positions), np_(m.q_segment_ids),
        np_(m.kv_positions), np_(m.kv_segment_ids), ref_bounds[0], ref_bounds[1],
        m.q_blocksize, kv_block, causal=m.causal, window_left=m.window_left,
        window_right=m.window_right, padding_segment_id=m.padding_segment_id, rows=rows,
        heads=heads, softmax_scale=softmax_scale)
    got, gl = to_np(out), to_np(lse)
    if rows is not None:
        idx = tuple(np.array(rows).T)
        got, ref, gl, ref_lse = got[idx], ref[idx], gl[idx], ref_lse[idx]
    if heads is not None:
        got, ref, gl, ref_lse = got[..., heads, :], ref[..., heads, :], gl[..., heads], ref_lse[..., heads]
    return got, ref, gl, ref_lse


@pytest.mark.parametrize("kv_block,D", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_small(sba, kv_block, D):
    w = workloads.blocksparse(device=DEV, B=2, T=1024, Hq=4, Hkv=2, D=D, mean_doc=300,
                              pad_tail=70, window=(256, 0), seed=500 + kv_block + D)
    assert_attention_close(*_run(sba, w, kv_block=kv_block), what=f"bsa kb={kv_block} D={D}")


@pytest.mark.parametrize("kv_block,D", [(128, 128), (64, 64)])
def test_large_logits_rescale(sba, kv_block, D):
    """Scale 0.6 makes logits ~5-7x larger than 1/sqrt(D): running maxima jump by
    more than 2^8 between blocks, exercising the lazy rescale of O in TMEM."""
    w = workloads.blocksparse(device=DEV, B=1, T=1024, Hq=4, Hkv=1, D=D, mean_doc=500,
                              pad_tail=10, window=(300, 0), seed=700 + kv_block + D)
    assert_attention_close(*_run(sba, w, kv_block=kv_block, softmax_scale=0.6),
                           what=f"bsa large logits kb={kv_block} D={D}")


@pytest.mark.parametrize("window", [(-1, -1), (200, 50), (0, 0)])
def test_windows_and_noncausal(sba, window):
    w = workloads.blocksparse(device=DEV, B=1, T=768, Hq=2, Hkv=1, D=128, mean_doc=1000,
                              pad_tail=0, window=window, seed=600)
    w.mask.causal = window[0] != 200
    assert_attention_close(*_run(sba, w), what=f"bsa window {window}")


def test_full_size_sampled(sba):
    """B=4, T=16384, Hq=32, Hkv=8, window (1024, 0): 48 sampled tokens, all heads."""
    w = workloads.blocksparse(device=DEV)
    rng = np.random.default_rng(3)
    rows = [(int(b), int(t)) for b, t in zip(rng.integers(0, 4, 48), rng.integers(0, 16384, 48))]
    rows += [(0, 0), (3, 16383), (1, 16083), (2, 16084)]
    assert_attention_close(*_run(sba, w, rows=rows), what="bsa full sampled")


def test_first_item_of_every_cta(sba):
    """128 work items (B=2, 8 query blocks, 8 KV heads, one head pair each) on at most
    152 persistent CTAs: every CTA runs exactly one item, its first, so a hazard on a
    CTA's first item (operands read before they land, stale shared or tensor memory)
    shows in every row.  Every query block holds padding rows and a segment change.
    Run twice: the results must also be identical."""
    w = workloads.blocksparse(device=DEV, B=2, T=1024, Hq=16, Hkv=8, D=128, mean_doc=90,
                              pad_tail=0, window=(300, 0), seed=808)
    seg = w.mask.q_segment_ids.cpu().numpy().copy()
    for qb in range(8):
        seg[:, qb * 128 + 100:qb * 128 + 112] = -1  # padding inside every query block
    t = torch.from_numpy(seg.astype(np.int32)).to(DEV)
    w.mask.q_segment_ids = t
    w.mask.kv_segment_ids = t.clone()
    got, ref, gl, rl = _run(sba, w)
    assert_attention_close(got, ref, gl, rl, what="first items")
    got2, _, gl2, _ = _run(sba, w)
    assert np.array_equal(got, got2) and np.array_equal(gl, gl2), "second launch differs"


@pytest.mark.parametrize("kv_block", [128, 64])
def test_unsorted_segments_and_positions(sba, kv_block):
    """Key blocks whose positions are not consecutive or whose segment ids are not
    sorted take the per-key mask test; the others the per-row column interval.  Mixed
    here: random segment ids in half the rows' span, positions swapped inside a few
    blocks, padding tokens scattered."""
    w = workloads.blocksparse(device=DEV, B=2, T=1024, Hq=4, Hkv=2, D=128, mean_doc=400,
                              pad_tail=20, window=(-1, -1), seed=880 + kv_block)
    rng = np.random.default_rng(kv_block)
    seg = w.mask.q_segment_ids.cpu().numpy().copy()
    pos = w.mask.q_positions.cpu().numpy().copy()
    seg[:, 512:] = rng.integers(0, 3, size=(2, 512))
    seg[rng.random(seg.shape) < 0.03] = -1
    for blk in (1, 3, 6):
        a, b = blk * 128 + 5, blk * 128 + 70
        pos[:, [a, b]] = pos[:, [b, a]]
    to = lambda a: torch.from_numpy(a.astype(np.int32)).to(DEV)
    w.mask.q_segment_ids, w.mask.kv_segment_ids = to(seg), to(seg)
    w.mask.q_positions, w.mask.kv_positions = to(pos), to(pos)
    w.mask.causal = True
    assert_attention_close(*_run(sba, w, kv_block=kv_block), what=f"unsorted kb={kv_block}")
