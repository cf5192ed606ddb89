"""Pins for the block-sparse attention and ragged-decode oracles (CPU only)."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import blocksparse_attention, ragged_decode_attention, sparse_mask_bounds


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa_heads(q, k, v, mask, scale):
    """q [T, H, D], k/v [S, H, D], mask [T, S] (shared by heads)."""
    qt = torch.from_numpy(np.ascontiguousarray(q)).permute(1, 0, 2)
    kt = torch.from_numpy(np.ascontiguousarray(k)).permute(1, 0, 2)
    vt = torch.from_numpy(np.ascontiguousarray(v)).permute(1, 0, 2)
    m = torch.from_numpy(mask)
    out = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    scores = ((qt @ kt.transpose(1, 2)) * scale).masked_fill(~m, -math.inf)
    return out.permute(1, 0, 2).numpy(), torch.logsumexp(scores, -1).permute(1, 0).numpy()


# --------------------------------------------------------------------------- block-sparse

def test_blocksparse_full_range_equals_causal_dense():
    T, blk, Hq, Hkv, D = 96, 16, 4, 2, 8
    q, k, v = _rand((1, T, Hq, D), 1), _rand((1, T, Hkv, D), 2), _rand((1, T, Hkv, D), 3)
    pos = np.arange(T)[None]
    seg = np.zeros((1, T), np.int64)
    nb = T // blk
    lower = np.zeros((1, 1, nb), np.int32)
    upper = np.full((1, 1, nb), nb, np.int32)
    out, lse = blocksparse_attention(q, k, v, pos, seg, pos, seg, lower, upper, blk, blk,
                                     causal=True, softmax_scale=0.3)
    ref, ref_lse = _sdpa_heads(q[0], np.repeat(k[0], 2, 1), np.repeat(v[0], 2, 1),
                               np.tril(np.ones((T, T), bool)), 0.3)
    np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("window", [(-1, -1), (32, 0), (48, 16)])
def test_blocksparse_with_oracle_bounds_equals_dense_token_mask(window):
    """Documents + padding + window: with the bounds from the SparseMask oracle
    (window a multiple of the block), restricting to [lower, upper) drops no
    attending pair, so the result equals dense attention under the token mask."""
    rng = np.random.default_rng(4)
    T, blk, Hq, Hkv, D = 160, 16, 2, 1, 8
    seg = np.full(T, -1, np.int64)
    off, d = 0, 0
    while off < T - 12:
        L = int(rng.integers(5, 50))
        seg[off:min(off + L, T - 12)] = d
        off, d = off + L, d + 1
    pos = np.arange(T)
    wl, wr = window
    lo, up, lof, upf = sparse_mask_bounds(pos[None], seg[None], pos[None], seg[None], blk, blk,
                                          causal=True, window_left=wl, window_right=wr)
    q, k, v = _rand((1, T, Hq, D), 5), _rand((1, T, Hkv, D), 6), _rand((1, T, Hkv, D), 7)
    out, lse = blocksparse_attention(q, k, v, pos[None], seg[None], pos[None], seg[None], lo, up,
                                     blk, blk, causal=True, window_left=wl, window_right=wr)
    m = (seg[:, None] == seg[None, :]) & (seg[:, None] != -1) & (pos[None, :] <= pos[:, None])
    if wl >= 0:
        m &= pos[:, None] - pos[None, :] <= wl
    if wr >= 0:
        m &= pos[None, :] - pos[:, None] <= wr
    rows = m.any(1)
    ref, ref_lse = _sdpa_heads(q[0][rows], np.repeat(k[0], 2, 1), np.repeat(v[0], 2, 1), m[rows],
                               1 / math.sqrt(D))
    np.testing.assert_allclose(out[0][rows], ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse[0][rows], ref_lse, rtol=1e-10, atol=1e-12)
    assert np.all(out[0][~rows] == 0) and np.all(np.isneginf(lse[0][~rows]))


def test_blocksparse_bounds_restrict_keys():
    """Keys outside [lower, upper) are not seen even if the token mask allows them."""
    T, blk, D = 32, 8, 4
    q, k, v = _rand((1, T, 1, D), 8), _rand((1, T, 1, D), 9), _rand((1, T, 1, D), 10)
    pos = np.arange(T)[None]
    seg = np.zeros((1, T), np.int64)
    lower = np.array([[[0, 1, 3, 3]]], np.int32)
    upper = np.array([[[1, 2, 3, 4]]], np.int32)   # block 2 sees nothing
    out, lse = blocksparse_attention(q, k, v, pos, seg, pos, seg, lower, upper, blk, blk)
    assert np.all(out[0, 16:24] == 0) and np.all(np.isneginf(lse[0, 16:24]))
    # query 12 (block 1) sees keys 8..12 only
    s = (k[0, 8:13, 0] @ q[0, 12, 0]) / 2.0
    w = np.exp(s - s.max())
    np.testing.assert_allclose(out[0, 12, 0], (w / w.sum()) @ v[0, 8:13, 0], rtol=1e-12)


# --------------------------------------------------------------------------- decode

def _decode_inputs(B=3, Hq=4, Hkv=2, D=8, S=64, seed=11):
    return _rand((B, Hq, D), seed), _rand((B, S, Hkv, D), seed + 1), _rand((B, S, Hkv, D), seed + 2)


def test_decode_plain_equals_sdpa():
    q, k, v = _decode_inputs()
    start = np.array([0, 5, 17])
    end = np.array([64, 30, 18])
    out, lse = ragged_decode_attention(q, k, v, start, end, softmax_scale=0.4)
    for b in range(3):
        sl = slice(start[b], end[b])
        ref, ref_lse = _sdpa_heads(q[b][None], np.repeat(k[b, sl], 2, 1), np.repeat(v[b, sl], 2, 1),
                                   np.ones((1, end[b] - start[b]), bool), 0.4)
        np.testing.assert_allclose(out[b], ref[0], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse[0], rtol=1e-10, atol=1e-12)
    # a single key: out = v exactly
    np.testing.assert_array_equal(out[2], np.repeat(v[2, 17], 2, 0))


def test_decode_window_matches_sliced_range():
    q, k, v = _decode_inputs(seed=12)
    start, end = np.zeros(3, int), np.array([64, 40, 10])
    out, _ = ragged_decode_attention(q, k, v, start, end, window_left=7, window_right=0)
    for b in range(3):
        lo = max(0, end[b] - 1 - 7)
        ref, _ = ragged_decode_attention(q[b:b + 1], k[b:b + 1], v[b:b + 1], [lo], [end[b]])
        np.testing.assert_allclose(out[b], ref[0], rtol=1e-12, atol=1e-14)


def test_decode_cap_limits():
    q, k, v = _decode_inputs(seed=13)
    start, end = np.zeros(3, int), np.array([64, 33, 2])
    plain, plain_lse = ragged_decode_attention(q, k, v, start, end)
    big, big_lse = ragged_decode_attention(q, k, v, start, end, logits_soft_cap=1e9)
    np.testing.assert_allclose(big, plain, rtol=1e-9, atol=1e-12)
    # a tiny cap flattens every logit to ~0: uniform weights over the keys
    tiny, tiny_lse = ragged_decode_attention(q, k, v, start, end, logits_soft_cap=1e-7)
    for b in range(3):
        mean_v = np.repeat(v[b, :end[b]].mean(0), 2, 0)
        np.testing.assert_allclose(tiny[b], mean_v, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(tiny_lse[b], math.log(end[b]), atol=1e-6)
    # cap 2: every softmax weight ratio is bounded by e^(2 * 2)
    capped, _ = ragged_decode_attention(q * 30, k, v, start, end, logits_soft_cap=2.0)
    assert np.all(np.isfinite(capped))


def test_decode_sinks():
    q, k, v = _decode_inputs(B=2, Hq=4, Hkv=2, S=64, seed=14)
    start, end = np.zeros(2, int), np.array([64, 50])
    nowin, _ = ragged_decode_attention(q, k, v, start, end)
    # zero biases with a window covering the sinks == no sinks
    zero = np.zeros((4, 3))
    out, _ = ragged_decode_attention(q, k, v, start, end, window_left=100, sink_bias=zero)
    np.testing.assert_allclose(out, nowin, rtol=1e-12, atol=1e-14)
    # window excludes the sinks, bias -1e30: sinks drop out -> equals the window alone
    out2, _ = ragged_decode_attention(q, k, v, start, end, window_left=5, sink_bias=np.full(3, -1e30))
    win, _ = ragged_decode_attention(q, k, v, start, end, window_left=5)
    np.testing.assert_allclose(out2, win, rtol=1e-12, atol=1e-14)
    # a huge per-head bias on one sink, added after the (tiny) cap: that sink wins,
    # for head h sink h % 3
    bias = np.zeros((4, 3))
    for h in range(4):
        bias[h, h % 3] = 1e3
    out3, lse3 = ragged_decode_attention(q, k, v, start, end, window_left=5, logits_soft_cap=1e-3,
                                         sink_bias=bias)
    for b in range(2):
        for h in range(4):
            np.testing.assert_allclose(out3[b, h], v[b, h % 3, h // 2], rtol=1e-12, atol=1e-12)
    # sinks are kept although outside the window: 3 sinks + 6 window keys
    counts = ragged_decode_attention(q, k, v, start, end, window_left=5, logits_soft_cap=1e-9,
                                     sink_bias=np.zeros(3))[1]
    np.testing.assert_allclose(counts, math.log(9), atol=1e-6)


def test_decode_empty_row():
    q, k, v = _decode_inputs(B=2, seed=15)
    out, lse = ragged_decode_attention(q, k, v, np.array([4, 0]), np.array([4, 3]))
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))
