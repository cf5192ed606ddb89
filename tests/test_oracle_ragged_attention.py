"""Pins for the ragged multi-query attention oracle (CPU only).

Every expected value here comes from something other than the oracle's own loop:
torch's scaled-dot-product attention in float64 under masks built with
``tril`` / ``triu`` from the query positions, closed forms, or the separately
written decode oracle.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import ragged_decode_attention
from oracle.ragged_attention import query_position, ragged_flash_attention


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, mask, scale):
    """q [Q, H, D], k/v [K, H, D], mask [Q, K] bool (shared by heads)."""
    qt = torch.from_numpy(np.ascontiguousarray(q)).permute(1, 0, 2)
    kt = torch.from_numpy(np.ascontiguousarray(k)).permute(1, 0, 2)
    vt = torch.from_numpy(np.ascontiguousarray(v)).permute(1, 0, 2)
    m = mask.to(torch.bool)
    out = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    scores = ((qt @ kt.transpose(1, 2)) * scale).masked_fill(~m, -math.inf)
    return out.permute(1, 0, 2).numpy(), torch.logsumexp(scores, -1).permute(1, 0).numpy()


def _band(Q, K, start, end, left, right):
    """[Q, K] mask of queries at end - Q + i: keys in [start, end) and the band
    [p - left, p + right] (None = unbounded), built from tril / triu diagonals."""
    m = torch.ones(Q, K, dtype=torch.float64)
    off = end - Q                         # query i sits on diagonal i + off
    if right is not None:
        m = m.tril(diagonal=off + right)
    if left is not None:
        m = m.triu(diagonal=off - left)
    m[:, :start] = 0
    m[:, end:] = 0
    return m > 0


def test_query_positions_are_the_last_q_tokens():
    assert [query_position(10, 3, i) for i in range(3)] == [7, 8, 9]
    assert query_position(5, 1, 0) == 4          # a single query is the decode query


def test_full_causal_self_attention_equals_sdpa():
    """Q = K, the whole cache in range, right window 0: plain causal attention."""
    K, H, D = 40, 3, 8
    q, k, v = _rand((1, K, H, D), 1), _rand((1, K, H, D), 2), _rand((1, K, H, D), 3)
    out, lse = ragged_flash_attention(q, k, v, [0], [K], softmax_scale=0.37,
                                      window_left=-1, window_right=0)
    qt, kt, vt = (torch.from_numpy(x[0]).permute(1, 0, 2) for x in (q, k, v))
    ref = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.37)
    np.testing.assert_allclose(out[0], ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    causal = torch.ones(K, K, dtype=torch.bool).tril()
    _, ref_lse = _sdpa(q[0], k[0], v[0], causal, 0.37)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=0, atol=1e-12)


def test_no_window_every_query_sees_the_whole_range():
    B, Q, K, H, D = 2, 3, 30, 2, 8
    q, k, v = _rand((B, Q, H, D), 4), _rand((B, K, H, D), 5), _rand((B, K, H, D), 6)
    start, end = [4, 0], [21, 30]
    out, lse = ragged_flash_attention(q, k, v, start, end)
    for b in range(B):
        mask = torch.zeros(Q, K, dtype=torch.bool)
        mask[:, start[b]:end[b]] = True
        ref, ref_lse = _sdpa(q[b], k[b], v[b], mask, 1 / math.sqrt(D))
        np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], ref_lse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("left,right", [(5, 0), (0, 0), (7, 2), (None, 3), (4, None)])
def test_window_band_equals_masked_sdpa(left, right):
    B, Q, K, H, D = 1, 6, 48, 2, 8
    q, k, v = _rand((B, Q, H, D), 7), _rand((B, K, H, D), 8), _rand((B, K, H, D), 9)
    start, end = 3, 41
    out, lse = ragged_flash_attention(
        q, k, v, [start], [end], softmax_scale=0.5,
        window_left=-1 if left is None else left, window_right=-1 if right is None else right)
    mask = _band(Q, K, start, end, left, right)
    ref, ref_lse = _sdpa(q[0], k[0], v[0], mask, 0.5)
    np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=0, atol=1e-12)


def test_single_query_equals_decode_oracle():
    B, K, Hq, Hkv, D = 3, 64, 4, 2, 16
    q, k, v = _rand((B, 1, Hq, D), 10), _rand((B, K, Hkv, D), 11), _rand((B, K, Hkv, D), 12)
    bias = 0.3 * _rand((Hq, 3), 13)
    start, end = [0, 5, 2], [64, 40, 9]
    kw = dict(softmax_scale=0.2, window_left=9, window_right=0, logits_soft_cap=2.0,
              sink_bias=bias)
    out, lse = ragged_flash_attention(q, k, v, start, end, **kw)
    ref, ref_lse = ragged_decode_attention(q[:, 0], k, v, start, end, **kw)
    np.testing.assert_allclose(out[:, 0], ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[:, 0], ref_lse, rtol=0, atol=1e-12)


def test_gqa_equals_repeated_kv_heads():
    B, Q, K, Hq, Hkv, D = 1, 4, 32, 6, 2, 8
    q, k, v = _rand((B, Q, Hq, D), 14), _rand((B, K, Hkv, D), 15), _rand((B, K, Hkv, D), 16)
    kw = dict(window_left=6, window_right=0)
    out, lse = ragged_flash_attention(q, k, v, [2], [29], **kw)
    rep, rep_lse = ragged_flash_attention(q, np.repeat(k, 3, 2), np.repeat(v, 3, 2), [2], [29], **kw)
    np.testing.assert_allclose(out, rep, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, rep_lse, rtol=0, atol=1e-13)


def test_soft_cap_limits():
    B, Q, K, H, D = 1, 3, 20, 2, 8
    q, k, v = 3 * _rand((B, Q, H, D), 17), _rand((B, K, H, D), 18), _rand((B, K, H, D), 19)
    kw = dict(window_left=4, window_right=0)
    plain, plain_lse = ragged_flash_attention(q, k, v, [0], [K], **kw)
    huge, huge_lse = ragged_flash_attention(q, k, v, [0], [K], logits_soft_cap=1e30, **kw)
    np.testing.assert_allclose(huge, plain, rtol=0, atol=1e-12)
    np.testing.assert_allclose(huge_lse, plain_lse, rtol=0, atol=1e-12)
    # cap -> 0: every logit is ~0, so the weights are uniform over the 5 window keys
    tiny, tiny_lse = ragged_flash_attention(q, k, v, [0], [K], logits_soft_cap=1e-9, **kw)
    for i in range(Q):
        p = K - Q + i
        np.testing.assert_allclose(tiny[0, i], v[0, p - 4:p + 1].mean(0), rtol=0, atol=1e-8)
        np.testing.assert_allclose(tiny_lse[0, i], math.log(5), rtol=0, atol=1e-8)


def test_sinks_outside_the_window_and_their_bias():
    B, Q, K, H, D = 1, 4, 40, 2, 8
    q, k, v = _rand((B, Q, H, D), 20), _rand((B, K, H, D), 21), _rand((B, K, H, D), 22)
    left = 5
    # zero bias: the sinks are ordinary extra keys next to each query's band
    out, lse = ragged_flash_attention(q, k, v, [0], [K], window_left=left, window_right=0,
                                      sink_bias=np.zeros(3))
    mask = _band(Q, K, 0, K, left, 0)
    mask[:, :3] = True
    ref, ref_lse = _sdpa(q[0], k[0], v[0], mask, 1 / math.sqrt(D))
    np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=0, atol=1e-12)
    # a -1e30 bias removes the sinks again
    gone, gone_lse = ragged_flash_attention(q, k, v, [0], [K], window_left=left, window_right=0,
                                            sink_bias=np.full((H, 3), -1e30))
    plain, plain_lse = ragged_flash_attention(q, k, v, [0], [K], window_left=left, window_right=0)
    np.testing.assert_allclose(gone, plain, rtol=0, atol=1e-12)
    np.testing.assert_allclose(gone_lse, plain_lse, rtol=0, atol=1e-12)
    # a per-head bias b on sink 0 only: exp(b) weighs that key, closed form for one key
    only = ragged_flash_attention(q, k, v, [0], [K], window_left=0, window_right=0,
                                  sink_bias=np.array([[2.0], [-1.0]]))
    for i in range(Q):
        p = K - Q + i
        for h, b in ((0, 2.0), (1, -1.0)):
            s0 = q[0, i, h] @ k[0, 0, h] / math.sqrt(D) + b
            sp = q[0, i, h] @ k[0, p, h] / math.sqrt(D)
            w0 = 1 / (1 + math.exp(sp - s0))
            np.testing.assert_allclose(only[0][0, i, h], w0 * v[0, 0, h] + (1 - w0) * v[0, p, h],
                                       rtol=0, atol=1e-12)
            np.testing.assert_allclose(only[1][0, i, h], max(s0, sp) + math.log1p(math.exp(-abs(s0 - sp))),
                                       rtol=0, atol=1e-12)


def test_queries_before_the_range_are_empty():
    """Q larger than the row's range: with a right window of 0 the first queries sit
    before ``start`` and see nothing."""
    B, Q, K, H, D = 1, 6, 16, 2, 4
    q, k, v = _rand((B, Q, H, D), 23), _rand((B, K, H, D), 24), _rand((B, K, H, D), 25)
    out, lse = ragged_flash_attention(q, k, v, [8], [11], window_right=0)
    # positions 5..10: queries 0..2 are left of start = 8
    assert np.all(np.isneginf(lse[0, :3])) and np.all(out[0, :3] == 0.0)
    # query 3 sits at 8 = start: one key, out = v exactly, lse = its logit
    np.testing.assert_array_equal(out[0, 3], v[0, 8])
    np.testing.assert_allclose(lse[0, 3], np.einsum("hd,hd->h", q[0, 3], k[0, 8]) / 2.0,
                               rtol=0, atol=1e-14)
    # an empty range gives empty rows everywhere
    out, lse = ragged_flash_attention(q, k, v, [5], [5])
    assert np.all(np.isneginf(lse)) and np.all(out == 0.0)
