"""Pins for the fp64 NSA selection backward oracle (CPU only).

The gradients are checked against things other than the oracle's own formulas:
central finite differences of the forward oracle (itself pinned in
test_oracle_nsa.py), torch float64 autograd of attention under a dense mask built
straight from the index array, torch autograd of causal scaled-dot-product
attention when every block is selected, and the invariances the definition implies
(order, -1 padding and duplicates of the indices; GQA as repeated KV heads; packed
sequences as separate ones; rows with nothing selected contribute nothing).
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import nsa_select_attention
from oracle.nsa_backward import nsa_select_attention_backward


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _messy_indices(rng, B, T, Hkv, S, bs, T_len=None):
    """Random ids including -1, out-of-range, future blocks and duplicates."""
    nb = -(-(T_len or T) // bs)
    idx = rng.integers(-2, nb + 2, size=(B, T, Hkv, S)).astype(np.int32)
    idx[..., 1] = idx[..., 0]  # a duplicate in every list
    counts = rng.integers(0, S + 2, size=(B, T, Hkv)).astype(np.int32)
    return idx, counts


def _dense_mask(idx, counts, T, bs, causal):
    """[B, Hkv, T, T] bool: token t may see key k (built from the index array with
    array operations, independently of the oracle's key-set code)."""
    B, _, Hkv, S = idx.shape
    nb = -(-T // bs)
    slot = np.arange(S)[None, None, None, :]
    use = (slot < np.clip(counts, 0, S)[..., None]) & (idx >= 0) & (idx < nb)
    chosen = np.zeros((B, T, Hkv, nb + 1), dtype=bool)
    safe = np.where(use, idx, nb)
    np.put_along_axis(chosen, safe, True, axis=-1)
    chosen = chosen[..., :nb]                                  # [B, T, Hkv, nb]
    key_blk = np.arange(T) // bs                               # [T]
    m = chosen[..., key_blk]                                   # [B, T, Hkv, T]
    if causal:
        m &= np.tril(np.ones((T, T), dtype=bool))[None, :, None, :]
    return m.transpose(0, 2, 1, 3)


def _torch_grads(q, k, v, mask, do, scale):
    """Autograd of softmax attention under a dense mask, float64.  q [B,T,Hq,D], k/v
    [B,T,Hkv,D], mask [B,Hkv,T,T]; rows with no key give output 0."""
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    kr = kt.repeat_interleave(G, dim=2)
    vr = vt.repeat_interleave(G, dim=2)
    m = torch.from_numpy(mask).repeat_interleave(G, dim=1)          # [B, Hq, T, T]
    scores = torch.einsum("bqhd,bkhd->bhqk", qt, kr) * scale
    scores = scores.masked_fill(~m, -math.inf)
    any_key = m.any(dim=-1, keepdim=True)
    p = torch.softmax(torch.where(any_key, scores, torch.zeros_like(scores)), dim=-1)
    p = torch.where(m, p, torch.zeros_like(p))
    out = torch.einsum("bhqk,bkhd->bqhd", p, vr)
    (out * torch.from_numpy(do)).sum().backward()
    return qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


@pytest.mark.parametrize("T,bs,Hq,Hkv,D,S,causal", [(40, 8, 4, 2, 6, 4, True), (33, 16, 3, 1, 5, 3, False),
                                                    (64, 32, 2, 2, 4, 2, True)])
def test_matches_autograd_of_dense_mask(T, bs, Hq, Hkv, D, S, causal):
    rng = np.random.default_rng(T + bs)
    B = 2
    q, k, v = _rand((B, T, Hq, D), 1), _rand((B, T, Hkv, D), 2), _rand((B, T, Hkv, D), 3)
    do = _rand((B, T, Hq, D), 4)
    idx, counts = _messy_indices(rng, B, T, Hkv, S, bs)
    scale = 0.41
    dq, dk, dv = nsa_select_attention_backward(q, k, v, idx, counts, bs, do, causal=causal,
                                               softmax_scale=scale)
    rq, rk, rv = _torch_grads(q, k, v, _dense_mask(idx, counts, T, bs, causal), do, scale)
    np.testing.assert_allclose(dq, rq, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, rk, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, rv, rtol=1e-9, atol=1e-11)


def test_central_finite_differences():
    """d/dx of sum(out * W) by central differences of the forward oracle, every
    element of q, k and v, h = 1e-5 (truncation error ~h^2)."""
    rng = np.random.default_rng(7)
    B, T, Hq, Hkv, D, bs, S = 1, 24, 4, 2, 3, 8, 3
    q, k, v = _rand((B, T, Hq, D), 11), _rand((B, T, Hkv, D), 12), _rand((B, T, Hkv, D), 13)
    W = _rand((B, T, Hq, D), 14)
    idx, counts = _messy_indices(rng, B, T, Hkv, S, bs)
    scale = 0.7

    def loss(qq, kk, vv):
        out, _ = nsa_select_attention(qq, kk, vv, idx, counts, bs, softmax_scale=scale)
        return float((out * W).sum())

    dq, dk, dv = nsa_select_attention_backward(q, k, v, idx, counts, bs, W, softmax_scale=scale)
    h = 1e-5
    for x, g, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
        num = np.zeros_like(x)
        for i in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[i] += h
            xm[i] -= h
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            num[i] = (loss(*args_p) - loss(*args_m)) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_all_blocks_equals_causal_sdpa_autograd():
    B, T, Hq, Hkv, D, bs = 1, 96, 4, 2, 8, 32
    q, k, v = _rand((B, T, Hq, D), 21), _rand((B, T, Hkv, D), 22), _rand((B, T, Hkv, D), 23)
    do = _rand((B, T, Hq, D), 24)
    nb = T // bs
    idx = np.broadcast_to(np.arange(nb, dtype=np.int32), (B, T, Hkv, nb)).copy()
    dq, dk, dv = nsa_select_attention_backward(q, k, v, idx, nb, bs, do)
    qt = torch.tensor(q, requires_grad=True)
    kt = torch.tensor(k, requires_grad=True)
    vt = torch.tensor(v, requires_grad=True)
    G = Hq // Hkv
    out = F.scaled_dot_product_attention(qt.transpose(1, 2), kt.repeat_interleave(G, 2).transpose(1, 2),
                                         vt.repeat_interleave(G, 2).transpose(1, 2), is_causal=True)
    (out.transpose(1, 2) * torch.from_numpy(do)).sum().backward()
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_invariant_to_order_padding_and_duplicates():
    rng = np.random.default_rng(31)
    B, T, Hq, Hkv, D, bs, S = 1, 64, 2, 1, 4, 16, 3
    q, k, v = _rand((B, T, Hq, D), 31), _rand((B, T, Hkv, D), 32), _rand((B, T, Hkv, D), 33)
    do = _rand((B, T, Hq, D), 34)
    idx = rng.integers(0, 4, size=(B, T, Hkv, S)).astype(np.int32)
    counts = np.full((B, T, Hkv), S, np.int32)
    base = nsa_select_attention_backward(q, k, v, idx, counts, bs, do)
    perm = idx[..., ::-1].copy()
    padded = np.concatenate([idx, np.full((B, T, Hkv, 2), -1, np.int32)], axis=-1)
    dup = np.concatenate([idx, idx[..., :1]], axis=-1)
    for alt, cnt in ((perm, counts), (padded, counts + 2), (dup, counts + 1)):
        got = nsa_select_attention_backward(q, k, v, alt, cnt, bs, do)
        for g, r in zip(got, base):
            np.testing.assert_allclose(g, r, rtol=1e-12, atol=1e-13)


def test_gqa_equals_repeated_kv_heads():
    rng = np.random.default_rng(41)
    B, T, Hkv, G, D, bs, S = 1, 48, 1, 3, 4, 16, 2
    q, k, v = _rand((B, T, Hkv * G, D), 41), _rand((B, T, Hkv, D), 42), _rand((B, T, Hkv, D), 43)
    do = _rand((B, T, Hkv * G, D), 44)
    idx = rng.integers(0, 3, size=(B, T, Hkv, S)).astype(np.int32)
    dq, dk, dv = nsa_select_attention_backward(q, k, v, idx, S, bs, do)
    # the same with one KV head per query head (K/V repeated): dk/dv sum over the copies
    rq, rk, rv = nsa_select_attention_backward(q, np.repeat(k, G, 2), np.repeat(v, G, 2),
                                               np.repeat(idx, G, 2), S, bs, do)
    np.testing.assert_allclose(dq, rq, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk, rk.reshape(B, T, Hkv, G, D).sum(3), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv, rv.reshape(B, T, Hkv, G, D).sum(3), rtol=1e-12, atol=1e-13)


def test_varlen_equals_separate_sequences():
    rng = np.random.default_rng(51)
    lens = [37, 20, 55]
    Hq, Hkv, D, bs, S = 2, 1, 4, 16, 3
    T = sum(lens)
    cu = np.cumsum([0] + lens)
    q, k, v = _rand((1, T, Hq, D), 51), _rand((1, T, Hkv, D), 52), _rand((1, T, Hkv, D), 53)
    do = _rand((1, T, Hq, D), 54)
    idx = rng.integers(-1, 4, size=(1, T, Hkv, S)).astype(np.int32)
    dq, dk, dv = nsa_select_attention_backward(q, k, v, idx, S, bs, do, cu_seqlens=cu)
    for s in range(len(lens)):
        sl = slice(cu[s], cu[s + 1])
        rq, rk, rv = nsa_select_attention_backward(q[:, sl], k[:, sl], v[:, sl], idx[:, sl], S, bs,
                                                   do[:, sl])
        np.testing.assert_allclose(dq[:, sl], rq, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dk[:, sl], rk, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(dv[:, sl], rv, rtol=1e-12, atol=1e-13)


def test_rows_with_nothing_selected_contribute_nothing():
    """Tokens whose lists hold only -1 (or only future blocks under causal masking)
    have a constant output: their dq is 0 and their d_out does not reach dk / dv."""
    B, T, Hq, Hkv, D, bs, S = 1, 64, 2, 1, 4, 16, 2
    q, k, v = _rand((B, T, Hq, D), 61), _rand((B, T, Hkv, D), 62), _rand((B, T, Hkv, D), 63)
    do = _rand((B, T, Hq, D), 64)
    idx = np.zeros((B, T, Hkv, S), np.int32)
    empty = [3, 10, 40]
    idx[0, empty[0]] = -1
    idx[0, empty[1]] = 2          # future block only
    idx[0, empty[1], :, 1] = 3
    idx[0, empty[2]] = -1
    dq, dk, dv = nsa_select_attention_backward(q, k, v, idx, S, bs, do)
    assert np.all(dq[0, empty] == 0.0)
    do0 = do.copy()
    do0[0, empty] = 0.0
    _, rk, rv = nsa_select_attention_backward(q, k, v, idx, S, bs, do0)
    np.testing.assert_array_equal(dk, rk)
    np.testing.assert_array_equal(dv, rv)


def test_single_key_row_closed_form():
    """Token 0 sees only key 0: p = 1, so dv_0 gets d_out_0 exactly, ds = 0 gives
    dq_0 = 0, and key 0's dk receives nothing from token 0."""
    B, T, Hq, Hkv, D, bs = 1, 16, 1, 1, 4, 16
    q, k, v = _rand((B, T, Hq, D), 71), _rand((B, T, Hkv, D), 72), _rand((B, T, Hkv, D), 73)
    do = np.zeros((B, T, Hq, D))
    do[0, 0, 0] = _rand((D,), 74)
    idx = np.zeros((B, T, Hkv, 1), np.int32)
    dq, dk, dv = nsa_select_attention_backward(q, k, v, idx, 1, bs, do)
    np.testing.assert_array_equal(dq[0, 0, 0], np.zeros(D))
    np.testing.assert_allclose(dv[0, 0, 0], do[0, 0, 0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(dk[0, 0, 0], np.zeros(D), atol=1e-15)
