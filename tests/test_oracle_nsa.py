"""Pins for the fp64 NSA selection oracle (CPU only).

Each test checks the oracle against something other than itself: torch's
float64 scaled-dot-product attention (a library routine with an explicit
mask), a dense T x T mask built directly from the index array, closed forms,
and invariances the definition implies.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import nsa_select_attention


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, mask, scale):
    """q [T, H, D], k/v [T, H, D], mask [T, T] bool (query, key) -> out [T,H,D], lse [T,H]."""
    qt = torch.from_numpy(q).permute(1, 0, 2)
    kt = torch.from_numpy(k).permute(1, 0, 2)
    vt = torch.from_numpy(v).permute(1, 0, 2)
    m = torch.from_numpy(mask)
    out = F.scaled_dot_product_attention(qt, kt, vt, attn_mask=m, scale=scale)
    scores = (qt @ kt.transpose(1, 2)) * scale
    scores = scores.masked_fill(~m, -math.inf)
    lse = torch.logsumexp(scores, dim=-1)
    return out.permute(1, 0, 2).numpy(), lse.permute(1, 0).numpy()


def _expand_kv(x, G):
    return np.repeat(x, G, axis=2)


@pytest.mark.parametrize("T,bs,Hq,Hkv,D", [(200, 16, 4, 2, 8), (64, 64, 3, 1, 16), (130, 32, 8, 8, 4)])
def test_all_blocks_equals_causal_dense(T, bs, Hq, Hkv, D):
    """Every block selected => plain causal attention (torch SDPA, float64)."""
    B = 1
    q, k, v = _rand((B, T, Hq, D), 1), _rand((B, T, Hkv, D), 2), _rand((B, T, Hkv, D), 3)
    nb = -(-T // bs)
    idx = np.broadcast_to(np.arange(nb, dtype=np.int32), (B, T, Hkv, nb)).copy()
    scale = 0.37
    out, lse = nsa_select_attention(q, k, v, idx, nb, bs, softmax_scale=scale)
    G = Hq // Hkv
    mask = np.tril(np.ones((T, T), dtype=bool))
    ref, ref_lse = _sdpa(q[0], _expand_kv(k, G)[0], _expand_kv(v, G)[0], mask, scale)
    np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-10, atol=1e-12)


def test_default_scale_is_inverse_sqrt_d():
    T, bs, D = 48, 16, 9
    q, k, v = _rand((1, T, 2, D), 4), _rand((1, T, 1, D), 5), _rand((1, T, 1, D), 6)
    idx = np.broadcast_to(np.arange(3, dtype=np.int32), (1, T, 1, 3)).copy()
    out, lse = nsa_select_attention(q, k, v, idx, 3, bs)
    ref, ref_lse = _sdpa(q[0], _expand_kv(k, 2)[0], _expand_kv(v, 2)[0],
                         np.tril(np.ones((T, T), dtype=bool)), 1.0 / 3.0)
    np.testing.assert_allclose(out[0], ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse[0], ref_lse, rtol=1e-10, atol=1e-12)


def _dense_mask_from_indices(idx, counts, T, bs, causal):
    """Literal [T, Hkv, T] mask: key k visible iff its block is among the first
    ``count`` (valid) entries, k < T, and (causal) k <= t."""
    _, _, Hkv, S = idx.shape
    nb = -(-T // bs)
    key_block = np.arange(T) // bs
    mask = np.zeros((T, Hkv, T), dtype=bool)
    for t in range(T):
        for h in range(Hkv):
            c = int(counts[0, t, h])
            for e in idx[0, t, h, :c]:
                if 0 <= e < nb:
                    mask[t, h] |= key_block == e
    if causal:
        mask &= np.tril(np.ones((T, T), dtype=bool))[:, None, :]
    return mask


@pytest.mark.parametrize("causal", [True, False])
def test_random_selection_equals_dense_masked(causal):
    """Random indices (with -1, out-of-range, duplicates, future blocks) against
    a dense masked softmax built straight from the index array."""
    rng = np.random.default_rng(7)
    T, bs, Hq, Hkv, D, S = 150, 16, 4, 2, 8, 5
    nb = -(-T // bs)
    q, k, v = _rand((1, T, Hq, D), 8), _rand((1, T, Hkv, D), 9), _rand((1, T, Hkv, D), 10)
    idx = rng.integers(-2, nb + 2, size=(1, T, Hkv, S)).astype(np.int32)
    counts = rng.integers(0, S + 1, size=(1, T, Hkv)).astype(np.int32)
    out, lse = nsa_select_attention(q, k, v, idx, counts, bs, causal=causal, softmax_scale=0.5)
    mask = _dense_mask_from_indices(idx, counts, T, bs, causal)
    G = Hq // Hkv
    for h in range(Hq):
        m = mask[:, h // G, :]
        rows = m.any(axis=1)
        ref, ref_lse = _sdpa(q[0][rows][:, h:h + 1], k[0][:, h // G:h // G + 1],
                             v[0][:, h // G:h // G + 1], m[rows], 0.5)
        np.testing.assert_allclose(out[0][rows][:, h], ref[:, 0], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[0][rows][:, h], ref_lse[:, 0], rtol=1e-10, atol=1e-12)
        assert np.all(out[0][~rows][:, h] == 0.0)
        assert np.all(np.isneginf(lse[0][~rows][:, h]))


def test_order_padding_and_duplicates_invariance():
    rng = np.random.default_rng(11)
    T, bs, Hq, Hkv, D, S = 96, 8, 2, 1, 4, 6
    nb = T // bs
    q, k, v = _rand((1, T, Hq, D), 12), _rand((1, T, Hkv, D), 13), _rand((1, T, Hkv, D), 14)
    idx = np.full((1, T, Hkv, S), -1, dtype=np.int32)
    counts = np.zeros((1, T, Hkv), dtype=np.int32)
    for t in range(T):
        j = t // bs
        c = int(rng.integers(1, min(4, j + 1) + 1))
        picks = [j] + list(rng.choice(j, size=c - 1, replace=False)) if j else [0]
        idx[0, t, 0, :len(picks)] = picks
        counts[0, t, 0] = len(picks)
    base, base_lse = nsa_select_attention(q, k, v, idx, counts, bs)
    # reversed order of the valid entries
    rev = idx.copy()
    for t in range(T):
        c = counts[0, t, 0]
        rev[0, t, 0, :c] = idx[0, t, 0, :c][::-1]
    o2, l2 = nsa_select_attention(q, k, v, rev, counts, bs)
    np.testing.assert_array_equal(o2, base)
    np.testing.assert_array_equal(l2, base_lse)
    # count = S with -1 padding beyond the valid entries
    o3, l3 = nsa_select_attention(q, k, v, idx, S, bs)
    np.testing.assert_array_equal(o3, base)
    # duplicated entries
    dup = idx.copy()
    dup[0, :, 0, S - 1] = idx[0, :, 0, 0]
    o4, l4 = nsa_select_attention(q, k, v, dup, S, bs)
    np.testing.assert_array_equal(o4, base)
    np.testing.assert_array_equal(l4, base_lse)
    # entries after count are ignored even when they are valid blocks
    junk = idx.copy()
    for t in range(T):
        c = counts[0, t, 0]
        if c < S:
            junk[0, t, 0, c:] = 0
    o5, _ = nsa_select_attention(q, k, v, junk, counts, bs)
    np.testing.assert_array_equal(o5, base)


def test_first_token_closed_form():
    """Token 0 of a causal sequence sees only key 0: out = v0 exactly and
    LSE = scale * <q0, k0>."""
    T, bs, Hq, Hkv, D = 32, 8, 4, 2, 16
    q, k, v = _rand((2, T, Hq, D), 15), _rand((2, T, Hkv, D), 16), _rand((2, T, Hkv, D), 17)
    idx = np.zeros((2, T, Hkv, 2), dtype=np.int32)
    out, lse = nsa_select_attention(q, k, v, idx, 1, bs, softmax_scale=0.25)
    for b in range(2):
        for h in range(Hq):
            np.testing.assert_array_equal(out[b, 0, h], v[b, 0, h // 2])
            assert lse[b, 0, h] == pytest.approx(0.25 * float(q[b, 0, h] @ k[b, 0, h // 2]), rel=1e-14)


def test_empty_selection_gives_zero_and_neg_inf():
    T, bs = 16, 4
    q, k, v = _rand((1, T, 2, 4), 18), _rand((1, T, 1, 4), 19), _rand((1, T, 1, 4), 20)
    idx = np.full((1, T, 1, 2), -1, dtype=np.int32)
    out, lse = nsa_select_attention(q, k, v, idx, 2, bs)
    assert np.all(out == 0.0) and np.all(np.isneginf(lse))
    # a future block only (causal) is empty as well
    idx2 = np.full((1, T, 1, 1), 3, dtype=np.int32)
    out2, lse2 = nsa_select_attention(q, k, v, idx2, 1, bs)
    assert np.all(out2[0, :12] == 0.0) and np.all(np.isneginf(lse2[0, :12]))
    assert np.all(np.isfinite(lse2[0, 12:]))


def test_varlen_equals_separate_sequences():
    """Packing with cu_seqlens equals running each sequence on its own."""
    rng = np.random.default_rng(21)
    lens = [37, 64, 5, 90]
    bs, Hq, Hkv, D, S = 16, 4, 2, 8, 3
    T = sum(lens)
    q, k, v = _rand((1, T, Hq, D), 22), _rand((1, T, Hkv, D), 23), _rand((1, T, Hkv, D), 24)
    idx = np.full((1, T, Hkv, S), -1, dtype=np.int32)
    off = 0
    for L in lens:
        for t in range(L):
            j = t // bs
            idx[0, off + t, :, 0] = j
            idx[0, off + t, :, 1] = rng.integers(0, j + 1)
        off += L
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    packed, packed_lse = nsa_select_attention(q, k, v, idx, S, bs, cu_seqlens=cu)
    off = 0
    for L in lens:
        sl = slice(off, off + L)
        o, l = nsa_select_attention(q[:, sl], k[:, sl], v[:, sl], idx[:, sl], S, bs)
        np.testing.assert_array_equal(packed[:, sl], o)
        np.testing.assert_array_equal(packed_lse[:, sl], l)
        off += L


def test_gqa_equals_repeated_heads():
    """GQA with group G equals MHA on KV heads repeated G times with the
    indices repeated alongside (query head hq reads KV head hq // G)."""
    rng = np.random.default_rng(25)
    T, bs, Hq, Hkv, D, S = 64, 8, 6, 2, 4, 3
    G = Hq // Hkv
    q, k, v = _rand((1, T, Hq, D), 26), _rand((1, T, Hkv, D), 27), _rand((1, T, Hkv, D), 28)
    idx = rng.integers(0, T // bs, size=(1, T, Hkv, S)).astype(np.int32)
    a, la = nsa_select_attention(q, k, v, idx, S, bs)
    b, lb = nsa_select_attention(q, _expand_kv(k, G), _expand_kv(v, G), np.repeat(idx, G, axis=2), S, bs)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(la, lb, rtol=1e-13, atol=1e-14)


def test_selection_gate_scales_rows_and_leaves_lse():
    """The g_slc reading (parity unpinned: the pages give the gate's signature, not its
    effect): each (token, query head) output row is multiplied by its gate; rows with
    no admissible key stay 0 and the LSE is the ungated attention's.  This restates the
    reading; it does not pin it against the pages."""
    rng = np.random.default_rng(12)
    B, T, Hq, Hkv, D, bs = 1, 40, 4, 2, 8, 8
    q = rng.standard_normal((B, T, Hq, D))
    k = rng.standard_normal((B, T, Hkv, D))
    v = rng.standard_normal((B, T, Hkv, D))
    idx = rng.integers(-1, 5, size=(B, T, Hkv, 3))
    gate = rng.uniform(-2.0, 2.0, size=(B, T, Hq))
    gate[0, 5, 1] = 0.0
    o, l = nsa_select_attention(q, k, v, idx, 3, bs)
    og, lg = nsa_select_attention(q, k, v, idx, 3, bs, g_slc=gate)
    np.testing.assert_array_equal(lg, l)
    assert np.all(og[0, 5, 1] == 0.0)
    empty = np.isneginf(l)
    assert np.all(og[empty] == 0.0)
    # a gate of one is the ungated selection branch; any other gate scales its row
    ones = nsa_select_attention(q, k, v, idx, 3, bs, g_slc=np.ones((B, T, Hq)))[0]
    np.testing.assert_array_equal(ones, o)
    np.testing.assert_allclose(og, o * gate[..., None], rtol=0, atol=1e-12)
