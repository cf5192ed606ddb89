"""fp64 oracle: native-sparse-attention selection forward.  (TEST INFRASTRUCTURE)

Source: ejkernel.modules.operations.native_sparse_attention (operation API page),
``NativeSparseAttention.run`` and ``native_sparse_attention``: each query token
attends, per KV head, only to the key blocks of ``block_size`` tokens listed in
``block_indices[b, t, h_kv, :block_counts]``; query heads share KV heads (GQA);
``cu_seqlens`` packs variable-length sequences into one batch row; the output
has the query's shape.

This is the plain definition of the result, written out: for one output row the
explicit set of admissible keys is built first, then an ordinary softmax is
taken over exactly those keys.  Readings of points the page leaves open:

* index layout ``[B, T, Hkv, S]`` (the signature), block ids relative to the
  start of the token's own sequence;
* the entries taken are ``block_indices[..., :count]`` with ``count`` clipped
  to ``[0, S]``; entries outside ``[0, ceil(L / block_size))`` are ignored and
  the selection is a *set* (order and duplicates do not matter);
* causal masking keeps keys ``k <= t`` (sequence-relative positions);
* query head ``hq`` reads KV head ``hq // (Hq // Hkv)``;
* default ``softmax_scale`` is ``1 / sqrt(D)``;
* the log-sum-exp is natural-log; a row with no admissible key has output 0 and
  LSE ``-inf``.

The optional ``g_slc`` gate is a reading, parity unpinned: the page lists the
argument in the operation's signature but never states its effect, so nothing on
the pages can check the per-row multiplier used here (its test only restates it).
"""

from __future__ import annotations

import math

import numpy as np


def selected_key_set(idx_row, count, seq_len, block_size, t_rel, causal):
    """Sorted sequence-relative key positions one (token, KV head) may see.

    ``idx_row`` is ``block_indices[b, t, h_kv, :]``; ``count`` the matching
    ``block_counts`` entry; ``seq_len`` the token's sequence length;
    ``t_rel`` its position inside that sequence.
    """
    idx_row = np.asarray(idx_row).reshape(-1)
    count = max(0, min(int(count), idx_row.shape[0]))
    num_blocks = -(-int(seq_len) // int(block_size))
    blocks = set()
    for raw in idx_row[:count]:
        blk = int(raw)
        if 0 <= blk < num_blocks:
            blocks.add(blk)
    keys = []
    for blk in sorted(blocks):
        start = blk * block_size
        stop = min(start + block_size, seq_len)
        for key in range(start, stop):
            if causal and key > t_rel:
                break
            keys.append(key)
    return np.asarray(keys, dtype=np.int64)


def _softmax_rows(scores, values):
    """Plain softmax over the last axis of ``scores`` [G, n] applied to ``values`` [n, D]."""
    m = scores.max(axis=1, keepdims=True)
    e = np.exp(scores - m)
    l = e.sum(axis=1, keepdims=True)
    out = (e @ values) / l
    lse = (m + np.log(l))[:, 0]
    return out, lse


def nsa_select_attention(q, k, v, block_indices, block_counts, block_size, *,
                         cu_seqlens=None, causal=True, softmax_scale=None,
                         rows=None, g_slc=None):
    """Selection-branch attention output and LSE.

    Arguments (numpy, any float dtype; widened exactly to float64):
      q             [B, T, Hq, D]
      k, v          [B, T, Hkv, D]
      block_indices [B, T, Hkv, S] integer
      block_counts  int, or integer array [B, T, Hkv]
      cu_seqlens    None, or int array [N + 1] (then B must be 1)
      rows          None (all tokens) or iterable of (b, t) pairs to compute;
                    rows not computed are left NaN.
      g_slc         None, or the selection-branch gate [B, T, Hq]: the output of
                    (b, t, hq) is scaled by g_slc[b, t, hq] (the operation's g_slc
                    argument, read as a per-row gate of the selection output); the
                    LSE is the attention's and is not gated.

    Returns ``(out [B, T, Hq, D] float64, lse [B, T, Hq] float64)``.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    block_indices = np.asarray(block_indices)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if (softmax_scale is None or softmax_scale <= 0) else float(softmax_scale)
    scalar_count = np.isscalar(block_counts) or np.ndim(block_counts) == 0
    if not scalar_count:
        block_counts = np.asarray(block_counts)
    if cu_seqlens is not None:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        if B != 1:
            raise ValueError("cu_seqlens requires batch 1")
    out = np.full((B, T, Hq, D), np.nan)
    lse = np.full((B, T, Hq), np.nan)
    if rows is None:
        rows = [(b, t) for b in range(B) for t in range(T)]
    for b, t in rows:
        if cu_seqlens is not None:
            s = int(np.searchsorted(cu, t, side="right")) - 1
            bos, seq_len = int(cu[s]), int(cu[s + 1] - cu[s])
        else:
            bos, seq_len = 0, T
        t_rel = t - bos
        for hkv in range(Hkv):
            count = int(block_counts) if scalar_count else int(block_counts[b, t, hkv])
            keys = selected_key_set(block_indices[b, t, hkv], count, seq_len,
                                    block_size, t_rel, causal)
            heads = slice(hkv * G, (hkv + 1) * G)
            if keys.size == 0:
                out[b, t, heads] = 0.0
                lse[b, t, heads] = -np.inf
                continue
            kk = k[b, bos + keys, hkv]          # [n, D]
            vv = v[b, bos + keys, hkv]          # [n, D]
            scores = scale * (q[b, t, heads] @ kk.T)   # [G, n]
            o, l = _softmax_rows(scores, vv)
            out[b, t, heads] = o
            lse[b, t, heads] = l
    if g_slc is not None:
        out = out * np.asarray(g_slc, dtype=np.float64)[..., None]
    return out, lse
