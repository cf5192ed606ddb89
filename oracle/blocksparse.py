"""fp64 oracle: attention restricted by SparseMask block bounds.  (TEST INFRASTRUCTURE)

Source: ejkernel.kernels._triton.blocksparse_attention._mask (module source
page), the module docstring and the ``SparseMask`` docstring: key/value blocks
outside ``[lower, upper)`` of a query block are skipped entirely; blocks inside
``[lower_full, upper_full)`` need no per-token masking (an optimisation only:
it does not change the result); segment ids separate packed documents.

The page does not spell out the token-level mask.  Reading used here (the
plainest one consistent with the block rule): query token ``i`` attends key
token ``j`` iff

* the key block of ``j`` lies in ``[lower, upper)`` of the query block of ``i``;
* ``seg_q[i] == seg_kv[j]`` and neither is the padding segment id;
* causal: ``pos_kv[j] <= pos_q[i]``;
* window: ``pos_q[i] - pos_kv[j] <= window_left`` and
  ``pos_kv[j] - pos_q[i] <= window_right`` (each only when >= 0).

Then a plain softmax over exactly those keys; a row with none gives output 0
and LSE ``-inf``.  Query head ``hq`` reads KV head ``hq // (Hq // Hkv)``.
"""

from __future__ import annotations

import math

import numpy as np


def blocksparse_attention(q, k, v, q_positions, q_segment_ids, kv_positions,
                          kv_segment_ids, lower, upper, q_blocksize, kv_blocksize,
                          *, causal=True, window_left=-1, window_right=-1,
                          padding_segment_id=-1, softmax_scale=None, rows=None,
                          heads=None):
    """Output ``[B, Tq, Hq, D]`` and LSE ``[B, Tq, Hq]`` (float64).

    ``lower``/``upper`` are ``[B, 1, NBq]`` block bounds.  ``rows`` restricts the
    computation to a list of (b, t) pairs and ``heads`` to a list of query
    heads; everything not computed is NaN.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    q_pos = np.asarray(q_positions, dtype=np.int64)
    q_seg = np.asarray(q_segment_ids, dtype=np.int64)
    kv_pos = np.asarray(kv_positions, dtype=np.int64)
    kv_seg = np.asarray(kv_segment_ids, dtype=np.int64)
    lower = np.asarray(lower)
    upper = np.asarray(upper)
    B, Tq, Hq, D = q.shape
    Tkv, Hkv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if (softmax_scale is None or softmax_scale <= 0) else float(softmax_scale)
    pad = int(padding_segment_id)
    out = np.full((B, Tq, Hq, D), np.nan)
    lse = np.full((B, Tq, Hq), np.nan)
    if rows is None:
        rows = [(b, t) for b in range(B) for t in range(Tq)]
    head_list = list(range(Hq)) if heads is None else list(heads)
    for b, t in rows:
        qb = t // q_blocksize
        lo, up = int(lower[b, 0, qb]), int(upper[b, 0, qb])
        cand = np.arange(lo * kv_blocksize, min(up * kv_blocksize, Tkv), dtype=np.int64)
        keep = (kv_seg[b, cand] == q_seg[b, t]) & (q_seg[b, t] != pad) & (kv_seg[b, cand] != pad)
        if causal:
            keep &= kv_pos[b, cand] <= q_pos[b, t]
        if window_left >= 0:
            keep &= (q_pos[b, t] - kv_pos[b, cand]) <= window_left
        if window_right >= 0:
            keep &= (kv_pos[b, cand] - q_pos[b, t]) <= window_right
        keys = cand[keep]
        for hq in head_list:
            hkv = hq // G
            if keys.size == 0:
                out[b, t, hq] = 0.0
                lse[b, t, hq] = -np.inf
                continue
            s = scale * (k[b, keys, hkv] @ q[b, t, hq])
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            out[b, t, hq] = (e @ v[b, keys, hkv]) / l
            lse[b, t, hq] = m + math.log(l)
    return out, lse
