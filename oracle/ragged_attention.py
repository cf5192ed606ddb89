"""fp64 oracle: ragged multi-query attention.  (TEST INFRASTRUCTURE)

Source: ejkernel.kernels._xla.ragged_decode_attention._xla_impl_fwd (API page),
``ragged_flash_attention_xla``: queries ``[B, Q, H, D]`` against a key/value
cache ``[B, K, H, D]`` restricted per batch row to ``[sequence_start,
sequence_end)``, with an optional ``sliding_window=(left, right)``, a
``logits_soft_cap`` and ``softmax_aux`` sink biases (``[H, num_sinks]`` or
``[num_sinks]``); ``create_attention_mask`` builds one ``[B, Q, 1, K]`` mask
(ragged range, window, sinks that are always attendable) shared by the heads;
``block_size`` only chunks the computation.

Readings of what the page leaves open:
  * the Q queries of a row are its last Q tokens: query ``i`` sits at position
    ``p_i = end - Q + i`` (with Q = 1 this is the decode reading ``p = end - 1``);
  * there is no causal switch: key ``k`` is attendable by query ``i`` iff
    ``start <= k < end`` and either it is inside the inclusive window of ``p_i``
    (``k >= p_i - left`` when ``left >= 0``, ``k <= p_i + right`` when
    ``right >= 0``) or it is a sink (``k < num_sinks``); without a window every
    query of the row sees the whole range, and ``right = 0`` makes it causal;
  * logit order: ``s = scale * <q, k>``; ``s = cap * tanh(s / cap)`` when
    ``cap > 0``; then the sink bias for ``k < num_sinks``;
  * the key/value head count may divide the query head count (query head
    ``hq`` reads KV head ``hq // (Hq // Hkv)``); the page's case is Hkv = Hq;
  * a query with no attendable key gives output 0 and LSE ``-inf``; the LSE is
    natural-log.
"""

from __future__ import annotations

import math

import numpy as np


def query_position(end, q_len, i):
    """Position of query ``i`` of a row whose range ends at ``end`` (exclusive)."""
    return int(end) - int(q_len) + int(i)


def attendable_keys_at(p, start, end, window_left, window_right, num_sinks):
    """Sorted key positions a query at position ``p`` may attend."""
    keys = []
    for key in range(max(int(start), 0), int(end)):
        in_window = True
        if window_left is not None and window_left >= 0 and key < p - window_left:
            in_window = False
        if window_right is not None and window_right >= 0 and key > p + window_right:
            in_window = False
        if in_window or key < num_sinks:
            keys.append(key)
    return np.asarray(keys, dtype=np.int64)


def ragged_flash_attention(q, k, v, sequence_start, sequence_end, *,
                           softmax_scale=None, window_left=-1, window_right=-1,
                           logits_soft_cap=None, sink_bias=None, rows=None):
    """Output ``[B, Q, Hq, D]`` and LSE ``[B, Q, Hq]`` (float64).

    ``k``, ``v``: ``[B, K, Hkv, D]``.  ``sink_bias``: None, ``[num_sinks]`` or
    ``[Hq, num_sinks]``.  ``rows``: None (all) or an iterable of ``(b, i)``
    pairs to compute; the rest stays NaN.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Q, Hq, D = q.shape
    Hkv = k.shape[2]
    if Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if (softmax_scale is None or softmax_scale <= 0) else float(softmax_scale)
    if sink_bias is None:
        bias, num_sinks = None, 0
    else:
        bias = np.asarray(sink_bias, dtype=np.float64)
        num_sinks = bias.shape[-1]
        if bias.ndim == 1:
            bias = np.broadcast_to(bias, (Hq, num_sinks))
    cap = float(logits_soft_cap) if (logits_soft_cap is not None and logits_soft_cap > 0) else None
    out = np.full((B, Q, Hq, D), np.nan)
    lse = np.full((B, Q, Hq), np.nan)
    if rows is None:
        rows = [(b, i) for b in range(B) for i in range(Q)]
    for b, i in rows:
        p = query_position(sequence_end[b], Q, i)
        keys = attendable_keys_at(p, sequence_start[b], sequence_end[b], window_left,
                                  window_right, num_sinks)
        if keys.size == 0:
            out[b, i] = 0.0
            lse[b, i] = -np.inf
            continue
        for hq in range(Hq):
            hkv = hq // G
            kk = np.asarray(k[b, keys, hkv], dtype=np.float64)
            vv = np.asarray(v[b, keys, hkv], dtype=np.float64)
            s = scale * (kk @ q[b, i, hq])
            if cap is not None:
                s = cap * np.tanh(s / cap)
            if bias is not None:
                sink = keys < num_sinks
                s = s + np.where(sink, bias[hq, np.minimum(keys, num_sinks - 1)], 0.0)
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            out[b, i, hq] = (e @ vv) / l
            lse[b, i, hq] = m + math.log(l)
    return out, lse
