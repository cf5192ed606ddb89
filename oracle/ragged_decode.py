"""fp64 oracle: ragged single-token decode attention.  (TEST INFRASTRUCTURE)

Source: ejkernel.kernels._xla.ragged_decode_attention._xla_impl_fwd (API page):
``ragged_decode_mqa_xla`` / ``inner_decode_xla`` (query ``[B, Hq, D]``,
key/value cache ``[B, S, Hkv, D]``, per-row ``sequence_start`` /
``sequence_end``, optional ``sliding_window=(left, right)``,
``logits_soft_cap`` and ``softmax_aux`` sink biases ``[Hq, num_sinks]`` or
``[num_sinks]``), ``create_attention_mask`` (ragged range, window, sinks that
are always attendable), ``apply_logits_soft_cap`` and
``apply_attention_sinks_block`` (biases added to the scores of the sink
tokens, located by their position in the full sequence).

Readings of what the page leaves open:
  * the range ``[start, end)`` is half-open and the decoding query sits at
    position ``p = end - 1``;
  * key ``k`` is attendable iff ``start <= k < end`` and either it is inside the
    inclusive window (``k >= p - left`` when ``left >= 0`` and ``k <= p + right``
    when ``right >= 0``) or it is a sink (``k < num_sinks``);
  * logit order: ``s = scale * <q, k>``; soft cap ``s = cap * tanh(s / cap)``
    when ``cap > 0``; then the sink bias is added for ``k < num_sinks``;
  * query head ``hq`` reads KV head ``hq // (Hq // Hkv)``;
  * an empty row gives output 0 and LSE ``-inf``.
"""

from __future__ import annotations

import math

import numpy as np


def attendable_keys(start, end, window_left, window_right, num_sinks):
    """Sorted key positions one decode row may attend."""
    start, end = int(start), int(end)
    if end <= start:
        return np.zeros(0, dtype=np.int64)
    p = end - 1
    keys = []
    for key in range(max(start, 0), end):
        in_window = True
        if window_left is not None and window_left >= 0 and key < p - window_left:
            in_window = False
        if window_right is not None and window_right >= 0 and key > p + window_right:
            in_window = False
        if in_window or key < num_sinks:
            keys.append(key)
    return np.asarray(keys, dtype=np.int64)


def ragged_decode_attention(q, k, v, sequence_start, sequence_end, *,
                            softmax_scale=None, window_left=-1, window_right=-1,
                            logits_soft_cap=None, sink_bias=None, rows=None):
    """Decode output ``[B, Hq, D]`` and LSE ``[B, Hq]`` (float64).

    ``sink_bias`` is None, ``[num_sinks]`` (shared by all heads) or
    ``[Hq, num_sinks]``.  ``rows`` restricts the computation to a list of batch
    rows; rows not computed are NaN.
    """
    q = np.asarray(q, dtype=np.float64)
    B, Hq, D = q.shape
    Hkv = k.shape[2]
    G = Hq // Hkv
    scale = (1.0 / math.sqrt(D)) if (softmax_scale is None or softmax_scale <= 0) else float(softmax_scale)
    if sink_bias is None:
        bias = None
        num_sinks = 0
    else:
        bias = np.asarray(sink_bias, dtype=np.float64)
        num_sinks = bias.shape[-1]
        if bias.ndim == 1:
            bias = np.broadcast_to(bias, (Hq, num_sinks))
    cap = float(logits_soft_cap) if (logits_soft_cap is not None and logits_soft_cap > 0) else None
    out = np.full((B, Hq, D), np.nan)
    lse = np.full((B, Hq), np.nan)
    for b in (range(B) if rows is None else rows):
        keys = attendable_keys(sequence_start[b], sequence_end[b], window_left,
                               window_right, num_sinks)
        if keys.size == 0:
            out[b] = 0.0
            lse[b] = -np.inf
            continue
        for hq in range(Hq):
            hkv = hq // G
            kk = np.asarray(k[b, keys, hkv], dtype=np.float64)
            vv = np.asarray(v[b, keys, hkv], dtype=np.float64)
            s = scale * (kk @ q[b, hq])
            if cap is not None:
                s = cap * np.tanh(s / cap)
            if bias is not None:
                sink = keys < num_sinks
                s = s + np.where(sink, bias[hq, np.minimum(keys, num_sinks - 1)], 0.0)
            m = s.max()
            e = np.exp(s - m)
            l = e.sum()
            out[b, hq] = (e @ vv) / l
            lse[b, hq] = m + math.log(l)
    return out, lse
