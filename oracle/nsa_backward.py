"""fp64 oracle: gradients of the native-sparse-attention selection forward.  (TEST INFRASTRUCTURE)

Source: ejkernel.modules.operations.native_sparse_attention (operation API page),
``NativeSparseAttention.run`` / ``native_sparse_attention``: the operation is
differentiable with respect to its query, key and value inputs.  The page prints
no backward algorithm; the gradient is the one calculus fixes for the forward the
sibling module ``oracle.nsa`` defines, written out row by row over the same
explicit key set:

for one output row (token t, query head h, KV head h // G) with key set K,
    s_k  = scale * <q, k_k>,  p_k = exp(s_k - lse)  (the row's softmax),
    o    = sum_k p_k v_k,
    dv_k += p_k * do                      (for every k in K)
    dp_k  = <do, v_k>
    ds_k  = p_k * (dp_k - sum_j p_j dp_j)  (softmax Jacobian; sum_j p_j dp_j = <do, o>)
    dq   += scale * sum_k ds_k k_k
    dk_k += scale * ds_k * q
A row with an empty key set has a constant output (0) and contributes nothing.
The key set, its readings (set semantics, causal k <= t, sequence-relative
block ids, GQA map) and the default scale are those of ``oracle.nsa``.
"""

from __future__ import annotations

import math

import numpy as np

from .nsa import selected_key_set


def nsa_select_attention_backward(q, k, v, block_indices, block_counts, block_size, d_out, *,
                                  cu_seqlens=None, causal=True, softmax_scale=None, rows=None):
    """Gradients ``(dq, dk, dv)`` (float64, shapes of q, k, v) of
    ``sum(nsa_select_attention(q, k, v, ...)[0] * d_out)``.

    Arguments as for ``oracle.nsa.nsa_select_attention``; ``d_out`` has the
    output's shape ``[B, T, Hq, D]``.  ``rows`` (None = all) restricts the
    query rows whose contribution is accumulated: ``dq`` is then exact on those
    rows (NaN elsewhere) and ``dk`` / ``dv`` hold only their contributions.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(d_out, dtype=np.float64)
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
    dq = np.zeros_like(q) if rows is None else np.full_like(q, np.nan)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    if rows is None:
        rows = [(b, t) for b in range(B) for t in range(T)]
    for b, t in rows:
        if cu_seqlens is not None:
            s = int(np.searchsorted(cu, t, side="right")) - 1
            bos, seq_len = int(cu[s]), int(cu[s + 1] - cu[s])
        else:
            bos, seq_len = 0, T
        t_rel = t - bos
        dq[b, t] = 0.0
        for hkv in range(Hkv):
            count = int(block_counts) if scalar_count else int(block_counts[b, t, hkv])
            keys = selected_key_set(block_indices[b, t, hkv], count, seq_len, block_size,
                                    t_rel, causal)
            if keys.size == 0:
                continue
            rows_k = bos + keys
            kk = k[b, rows_k, hkv]                      # [n, D]
            vv = v[b, rows_k, hkv]                      # [n, D]
            for hq in range(hkv * G, (hkv + 1) * G):
                s_row = scale * (kk @ q[b, t, hq])      # [n]
                m = s_row.max()
                e = np.exp(s_row - m)
                p = e / e.sum()                         # softmax over the key set
                dp = vv @ do[b, t, hq]                  # <do, v_k>
                ds = p * (dp - p @ dp)
                dq[b, t, hq] = scale * (ds @ kk)
                dk[b, rows_k, hkv] += scale * np.outer(ds, q[b, t, hq])
                dv[b, rows_k, hkv] += np.outer(p, do[b, t, hq])
    return dq, dk, dv
