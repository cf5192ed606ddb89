"""int64 oracle: SparseMask block bounds, forward and dK/dV.  (TEST INFRASTRUCTURE)

Source: ejkernel.kernels._triton.blocksparse_attention._mask (module source
page): the ``SparseMask`` dataclass, the ``_compute_sparse_mask`` kernel (taken
with the query blocks as the outer operand for the forward / dQ bounds and with
the key/value blocks as the outer operand when ``calculate_dkdv_mask`` is set),
and the padding, padding-segment remap and clip/fix-up steps of
``define_sparse_mask_fn``.

The bounds are a block-level heuristic with an exact integer result, so this
module takes the page's steps in the page's order, in plain loops:

1. pad both sides to a block multiple (query positions with -1, key/value
   positions with the int32 maximum, segment ids with the padding id);
2. remap the padding segment id to ``padded_kv_len + 1`` on both sides;
3. per outer block, take min/max of positions and segment ids; a block made
   only of padding gets bounds (0, 0, 0, 0);
4. sweep every inner block, evaluate the attend and full predicates
   (segment-range overlap, causal, inclusive left/right window, inner block made
   only of padding) and min/max-accumulate the four bounds;
5. clip and order the bounds as the fix-up step does.

Readings of what the page leaves open (each is also listed in the design notes):
  * the padding segment id is an argument (default -1);
  * padding tokens receive the padding segment id;
  * window tests are inclusive, -1 means unbounded;
  * position arithmetic is done in 64-bit integers.
The window-left attend test compares the *smallest* key position of a block
with ``min(query positions) - window_left``; it is reproduced as written, so a
key block that straddles the window edge may be left out.  The kv-outer
(dK/dV) predicates are likewise taken as printed; they are not the transposed
forward tests (under causal masking their left-window attend test never prunes
a block, and their full tests compare the smallest positions).
"""

from __future__ import annotations

import numpy as np

INT32_MAX = 2**31 - 1


def _pad_to_block(values, block, fill):
    B, T = values.shape
    Tp = -(-T // block) * block
    out = np.full((B, Tp), fill, dtype=np.int64)
    out[:, :T] = values
    return out


def sparse_mask_bounds(q_positions, q_segment_ids, kv_positions, kv_segment_ids,
                       q_blocksize, kv_blocksize, *, causal=True,
                       window_left=-1, window_right=-1, padding_segment_id=-1,
                       calculate_dkdv_mask=False):
    """SparseMask bounds.

    Inputs are integer arrays ``[B, Tq]`` (query side) and ``[B, Tkv]``
    (key/value side).  Forward (``calculate_dkdv_mask=False``): the query blocks
    are the outer operand and the result is four int32 arrays ``[B, 1, NBq]``
    (``lower, upper, lower_full, upper_full`` ranges of key/value blocks).
    Backward dK/dV (``calculate_dkdv_mask=True``): the key/value blocks are the
    outer operand and the result is ``[B, 1, NBkv]`` ranges of query blocks, with
    the kv-outer position predicates of the page.
    """
    q_pos = np.asarray(q_positions, dtype=np.int64)
    q_seg = np.asarray(q_segment_ids, dtype=np.int64)
    kv_pos = np.asarray(kv_positions, dtype=np.int64)
    kv_seg = np.asarray(kv_segment_ids, dtype=np.int64)
    pad = int(padding_segment_id)

    # Step 1: pad to block multiples.
    q_pos = _pad_to_block(q_pos, q_blocksize, -1)
    q_seg = _pad_to_block(q_seg, q_blocksize, pad)
    kv_pos = _pad_to_block(kv_pos, kv_blocksize, INT32_MAX)
    kv_seg = _pad_to_block(kv_seg, kv_blocksize, pad)
    Tkv = kv_pos.shape[1]

    # Step 2: padding segment id -> padded kv length + 1 (on both sides, either way).
    pad_inner = Tkv + 1
    q_seg = np.where(q_seg == pad, pad_inner, q_seg)
    kv_seg = np.where(kv_seg == pad, pad_inner, kv_seg)

    if calculate_dkdv_mask:
        return _bounds(kv_pos, kv_seg, q_pos, q_seg, kv_blocksize, q_blocksize, False,
                       causal, window_left, window_right, pad_inner)
    return _bounds(q_pos, q_seg, kv_pos, kv_seg, q_blocksize, kv_blocksize, True,
                   causal, window_left, window_right, pad_inner)


def _position_predicates(query_is_outer, causal, window_left, window_right,
                         o_min, o_max, i_min, i_max):
    """(attend, full) position tests of one (outer block, inner block) pair, as the
    page's kernel states them for each choice of outer operand."""
    attend_pos, full_pos = True, True
    if query_is_outer:      # outer = query block, inner = key/value block
        if causal:
            attend_pos = o_max >= i_min
            full_pos = o_min >= i_max
        if window_left >= 0:
            attend_pos = attend_pos and (i_min >= o_min - window_left)
            full_pos = full_pos and (i_min >= o_max - window_left)
        if window_right >= 0:
            attend_pos = attend_pos and (i_max <= o_max + window_right)
            full_pos = full_pos and (i_max <= o_min + window_right)
    else:                   # outer = key/value block, inner = query block
        if causal:
            attend_pos = i_max >= o_min
            full_pos = i_min >= o_max
        if window_left >= 0:
            attend_pos = attend_pos and (i_max >= o_min - window_left)
            full_pos = full_pos and (i_min >= o_min - window_left)
        if window_right >= 0:
            attend_pos = attend_pos and (i_min <= o_max + window_right)
            full_pos = full_pos and (i_max <= o_max + window_right)
    return attend_pos, full_pos


def _bounds(o_pos, o_seg, i_pos, i_seg, o_block, i_block, query_is_outer, causal,
            window_left, window_right, pad_inner):
    B, To = o_pos.shape
    Ti = i_pos.shape[1]
    nbo = To // o_block
    nbi = Ti // i_block
    lower = np.zeros((B, 1, nbo), dtype=np.int64)
    upper = np.zeros((B, 1, nbo), dtype=np.int64)
    lower_full = np.zeros((B, 1, nbo), dtype=np.int64)
    upper_full = np.zeros((B, 1, nbo), dtype=np.int64)

    for b in range(B):
        for j in range(nbo):
            # Step 3: summaries of the outer block.
            os_ = slice(j * o_block, (j + 1) * o_block)
            o_seg_min, o_seg_max = int(o_seg[b, os_].min()), int(o_seg[b, os_].max())
            o_same = o_seg_min == o_seg_max
            if o_same and o_seg_min == pad_inner:
                continue  # all four bounds stay 0
            o_pos_min, o_pos_max = int(o_pos[b, os_].min()), int(o_pos[b, os_].max())

            up, lo, up_full, lo_full = 0, nbi, 0, nbi
            # Step 4: sweep the inner blocks.
            for i in range(nbi):
                is_ = slice(i * i_block, (i + 1) * i_block)
                i_seg_min, i_seg_max = int(i_seg[b, is_].min()), int(i_seg[b, is_].max())
                i_same = i_seg_min == i_seg_max
                attend_seg = (i_seg_min <= o_seg_max) and (o_seg_min <= i_seg_max)
                full_seg = o_same and i_same
                i_pos_min, i_pos_max = int(i_pos[b, is_].min()), int(i_pos[b, is_].max())
                attend_pos, full_pos = _position_predicates(
                    query_is_outer, causal, window_left, window_right,
                    o_pos_min, o_pos_max, i_pos_min, i_pos_max)

                attend = attend_pos and attend_seg and not (i_seg_min == pad_inner)
                full = full_seg and full_pos and attend
                if attend:
                    up = max(up, i + 1)
                    lo = min(lo, i)
                if full:
                    up_full = max(up_full, i + 1)
                    lo_full = min(lo_full, i)

            # Step 5: clip / order fix-up.
            lo = min(max(lo, 0), nbi)
            up = min(max(up, 0), nbi)
            lo = min(lo, up)
            lo_full = max(min(max(lo_full, 0), nbi), lo)
            up_full = min(max(min(max(up_full, 0), nbi), lo_full), up)
            lower[b, 0, j] = lo
            upper[b, 0, j] = up
            lower_full[b, 0, j] = lo_full
            upper_full[b, 0, j] = up_full

    cast = lambda a: a.astype(np.int32)
    return cast(lower), cast(upper), cast(lower_full), cast(upper_full)
