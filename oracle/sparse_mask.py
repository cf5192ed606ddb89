"""fp64/int64 oracle: SparseMask block bounds for the forward pass.  (TEST INFRASTRUCTURE)

Source: ejkernel.kernels._triton.blocksparse_attention._mask (module source
page): the ``SparseMask`` dataclass, the ``_compute_sparse_mask`` kernel taken
with the query as the outer operand, and the padding, padding-segment remap and
clip/fix-up steps of ``define_sparse_mask_fn``.

The bounds are a block-level heuristic with an exact integer result, so this
module takes the page's steps in the page's order, in plain loops:

1. pad both sides to a block multiple (query positions with -1, key/value
   positions with the int32 maximum, segment ids with the padding id);
2. remap the padding segment id to ``padded_kv_len + 1`` on both sides;
3. per query ("outer") block, take min/max of positions and segment ids; a
   block made only of padding gets bounds (0, 0, 0, 0);
4. sweep every key/value ("inner") block, evaluate the attend and full
   predicates (segment-range overlap, causal, inclusive left/right window,
   padding) and min/max-accumulate the four bounds;
5. clip and order the bounds as the fix-up step does.

Readings of what the page leaves open (each is also listed in the design notes):
  * the padding segment id is an argument (default -1);
  * padding tokens receive the padding segment id;
  * window tests are inclusive, -1 means unbounded;
  * position arithmetic is done in 64-bit integers.
The window-left attend test compares the *smallest* key position of a block
with ``min(query positions) - window_left``; it is reproduced as written, so a
key block that straddles the window edge may be left out.
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
                       window_left=-1, window_right=-1, padding_segment_id=-1):
    """Forward SparseMask bounds.

    Inputs are integer arrays ``[B, Tq]`` (query side) and ``[B, Tkv]``
    (key/value side).  Returns four int32 arrays of shape ``[B, 1, NBq]``:
    ``lower, upper, lower_full, upper_full`` with ``NBq = ceil(Tq / q_blocksize)``.
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
    B, Tq = q_pos.shape
    Tkv = kv_pos.shape[1]
    nbq = Tq // q_blocksize
    nbkv = Tkv // kv_blocksize

    # Step 2: padding segment id -> padded kv length + 1.
    pad_inner = Tkv + 1
    q_seg = np.where(q_seg == pad, pad_inner, q_seg)
    kv_seg = np.where(kv_seg == pad, pad_inner, kv_seg)

    use_window = window_left >= 0 or window_right >= 0
    lower = np.zeros((B, 1, nbq), dtype=np.int64)
    upper = np.zeros((B, 1, nbq), dtype=np.int64)
    lower_full = np.zeros((B, 1, nbq), dtype=np.int64)
    upper_full = np.zeros((B, 1, nbq), dtype=np.int64)

    for b in range(B):
        for j in range(nbq):
            # Step 3: summaries of the query (outer) block.
            qs = slice(j * q_blocksize, (j + 1) * q_blocksize)
            o_seg_min, o_seg_max = int(q_seg[b, qs].min()), int(q_seg[b, qs].max())
            o_same = o_seg_min == o_seg_max
            if o_same and o_seg_min == pad_inner:
                continue  # all four bounds stay 0
            o_pos_min, o_pos_max = int(q_pos[b, qs].min()), int(q_pos[b, qs].max())

            up, lo, up_full, lo_full = 0, nbkv, 0, nbkv
            # Step 4: sweep the key/value (inner) blocks.
            for i in range(nbkv):
                ks = slice(i * kv_blocksize, (i + 1) * kv_blocksize)
                i_seg_min, i_seg_max = int(kv_seg[b, ks].min()), int(kv_seg[b, ks].max())
                i_same = i_seg_min == i_seg_max
                attend_seg = (i_seg_min <= o_seg_max) and (o_seg_min <= i_seg_max)
                full_seg = o_same and i_same
                i_pos_min, i_pos_max = int(kv_pos[b, ks].min()), int(kv_pos[b, ks].max())

                if causal:
                    attend_pos = o_pos_max >= i_pos_min
                    full_pos = o_pos_min >= i_pos_max
                else:
                    attend_pos = True
                    full_pos = True
                if use_window:
                    if window_left >= 0:
                        attend_pos = attend_pos and (i_pos_min >= o_pos_min - window_left)
                        full_pos = full_pos and (i_pos_min >= o_pos_max - window_left)
                    if window_right >= 0:
                        attend_pos = attend_pos and (i_pos_max <= o_pos_max + window_right)
                        full_pos = full_pos and (i_pos_max <= o_pos_min + window_right)

                attend = attend_pos and attend_seg and not (i_seg_min == pad_inner)
                full = full_seg and full_pos and attend
                if attend:
                    up = max(up, i + 1)
                    lo = min(lo, i)
                if full:
                    up_full = max(up_full, i + 1)
                    lo_full = min(lo_full, i)

            # Step 5: clip / order fix-up.
            lo = min(max(lo, 0), nbkv)
            up = min(max(up, 0), nbkv)
            lo = min(lo, up)
            lo_full = max(min(max(lo_full, 0), nbkv), lo)
            up_full = min(max(min(max(up_full, 0), nbkv), lo_full), up)
            lower[b, 0, j] = lo
            upper[b, 0, j] = up
            lower_full[b, 0, j] = lo_full
            upper_full[b, 0, j] = up_full

    cast = lambda a: a.astype(np.int32)
    return cast(lower), cast(upper), cast(lower_full), cast(upper_full)
