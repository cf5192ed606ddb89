"""Pins for the SparseMask bounds oracle (CPU only).

The block rule is a conservative heuristic; where it is exact (positions
``arange``, windows that are multiples of the block, contiguous documents) the
bounds must equal the block ranges found by brute force over token pairs.  The
worked example printed on the mask page pins lower/upper directly.
"""

import os

import numpy as np
import pytest

from oracle import sparse_mask_bounds

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sparse_mask_causal_4block.txt")


def _brute_blocks(qp, qs, kp, ks, qb, kb, causal, wl, wr, pad=-1):
    """Per query block: sets of key blocks with ANY / ALL token pairs attending."""
    Tq, Tkv = qp.shape[0], kp.shape[0]
    att = (qs[:, None] == ks[None, :]) & (qs[:, None] != pad) & (ks[None, :] != pad)
    if causal:
        att &= kp[None, :] <= qp[:, None]
    if wl >= 0:
        att &= qp[:, None] - kp[None, :] <= wl
    if wr >= 0:
        att &= kp[None, :] - qp[:, None] <= wr
    nbq, nbk = -(-Tq // qb), -(-Tkv // kb)
    anyset, allset = [], []
    for j in range(nbq):
        a, f = set(), set()
        rows = att[j * qb:(j + 1) * qb]
        for i in range(nbk):
            blk = rows[:, i * kb:(i + 1) * kb]
            if blk.any():
                a.add(i)
            if blk.all():
                f.add(i)
        anyset.append(a)
        allset.append(f)
    return anyset, allset


def _as_sets(lo, up, lof, upf):
    return set(range(int(lo), int(up))), set(range(int(lof), int(upf)))


def test_page_example_causal_four_blocks():
    rows = np.loadtxt(GOLDEN, dtype=np.int64, comments="#")
    nb, block = 4, 64
    T = nb * block
    pos = np.arange(T)[None, :]
    seg = np.zeros((1, T), dtype=np.int64)
    lo, up, lof, upf = sparse_mask_bounds(pos, seg, pos, seg, block, block, causal=True)
    assert lo.shape == (1, 1, nb) and lo.dtype == np.int32
    for j, lower, upper in rows:
        assert (lo[0, 0, j], up[0, 0, j]) == (lower, upper)
    # Full bounds: by brute force, block j is fully attended by the blocks before it.
    anyset, allset = _brute_blocks(pos[0], seg[0], pos[0], seg[0], block, block, True, -1, -1)
    for j in range(nb):
        a, f = _as_sets(lo[0, 0, j], up[0, 0, j], lof[0, 0, j], upf[0, 0, j])
        assert a == anyset[j] and f == allset[j]
    # exact integers (an empty full range is reported as (NB, upper) for block 0)
    assert lof[0, 0].tolist() == [4, 0, 0, 0] and upf[0, 0].tolist() == [1, 1, 2, 3]


def test_noncausal_single_segment_attends_everything():
    T, qb, kb = 300, 32, 64
    pos = np.arange(T)[None, :]
    seg = np.full((1, T), 5)
    lo, up, lof, upf = sparse_mask_bounds(pos, seg, pos, seg, qb, kb, causal=False)
    nbk = -(-T // kb)
    assert np.all(lo == 0) and np.all(up == nbk)
    # the ragged last kv block holds padding tokens -> its segment range is not a
    # single segment, so it is attended but not full
    assert np.all(lof[0, 0, :-1] == 0) and np.all(upf[0, 0, :-1] == nbk - 1)
    # the ragged last query block mixes real tokens and padding: nothing is full
    assert lof[0, 0, -1] >= upf[0, 0, -1]


def test_all_padding_block_and_nothing_attended():
    qb = kb = 8
    T = 32
    pos = np.arange(T)[None, :]
    qseg = np.zeros((1, T), dtype=np.int64)
    qseg[0, 24:] = -1                    # last query block is all padding
    kseg = np.full((1, T), 3)            # keys live in another document
    kseg[0, :8] = 0
    lo, up, lof, upf = sparse_mask_bounds(pos, qseg, pos, kseg, qb, kb, causal=True)
    # block 3: all padding -> zeros
    assert (lo[0, 0, 3], up[0, 0, 3], lof[0, 0, 3], upf[0, 0, 3]) == (0, 0, 0, 0)
    # blocks 1, 2: segment 0 only, keys of segment 0 live in kv block 0 -> attended & full
    for j in (1, 2):
        assert (lo[0, 0, j], up[0, 0, j], lof[0, 0, j], upf[0, 0, j]) == (0, 1, 0, 1)
    # nothing attended: (0, 0, NB, 0)
    kseg2 = np.full((1, T), 7)
    lo, up, lof, upf = sparse_mask_bounds(pos, qseg, pos, kseg2, qb, kb, causal=True)
    for j in range(3):
        assert (lo[0, 0, j], up[0, 0, j], lof[0, 0, j], upf[0, 0, j]) == (0, 0, 4, 0)


@pytest.mark.parametrize("block,wl,wr,causal", [
    (16, -1, -1, True), (16, 32, 0, True), (8, 24, -1, True), (16, 16, 32, False),
    (32, 64, 0, True), (16, -1, 48, False)])
def test_brute_force_single_segment(block, wl, wr, causal):
    T = 160
    pos = np.arange(T)
    seg = np.zeros(T, dtype=np.int64)
    lo, up, lof, upf = sparse_mask_bounds(pos[None], seg[None], pos[None], seg[None], block, block,
                                          causal=causal, window_left=wl, window_right=wr)
    anyset, allset = _brute_blocks(pos, seg, pos, seg, block, block, causal, wl, wr)
    for j in range(len(anyset)):
        a, f = _as_sets(lo[0, 0, j], up[0, 0, j], lof[0, 0, j], upf[0, 0, j])
        assert a == anyset[j], j
        assert f == allset[j], j


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_brute_force_packed_documents_noncausal(seed):
    rng = np.random.default_rng(seed)
    T, qb, kb = 256, 16, 32
    lens = []
    while sum(lens) < T - 20:
        lens.append(int(rng.integers(1, 60)))
    seg = np.full(T, -1, dtype=np.int64)
    off = 0
    for d, L in enumerate(lens):
        seg[off:min(off + L, T - 20)] = d
        off += L
        if off >= T - 20:
            break
    pos = np.arange(T)
    lo, up, lof, upf = sparse_mask_bounds(pos[None], seg[None], pos[None], seg[None], qb, kb,
                                          causal=False)
    anyset, allset = _brute_blocks(pos, seg, pos, seg, qb, kb, False, -1, -1)
    for j in range(len(anyset)):
        a, f = _as_sets(lo[0, 0, j], up[0, 0, j], lof[0, 0, j], upf[0, 0, j])
        if not anyset[j]:
            continue  # all-padding query block: checked separately
        assert a == anyset[j], j
        assert f == allset[j], j


def test_left_window_edge_reading():
    """The attend test on the left window edge compares the smallest key
    position of a block with min(query) - window_left: a straddling block is
    dropped although one of its token pairs lies inside the window."""
    block, wl = 4, 5
    T = 16
    pos = np.arange(T)[None, :]
    seg = np.zeros((1, T), dtype=np.int64)
    lo, up, lof, upf = sparse_mask_bounds(pos, seg, pos, seg, block, block, causal=True,
                                          window_left=wl)
    # query block 2 = positions 8..11; key block 0 = 0..3: pair (8, 3) is in the
    # window, yet 0 >= 8 - 5 fails, so the block range starts at 1.
    assert (lo[0, 0, 2], up[0, 0, 2]) == (1, 3)


def test_ragged_lengths_are_padded():
    """Tq, Tkv not multiples of the block: query padding has position -1 and
    key padding the int32 maximum, both with the padding segment."""
    Tq, Tkv, qb, kb = 10, 13, 4, 4
    qp, kp = np.arange(Tq)[None], np.arange(Tkv)[None]
    qs, ks = np.zeros((1, Tq), np.int64), np.zeros((1, Tkv), np.int64)
    lo, up, lof, upf = sparse_mask_bounds(qp, qs, kp, ks, qb, kb, causal=True)
    assert lo.shape == (1, 1, 3)
    # last query block holds positions 8, 9 and two pads (-1): min position -1
    # makes no key block full; the block's max position 9 reaches kv block 2.
    assert (lo[0, 0, 2], up[0, 0, 2], lof[0, 0, 2], upf[0, 0, 2]) == (0, 3, 4, 3)
    # first query block: keys 0..3 attended, none full (diagonal); 4 kv blocks after padding
    assert (lo[0, 0, 0], up[0, 0, 0], lof[0, 0, 0], upf[0, 0, 0]) == (0, 1, 4, 1)
    # kv block 3 (key 12 + three pads) is never full and only attended when the
    # query block's max position reaches 12
    assert up.max() == 3


# --------------------------------------------------------------------------- dK/dV bounds
# With the key/value blocks as the outer operand, kv block i gets the range of query
# blocks j that attend it.

def _brute_kv_blocks(qp, qs, kp, ks, qb, kb, causal, wl, wr, pad=-1):
    """Per kv block: sets of query blocks with ANY / ALL token pairs attending."""
    anyset, allset = _brute_blocks(qp, qs, kp, ks, qb, kb, causal, wl, wr, pad)
    nbk = -(-kp.shape[0] // kb)
    return ([{j for j, a in enumerate(anyset) if i in a} for i in range(nbk)],
            [{j for j, f in enumerate(allset) if i in f} for i in range(nbk)])


def test_dkdv_page_example_transposed():
    """The page's causal four-block example read from the key side: kv block i is
    attended by query blocks i..3 and fully by the blocks after it."""
    nb, block = 4, 64
    pos = np.arange(nb * block)[None, :]
    seg = np.zeros_like(pos)
    lo, up, lof, upf = sparse_mask_bounds(pos, seg, pos, seg, block, block, causal=True,
                                          calculate_dkdv_mask=True)
    assert lo.shape == (1, 1, nb) and lo.dtype == np.int32
    assert lo[0, 0].tolist() == [0, 1, 2, 3] and up[0, 0].tolist() == [4, 4, 4, 4]
    # full: query blocks after i; for i = 3 the empty range is reported as (4, 4)
    assert lof[0, 0].tolist() == [1, 2, 3, 4] and upf[0, 0].tolist() == [4, 4, 4, 4]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_dkdv_is_the_transpose_of_the_forward_relation(causal, seed):
    """Without a window every predicate of the rule is symmetric in its two operands,
    so kv block i's query range is exactly the set of query blocks whose forward range
    contains i (documents are contiguous, so every set is an interval)."""
    rng = np.random.default_rng(seed)
    T, qb, kb = 700, 32, 64
    lens = rng.integers(20, 300, size=8)
    seg = np.repeat(np.arange(8), lens)[:T - 37]
    seg = np.concatenate([seg, np.full(T - seg.size, -1)])[None, :]
    pos = np.arange(T)[None, :]
    f = sparse_mask_bounds(pos, seg, pos, seg, qb, kb, causal=causal)
    d = sparse_mask_bounds(pos, seg, pos, seg, qb, kb, causal=causal, calculate_dkdv_mask=True)
    nbq, nbk = f[0].shape[2], d[0].shape[2]
    for i in range(nbk):
        att = [j for j in range(nbq) if f[0][0, 0, j] <= i < f[1][0, 0, j]]
        full = [j for j in range(nbq) if f[2][0, 0, j] <= i < f[3][0, 0, j]]
        got_att = set(range(d[0][0, 0, i], d[1][0, 0, i]))
        got_full = set(range(d[2][0, 0, i], d[3][0, 0, i]))
        assert got_att == set(att), (i, got_att, att)
        assert got_full == set(full), (i, got_full, full)


@pytest.mark.parametrize("block,causal", [(32, True), (64, False), (16, True)])
def test_dkdv_brute_force_without_window(block, causal):
    T = 5 * block + 7
    pos = np.arange(T)
    seg = np.zeros(T, dtype=np.int64)
    lo, up, lof, upf = sparse_mask_bounds(pos[None], seg[None], pos[None], seg[None], block,
                                          block, causal=causal, calculate_dkdv_mask=True)
    anyset, allset = _brute_kv_blocks(pos, seg, pos, seg, block, block, causal, -1, -1)
    for i in range(lo.shape[2]):
        a, f = _as_sets(lo[0, 0, i], up[0, 0, i], lof[0, 0, i], upf[0, 0, i])
        assert a == anyset[i]
        # a padded tail block (either side) mixes a segment with padding, so it is
        # never part of a full pair; elsewhere the full set is exact
        last = lo.shape[2] - 1
        if i < last:
            assert f == allset[i] - {last}
        else:
            assert f == set()


@pytest.mark.parametrize("w", [64, 128, 192])
def test_dkdv_symmetric_window_noncausal_is_exact(w):
    """Non-causal with equal left and right windows (multiples of the block): the
    printed kv-outer tests then reduce to |q - k| <= w per block pair, which matches
    brute force over token pairs."""
    T, block = 8 * 64, 64
    pos = np.arange(T)
    seg = np.zeros(T, dtype=np.int64)
    lo, up, lof, upf = sparse_mask_bounds(pos[None], seg[None], pos[None], seg[None], block,
                                          block, causal=False, window_left=w, window_right=w,
                                          calculate_dkdv_mask=True)
    anyset, _ = _brute_kv_blocks(pos, seg, pos, seg, block, block, False, w, w)
    for i in range(lo.shape[2]):
        assert set(range(lo[0, 0, i], up[0, 0, i])) == anyset[i]


def test_dkdv_left_window_does_not_prune_under_causal():
    """The printed kv-outer left-window attend test (largest query position >=
    smallest key position - left) is implied by the causal attend test, so a left
    window leaves the dK/dV attend range causal: kv block i keeps query blocks i..NB."""
    T, block = 8 * 64, 64
    pos = np.arange(T)[None, :]
    seg = np.zeros_like(pos)
    lo, up, _, _ = sparse_mask_bounds(pos, seg, pos, seg, block, block, causal=True,
                                      window_left=64, calculate_dkdv_mask=True)
    assert lo[0, 0].tolist() == list(range(8)) and up[0, 0].tolist() == [8] * 8


def test_dkdv_padding_blocks():
    """An all-padding kv block gets (0, 0, 0, 0); all-padding query blocks are never
    attended; different query and kv lengths give ragged tails on both sides."""
    Tq, Tkv, qb, kb = 200, 300, 32, 64
    qpos, kpos = np.arange(Tq)[None], np.arange(Tkv)[None]
    qseg = np.zeros((1, Tq), dtype=np.int64)
    kseg = np.zeros((1, Tkv), dtype=np.int64)
    qseg[0, 160:] = -1                   # query blocks 5 and 6 are all padding
    kseg[0, 256:] = -1                   # kv block 4 is all padding
    lo, up, lof, upf = sparse_mask_bounds(qpos, qseg, kpos, kseg, qb, kb, causal=False,
                                          calculate_dkdv_mask=True)
    assert lo.shape == (1, 1, 5)
    assert (lo[0, 0, 4], up[0, 0, 4], lof[0, 0, 4], upf[0, 0, 4]) == (0, 0, 0, 0)
    assert np.all(up[0, 0, :4] == 5) and np.all(lo[0, 0, :4] == 0)


def test_dkdv_one_sided_windows_as_printed():
    """Hand evaluation of the printed kv-outer window tests (non-causal, one segment,
    positions arange, block 64, 8 blocks).  Left window 64: attend needs
    max q >= min k - 64 and full needs min q >= min k - 64, both j >= i - 1.  Right
    window 64: attend needs min q <= max k + 64 and full needs max q <= max k + 64,
    both j <= i + 1.  (The tests bound the opposite side of the transposed forward
    rule; a swapped min/max in either full test moves the full range by one block.)"""
    T, block, nb = 8 * 64, 64, 8
    pos = np.arange(T)[None, :]
    seg = np.zeros_like(pos)
    lo, up, lof, upf = sparse_mask_bounds(pos, seg, pos, seg, block, block, causal=False,
                                          window_left=64, calculate_dkdv_mask=True)
    want_lo = [max(i - 1, 0) for i in range(nb)]
    assert lo[0, 0].tolist() == want_lo and up[0, 0].tolist() == [nb] * nb
    assert lof[0, 0].tolist() == want_lo and upf[0, 0].tolist() == [nb] * nb
    lo, up, lof, upf = sparse_mask_bounds(pos, seg, pos, seg, block, block, causal=False,
                                          window_right=64, calculate_dkdv_mask=True)
    want_up = [min(i + 2, nb) for i in range(nb)]
    assert lo[0, 0].tolist() == [0] * nb and up[0, 0].tolist() == want_up
    assert lof[0, 0].tolist() == [0] * nb and upf[0, 0].tolist() == want_up
