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
