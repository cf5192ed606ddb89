"""GPU parity: SparseMask bounds kernel (forward and dK/dV) vs the oracle, bit-exact."""

import os

import numpy as np
import pytest
import torch

import oracle
from selected_block_attention_gb300 import workloads

pytestmark = pytest.mark.gpu
DEV = "cuda"
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "sparse_mask_causal_4block.txt")


@pytest.fixture(scope="module")
def sba():
    import __graft_entry__

    __graft_entry__.build()
    import selected_block_attention_gb300 as m

    return m


def _check(sba, qp, qs, kp, ks, qb, kb, **kw):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)
    got = sba.sparse_mask_bounds(t(qp), t(qs), t(kp), t(ks), qb, kb, **kw)
    sba.check_error()
    ref = oracle.sparse_mask_bounds(qp, qs, kp, ks, qb, kb, **kw)
    for name, g, r in zip(("lower", "upper", "lower_full", "upper_full"), got, ref):
        np.testing.assert_array_equal(g.cpu().numpy(), r, err_msg=name)
    return got


def test_page_example(sba):
    rows = np.loadtxt(GOLDEN, dtype=np.int64, comments="#")
    pos = np.arange(256)[None]
    seg = np.zeros((1, 256), np.int64)
    lo, up, _, _ = _check(sba, pos, seg, pos, seg, 64, 64, causal=True)
    for j, lower, upper in rows:
        assert (int(lo[0, 0, j]), int(up[0, 0, j])) == (lower, upper)


def test_full_size_workload(sba):
    """B=4, T=16384, block 128, window (1024, 0), documents + 300 padding tokens."""
    m = workloads.mask(device="cpu")
    _check(sba, m.q_positions.numpy(), m.q_segment_ids.numpy(), m.kv_positions.numpy(),
           m.kv_segment_ids.numpy(), 128, 128, causal=True, window_left=1024, window_right=0,
           padding_segment_id=-1)


@pytest.mark.parametrize("seed", range(6))
def test_random_ragged(sba, seed):
    """Ragged lengths (scalar load path), odd block sizes, windows both sides,
    non-causal, shuffled positions, several documents and padding."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 4))
    Tq, Tkv = int(rng.integers(1, 700)), int(rng.integers(1, 700))
    qb, kb = int(rng.choice([7, 16, 33, 64, 128])), int(rng.choice([5, 16, 32, 100, 128]))
    qp = np.sort(rng.integers(-5, 900, size=(B, Tq)), axis=1)
    kp = np.sort(rng.integers(-5, 900, size=(B, Tkv)), axis=1)
    if seed % 2:
        rng.shuffle(qp, axis=1)
    qs = np.sort(rng.integers(0, 6, size=(B, Tq)), axis=1)
    ks = np.sort(rng.integers(0, 6, size=(B, Tkv)), axis=1)
    qs[:, -int(rng.integers(0, 40)) or Tq:] = -1
    ks[:, -int(rng.integers(0, 40)) or Tkv:] = -1
    wl = int(rng.choice([-1, 0, 37, 128]))
    wr = int(rng.choice([-1, 0, 64]))
    _check(sba, qp, qs, kp, ks, qb, kb, causal=bool(seed % 3), window_left=wl, window_right=wr,
           padding_segment_id=-1)


def test_multiple_of_four_vector_path(sba):
    rng = np.random.default_rng(9)
    T = 4096
    seg = np.sort(rng.integers(0, 12, size=(2, T)), axis=1)
    seg[:, -100:] = 77  # another padding id
    pos = np.broadcast_to(np.arange(T), (2, T))
    _check(sba, pos, seg, pos, seg, 64, 128, causal=True, window_left=300, window_right=-1,
           padding_segment_id=77)


def test_many_kv_blocks_chunked(sba):
    """More key blocks than one shared-memory chunk holds (1024)."""
    T = 40000
    pos = np.arange(T)[None]
    seg = (np.arange(T) // 5000)[None]
    _check(sba, pos, seg, pos, seg, 512, 32, causal=True, window_left=2000, window_right=-1)


@pytest.mark.parametrize("dkdv", [False, True])
@pytest.mark.parametrize("seed", range(8))
def test_random_unsorted(sba, seed, dkdv):
    """Positions and segment ids in no order at all (the candidate-range pruning must hold
    for any input, not only monotone ones), padding scattered inside the rows, both
    window sides, causal or not."""
    rng = np.random.default_rng(300 + seed)
    B = int(rng.integers(1, 5))
    Tq, Tkv = int(rng.integers(200, 3000)), int(rng.integers(200, 3000))
    qb, kb = int(rng.choice([4, 16, 33, 64])), int(rng.choice([4, 16, 31, 64]))
    span = int(rng.choice([50, 3000, 1 << 30]))
    qp = rng.integers(-span, span, size=(B, Tq))
    kp = rng.integers(-span, span, size=(B, Tkv))
    if seed % 4 == 1:  # mostly sorted with a few swaps
        qp.sort(axis=1); kp.sort(axis=1)
        for a in (qp, kp):
            for _ in range(5):
                i, j = rng.integers(0, a.shape[1], 2)
                a[:, [i, j]] = a[:, [j, i]]
    qs = rng.integers(0, 8, size=(B, Tq))
    ks = rng.integers(0, 8, size=(B, Tkv))
    if seed % 2:
        qs.sort(axis=1); ks.sort(axis=1)
    qs[rng.random((B, Tq)) < 0.05] = -1
    ks[rng.random((B, Tkv)) < 0.05] = -1
    wl = int(rng.choice([-1, 0, 37, 1000]))
    wr = int(rng.choice([-1, 0, 64, 2000]))
    _check(sba, qp, qs, kp, ks, qb, kb, causal=bool(seed % 3), window_left=wl, window_right=wr,
           padding_segment_id=-1, calculate_dkdv_mask=dkdv)


@pytest.mark.parametrize("dkdv", [False, True])
def test_more_inner_blocks_than_shared_memory_holds(sba, dkdv):
    """5,000 inner blocks per row: beyond the 4,096 the one-cluster-per-row kernel keeps
    in shared memory, so the chunked kernel runs."""
    T = 40000
    pos = np.arange(T)[None]
    seg = (np.arange(T) // 5000)[None]
    qb, kb = (512, 8) if not dkdv else (8, 512)
    _check(sba, pos, seg, pos, seg, qb, kb, causal=True, window_left=2000, window_right=-1,
           calculate_dkdv_mask=dkdv)


def test_many_batch_rows(sba):
    """300 batch rows (one cluster each), ragged tail, both directions."""
    m = workloads.mask(device="cpu", B=300, T=1000, mean_doc=150, pad_tail=37, block=64,
                       window=(200, 0))
    a = [m.q_positions.numpy(), m.q_segment_ids.numpy(), m.kv_positions.numpy(),
         m.kv_segment_ids.numpy()]
    for dkdv in (False, True):
        _check(sba, *a, 64, 32, causal=True, window_left=200, window_right=0,
               calculate_dkdv_mask=dkdv)


def test_scaled_sweep_sampled(sba):
    """The scaled bandwidth workload (B=64, T=131072, block 128, window (1024, 0)) in the
    launch the bench times; the oracle checks rows 0, 31 and 63 (one long row costs it
    a few seconds)."""
    m = workloads.mask(device=DEV, B=64, T=131072)
    got = sba.sparse_mask_bounds(m.q_positions, m.q_segment_ids, m.kv_positions, m.kv_segment_ids,
                                 128, 128, causal=True, window_left=1024, window_right=0)
    sba.check_error()
    for b in (0, 31, 63):
        sl = lambda t: t[b:b + 1].cpu().numpy()
        ref = oracle.sparse_mask_bounds(sl(m.q_positions), sl(m.q_segment_ids), sl(m.kv_positions),
                                        sl(m.kv_segment_ids), 128, 128, causal=True,
                                        window_left=1024, window_right=0)
        for name, g, r in zip(("lower", "upper", "lower_full", "upper_full"), got, ref):
            np.testing.assert_array_equal(g[b:b + 1].cpu().numpy(), r, err_msg=f"{name} row {b}")


# --------------------------------------------------------------------------- dK/dV bounds

def test_dkdv_page_example_transposed(sba):
    pos = np.arange(256)[None]
    seg = np.zeros((1, 256), np.int64)
    lo, up, lof, upf = _check(sba, pos, seg, pos, seg, 64, 64, causal=True,
                              calculate_dkdv_mask=True)
    assert lo[0, 0].tolist() == [0, 1, 2, 3] and up[0, 0].tolist() == [4] * 4
    assert lof[0, 0].tolist() == [1, 2, 3, 4] and upf[0, 0].tolist() == [4] * 4


def test_dkdv_full_size_workload(sba):
    """The forward workload's inputs (B=4, T=16384, block 128, window (1024, 0))."""
    m = workloads.mask(device="cpu")
    _check(sba, m.q_positions.numpy(), m.q_segment_ids.numpy(), m.kv_positions.numpy(),
           m.kv_segment_ids.numpy(), 128, 128, causal=True, window_left=1024, window_right=0,
           padding_segment_id=-1, calculate_dkdv_mask=True)


@pytest.mark.parametrize("seed", range(6))
def test_dkdv_random_ragged(sba, seed):
    rng = np.random.default_rng(100 + seed)
    B = int(rng.integers(1, 4))
    Tq, Tkv = int(rng.integers(1, 700)), int(rng.integers(1, 700))
    qb, kb = int(rng.choice([7, 16, 33, 64, 128])), int(rng.choice([5, 16, 32, 100, 128]))
    qp = np.sort(rng.integers(-5, 900, size=(B, Tq)), axis=1)
    kp = np.sort(rng.integers(-5, 900, size=(B, Tkv)), axis=1)
    if seed % 2:
        rng.shuffle(kp, axis=1)
    qs = np.sort(rng.integers(0, 6, size=(B, Tq)), axis=1)
    ks = np.sort(rng.integers(0, 6, size=(B, Tkv)), axis=1)
    qs[:, -int(rng.integers(0, 40)) or Tq:] = -1
    ks[:, -int(rng.integers(0, 40)) or Tkv:] = -1
    wl = int(rng.choice([-1, 0, 37, 128]))
    wr = int(rng.choice([-1, 0, 64]))
    _check(sba, qp, qs, kp, ks, qb, kb, causal=bool(seed % 3), window_left=wl, window_right=wr,
           padding_segment_id=-1, calculate_dkdv_mask=True)


def test_dkdv_many_query_blocks_chunked(sba):
    """More query blocks (the inner operand here) than one shared-memory chunk holds."""
    T = 40000
    pos = np.arange(T)[None]
    seg = (np.arange(T) // 5000)[None]
    _check(sba, pos, seg, pos, seg, 32, 512, causal=True, window_left=2000, window_right=-1,
           calculate_dkdv_mask=True)


def test_l2_read_probe_reads_everything(sba):
    """The roofline's L2 probe XORs every 32-bit word it reads into its sink: an even
    number of passes over any buffer gives 0, an odd number the XOR of the buffer."""
    vals = (np.arange(1 << 16, dtype=np.int64) * 2654435761) % (1 << 31)
    buf = torch.from_numpy(vals.astype(np.int32)).to(DEV)
    want = int(np.bitwise_xor.reduce(vals.astype(np.uint32)))
    for reps, expect in ((1, want), (2, 0), (3, want)):
        sink = torch.zeros(1, dtype=torch.int32, device=DEV)
        sba.l2_read_probe(buf, reps, sink)
        sba.check_error()
        assert int(sink.cpu().numpy().astype(np.uint32)[0]) == expect
