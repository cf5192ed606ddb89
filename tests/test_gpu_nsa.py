"""GPU parity: NSA selection forward (C ABI through the binding) vs the fp64 oracle."""

import numpy as np
import pytest
import torch

import oracle
from selected_block_attention_gb300 import workloads
from tests._parity import assert_attention_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sba():
    import __graft_entry__

    __graft_entry__.build()
    import selected_block_attention_gb300 as m

    return m


DEV = "cuda"


def _run(sba, w, rows=None):
    out, lse = sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts, w.block_size,
                                  cu_seqlens=w.cu_seqlens, causal=w.causal)
    sba.check_error()
    counts = w.block_counts if isinstance(w.block_counts, int) else w.block_counts.cpu().numpy()
    cu = None if w.cu_seqlens is None else w.cu_seqlens.cpu().numpy()
    ref, ref_lse = oracle.nsa_select_attention(
        to_np(w.q), to_np(w.k), to_np(w.v),
        w.block_indices.cpu().numpy(), counts, w.block_size, cu_seqlens=cu, causal=w.causal,
        rows=rows)
    got, got_lse = to_np(out), to_np(lse)
    if rows is not None:
        idx = tuple(np.array(rows).T)
        return got[idx], ref[idx], got_lse[idx], ref_lse[idx]
    return got, ref, got_lse, ref_lse


def test_tiny_fp32_full(sba):
    """The 256-token fp32 workload (tf32 tensor cores), every row."""
    w = workloads.nsa_tiny(device=DEV)
    assert_attention_close(*_run(sba, w), what="nsa_tiny")


@pytest.mark.parametrize("bs", [32, 64, 128])
@pytest.mark.parametrize("D", [64, 128])
def test_bf16_small_shapes(sba, bs, D):
    """GQA 16:2 (G=8), ragged T, counts array, all block sizes, D 64/128."""
    w = workloads.nsa_prefill(device=DEV, B=2, T=333, Hq=16, Hkv=2, D=D, block_size=bs, S=6,
                              max_count=6, seed=100 + bs + D)
    got, ref, gl, rl = _run(sba, w)
    assert_attention_close(got, ref, gl, rl, what=f"bs={bs} D={D}")


@pytest.mark.parametrize("G", [1, 4, 16])
def test_bf16_group_sizes(sba, G):
    w = workloads.nsa_prefill(device=DEV, B=1, T=520, Hq=2 * G, Hkv=2, D=128, block_size=64,
                              S=16, max_count=16, seed=200 + G)
    assert_attention_close(*_run(sba, w), what=f"G={G}")


def test_messy_indices(sba):
    """-1 entries, out-of-range ids, future blocks (causal), duplicates, counts above S
    and below 0, empty selections."""
    rng = np.random.default_rng(5)
    w = workloads.nsa_prefill(device=DEV, B=2, T=400, Hq=8, Hkv=2, D=128, block_size=64, S=8,
                              max_count=8, seed=7)
    nb = -(-400 // 64)
    idx = rng.integers(-3, nb + 3, size=(2, 400, 2, 8)).astype(np.int32)
    idx[:, :, :, 7] = idx[:, :, :, 0]  # duplicates
    counts = rng.integers(-2, 11, size=(2, 400, 2)).astype(np.int32)
    counts[0, :20] = 0                  # empty rows
    w.block_indices = torch.from_numpy(idx).to(DEV)
    w.block_counts = torch.from_numpy(counts).to(DEV)
    got, ref, gl, rl = _run(sba, w)
    assert np.isneginf(rl).any()
    assert_attention_close(got, ref, gl, rl, what="messy")


def test_scalar_count_and_noncausal(sba):
    w = workloads.nsa_prefill(device=DEV, B=1, T=256, Hq=4, Hkv=1, D=128, block_size=32, S=5,
                              max_count=5, seed=9)
    w.block_counts = 3
    w.causal = False
    assert_attention_close(*_run(sba, w), what="scalar count, non-causal")


def test_varlen_small(sba):
    w = workloads.nsa_varlen(device=DEV, lengths=[100, 257, 1, 64, 190], Hq=8, Hkv=2, D=128,
                             block_size=64, S=4, count=4, seed=11)
    assert_attention_close(*_run(sba, w), what="varlen small")


def test_prefill_full_size_sampled(sba):
    """The B=2, T=8192, Hq=64, Hkv=4 workload in the benchmark's launch
    configuration; 96 sampled tokens (every head) against the oracle."""
    w = workloads.nsa_prefill(device=DEV)
    rng = np.random.default_rng(1)
    rows = [(int(b), int(t)) for b, t in zip(rng.integers(0, 2, 96), rng.integers(0, 8192, 96))]
    rows += [(0, 0), (1, 8191), (0, 63), (0, 64)]
    got, ref, gl, rl = _run(sba, w, rows=rows)
    assert_attention_close(got, ref, gl, rl, what="prefill sampled")


def test_varlen_full_size_sampled(sba):
    w = workloads.nsa_varlen(device=DEV)
    T = w.q.shape[1]
    rng = np.random.default_rng(2)
    cu = w.cu_seqlens.cpu().numpy()
    rows = [(0, int(t)) for t in rng.integers(0, T, 64)]
    rows += [(0, int(c)) for c in cu[:-1]] + [(0, int(c) - 1) for c in cu[1:]]
    got, ref, gl, rl = _run(sba, w, rows=rows)
    assert_attention_close(got, ref, gl, rl, what="varlen sampled")


def test_rejects_bad_arguments(sba):
    w = workloads.nsa_prefill(device=DEV, B=1, T=64, Hq=4, Hkv=1, D=128, block_size=64, S=2,
                              max_count=2, seed=3)
    with pytest.raises(sba.SBAError):
        sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts, 48)
    with pytest.raises(ValueError):
        sba.nsa_select_fwd(w.q.cpu(), w.k, w.v, w.block_indices, w.block_counts, 64)
