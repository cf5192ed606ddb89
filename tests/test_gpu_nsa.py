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


def _run(sba, w, rows=None, softmax_scale=None):
    out, lse = sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts, w.block_size,
                                  cu_seqlens=w.cu_seqlens, causal=w.causal,
                                  softmax_scale=softmax_scale)
    sba.check_error()
    counts = w.block_counts if isinstance(w.block_counts, int) else w.block_counts.cpu().numpy()
    cu = None if w.cu_seqlens is None else w.cu_seqlens.cpu().numpy()
    ref, ref_lse = oracle.nsa_select_attention(
        to_np(w.q), to_np(w.k), to_np(w.v),
        w.block_indices.cpu().numpy(), counts, w.block_size, cu_seqlens=cu, causal=w.causal,
        softmax_scale=softmax_scale, rows=rows)
    got, got_lse = to_np(out), to_np(lse)
    if rows is not None:
        idx = tuple(np.array(rows).T)
        return got[idx], ref[idx], got_lse[idx], ref_lse[idx]
    return got, ref, got_lse, ref_lse


def test_tiny_fp32_full(sba):
    """The 256-token fp32 workload (exact fp32 on CUDA cores), every row."""
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


def test_union_full_sort_capacity(sba):
    """G=8 puts 16 tokens in one item; S=32 entries each (with repeats across tokens and
    within a token) fill the 512-entry union sort."""
    rng = np.random.default_rng(21)
    T, bs = 700, 32
    w = workloads.nsa_prefill(device=DEV, B=1, T=T, Hq=16, Hkv=2, D=128, block_size=bs, S=32,
                              max_count=32, seed=21)
    nb = -(-T // bs)
    own = (np.arange(T) // bs)[None, :, None, None]
    idx = rng.integers(0, nb, size=(1, T, 2, 32))
    idx = np.minimum(idx, own).astype(np.int32)      # mostly past blocks, many repeats
    idx[..., 0] = own[..., 0]
    w.block_indices = torch.from_numpy(idx).to(DEV)
    w.block_counts = torch.full((1, T, 2), 32, dtype=torch.int32, device=DEV)
    assert_attention_close(*_run(sba, w), what="union sort capacity")


@pytest.mark.parametrize("bs", [32, 64, 128])
def test_union_dense_selection(sba, bs):
    """Every token selects every block up to its own: equals causal dense attention,
    and every union block is shared by all tokens of an item."""
    T = 640
    nb = -(-T // bs)
    w = workloads.nsa_prefill(device=DEV, B=1, T=T, Hq=32, Hkv=2, D=128, block_size=bs, S=nb,
                              max_count=nb, seed=30 + bs) if nb <= 32 else None
    if w is None:
        pytest.skip("more blocks than selection slots")
    idx = np.tile(np.arange(nb, dtype=np.int32), (1, T, 2, 1))
    w.block_indices = torch.from_numpy(idx).to(DEV)
    w.block_counts = nb
    assert_attention_close(*_run(sba, w), what=f"dense bs={bs}")


@pytest.mark.parametrize("G", [3, 12])
def test_union_odd_group_sizes(sba, G):
    """G that does not divide 128: items of 128 // G tokens (at most 16), rows below 128."""
    w = workloads.nsa_prefill(device=DEV, B=2, T=300, Hq=2 * G, Hkv=2, D=64, block_size=64,
                              S=8, max_count=8, seed=40 + G)
    assert_attention_close(*_run(sba, w), what=f"G={G}")


def test_union_large_logits_rescale(sba):
    """Scale 0.5 on N(0,1) data makes per-tile maxima jump by more than 2^8 in log2
    units between tiles, exercising the lazy rescale of O in TMEM.  Such a peaked
    softmax copies single V values into the output, and for |v| > 4 the bf16 rounding
    of the output alone costs up to 2^-6; V is halved (exactly) so the absolute bound
    measures the rescale and not the output format."""
    w = workloads.nsa_prefill(device=DEV, B=1, T=1024, Hq=32, Hkv=2, D=128, block_size=64,
                              S=16, max_count=16, seed=50)
    w.v = w.v * 0.5
    assert_attention_close(*_run(sba, w, softmax_scale=0.5), what="large logits")


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


@pytest.mark.parametrize("case", ["bf16", "f32"])
def test_selection_gate(sba, case):
    """g_slc scales each output row of the selection branch; the LSE is ungated."""
    if case == "bf16":
        w = workloads.nsa_prefill(device=DEV, B=2, T=300, Hq=32, Hkv=2, D=128, block_size=64,
                                  S=6, max_count=6, seed=60)
    else:
        w = workloads.nsa_tiny(device=DEV)
    # gates in (0, 1), as a sigmoid gate produces them (the absolute bound would
    # otherwise scale with |gate|)
    gate = torch.sigmoid(workloads.randn(tuple(w.q.shape[:3]), torch.float32, DEV, seed=61)).to(w.q.dtype)
    out, lse = sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts, w.block_size,
                                  causal=w.causal, g_slc=gate)
    sba.check_error()
    counts = w.block_counts if isinstance(w.block_counts, int) else w.block_counts.cpu().numpy()
    ref, ref_lse = oracle.nsa_select_attention(
        to_np(w.q), to_np(w.k), to_np(w.v), w.block_indices.cpu().numpy(), counts, w.block_size,
        causal=w.causal, g_slc=to_np(gate))
    assert_attention_close(to_np(out), ref, to_np(lse), ref_lse, what=f"gate {case}")


@pytest.mark.parametrize("B,dtype,gate,counts_tensor,with_lse,pinned", [
    (3, torch.bfloat16, True, True, True, True),      # three row chunks, gate, counts array
    (6, torch.bfloat16, False, False, False, True),   # 4 chunks of 1-2 rows, scalar count, no LSE
    (1, torch.float32, False, True, True, False),     # fp32, one chunk, pageable host memory
])
def test_host_entry_against_oracle(sba, B, dtype, gate, counts_tensor, with_lse, pinned):
    """The host-buffer entry point (inputs and outputs in host memory, batch rows staged
    and computed in chunks) against the fp64 oracle, every row.  Chunks change which
    tokens share an item (items are windows of consecutive tokens), so the result is
    held to the attention tolerances, not to the device entry's bits."""
    w = workloads.nsa_prefill(device=DEV, B=B, T=300, Hq=8, Hkv=2, D=128, block_size=64, S=5,
                              max_count=5, seed=300 + B, dtype=dtype)
    counts = w.block_counts if counts_tensor else 3
    g = None
    if gate:
        g = torch.sigmoid(workloads.randn(tuple(w.q.shape[:3]), torch.float32, DEV, seed=301)).to(dtype)
    host = lambda t: None if t is None else (t.cpu().pin_memory() if pinned else t.cpu())
    out, lse = sba.nsa_select_fwd_host(
        host(w.q), host(w.k), host(w.v), host(w.block_indices),
        host(counts) if counts_tensor else counts, w.block_size, causal=True, g_slc=host(g),
        return_lse=with_lse)
    torch.cuda.synchronize()
    sba.check_error()
    assert not out.is_cuda and out.is_pinned() == pinned
    ref, ref_lse = oracle.nsa_select_attention(
        to_np(w.q), to_np(w.k), to_np(w.v), w.block_indices.cpu().numpy(),
        w.block_counts.cpu().numpy() if counts_tensor else counts, w.block_size, causal=True,
        g_slc=None if g is None else to_np(g))
    if with_lse:
        assert_attention_close(to_np(out), ref, to_np(lse), ref_lse, what=f"host entry B={B}")
    else:
        assert lse is None
        assert_attention_close(to_np(out), ref, what=f"host entry B={B}")


def test_host_entry_in_stream_order(sba):
    """Two back-to-back host calls that share one workspace, synchronized once at the
    end: each call starts after the work already on the stream, so the second call's
    staging copies wait for the first call's kernels and copies.  With T = 256 (a
    multiple of the 32-token item window at G = 4) the row chunks form the same items
    as one whole-batch launch, so both results equal the device entry's bit for bit."""
    w1 = workloads.nsa_prefill(device=DEV, B=2, T=256, Hq=8, Hkv=2, D=128, S=4, max_count=4, seed=401)
    w2 = workloads.nsa_prefill(device=DEV, B=2, T=256, Hq=8, Hkv=2, D=128, S=4, max_count=4, seed=402)
    res = []
    ws = torch.empty(sba.nsa_select_host_workspace_size(2, 256, 8, 2, 128, 4), dtype=torch.uint8,
                     device=DEV)
    for w in (w1, w2):
        pin = lambda t: t.cpu().pin_memory()
        res.append(sba.nsa_select_fwd_host(pin(w.q), pin(w.k), pin(w.v), pin(w.block_indices),
                                           pin(w.block_counts), w.block_size, workspace=ws))
    torch.cuda.synchronize()
    sba.check_error()
    for w, (out, lse) in zip((w1, w2), res):
        ref_out, ref_lse = sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts,
                                              w.block_size)
        assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())


def test_first_item_of_every_cta(sba):
    """128 work items (1,024 tokens in groups of 8, one KV head) on at most 152
    persistent CTAs: every CTA runs exactly one item, its first.  Run twice: identical."""
    w = workloads.nsa_prefill(device=DEV, B=1, T=1024, Hq=16, Hkv=1, D=128, seed=909)
    got, ref, gl, rl = _run(sba, w)
    assert_attention_close(got, ref, gl, rl, what="nsa first items")
    got2, _, gl2, _ = _run(sba, w)
    assert np.array_equal(got, got2) and np.array_equal(gl, gl2), "second launch differs"


@pytest.mark.parametrize("B,causal,gate", [(1, True, False), (2, True, True), (2, False, False)])
def test_host_entry_split_along_tokens(sba, B, causal, gate):
    """T = 1024 (a multiple of 128): the host entry stages (batch row, token range)
    chunks, each computed once the K/V prefix it needs has arrived (without causal
    masking, the whole row's K/V with the row's first chunk).  The chunks hold whole
    item windows, so the result equals the device entry bit for bit; and the oracle."""
    w = workloads.nsa_prefill(device=DEV, B=B, T=1024, Hq=32, Hkv=2, D=128, seed=450 + B)
    g = None
    if gate:
        g = torch.sigmoid(workloads.randn(tuple(w.q.shape[:3]), torch.float32, DEV, seed=451)).to(w.q.dtype)
    pin = lambda t: None if t is None else t.cpu().pin_memory()
    out, lse = sba.nsa_select_fwd_host(pin(w.q), pin(w.k), pin(w.v), pin(w.block_indices),
                                       pin(w.block_counts), w.block_size, causal=causal, g_slc=pin(g))
    torch.cuda.synchronize()
    sba.check_error()
    ref_out, ref_lse = sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts,
                                          w.block_size, causal=causal, g_slc=g)
    sba.check_error()
    assert torch.equal(out, ref_out.cpu()) and torch.equal(lse, ref_lse.cpu())
    rows = [(b, t) for b in range(B) for t in (0, 1, 255, 256, 511, 700, 1023)]
    ref, rl = oracle.nsa_select_attention(
        to_np(w.q), to_np(w.k), to_np(w.v), w.block_indices.cpu().numpy(),
        w.block_counts.cpu().numpy(), w.block_size, causal=causal, rows=rows,
        g_slc=None if g is None else to_np(g))
    idx = tuple(np.array(rows).T)
    assert_attention_close(to_np(out)[idx], ref[idx], to_np(lse)[idx], rl[idx], what="host split")
