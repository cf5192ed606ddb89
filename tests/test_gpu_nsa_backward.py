"""GPU parity: NSA selection backward (dq, dk, dv) vs the fp64 oracle.

The forward's out / LSE come from the GPU forward (the backward consumes what the
forward produced, as in training); the oracle recomputes everything from q, k, v in
float64.  Gradients are bf16 outputs whose magnitudes grow with the number of tokens
summed into a key (dk, dv), so the bar is relative: max abs error <= 2e-2 x max(1,
max |ref|) and relative Frobenius error <= 5e-3.
"""

import numpy as np
import pytest
import torch

import oracle
from selected_block_attention_gb300 import workloads
from tests._parity import to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
REL_FRO = 5e-3
MAX_ABS_REL = 2e-2


@pytest.fixture(scope="module")
def sba():
    import __graft_entry__

    __graft_entry__.build()
    import selected_block_attention_gb300 as m

    return m


def assert_grad_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite gradient"
    err = np.abs(got - ref).max() if got.size else 0.0
    bar = MAX_ABS_REL * max(1.0, np.abs(ref).max() if ref.size else 0.0)
    denom = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / denom if denom > 0 else np.linalg.norm(got)
    assert err <= bar, f"{what}: max abs error {err:.3g} > {bar:.3g}"
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3g}"
    return err, rel


def _run(sba, w, seed=0, causal=True):
    kw = dict(cu_seqlens=w.cu_seqlens, causal=causal)
    out, lse = sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts, w.block_size, **kw)
    g = torch.Generator(device=DEV).manual_seed(seed)
    do = torch.randn(w.q.shape, generator=g, device=DEV, dtype=torch.float32).to(w.q.dtype)
    dq, dk, dv = sba.nsa_select_bwd(w.q, w.k, w.v, out, lse, do, w.block_indices, w.block_counts,
                                    w.block_size, **kw)
    sba.check_error()
    return do, dq, dk, dv


def _oracle(w, do, causal=True, rows=None):
    counts = w.block_counts if isinstance(w.block_counts, int) else w.block_counts.cpu().numpy()
    cu = None if w.cu_seqlens is None else w.cu_seqlens.cpu().numpy()
    return oracle.nsa_select_attention_backward(
        to_np(w.q), to_np(w.k), to_np(w.v), w.block_indices.cpu().numpy(), counts, w.block_size,
        to_np(do), cu_seqlens=cu, causal=causal, rows=rows)


def _messy(w, seed):
    """Indices with -1, out-of-range and future blocks and a duplicate per list."""
    rng = np.random.default_rng(seed)
    idx = w.block_indices.cpu().numpy().copy()
    B, T, Hkv, S = idx.shape
    nb = -(-T // w.block_size)
    noise = rng.integers(-2, nb + 2, size=idx.shape)
    pick = rng.random(idx.shape) < 0.25
    idx[pick] = noise[pick]
    idx[..., 1] = idx[..., 0]
    w.block_indices = torch.from_numpy(idx.astype(np.int32)).to(DEV)
    w.block_counts = torch.from_numpy(rng.integers(0, S + 2, size=(B, T, Hkv)).astype(np.int32)).to(DEV)
    return w


@pytest.mark.parametrize("Hq,Hkv", [(16, 1), (16, 2), (8, 1)])
def test_small_all_elements(sba, Hq, Hkv):
    w = workloads.nsa_prefill(device=DEV, B=2, T=640, Hq=Hq, Hkv=Hkv, D=128, seed=1000 + Hq + Hkv)
    do, dq, dk, dv = _run(sba, w, seed=1)
    rq, rk, rv = _oracle(w, do)
    assert_grad_close(to_np(dq), rq, "dq")
    assert_grad_close(to_np(dk), rk, "dk")
    assert_grad_close(to_np(dv), rv, "dv")


def test_group_windows_with_a_short_last_window(sba):
    """B=3, Hkv=2: six (batch row, KV head) groups, so the dK/dV items' windows of four
    groups end with a window of two; every element against the oracle."""
    w = workloads.nsa_prefill(device=DEV, B=3, T=384, Hq=16, Hkv=2, D=128, seed=1050)
    do, dq, dk, dv = _run(sba, w, seed=2)
    rq, rk, rv = _oracle(w, do)
    assert_grad_close(to_np(dq), rq, "dq")
    assert_grad_close(to_np(dk), rk, "dk")
    assert_grad_close(to_np(dv), rv, "dv")


@pytest.mark.parametrize("causal", [True, False])
def test_messy_indices_ragged_tail(sba, causal):
    """-1, out of range, future blocks, duplicates, counts beyond S; T not a multiple of
    the block or of the tokens per item."""
    w = _messy(workloads.nsa_prefill(device=DEV, B=1, T=1000, Hq=16, Hkv=2, D=128, seed=1100), 1101)
    do, dq, dk, dv = _run(sba, w, seed=2, causal=causal)
    rq, rk, rv = _oracle(w, do, causal=causal)
    assert_grad_close(to_np(dq), rq, "dq")
    assert_grad_close(to_np(dk), rk, "dk")
    assert_grad_close(to_np(dv), rv, "dv")


def test_varlen_small(sba):
    w = workloads.nsa_varlen(device=DEV, num_seqs=4, min_len=70, max_len=400, Hq=16, Hkv=2, seed=1200)
    do, dq, dk, dv = _run(sba, w, seed=3)
    rq, rk, rv = _oracle(w, do)
    assert_grad_close(to_np(dq), rq, "dq")
    assert_grad_close(to_np(dk), rk, "dk")
    assert_grad_close(to_np(dv), rv, "dv")


def _selectors(w, b, hkv, blk):
    """(b, t) rows whose (filtered) selection for KV head hkv contains key block blk of
    batch row b (fixed-length rows)."""
    idx = w.block_indices.cpu().numpy()[b, :, hkv]
    cnt = w.block_counts.cpu().numpy()[b, :, hkv]
    S = idx.shape[-1]
    t = np.arange(idx.shape[0])
    use = (np.arange(S)[None, :] < np.clip(cnt, 0, S)[:, None]) & (idx == blk)
    hit = use.any(axis=1) & (blk * w.block_size <= t)
    return [(b, int(x)) for x in t[hit]]


def test_prefill_full_size_sampled(sba):
    """B=2, T=8192, Hq=64, Hkv=4 (the benchmark launch): dq on sampled tokens; dk, dv
    exactly on three key blocks, each from all the tokens that selected it."""
    w = workloads.nsa_prefill(device=DEV)
    do, dq, dk, dv = _run(sba, w, seed=4)
    rng = np.random.default_rng(5)
    rows = [(int(b), int(t)) for b, t in zip(rng.integers(0, 2, 24), rng.integers(0, 8192, 24))]
    rows += [(0, 0), (1, 8191), (0, 64)]
    rq, _, _ = _oracle(w, do, rows=rows)
    idx = tuple(np.array(rows).T)
    assert_grad_close(to_np(dq)[idx], rq[idx], "dq sampled")
    for b, hkv, blk in ((0, 1, 120), (1, 3, 127), (1, 0, 90)):
        sel = _selectors(w, b, hkv, blk)
        assert sel, "block chosen by nobody"
        _, rk, rv = _oracle(w, do, rows=sel)
        ks = slice(blk * 64, blk * 64 + 64)
        assert_grad_close(to_np(dk)[b, ks, hkv], rk[b, ks, hkv], f"dk block {blk}")
        assert_grad_close(to_np(dv)[b, ks, hkv], rv[b, ks, hkv], f"dv block {blk}")


def test_unselected_keys_get_zero(sba):
    """Keys of blocks nobody selected (every token selects only its own block) get
    zero dk / dv; dq is the single-block softmax gradient."""
    w = workloads.nsa_prefill(device=DEV, B=1, T=512, Hq=16, Hkv=1, D=128, seed=1300)
    idx = np.full(w.block_indices.shape, -1, np.int32)
    idx[0, :, 0, 0] = np.arange(512) // 64
    idx[0, 300:, 0, 0] = 3  # tokens 300.. select block 3 only: blocks 4..7 unselected
    w.block_indices = torch.from_numpy(idx).to(DEV)
    do, dq, dk, dv = _run(sba, w, seed=6)
    assert torch.count_nonzero(dk[0, 320:, 0]).item() == 0
    assert torch.count_nonzero(dv[0, 320:, 0]).item() == 0
    rq, rk, rv = _oracle(w, do)
    assert_grad_close(to_np(dq), rq, "dq")
    assert_grad_close(to_np(dk), rk, "dk")
    assert_grad_close(to_np(dv), rv, "dv")
