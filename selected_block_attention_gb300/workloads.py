"""Seeded synthetic workloads (inputs only; none of the method's arithmetic).

These generators build the inputs of the five workload shapes the library is
measured and tested on.  They are shared by the tests, the benchmark and the
parity checks: the same materialised tensors go to the CUDA path and, copied to
the host, to the fp64 checker.  Structure (selection pattern, document lengths,
ragged ends) is drawn on the host with numpy's PCG64; dense float tensors are
drawn with a seeded ``torch.Generator`` on the requested device, so that the
8.6 GB decode cache need not pass through host memory.

Recipes (seed = ``0x5BA00000 + workload id`` unless given):

* ``nsa_tiny``     B=1 T=256 Hq=4 Hkv=1 D=64, fp32 N(0,1), block 64, causal;
                   tokens 0..63 select {own block}, later tokens {own block,
                   one uniform earlier block}; S=2.
* ``nsa_prefill``  B=2 T=8192 Hq=64 Hkv=4 D=128, bf16 N(0,1), block 64,
                   causal; per (b, t, kv head) count ~ U{1..16} clipped to the
                   blocks available, own block + distinct uniform earlier
                   blocks, shuffled, padded to S=16 with -1; counts array.
* ``nsa_varlen``   8 sequences, lengths U[1024, 16384], packed (B=1) with int32
                   ``cu_seqlens``; Hq=32 Hkv=2 D=128 bf16, block 64; scalar
                   count 16, per token min(16, j+1) entries valid and -1 after.
* ``mask``         B=4 T=16384, positions arange, documents with geometric
                   lengths (mean 2048) covering T-300 tokens, last 300 tokens
                   padding (segment -1); causal, window (1024, 0), block 128.
* ``blocksparse``  the ``mask`` workload plus Hq=32 Hkv=8 D=128 bf16 N(0,1).
* ``decode``       B=64 Hq=32 Hkv=8 D=128 S=32768 bf16 N(0,1); start 0, end
                   ~ U{1..32768}; window (4096, 0); cap 50; 4 sinks with
                   per-head biases N(0, 0.1).

Every generator takes size overrides so the tests can run the same recipe at
small sizes.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

SEED_BASE = 0x5BA00000


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0xFFFFFFFFFFFF)
    return g


def randn(shape, dtype, device, seed, std=1.0):
    """N(0, std^2) tensor of ``dtype`` drawn in fp32 on ``device``."""
    g = _gen(device, seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def select_blocks(rng, own_block, count, S):
    """Own block plus ``count - 1`` distinct uniform earlier blocks, shuffled,
    padded with -1 to length S.  Vectorised over the leading axis."""
    own_block = np.asarray(own_block, dtype=np.int64)
    count = np.asarray(count, dtype=np.int64)
    n = own_block.shape[0]
    out = np.full((n, S), -1, dtype=np.int32)
    chunk = 8192
    for c0 in range(0, n, chunk):
        own_c = own_block[c0:c0 + chunk]
        width = max(int(own_c.max()) if own_c.size else 0, 1)
        keys = rng.random((own_c.shape[0], width))
        keys[np.arange(width)[None, :] >= own_c[:, None]] = np.inf  # only blocks < own
        order = np.argsort(keys, axis=1, kind="stable")  # uniform random distinct picks
        for r in range(own_c.shape[0]):
            c = int(count[c0 + r])
            picks = np.empty(c, dtype=np.int64)
            picks[0] = own_c[r]
            if c > 1:
                picks[1:] = order[r, : c - 1]
            rng.shuffle(picks)
            out[c0 + r, :c] = picks
    return out


@dataclass
class NSAWorkload:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    block_indices: torch.Tensor            # int32 [B, T, Hkv, S]
    block_counts: object                   # int32 tensor [B, T, Hkv] or int
    block_size: int
    cu_seqlens: torch.Tensor | None = None  # int32 [N + 1]
    causal: bool = True
    softmax_scale: float | None = None
    name: str = ""
    meta: dict = field(default_factory=dict)


def nsa_tiny(device="cpu", seed=SEED_BASE + 1, T=256, Hq=4, Hkv=1, D=64,
             block_size=64, dtype=torch.float32):
    rng = np.random.Generator(np.random.PCG64(seed))
    B = 1
    t = np.arange(T)
    own = t // block_size
    count = np.where(own == 0, 1, 2)
    idx = np.full((B, T, Hkv, 2), -1, dtype=np.int32)
    for h in range(Hkv):
        idx[0, :, h, :] = select_blocks(rng, own, count, 2)
    counts = np.broadcast_to(count[None, :, None], (B, T, Hkv)).astype(np.int32).copy()
    return NSAWorkload(
        q=randn((B, T, Hq, D), dtype, device, seed + 11),
        k=randn((B, T, Hkv, D), dtype, device, seed + 12),
        v=randn((B, T, Hkv, D), dtype, device, seed + 13),
        block_indices=torch.from_numpy(idx).to(device),
        block_counts=torch.from_numpy(counts).to(device),
        block_size=block_size, name=f"nsa_tiny B=1 T={T} Hq={Hq} Hkv={Hkv} D={D} bs={block_size} fp32 causal")


def nsa_prefill(device="cpu", seed=SEED_BASE + 2, B=2, T=8192, Hq=64, Hkv=4, D=128,
                block_size=64, S=16, max_count=16, dtype=torch.bfloat16):
    rng = np.random.Generator(np.random.PCG64(seed))
    t = np.arange(T)
    own = np.broadcast_to((t // block_size)[None, :, None], (B, T, Hkv)).reshape(-1)
    count = rng.integers(1, max_count + 1, size=own.shape[0])
    count = np.minimum(count, own + 1)
    idx = select_blocks(rng, own, count, S).reshape(B, T, Hkv, S)
    counts = count.reshape(B, T, Hkv).astype(np.int32)
    return NSAWorkload(
        q=randn((B, T, Hq, D), dtype, device, seed + 11),
        k=randn((B, T, Hkv, D), dtype, device, seed + 12),
        v=randn((B, T, Hkv, D), dtype, device, seed + 13),
        block_indices=torch.from_numpy(idx).to(device),
        block_counts=torch.from_numpy(counts).to(device),
        block_size=block_size,
        name=f"nsa_prefill B={B} T={T} Hq={Hq} Hkv={Hkv} D={D} bs={block_size} bf16 causal")


def nsa_varlen(device="cpu", seed=SEED_BASE + 3, num_seqs=8, min_len=1024, max_len=16384,
               Hq=32, Hkv=2, D=128, block_size=64, S=16, count=16, dtype=torch.bfloat16,
               lengths=None):
    rng = np.random.Generator(np.random.PCG64(seed))
    if lengths is None:
        lengths = rng.integers(min_len, max_len + 1, size=num_seqs)
    lengths = np.asarray(lengths, dtype=np.int64)
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(lengths)
    T = int(cu[-1])
    own = np.concatenate([np.arange(L) // block_size for L in lengths])
    own = np.broadcast_to(own[:, None], (T, Hkv)).reshape(-1)
    cnt = np.minimum(count, own + 1)
    idx = select_blocks(rng, own, cnt, S).reshape(1, T, Hkv, S)
    return NSAWorkload(
        q=randn((1, T, Hq, D), dtype, device, seed + 11),
        k=randn((1, T, Hkv, D), dtype, device, seed + 12),
        v=randn((1, T, Hkv, D), dtype, device, seed + 13),
        block_indices=torch.from_numpy(idx).to(device),
        block_counts=int(count), block_size=block_size,
        cu_seqlens=torch.from_numpy(cu.astype(np.int32)).to(device),
        name=f"nsa_varlen N={len(lengths)} T={T} Hq={Hq} Hkv={Hkv} D={D} bs={block_size} bf16 causal",
        meta={"lengths": [int(x) for x in lengths]})


@dataclass
class MaskWorkload:
    q_positions: torch.Tensor     # int32 [B, T]
    q_segment_ids: torch.Tensor
    kv_positions: torch.Tensor
    kv_segment_ids: torch.Tensor
    q_blocksize: int
    kv_blocksize: int
    causal: bool
    window_left: int
    window_right: int
    padding_segment_id: int
    name: str = ""


def packed_segments(rng, B, T, mean_len, pad_tail, pad_id=-1):
    """Segment ids 0, 1, 2, ... per document; geometric document lengths on
    {1, 2, ...} with the given mean (inverse CDF of uniforms); the last
    ``pad_tail`` tokens of each row carry ``pad_id``."""
    p = 1.0 / mean_len
    seg = np.full((B, T), pad_id, dtype=np.int64)
    real = T - pad_tail
    for b in range(B):
        pos, sid = 0, 0
        while pos < real:
            u = rng.random()
            length = int(np.floor(np.log1p(-u) / np.log1p(-p))) + 1
            stop = min(pos + length, real)
            seg[b, pos:stop] = sid
            pos, sid = stop, sid + 1
    return seg


def mask(device="cpu", seed=SEED_BASE + 4, B=4, T=16384, mean_doc=2048, pad_tail=300,
         block=128, window=(1024, 0), causal=True, pad_id=-1):
    rng = np.random.Generator(np.random.PCG64(seed))
    seg = packed_segments(rng, B, T, mean_doc, pad_tail, pad_id)
    pos = np.broadcast_to(np.arange(T)[None, :], (B, T))
    to = lambda a: torch.from_numpy(np.ascontiguousarray(a).astype(np.int32)).to(device)
    return MaskWorkload(to(pos), to(seg), to(pos), to(seg), block, block, causal,
                        window[0], window[1], pad_id,
                        name=f"sparse_mask B={B} T={T} block={block} window={window} causal")


@dataclass
class BlockSparseWorkload:
    mask: MaskWorkload
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    name: str = ""


def blocksparse(device="cpu", seed=SEED_BASE + 4, B=4, T=16384, Hq=32, Hkv=8, D=128,
                mean_doc=2048, pad_tail=300, block=128, window=(1024, 0),
                dtype=torch.bfloat16):
    m = mask(device, seed, B, T, mean_doc, pad_tail, block, window)
    return BlockSparseWorkload(
        m, randn((B, T, Hq, D), dtype, device, seed + 11),
        randn((B, T, Hkv, D), dtype, device, seed + 12),
        randn((B, T, Hkv, D), dtype, device, seed + 13),
        name=f"blocksparse_attn B={B} T={T} Hq={Hq} Hkv={Hkv} D={D} block={block} window={window} bf16")


@dataclass
class DecodeWorkload:
    q: torch.Tensor               # [B, Hq, D]
    k: torch.Tensor               # [B, S, Hkv, D]
    v: torch.Tensor
    sequence_start: torch.Tensor  # int32 [B]
    sequence_end: torch.Tensor    # int32 [B]
    window_left: int
    window_right: int
    logits_soft_cap: float
    sink_bias: torch.Tensor | None  # fp32 [Hq, num_sinks]
    name: str = ""


def decode(device="cpu", seed=SEED_BASE + 5, B=64, Hq=32, Hkv=8, D=128, S=32768,
           window=(4096, 0), cap=50.0, num_sinks=4, sink_std=0.1, dtype=torch.bfloat16,
           ends=None):
    rng = np.random.Generator(np.random.PCG64(seed))
    if ends is None:
        ends = rng.integers(1, S + 1, size=B)
    ends = np.asarray(ends, dtype=np.int32)
    starts = np.zeros(B, dtype=np.int32)
    sink = randn((Hq, num_sinks), torch.float32, device, seed + 14, std=sink_std) if num_sinks else None
    return DecodeWorkload(
        q=randn((B, Hq, D), dtype, device, seed + 11),
        k=randn((B, S, Hkv, D), dtype, device, seed + 12),
        v=randn((B, S, Hkv, D), dtype, device, seed + 13),
        sequence_start=torch.from_numpy(starts).to(device),
        sequence_end=torch.from_numpy(ends).to(device),
        window_left=window[0], window_right=window[1], logits_soft_cap=cap,
        sink_bias=sink,
        name=f"ragged_decode B={B} Hq={Hq} Hkv={Hkv} D={D} S={S} window={window} cap={cap} sinks={num_sinks} bf16")


@dataclass
class RaggedAttentionWorkload:
    q: torch.Tensor               # [B, Q, Hq, D]
    k: torch.Tensor               # [B, S, Hkv, D]
    v: torch.Tensor
    sequence_start: torch.Tensor  # int32 [B]
    sequence_end: torch.Tensor    # int32 [B]
    window_left: int
    window_right: int
    logits_soft_cap: float
    sink_bias: torch.Tensor | None  # fp32 [Hq, num_sinks]
    name: str = ""


def ragged_attention(device="cpu", seed=SEED_BASE + 6, B=64, Q=4, Hq=32, Hkv=8, D=128, S=32768,
                     window=(4096, 0), cap=50.0, num_sinks=4, sink_std=0.1,
                     dtype=torch.bfloat16, ends=None, starts=None):
    """Q query tokens per row against a KV cache (multi-token decode / chunked prefill).
    Default: 64 rows verifying 4 tokens each; ends ~ U{Q..S}, so every query has a
    position inside the cache."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if ends is None:
        ends = rng.integers(min(Q, S), S + 1, size=B)
    ends = np.asarray(ends, dtype=np.int32)
    starts = np.zeros(B, dtype=np.int32) if starts is None else np.asarray(starts, dtype=np.int32)
    sink = randn((Hq, num_sinks), torch.float32, device, seed + 14, std=sink_std) if num_sinks else None
    return RaggedAttentionWorkload(
        q=randn((B, Q, Hq, D), dtype, device, seed + 11),
        k=randn((B, S, Hkv, D), dtype, device, seed + 12),
        v=randn((B, S, Hkv, D), dtype, device, seed + 13),
        sequence_start=torch.from_numpy(starts).to(device),
        sequence_end=torch.from_numpy(ends).to(device),
        window_left=window[0], window_right=window[1], logits_soft_cap=cap,
        sink_bias=sink,
        name=f"ragged_attention B={B} Q={Q} Hq={Hq} Hkv={Hkv} D={D} S={S} window={window} "
             f"cap={cap} sinks={num_sinks} bf16")
