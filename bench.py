"""Benchmark: selected-block sparse attention on GB300.

Headline (``value``): NSA selection forward TFLOP/s on the B=2, T=8192, Hq=64,
Hkv=4, D=128, block 64 causal prefill (bf16), inputs resident in HBM, L2 flushed
between steps (a 256 MB buffer is rewritten and another 256 MB read before each
timed step, outside the step's events, so the step starts with a clean L2).  FLOPs are algorithmic: 4 * D * (number of admissible keys) per
(token, query head), i.e. the work the selection defines, not padded tiles.

The same JSON line carries ``roofline`` (dominant kernel vs the measured peak),
``cpu_baseline`` (the fp64 oracle on a bounded sample, host cores), ``e2e`` (same
metric with host buffers, copies inside the timed region), ``clocks`` (nvidia-smi
sampled during the timed region) and ``rows``: the other workloads of the path
(varlen NSA, SparseMask bounds, block-sparse attention, ragged decode, ragged
multi-query attention), each timed the same way.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --case {nsa_prefill,nsa_varlen,nsa_bwd,blocksparse,mask_sweep,decode,ragged_q4,ragged_chunk512}
                  [--repeat R]
                  [--decode-batch B]      # profiling: launches only, no JSON line

``--impl reference`` times the fp64 CPU oracle on the same workload (bounded
sample per step, host cores) and prints the same line with ``"impl": "reference"``.
Under torchrun (N > 1) every rank runs its own replica (weak scaling, no
collective on the data path); rank 0 prints.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selected_block_attention_gb300 import workloads  # noqa: E402

METRIC = "selected-block sparse attn fwd TFLOP/s & HBM GB/s vs roofline; decode tok/s"
L2_FLUSH_BYTES = 256 << 20
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- helpers
def log(msg):
    print(f"[bench {time.strftime('%H:%M:%S')}] {msg}", file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in PEAKS_FALLBACK}, "measured"
    except Exception:
        return dict(PEAKS_FALLBACK), "fallback"


def nsa_work(w):
    """(F_alg FLOPs, HBM bytes, gathered K/V bytes, token groups) from the inputs."""
    idx = w.block_indices.cpu().numpy().astype(np.int64)
    B, T, Hkv, S = idx.shape
    Hq, D = w.q.shape[2], w.q.shape[3]
    G = Hq // Hkv
    bs = w.block_size
    if isinstance(w.block_counts, int):
        counts = np.full((B, T, Hkv), w.block_counts, dtype=np.int64)
    else:
        counts = w.block_counts.cpu().numpy().astype(np.int64)
    if w.cu_seqlens is not None:
        cu = w.cu_seqlens.cpu().numpy().astype(np.int64)
        seq = np.searchsorted(cu, np.arange(T), side="right") - 1
        t_rel = np.arange(T) - cu[seq]
        L = (cu[seq + 1] - cu[seq])
    else:
        t_rel = np.arange(T)
        L = np.full(T, T)
    t_rel = np.broadcast_to(t_rel[None, :, None, None], idx.shape)
    Lb = np.broadcast_to(L[None, :, None, None], idx.shape)
    slot = np.arange(S)[None, None, None, :]
    valid = (slot < np.minimum(counts, S)[..., None]) & (idx >= 0) & (idx * bs < Lb)
    if w.causal:
        valid &= idx * bs <= t_rel
    hi = np.minimum(idx * bs + bs, Lb)
    if w.causal:
        hi = np.minimum(hi, t_rel + 1)
    keys = np.where(valid, hi - idx * bs, 0).sum()
    n_blocks = valid.sum()
    elt = w.q.element_size()
    flops = 4.0 * D * G * float(keys)
    hbm = (w.q.numel() * 2 + w.k.numel() + w.v.numel()) * elt + B * T * Hq * 4 + idx.size * 4 + \
        (0 if isinstance(w.block_counts, int) else counts.size * 4)
    gather = float(n_blocks) * bs * D * 2 * elt
    return flops, float(hbm), gather, int(B * T * Hkv)


def nsa_selected_pairs(w, rows=128):
    """Per (batch row, KV head, key block): the number of tokens whose filtered selection
    holds it; "chunks" = the dK/dV kernel's chunks of rows // G tokens over all of them."""
    idx = w.block_indices.cpu().numpy().astype(np.int64)
    B, T, Hkv, S = idx.shape
    G = w.q.shape[2] // Hkv
    bs = w.block_size
    counts = (np.full((B, T, Hkv), w.block_counts, dtype=np.int64) if isinstance(w.block_counts, int)
              else w.block_counts.cpu().numpy().astype(np.int64))
    t = np.arange(T)[None, :, None, None]
    valid = (np.arange(S)[None, None, None, :] < np.minimum(counts, S)[..., None]) & (idx >= 0) & \
        (idx * bs < T) & (idx * bs <= t)
    nb = -(-T // bs)
    slot = (np.arange(B)[:, None, None, None] * Hkv + np.arange(Hkv)[None, None, :, None]) * nb + idx
    # a duplicate entry in one token's list counts once
    tok = np.broadcast_to(np.arange(B * T).reshape(B, T, 1, 1), idx.shape)
    pairs = np.unique(slot[valid] * (B * T) + tok[valid])
    per_slot = np.bincount(pairs // (B * T))
    nt = rows // G
    return {"pairs": int(pairs.size), "chunks": int((-(-per_slot // nt)).sum())}


def union_tiles(w, rows=128, tile_keys=64):
    """Tiles the union walk executes: per (item, KV head), the number of distinct selected
    blocks (each block of <= 64 keys is one 64-key tile).  An item holds NT = rows // G
    tokens: for G >= 8 the tokens of each window of 8 * NT tokens ranked by selection
    count (clipped to [0, S], ties by position), NT consecutive ranks per item, as the
    kernel forms them; otherwise NT consecutive tokens."""
    idx = w.block_indices.cpu().numpy().astype(np.int64)
    B, T, Hkv, S = idx.shape
    G = w.q.shape[2] // Hkv
    NT = min(16, rows // G)
    bs = w.block_size
    counts = (np.full((B, T, Hkv), w.block_counts, dtype=np.int64) if isinstance(w.block_counts, int)
              else w.block_counts.cpu().numpy().astype(np.int64))
    if w.cu_seqlens is not None:
        cu = w.cu_seqlens.cpu().numpy().astype(np.int64)
        seq = np.searchsorted(cu, np.arange(T), side="right") - 1
        start, L = cu[seq], cu[seq + 1] - cu[seq]
    else:
        start, L = np.zeros(T, dtype=np.int64), np.full(T, T)
    t_rel = (np.arange(T) - start)[None, :, None, None]
    valid = (np.arange(S)[None, None, None, :] < np.minimum(counts, S)[..., None]) & (idx >= 0) & \
        (idx * bs < L[None, :, None, None])
    if w.causal:
        valid &= idx * bs <= t_rel
    tok = (np.arange(B)[:, None] * T + np.arange(T)[None, :])[:, :, None, None]
    first_row = np.broadcast_to(tok - t_rel + idx * bs, idx.shape)  # absolute first key row
    if G >= 8:
        wn = 8 * NT
        n_tok = B * T
        nw = -(-n_tok // wn)
        cnt = np.full((nw * wn, Hkv), 0xFFFF, dtype=np.int64)
        cnt[:n_tok] = np.clip(counts.reshape(n_tok, Hkv), 0, S)
        li = np.arange(nw * wn) % wn
        key = (cnt << 8) | li[:, None]
        order = np.argsort(key.reshape(nw, wn, Hkv), axis=1, kind="stable")
        rank = np.empty_like(order)
        np.put_along_axis(rank, order, np.arange(wn)[None, :, None], axis=1)
        grp = (np.arange(nw)[:, None, None] * 8 + rank // NT).reshape(nw * wn, Hkv)[:n_tok]
        group = np.broadcast_to(grp.reshape(B, T, Hkv)[..., None], idx.shape)
    else:
        group = np.broadcast_to(tok // NT, idx.shape)
    head = np.broadcast_to(np.arange(Hkv)[None, None, :, None], idx.shape)
    item = group[valid] * Hkv + head[valid]
    pairs = np.unique(item * (B * T + bs) + first_row[valid])  # distinct (item, block)
    per_item = np.bincount(pairs // (B * T + bs))
    if bs >= tile_keys:
        return int(per_item.sum()) * (bs // tile_keys)
    return int((-(-per_item * bs // tile_keys)).sum())


def profile_traffic(summary_name, source_rel):
    """DRAM bytes per launch from a committed ncu summary, or None when the kernel
    source changed since the capture (the summary records the source's SHA-256)."""
    import hashlib
    try:
        text = open(os.path.join(ROOT, "profiles", summary_name)).read()
        src = open(os.path.join(ROOT, source_rel), "rb").read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip().strip("-* `")] = v.strip().strip("`")
    if fields.get("source_sha256") != hashlib.sha256(src).hexdigest():
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def world_max(x, device):
    """Maximum of a per-rank float over all ranks (the rank's own value when alone)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    if torch.distributed.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_value(units_per_rank, world, ms_max, scale=1e12):
    """Whole-job throughput: all ranks' units over the slowest rank's step time."""
    return units_per_rank * world / (ms_max * 1e-3) / scale


class ClockSampler:
    """nvidia-smi clocks / throttle reasons, sampled every 50 ms in a thread."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        sel = [p for t, p in self.samples if t0 <= t <= t1]
        if not sel:  # region shorter than one sample period: nearest samples
            sel = [p for t, p in sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in sel if num(p[1]) is not None]
        mx = [num(p[2]) for p in sel if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in sel for n, v in zip(names, p[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(sel)}


HOLD_CYCLES = 400_000  # ~0.2 ms of GPU spin ahead of each timed step


class L2Flush:
    """Between timed steps: rewrite a buffer larger than L2 (evicts every input line),
    then read a second one, so the rewritten lines are written back to HBM before the
    step starts: the step begins with a clean L2 that holds none of its inputs (no
    write-back of someone else's dirty lines inside the timed region)."""

    def __init__(self, dev):
        self.w = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.zeros((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.add_(1)
        torch.sum(self.r, dim=0, out=self.sink)


def timed_steps(fn, steps, warmup, flush, stream):
    """Per-step device time (ms) with CUDA events on ``stream``; the L2 flush runs
    before every step, outside its events.  A short GPU spin ahead of the flush keeps
    the device busy while the host enqueues the step, so the events bracket the step's
    own GPU work and not the host's argument marshalling (host cost is what the
    end-to-end figure measures)."""
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        torch.cuda._sleep(HOLD_CYCLES)
        flush()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def decode_work(w):
    ends = w.sequence_end.cpu().numpy().astype(np.int64)
    starts = w.sequence_start.cpu().numpy().astype(np.int64)
    num_sinks = 0 if w.sink_bias is None else w.sink_bias.shape[-1]
    nkeys = 0
    for s, e in zip(starts, ends):
        if e <= s:
            continue
        lo = max(s, e - 1 - w.window_left) if w.window_left >= 0 else s
        nkeys += (e - lo) + max(0, min(num_sinks, lo, e) - s)
    B, Hq, D = w.q.shape
    Hkv = w.k.shape[2]
    kv_bytes = float(nkeys) * Hkv * D * 2 * 2
    flops = 4.0 * D * (Hq // Hkv) * Hkv * nkeys
    return kv_bytes + w.q.numel() * 2 * 2 + B * Hq * 4, flops


def ragged_attention_work(w):
    """Algorithmic bytes and FLOPs of one multi-query call: per (row, query) the keys in
    its window [p - left, p + right] inside [start, end) plus in-range sinks outside it;
    HBM bytes = K/V of the union of a row's query windows (read once) + Q + O + LSE."""
    ends = w.sequence_end.cpu().numpy().astype(np.int64)
    starts = np.maximum(w.sequence_start.cpu().numpy().astype(np.int64), 0)
    B, Q, Hq, D = w.q.shape
    Hkv = w.k.shape[2]
    ns = 0 if w.sink_bias is None else w.sink_bias.shape[-1]
    wl, wr = w.window_left, w.window_right
    pair_keys, union_keys = 0, 0

    def window(lo_pos, hi_pos, s, e):
        lo = np.maximum(s, lo_pos - wl) if wl >= 0 else s
        hi = np.minimum(e, hi_pos + wr + 1) if wr >= 0 else e
        hi = np.maximum(hi, lo)
        sinks_out = max(0, min(ns, e, lo) - s) + max(0, min(ns, e) - max(hi, s))
        return hi - lo, sinks_out

    for s, e in zip(starts, ends):
        if e <= s:
            continue
        for i in range(Q):
            n, extra = window(e - Q + i, e - Q + i, s, e)
            pair_keys += int(n) + extra
        n, extra = window(e - Q, e - 1, s, e)
        union_keys += int(n) + extra
    kv_bytes = float(union_keys) * Hkv * D * 2 * 2
    flops = 4.0 * D * Hq * pair_keys
    return kv_bytes + 2 * w.q.numel() * 2 + B * Q * Hq * 4, flops


def blocksparse_flops(w):
    m = w.mask
    pos = m.q_positions.cpu().numpy().astype(np.int64)
    seg = m.q_segment_ids.cpu().numpy().astype(np.int64)
    B, T = pos.shape
    Hq, D = w.q.shape[2], w.q.shape[3]
    total = 0
    for b in range(B):
        s = seg[b]
        start = np.zeros(T, dtype=np.int64)
        change = np.r_[True, s[1:] != s[:-1]]
        start_idx = np.maximum.accumulate(np.where(change, np.arange(T), 0))
        n = pos[b] - pos[b][start_idx] + 1
        if m.window_left >= 0:
            n = np.minimum(n, m.window_left + 1)
        total += np.where(s != m.padding_segment_id, n, 0).sum()
    return 4.0 * D * Hq * float(total)


# ----------------------------------------------------------------------------- arms
def l2_read_gbs(sba, dev, stream, mb=48, reps=200):
    """L2-to-SM read bandwidth from the library's probe: a 48 MB buffer (under half of
    the 129 MB L2) read `reps` times (about 10 GB in all, so launch overhead is
    negligible) with 16-byte L1-bypassing loads on every SM, after
    one warm-up pass; best of 3 timings."""
    buf = torch.ones(mb * (1 << 20) // 4, dtype=torch.int32, device=dev)
    sink = torch.zeros(1, dtype=torch.int32, device=dev)
    sba.l2_read_probe(buf, 1, sink)
    best = None
    for _ in range(3):
        s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        sba.l2_read_probe(buf, reps, sink)
        e0.record(stream)
        e0.synchronize()
        ms = s0.elapsed_time(e0)
        best = ms if best is None else min(best, ms)
    sba.check_error(dev)
    return reps * buf.numel() * 4 / (best * 1e-3) / 1e9


def run_cuda(args, rank, world, local_rank):
    import selected_block_attention_gb300 as sba
    from selected_block_attention_gb300 import _build

    _build.build()
    sba.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()
    flush = L2Flush(dev)

    w = workloads.nsa_prefill(device=dev)
    flops, hbm_bytes, gather_bytes, groups = nsa_work(w)
    log(f"prefill inputs ready: {flops / 1e12:.4f} TFLOP/step")
    out = torch.empty_like(w.q)
    lse = torch.empty(w.q.shape[:3], dtype=torch.float32, device=dev)

    def step():
        sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts, w.block_size,
                           causal=True, out=out, lse=lse)

    sampler = ClockSampler(local_rank if world > 1 else int(os.environ.get("SBA_GPU_INDEX", "0")))
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    times = timed_steps(step, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    sba.check_error(dev)
    ms = sum(times) / len(times)
    ms_max = world_max(ms, dev)
    clocks = sampler.summary(t0, t1)
    sampler.stop()
    log(f"timed steps done: {ms:.4f} ms/step")
    value = aggregate_value(flops, world, ms_max)
    n_tiles = union_tiles(w)
    exec_flops = 4.0 * 128 * 64 * w.q.shape[3] * n_tiles  # QK + PV of every union tile

    # e2e through the C ABI's host-buffer entry point (pinned host tensors): the library
    # copies every input to the device and the outputs back inside the timed region
    host = {n: getattr(w, n).cpu().pin_memory() for n in ("q", "k", "v", "block_indices", "block_counts")}
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    B, T, Hq, D = w.q.shape
    ws = torch.empty(sba.nsa_select_host_workspace_size(B, T, Hq, w.k.shape[2], D,
                                                        w.block_indices.shape[-1]),
                     dtype=torch.uint8, device=dev)

    def e2e_step():
        sba.nsa_select_fwd_host(host["q"], host["k"], host["v"], host["block_indices"],
                                host["block_counts"], w.block_size, causal=True, out=out_h,
                                lse=lse_h, workspace=ws, device=dev)

    e2e_steps = max(3, min(args.steps, 10))
    e2e_times = timed_steps(e2e_step, e2e_steps, 3, flush, stream)
    e2e_ms = sum(e2e_times) / len(e2e_times)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()

    log(f"e2e done: {e2e_ms:.4f} ms/step")
    bw_l2 = l2_read_gbs(sba, dev, stream)
    log(f"L2 read bandwidth {bw_l2:.0f} GB/s")
    union_bytes = float(n_tiles) * 64 * w.q.shape[3] * 2 * 2  # K and V of every union tile
    terms = {"tensor": flops / (peaks["bf16_tflops"] * 1e12) * 1e6,
             "hbm": hbm_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6,
             "l2_gather": gather_bytes / (bw_l2 * 1e9) * 1e6}
    t_roof = max(terms.values())
    exec_floor_us = max(exec_flops / (peaks["bf16_tflops"] * 1e12),
                        union_bytes / (bw_l2 * 1e9)) * 1e6
    rows = {} if args.no_rows else measure_rows(sba, dev, stream, flush, peaks, args, bw_l2)

    result = {
        "metric": METRIC,
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": "nsa_select_prefill B=2 T=8192 Hq=64 Hkv=4 D=128 block_size=64 causal, "
                        "counts U{1..16} clipped, own block + distinct uniform earlier blocks",
            "tokens": w.q.shape[0] * w.q.shape[1], "token_groups": groups,
            "flop_per_step": flops, "l2": "flushed before every timed step: a 256 MB buffer rewritten, then another 256 MB read (clean L2, no input resident)",
            "parallelism": f"replicas x{world}"},
        "roofline": {
            "bound": "tensor",
            "achieved": round(flops / (ms * 1e-3) / 1e12, 3),
            "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s",
            "frac": round(flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "traffic": profile_traffic("nsa_union_kernel_prefill.md",
                                       "selected_block_attention_gb300/csrc/nsa_select.cu"),
            "traffic_source": "stored: dram__bytes_read.sum + dram__bytes_write.sum of one ncu "
                              "capture (profiles/nsa_union_kernel_prefill.md), reported only while "
                              "the kernel source still has the SHA-256 recorded there",
            "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed alone)",
            "kernel": "nsa_union_kernel<128,64>",
            "union_tiles": int(n_tiles),
            "executed_mma_tflops": round(exec_flops / (ms * 1e-3) / 1e12, 1),
            "executed_mma_frac": round(exec_flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            # the union walk's own floor: its executed MMA work at the tensor peak or its
            # gathered K/V bytes at the measured L2 read bandwidth, whichever is larger
            "exec_floor_us": round(exec_floor_us, 2),
            "frac_exec_floor": round(exec_floor_us / (ms * 1e3), 4),
            # t_roof = max(F_alg / P_tensor, B_hbm / BW_hbm, B_gather / BW_l2) with the
            # per-token selection gather and the probe's L2 read bandwidth: the floor of a
            # kernel that gathers each token's blocks separately, which the union walk does
            # not (frac is the tensor-peak fraction; frac_exec_floor the union walk's own)
            "terms_us": {k: round(v, 2) for k, v in terms.items()},
            "l2_read_gbs": round(bw_l2, 1),
            "t_roof_us": round(t_roof, 2),
            "frac_t_roof": round(t_roof / (ms * 1e3), 4),
            "union_gather_bytes": union_bytes,
            "union_gather_us_at_l2": round(union_bytes / (bw_l2 * 1e9) * 1e6, 2),
            "hbm_achieved_gbs": round(hbm_bytes / (ms * 1e-3) / 1e9, 1),
            "hbm_frac": round(hbm_bytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "gathered_kv_bytes": gather_bytes,
            "gather_achieved_gbs": round(gather_bytes / (ms * 1e-3) / 1e9, 1),
        },
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "path": "sba_nsa_select_fwd_host: pinned host buffers, copies of (batch row, token range) "
                        "chunks overlapped with the computation (K/V prefix copied once)"},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "rows": rows,
    }
    return result


def t_roof_terms(flops, hbm_bytes, peaks, gather_bytes=None, bw_l2=None):
    """Roofline terms in us (tensor, HBM, and the per-token gather at the measured L2
    read bandwidth when given) and their maximum."""
    terms = {"tensor": flops / (peaks["bf16_tflops"] * 1e12) * 1e6,
             "hbm": hbm_bytes / (peaks["hbm_gbs"] * 1e9) * 1e6}
    if gather_bytes is not None:
        terms["l2_gather"] = gather_bytes / (bw_l2 * 1e9) * 1e6
    return {k: round(v, 2) for k, v in terms.items()}, max(terms.values())


def measure_rows(sba, dev, stream, flush, peaks, args, bw_l2):
    rows = {}
    steps, warm = max(3, min(args.steps, 20)), 3

    # the fp32 correctness workload (B=1 T=256 Hq=4 Hkv=1 D=64, CUDA cores): latency only
    w = workloads.nsa_tiny(device=dev)
    flops, hbm, _g, _n = nsa_work(w)
    t = timed_steps(lambda: sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts,
                                               w.block_size, causal=True),
                    steps, warm, flush, stream)
    ms = sum(t) / len(t)
    log(f"nsa tiny {ms * 1e3:.2f} us")
    rows["nsa_select_tiny_fp32"] = {
        "workload": w.name, "us": round(ms * 1e3, 2), "GFLOP/s": round(flops / ms / 1e6, 2),
        "hbm_bytes": int(hbm), "bound": "launch latency (0.7 MB, fp32 on CUDA cores)"}
    del w

    # NSA selection backward on the prefill workload (dq, dk, dv from the forward's out / LSE)
    w = workloads.nsa_prefill(device=dev)
    flops, hbm, _g, _n = nsa_work(w)
    out, lse = sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts, w.block_size,
                                  causal=True)
    gen = torch.Generator(device=dev).manual_seed(7)
    do = torch.randn(w.q.shape, generator=gen, device=dev, dtype=torch.float32).to(w.q.dtype)
    B, T, Hq, D = w.q.shape
    Hkv = w.k.shape[2]
    bws = torch.empty(sba.nsa_select_bwd_workspace_size(B, T, Hq, Hkv, w.block_indices.shape[-1]),
                      dtype=torch.uint8, device=dev)
    dq, dk, dv = torch.empty_like(w.q), torch.empty_like(w.k), torch.empty_like(w.v)
    t = timed_steps(lambda: sba.nsa_select_bwd(w.q, w.k, w.v, out, lse, do, w.block_indices,
                                               w.block_counts, w.block_size, causal=True, dq=dq,
                                               dk=dk, dv=dv, workspace=bws),
                    steps, warm, flush, stream)
    ms = sum(t) / len(t)
    bflops = 2.5 * flops  # S and dP recomputed, dV, dK, dQ: 10 D per (row, key) vs 4 D forward
    n_tiles = union_tiles(w)
    # executed MMA work: dQ kernel 3 MMAs (S, dP, dQ) of 128 x 64 x 128 per union tile;
    # dK/dV kernel 4 such MMAs per chunk of 8 tokens of a block's token list
    sel = nsa_selected_pairs(w)
    exec_fl = 2.0 * 128 * 64 * D * (3 * n_tiles + 4 * sel["chunks"])
    bhbm = hbm + 2 * (w.q.numel() + w.k.numel() + w.v.numel()) * 2  # + d_out, dq, dk, dv
    log(f"nsa backward {ms:.4f} ms")
    rows["nsa_select_bwd"] = {
        "workload": w.name + " (dq, dk, dv)", "ms": round(ms, 4),
        "TFLOP/s": round(bflops / ms / 1e9, 2),
        "frac_tensor": round(bflops / ms / 1e9 / peaks["bf16_tflops"], 4),
        "executed_mma_tflops": round(exec_fl / ms / 1e9, 1),
        "executed_mma_frac": round(exec_fl / ms / 1e9 / peaks["bf16_tflops"], 4),
        "hbm_bytes": int(bhbm), "kernels_per_call": 5, "memsets_per_call": 1,
        "flop_per_call": bflops, "token_list_chunks": sel["chunks"]}
    del w, out, lse, do, dq, dk, dv, bws
    torch.cuda.empty_cache()

    # varlen NSA (8 packed sequences)
    w = workloads.nsa_varlen(device=dev)
    flops, hbm, gather, groups = nsa_work(w)
    t = timed_steps(lambda: sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts,
                                               w.block_size, cu_seqlens=w.cu_seqlens),
                    steps, warm, flush, stream)
    ms = sum(t) / len(t)
    log(f"varlen nsa {ms:.4f} ms")
    terms, t_roof = t_roof_terms(flops, hbm, peaks, gather, bw_l2)
    # the union walk's own floor: its executed MMA work at the tensor peak, or the K/V of
    # its union tiles at the L2 read bandwidth (as for the headline)
    vt = union_tiles(w)
    v_exec = 4.0 * 128 * 64 * w.q.shape[3] * vt
    v_floor_us = max(v_exec / (peaks["bf16_tflops"] * 1e12),
                     vt * 64.0 * w.q.shape[3] * 2 * 2 / (bw_l2 * 1e9)) * 1e6
    rows["nsa_select_varlen"] = {
        "workload": w.name, "ms": round(ms, 4), "TFLOP/s": round(flops / ms / 1e9, 2),
        "frac_tensor": round(flops / ms / 1e9 / peaks["bf16_tflops"], 4),
        "union_tiles": vt, "executed_mma_frac": round(v_exec / ms / 1e9 / peaks["bf16_tflops"], 4),
        "exec_floor_us": round(v_floor_us, 2), "frac_exec_floor": round(v_floor_us / (ms * 1e3), 4),
        "hbm_GB/s": round(hbm / ms / 1e6, 1), "gather_GB/s": round(gather / ms / 1e6, 1),
        "terms_us": terms, "t_roof_us": round(t_roof, 2),
        "frac_t_roof": round(t_roof / (ms * 1e3), 4),
        "t_roof_note": "l2_gather term = per-token gather of every selected block, which the "
                       "union walk does not pay; frac_exec_floor is the kernel's own floor"}
    del w
    torch.cuda.empty_cache()

    # SparseMask bounds + block-sparse attention
    w = workloads.blocksparse(device=dev)
    m = w.mask
    bnd = {}

    def bounds():
        bnd["b"] = sba.sparse_mask_bounds(m.q_positions, m.q_segment_ids, m.kv_positions,
                                          m.kv_segment_ids, 128, 128, causal=True,
                                          window_left=1024, window_right=0)

    t = timed_steps(bounds, steps, warm, flush, stream)
    ms = sum(t) / len(t)
    in_bytes = 4 * m.q_positions.numel() * 4 + 4 * bnd["b"][0].numel() * 4
    log(f"bounds {ms * 1e3:.2f} us")
    rows["sparse_mask_bounds"] = {
        "workload": m.name, "us": round(ms * 1e3, 2), "GB/s": round(in_bytes / ms / 1e6, 1),
        "frac_hbm": round(in_bytes / ms / 1e6 / peaks["hbm_gbs"], 4)}
    t = timed_steps(lambda: sba.sparse_mask_bounds(
        m.q_positions, m.q_segment_ids, m.kv_positions, m.kv_segment_ids, 128, 128, causal=True,
        window_left=1024, window_right=0, calculate_dkdv_mask=True), steps, warm, flush, stream)
    ms = sum(t) / len(t)
    log(f"dkdv bounds {ms * 1e3:.2f} us")
    rows["sparse_mask_dkdv_bounds"] = {
        "workload": m.name + " (dK/dV, kv blocks outer)", "us": round(ms * 1e3, 2),
        "GB/s": round(in_bytes / ms / 1e6, 1),
        "frac_hbm": round(in_bytes / ms / 1e6 / peaks["hbm_gbs"], 4)}
    # the scaled sweep of the same recipe (B=64, T=131072): large enough to show bandwidth
    ms_w = workloads.mask(device=dev, B=64, T=131072)
    sweep = lambda: sba.sparse_mask_bounds(ms_w.q_positions, ms_w.q_segment_ids, ms_w.kv_positions,
                                           ms_w.kv_segment_ids, 128, 128, causal=True,
                                           window_left=1024, window_right=0)
    for key, dk in (("sparse_mask_bounds_b64_t128k", False), ("sparse_mask_dkdv_bounds_b64_t128k", True)):
        t = timed_steps(lambda: sba.sparse_mask_bounds(
            ms_w.q_positions, ms_w.q_segment_ids, ms_w.kv_positions, ms_w.kv_segment_ids, 128, 128,
            causal=True, window_left=1024, window_right=0, calculate_dkdv_mask=dk),
            steps, warm, flush, stream)
        ms = sum(t) / len(t)
        sw_bytes = 4 * ms_w.q_positions.numel() * 4 + 4 * 64 * 1024 * 4
        log(f"{key} {ms * 1e3:.2f} us")
        rows[key] = {
            "workload": ms_w.name + (" (dK/dV, kv blocks outer)" if dk else ""),
            "us": round(ms * 1e3, 2), "GB/s": round(sw_bytes / ms / 1e6, 1),
            "frac_hbm": round(sw_bytes / ms / 1e6 / peaks["hbm_gbs"], 4),
            "bytes": int(sw_bytes)}
    del ms_w, sweep
    lo, up, lof, upf = bnd["b"]
    fl = blocksparse_flops(w)
    t = timed_steps(lambda: sba.blocksparse_attn_fwd(w.q, w.k, w.v, m.q_positions, m.q_segment_ids,
                                                     m.kv_positions, m.kv_segment_ids, lo, up, lof,
                                                     upf, 128, 128, causal=True, window_left=1024,
                                                     window_right=0),
                    steps, warm, flush, stream)
    ms = sum(t) / len(t)
    log(f"blocksparse {ms:.4f} ms")
    # HBM bytes: Q, K, V read once, O and LSE written, positions / segment ids, bounds
    B, T, Hq, D = w.q.shape
    bsa_hbm = (2 * w.q.numel() * 2 + 2 * w.k.numel() * 2 + B * T * Hq * 4 + 4 * B * T * 4
               + 4 * lo.numel() * 4)
    terms, t_roof = t_roof_terms(fl, bsa_hbm, peaks)
    rows["blocksparse_attn"] = {
        "workload": w.name, "ms": round(ms, 4), "TFLOP/s": round(fl / ms / 1e9, 2),
        "frac_tensor": round(fl / ms / 1e9 / peaks["bf16_tflops"], 4),
        "hbm_bytes": int(bsa_hbm), "terms_us": terms, "t_roof_us": round(t_roof, 2),
        "frac_t_roof": round(t_roof / (ms * 1e3), 4)}
    del w, m, bnd
    torch.cuda.empty_cache()

    # ragged decode
    w = workloads.decode(device=dev)
    nbytes, dfl = decode_work(w)
    ws = torch.empty(sba.ragged_decode_workspace_size(64, 32, 32768, 128, w.window_left),
                     dtype=torch.uint8, device=dev)
    out = torch.empty_like(w.q)
    t = timed_steps(lambda: sba.ragged_decode_fwd(w.q, w.k, w.v, w.sequence_start, w.sequence_end,
                                                  window_left=w.window_left,
                                                  window_right=w.window_right,
                                                  logits_soft_cap=w.logits_soft_cap,
                                                  sink_bias=w.sink_bias, out=out, workspace=ws),
                    steps, warm, flush, stream)
    ms = sum(t) / len(t)
    log(f"decode {ms * 1e3:.2f} us")
    rows["ragged_decode"] = {
        "workload": w.name, "us": round(ms * 1e3, 2), "tok/s": round(w.q.shape[0] / (ms * 1e-3), 1),
        "GB/s": round(nbytes / ms / 1e6, 1), "frac_hbm": round(nbytes / ms / 1e6 / peaks["hbm_gbs"], 4),
        "kernels_per_call": 2, "memsets_per_call": 0}
    del w
    torch.cuda.empty_cache()

    # ragged multi-query attention: multi-token decode (4 tokens per row) and a chunked
    # prefill (512-token chunks, causal over the whole prefix)
    for key, w in (("ragged_attention_q4", workloads.ragged_attention(device=dev)),
                   ("ragged_attention_chunk512",
                    workloads.ragged_attention(device=dev, B=4, Q=512, S=16384, window=(-1, 0),
                                               cap=0.0, num_sinks=0, seed=514))):
        nbytes, mfl = ragged_attention_work(w)
        B, Q, Hq, D = w.q.shape
        ws = torch.empty(sba.ragged_flash_attention_workspace_size(
            B, Q, Hq, w.k.shape[1], D, w.window_left, w.window_right), dtype=torch.uint8, device=dev)
        out = torch.empty_like(w.q)
        t = timed_steps(lambda: sba.ragged_flash_attention_fwd(
            w.q, w.k, w.v, w.sequence_start, w.sequence_end, window_left=w.window_left,
            window_right=w.window_right, logits_soft_cap=w.logits_soft_cap, sink_bias=w.sink_bias,
            out=out, workspace=ws), steps, warm, flush, stream)
        ms = sum(t) / len(t)
        log(f"{key} {ms * 1e3:.2f} us")
        rows[key] = {
            "workload": w.name, "us": round(ms * 1e3, 2),
            "tok/s": round(B * Q / (ms * 1e-3), 1),
            "GB/s": round(nbytes / ms / 1e6, 1),
            "frac_hbm": round(nbytes / ms / 1e6 / peaks["hbm_gbs"], 4),
            "TFLOP/s": round(mfl / ms / 1e9, 2),
            "frac_tensor": round(mfl / ms / 1e9 / peaks["bf16_tflops"], 4),
            "kernels_per_call": 2 if w.q.shape[1] < 128 else 1, "memsets_per_call": 0}
        del w, ws, out
        torch.cuda.empty_cache()
    sba.check_error(dev)
    return rows


def run_case(args):
    """Launch one workload's kernels ``--repeat`` times (no timing JSON): the command the
    profiles are taken with.  Cases: nsa_prefill, nsa_varlen, blocksparse (bounds then
    attention), decode (``--decode-batch`` rows of the decode workload), ragged_q4 and
    ragged_chunk512 (the two multi-query workloads; ragged_q4 takes ``--decode-batch``
    rows)."""
    import selected_block_attention_gb300 as sba
    from selected_block_attention_gb300 import _build

    _build.build()
    sba.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.case in ("nsa_prefill", "nsa_varlen"):
        w = workloads.nsa_prefill(device=dev) if args.case == "nsa_prefill" else workloads.nsa_varlen(device=dev)
        fn = lambda: sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts,
                                        w.block_size, cu_seqlens=w.cu_seqlens)
    elif args.case == "blocksparse":
        w = workloads.blocksparse(device=dev)
        m = w.mask

        def fn():
            lo, up, lof, upf = sba.sparse_mask_bounds(m.q_positions, m.q_segment_ids, m.kv_positions,
                                                      m.kv_segment_ids, 128, 128, causal=True,
                                                      window_left=1024, window_right=0)
            sba.blocksparse_attn_fwd(w.q, w.k, w.v, m.q_positions, m.q_segment_ids, m.kv_positions,
                                     m.kv_segment_ids, lo, up, lof, upf, 128, 128, causal=True,
                                     window_left=1024, window_right=0)
    elif args.case == "nsa_bwd":
        w = workloads.nsa_prefill(device=dev)
        out, lse = sba.nsa_select_fwd(w.q, w.k, w.v, w.block_indices, w.block_counts, w.block_size)
        do = torch.randn_like(w.q)
        fn = lambda: sba.nsa_select_bwd(w.q, w.k, w.v, out, lse, do, w.block_indices, w.block_counts,
                                        w.block_size)
    elif args.case == "mask_sweep":
        m = workloads.mask(device=dev, B=64, T=131072)
        fn = lambda: sba.sparse_mask_bounds(m.q_positions, m.q_segment_ids, m.kv_positions,
                                            m.kv_segment_ids, 128, 128, causal=True,
                                            window_left=1024, window_right=0)
    elif args.case == "decode":
        w = workloads.decode(device=dev, B=args.decode_batch)

        def fn():
            sba.ragged_decode_fwd(w.q, w.k, w.v, w.sequence_start, w.sequence_end,
                                  window_left=w.window_left, window_right=w.window_right,
                                  logits_soft_cap=w.logits_soft_cap, sink_bias=w.sink_bias)
    elif args.case in ("ragged_q4", "ragged_chunk512"):
        w = (workloads.ragged_attention(device=dev, B=args.decode_batch) if args.case == "ragged_q4" else
             workloads.ragged_attention(device=dev, B=4, Q=512, S=16384, window=(-1, 0), cap=0.0,
                                        num_sinks=0, seed=514))

        def fn():
            sba.ragged_flash_attention_fwd(w.q, w.k, w.v, w.sequence_start, w.sequence_end,
                                           window_left=w.window_left, window_right=w.window_right,
                                           logits_soft_cap=w.logits_soft_cap, sink_bias=w.sink_bias)
    else:
        raise SystemExit(f"unknown case {args.case}")
    for i in range(args.repeat):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        print(f"{args.case} launch {i}: {s.elapsed_time(e):.4f} ms", file=sys.stderr)
    sba.check_error(dev)


# ----------------------------------------------------------------------------- oracle legs
# The fp64 oracle runs in worker processes started with "spawn" (never forked from a
# process that has touched the GPU), one per host core.  Every worker builds the same
# seeded prefill workload on the CPU (the dense values differ from the GPU-generated
# ones, the shapes, counts and selection structure are the recipe's) and evaluates the
# oracle on the rows it is handed; the algorithmic FLOPs of those rows are counted the
# same way as for the GPU line.
_ORACLE = {}


def _oracle_init():
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    w = workloads.nsa_prefill(device="cpu")
    _ORACLE["w"] = w
    _ORACLE["q"] = w.q.double().numpy()
    _ORACLE["k"] = w.k.double().numpy()
    _ORACLE["v"] = w.v.double().numpy()
    _ORACLE["idx"] = w.block_indices.numpy()
    _ORACLE["counts"] = w.block_counts.numpy()


def _row_flops(idx, counts, rows, bs, D, G):
    fl = 0.0
    for b, t in rows:
        hi = np.minimum(idx[b, t] * bs + bs, t + 1)
        valid = (np.arange(idx.shape[-1])[None, :] < counts[b, t][:, None]) & (idx[b, t] >= 0)
        fl += 4.0 * D * G * np.where(valid, hi - idx[b, t] * bs, 0).sum()
    return fl


def _oracle_rows(rows):
    """Oracle on the given (b, t) rows of the prefill workload; returns their FLOPs."""
    import oracle

    o = _ORACLE
    oracle.nsa_select_attention(o["q"], o["k"], o["v"], o["idx"], o["counts"], o["w"].block_size,
                                rows=rows)
    return _row_flops(o["idx"], o["counts"], rows, o["w"].block_size, o["q"].shape[3],
                      o["q"].shape[2] // o["k"].shape[2])


def _oracle_ping(_):
    return len(_ORACLE)


class OraclePool:
    """One spawn-started worker per host core, each holding the workload."""

    def __init__(self, cores=None):
        import multiprocessing as mp

        self.cores = cores or os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.cores, initializer=_oracle_init)
        self.pool.map(_oracle_ping, range(self.cores), chunksize=1)  # every worker ready

    def run(self, rows_per_worker, rng):
        """One parallel sample: rows_per_worker random tokens per worker.  Returns
        (FLOPs, wall seconds, rows)."""
        B, T = 2, 8192
        chunks = [[(int(b), int(t)) for b, t in zip(rng.integers(0, B, rows_per_worker),
                                                   rng.integers(0, T, rows_per_worker))]
                  for _ in range(self.cores)]
        t0 = time.perf_counter()
        fl = self.pool.map(_oracle_rows, chunks, chunksize=1)
        return float(sum(fl)), time.perf_counter() - t0, rows_per_worker * self.cores

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(pool, seconds):
    """fp64 oracle on all host cores over a bounded, seeded sample of prefill tokens."""
    rng = np.random.default_rng(0)
    flops, dt, rows = 0.0, 0.0, 0
    while dt < seconds:
        f, d, r = pool.run(32, rng)
        flops, dt, rows = flops + f, dt + d, rows + r
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": pool.cores,
            "kind": "oracle",
            "sample": f"{rows} random tokens (all 4 KV heads x 64 query heads) of the prefill "
                      f"workload, {dt:.1f} s, numpy float64, {pool.cores} processes x 1 thread"}


def run_reference(args):
    """The fp64 oracle on all host cores, same workload, bounded sample per step."""
    pool = OraclePool()
    rng = np.random.default_rng(0)
    per_worker = 32
    for _ in range(args.warmup):
        pool.run(per_worker, rng)
    tot_t, tot_f = 0.0, 0.0
    for _ in range(args.steps):
        f, d, _r = pool.run(per_worker, rng)
        tot_t += d
        tot_f += f
    pool.close()
    value = tot_f / tot_t / 1e12
    sample = (f"{per_worker * pool.cores} random tokens per step (all 4 KV heads x 64 query heads), "
              f"numpy float64, {pool.cores} processes x 1 thread")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "nsa_select_prefill B=2 T=8192 Hq=64 Hkv=4 D=128 block_size=64 causal "
                               "(bounded sample per step)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": pool.cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", default=None,
                    help="profiling mode: launch one workload --repeat times, no JSON line")
    ap.add_argument("--repeat", type=int, default=3)
    ap.add_argument("--decode-batch", type=int, default=64)
    args = ap.parse_args()
    if args.case is not None:
        run_case(args)
        return
    args.warmup = max(args.warmup, 3)

    if "WORLD_SIZE" not in os.environ and args.gpus > 1 and args.impl == "cuda":
        # launched without torchrun: start one rank per GPU on this node
        import socket

        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
               "--master-port", str(port), os.path.abspath(__file__), *sys.argv[1:]]
        raise SystemExit(subprocess.call(cmd))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "cuda" and world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} disagrees with WORLD_SIZE={world}")

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)))
        return

    # the oracle's worker processes start before the first GPU call (spawn in any case)
    pool = OraclePool() if rank == 0 and not args.no_cpu_baseline else None
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_cuda(args, rank, world, local_rank)
    if pool is not None:
        res["cpu_baseline"] = cpu_baseline(pool, args.cpu_seconds)
        pool.close()
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
