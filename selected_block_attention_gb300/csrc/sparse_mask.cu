// SparseMask block bounds: forward / dQ (query blocks outer) and dK/dV (key/value blocks
// outer).
//
// Follows "ejkernel.kernels._triton.blocksparse_attention._mask" (module source page):
// kernel _compute_sparse_mask (both choices of outer operand) and the padding /
// padding-segment remap / clip fix-up of define_sparse_mask_fn, fused into one launch.
//
// Main kernel (sparse_mask_cluster_kernel): one cluster of kCluster CTAs per batch row.
//   1. every block of the row is summarised exactly once (min/max of positions and of
//      remapped segment ids, coalesced 16-byte loads, several blocks in flight per
//      warp, warp min/max reductions): CTA r of the cluster takes the r-th slice of the
//      inner blocks, arrives on the cluster barrier, then takes the r-th slice of the
//      outer blocks (so waiting for the slowest peer overlaps its own reads);
//   2. after the cluster barrier each CTA copies the whole row of inner summaries out of
//      its peers' shared memory (distributed shared memory) and, in the same pass,
//      builds prefix maxima / suffix minima of the summary fields the attend test
//      compares;
//   3. per outer block (one lane each, so the searches of 32 outer blocks run side by
//      side) those monotone arrays give, by binary search, a candidate range of inner
//      blocks outside of which the attend test provably fails (e.g. under causal
//      masking, once every later key block starts after the query block's last
//      position, no later block can attend); the page's predicates are then evaluated
//      exactly on the candidates only (by the same lane when every range of the warp
//      is short, else one inner block per lane with warp min/max reductions) and
//      clipped as the fix-up does.
// Pruning never changes a result: a pruned block fails a necessary condition of the
// attend test, and a full block must attend.  Integer results are exact.
// Rows with more than kMaxInner inner blocks use the fallback kernel
// (sparse_mask_bounds_kernel): one warp per outer block, inner summaries recomputed per
// CTA in chunks.
#include <cooperative_groups.h>

#include <climits>

#include "common.cuh"

namespace sba {

static __device__ unsigned g_err_mask = 0;

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kChunk = 1024;  // inner-block summaries held in shared memory at once

struct BlockSummary {
  int pos_min, pos_max, seg_min, seg_max;
};

// Min/max of positions and remapped segment ids over tokens [t0, t0 + len) of one
// row; tokens at or beyond `valid` are padding (pos_fill, segment -> pad_remap).
__device__ __forceinline__ BlockSummary summarize_block(const int* __restrict__ pos,
                                                        const int* __restrict__ seg, long long t0,
                                                        int len, int valid, int pos_fill,
                                                        int pad_id, int pad_remap, bool vec) {
  const int lane = threadIdx.x & 31;
  int pmin = INT_MAX, pmax = INT_MIN, smin = INT_MAX, smax = INT_MIN;
  if (vec) {
    for (int o = lane * 4; o < len; o += 128) {
      long long t = t0 + o;
      int p4[4], s4[4];
      if (t < valid) {
        int4 pv = *reinterpret_cast<const int4*>(pos + t);
        int4 sv = *reinterpret_cast<const int4*>(seg + t);
        p4[0] = pv.x; p4[1] = pv.y; p4[2] = pv.z; p4[3] = pv.w;
        s4[0] = sv.x; s4[1] = sv.y; s4[2] = sv.z; s4[3] = sv.w;
      } else {
#pragma unroll
        for (int u = 0; u < 4; ++u) { p4[u] = pos_fill; s4[u] = pad_id; }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        int s = s4[u] == pad_id ? pad_remap : s4[u];
        pmin = min(pmin, p4[u]); pmax = max(pmax, p4[u]);
        smin = min(smin, s); smax = max(smax, s);
      }
    }
  } else {
    for (int o = lane; o < len; o += 32) {
      long long t = t0 + o;
      int p = pos_fill, s = pad_id;
      if (t < valid) { p = pos[t]; s = seg[t]; }
      s = s == pad_id ? pad_remap : s;
      pmin = min(pmin, p); pmax = max(pmax, p);
      smin = min(smin, s); smax = max(smax, s);
    }
  }
  BlockSummary r;
  r.pos_min = __reduce_min_sync(0xffffffffu, pmin);
  r.pos_max = __reduce_max_sync(0xffffffffu, pmax);
  r.seg_min = __reduce_min_sync(0xffffffffu, smin);
  r.seg_max = __reduce_max_sync(0xffffffffu, smax);
  return r;
}

// Position tests of one (outer block, inner block) pair, as the page's kernel states
// them for each choice of outer operand (kQueryOuter: the query block is outer).
template <bool kQueryOuter>
__device__ __forceinline__ void position_tests(bool causal, int window_left, int window_right,
                                               long long o_min, long long o_max, long long i_min,
                                               long long i_max, bool& attend, bool& full) {
  attend = true;
  full = true;
  if (kQueryOuter) {
    if (causal) { attend = o_max >= i_min; full = o_min >= i_max; }
    if (window_left >= 0) {
      attend = attend && (i_min >= o_min - window_left);
      full = full && (i_min >= o_max - window_left);
    }
    if (window_right >= 0) {
      attend = attend && (i_max <= o_max + window_right);
      full = full && (i_max <= o_min + window_right);
    }
  } else {
    if (causal) { attend = i_max >= o_min; full = i_min >= o_max; }
    if (window_left >= 0) {
      attend = attend && (i_max >= o_min - window_left);
      full = full && (i_min >= o_min - window_left);
    }
    if (window_right >= 0) {
      attend = attend && (i_min <= o_max + window_right);
      full = full && (i_max <= o_max + window_right);
    }
  }
}

// One outer side and one inner side: token arrays of one batch row set, their length,
// block size, block count and the position that pads them to a block multiple.
struct Side {
  const int* pos;
  const int* seg;
  int T, block, nb, pos_fill;
};

template <bool kQueryOuter>
__global__ void __launch_bounds__(kThreads)
sparse_mask_bounds_kernel(Side outer, Side inner, int causal, int window_left, int window_right,
                          int pad_id, int pad_remap, int* __restrict__ lower,
                          int* __restrict__ upper, int* __restrict__ lower_full,
                          int* __restrict__ upper_full, int vec_outer, int vec_inner) {
  __shared__ int s_kmin[kChunk], s_kmax[kChunk], s_ksmin[kChunk], s_ksmax[kChunk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int j = blockIdx.x * kWarps + warp;  // outer block of this warp
  const bool active = j < outer.nb;
  const int* op = outer.pos + (long long)b * outer.T;
  const int* os = outer.seg + (long long)b * outer.T;
  const int* ip = inner.pos + (long long)b * inner.T;
  const int* is = inner.seg + (long long)b * inner.T;
  const int nbi = inner.nb;

  // Outer block summary.
  BlockSummary o{0, 0, 0, 0};
  bool all_pad = false;
  if (active) {
    o = summarize_block(op, os, (long long)j * outer.block, outer.block, outer.T, outer.pos_fill,
                        pad_id, pad_remap, vec_outer != 0);
    all_pad = (o.seg_min == o.seg_max) && (o.seg_min == pad_remap);
  }
  const long long o_min = o.pos_min, o_max = o.pos_max;

  int up = 0, lo = nbi, up_full = 0, lo_full = nbi;
  for (int c0 = 0; c0 < nbi; c0 += kChunk) {
    const int cn = min(kChunk, nbi - c0);
    __syncthreads();
    for (int i = warp; i < cn; i += kWarps) {
      BlockSummary s = summarize_block(ip, is, (long long)(c0 + i) * inner.block, inner.block,
                                       inner.T, inner.pos_fill, pad_id, pad_remap, vec_inner != 0);
      if (lane == 0) {
        s_kmin[i] = s.pos_min; s_kmax[i] = s.pos_max;
        s_ksmin[i] = s.seg_min; s_ksmax[i] = s.seg_max;
      }
    }
    __syncthreads();
    if (!active || all_pad) continue;
    for (int i = lane; i < cn; i += 32) {
      const int is_min = s_ksmin[i], is_max = s_ksmax[i];
      const bool attend_seg = (is_min <= o.seg_max) && (o.seg_min <= is_max);
      const bool full_seg = (o.seg_min == o.seg_max) && (is_min == is_max);
      bool attend_pos, full_pos;
      position_tests<kQueryOuter>(causal != 0, window_left, window_right, o_min, o_max,
                                  s_kmin[i], s_kmax[i], attend_pos, full_pos);
      const bool attend = attend_pos && attend_seg && !(is_min == pad_remap);
      const bool full = full_seg && full_pos && attend;
      const int blk = c0 + i;
      if (attend) { up = max(up, blk + 1); lo = min(lo, blk); }
      if (full) { up_full = max(up_full, blk + 1); lo_full = min(lo_full, blk); }
    }
  }
  if (!active) return;
  up = __reduce_max_sync(0xffffffffu, up);
  lo = __reduce_min_sync(0xffffffffu, lo);
  up_full = __reduce_max_sync(0xffffffffu, up_full);
  lo_full = __reduce_min_sync(0xffffffffu, lo_full);
  if (lane != 0) return;
  const long long out = (long long)b * outer.nb + j;
  if (all_pad) {
    lower[out] = 0; upper[out] = 0; lower_full[out] = 0; upper_full[out] = 0;
    return;
  }
  // Clip / order fix-up.
  lo = min(max(lo, 0), nbi);
  up = min(max(up, 0), nbi);
  lo = min(lo, up);
  lo_full = max(min(max(lo_full, 0), nbi), lo);
  up_full = min(max(min(max(up_full, 0), nbi), lo_full), up);
  lower[out] = lo; upper[out] = up; lower_full[out] = lo_full; upper_full[out] = up_full;
}

// ------------------------------------------------------------------ cluster kernel
namespace cg = cooperative_groups;

constexpr int kCluster = 8;          // CTAs per batch row (portable cluster size)
constexpr int kCWarps = 8;
constexpr int kCThreads = kCWarps * 32;
constexpr int kMaxInner = 4096;      // inner blocks of a row held in shared memory
constexpr int kMaxOuterSlice = 1024; // outer blocks per CTA
constexpr int kUnroll = 4;           // blocks a warp summarises at once (loads in flight)

// Summaries (pos_min, pos_max, seg_min, seg_max) of up to kUnroll blocks of one row at
// once; blk[u] < 0 marks an unused slot.  Tokens at or beyond sd.T are padding.
__device__ __forceinline__ void summarize_unrolled(const int* __restrict__ pos,
                                                   const int* __restrict__ seg, const Side& sd,
                                                   const int (&blk)[kUnroll], bool vec,
                                                   int pad_id, int pad_remap,
                                                   int4 (&out)[kUnroll]) {
  const int lane = threadIdx.x & 31;
  int pmin[kUnroll], pmax[kUnroll], smin[kUnroll], smax[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    pmin[u] = INT_MAX; pmax[u] = INT_MIN; smin[u] = INT_MAX; smax[u] = INT_MIN;
  }
  if (vec) {
    for (int o = lane * 4; o < sd.block; o += 128) {
      int4 pv[kUnroll], sv[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long t = (long long)blk[u] * sd.block + o;
        if (blk[u] >= 0 && t < sd.T) {
          pv[u] = __ldcs(reinterpret_cast<const int4*>(pos + t));
          sv[u] = __ldcs(reinterpret_cast<const int4*>(seg + t));
        } else {
          pv[u] = make_int4(sd.pos_fill, sd.pos_fill, sd.pos_fill, sd.pos_fill);
          sv[u] = make_int4(pad_id, pad_id, pad_id, pad_id);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int p4[4] = {pv[u].x, pv[u].y, pv[u].z, pv[u].w};
        const int s4[4] = {sv[u].x, sv[u].y, sv[u].z, sv[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int sg = s4[e] == pad_id ? pad_remap : s4[e];
          pmin[u] = min(pmin[u], p4[e]); pmax[u] = max(pmax[u], p4[e]);
          smin[u] = min(smin[u], sg); smax[u] = max(smax[u], sg);
        }
      }
    }
  } else {
    for (int o = lane; o < sd.block; o += 32) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const long long t = (long long)blk[u] * sd.block + o;
        int pp = sd.pos_fill, sg = pad_id;
        if (blk[u] >= 0 && t < sd.T) { pp = pos[t]; sg = seg[t]; }
        sg = sg == pad_id ? pad_remap : sg;
        pmin[u] = min(pmin[u], pp); pmax[u] = max(pmax[u], pp);
        smin[u] = min(smin[u], sg); smax[u] = max(smax[u], sg);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u)
    out[u] = make_int4(__reduce_min_sync(0xffffffffu, pmin[u]), __reduce_max_sync(0xffffffffu, pmax[u]),
                       __reduce_min_sync(0xffffffffu, smin[u]), __reduce_max_sync(0xffffffffu, smax[u]));
}

// Summaries of blocks [b0, b0 + n) of one side into dst[0 .. n), kUnroll per warp step.
__device__ __forceinline__ void summarize_slice(const int* pos, const int* seg, const Side& sd,
                                                int b0, int n, bool vec, int pad_id,
                                                int pad_remap, int4* dst) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int base = warp * kUnroll; base < n; base += kCWarps * kUnroll) {
    int blk[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) blk[u] = base + u < n ? b0 + base + u : -1;
    int4 sm[kUnroll];
    summarize_unrolled(pos, seg, sd, blk, vec, pad_id, pad_remap, sm);
    if (lane == 0) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (base + u < n) dst[base + u] = sm[u];
    }
  }
}

// Gathers the row's inner summaries out of the cluster's shared memory and builds the
// six monotone arrays of the row in the same pass: out[0..2] = prefix maxima of
// pos_min, pos_max, seg_max (out[f][i] = max over v[0..i]) and out[3..5] = suffix minima
// of pos_min, pos_max, seg_min (out[f][i] = min over v[i..n-1]).  Thread t owns the
// contiguous chunk [t c, t c + c): it copies the chunk from its owners (block i lives
// in CTA i / islice at own_inner[i % islice]) into `all`, folds it, and the chunk totals
// are combined with warp shuffles (prefix: in thread order; suffix: in reverse thread
// order) and one exchange of warp totals through `tmp` (6 * kCWarps ints); then each
// thread rescans its chunk with its offset and writes it.  Ends with the CTA
// synchronised.
__device__ void gather_scans(cg::cluster_group& cluster, int4* own_inner, int islice, int4* all,
                             int n, int* const (&out)[6], int* tmp) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = (n + kCThreads - 1) / kCThreads;
  const int lo = min(tid * chunk, n), hi = min(lo + chunk, n);
  int run[6] = {INT_MIN, INT_MIN, INT_MIN, INT_MAX, INT_MAX, INT_MAX};
  for (int i0 = lo; i0 < hi; i0 += 4) {
    int4 x[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {  // remote loads first, so they are in flight together
      if (i0 + u < hi) {
        const int i = i0 + u;
        x[u] = *cluster.map_shared_rank(own_inner + i % islice, i / islice);
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (i0 + u < hi) {
        all[i0 + u] = x[u];
        run[0] = max(run[0], x[u].x); run[1] = max(run[1], x[u].y); run[2] = max(run[2], x[u].w);
        run[3] = min(run[3], x[u].x); run[4] = min(run[4], x[u].y); run[5] = min(run[5], x[u].z);
      }
    }
  }
  // inclusive scans of the chunk totals within the warp: prefix arrays towards higher
  // lanes, suffix arrays towards lower lanes
  int incl[6];
#pragma unroll
  for (int f = 0; f < 6; ++f) incl[f] = run[f];
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
#pragma unroll
    for (int f = 0; f < 3; ++f) {
      const int o = __shfl_up_sync(0xffffffffu, incl[f], d);
      if (lane >= d) incl[f] = max(incl[f], o);
    }
#pragma unroll
    for (int f = 3; f < 6; ++f) {
      const int o = __shfl_down_sync(0xffffffffu, incl[f], d);
      if (lane + d < 32) incl[f] = min(incl[f], o);
    }
  }
  if (lane == 31) {
#pragma unroll
    for (int f = 0; f < 3; ++f) tmp[f * kCWarps + warp] = incl[f];
  }
  if (lane == 0) {
#pragma unroll
    for (int f = 3; f < 6; ++f) tmp[f * kCWarps + warp] = incl[f];
  }
  __syncthreads();
  // exclusive offset of this thread: for the prefix arrays the totals of earlier warps
  // and earlier lanes, for the suffix arrays those of later warps and later lanes
  int ex[6];
#pragma unroll
  for (int f = 0; f < 6; ++f) {
    const bool pre = f < 3;
    int wt = pre ? (lane < warp ? tmp[f * kCWarps + lane] : INT_MIN)
                 : (lane > warp && lane < kCWarps ? tmp[f * kCWarps + lane] : INT_MAX);
#pragma unroll
    for (int d = 16; d >= 1; d >>= 1) {
      const int o = __shfl_xor_sync(0xffffffffu, wt, d);
      wt = pre ? max(wt, o) : min(wt, o);
    }
    int e;
    if (pre) {
      e = __shfl_up_sync(0xffffffffu, incl[f], 1);
      if (lane == 0) e = INT_MIN;
      ex[f] = max(e, wt);
    } else {
      e = __shfl_down_sync(0xffffffffu, incl[f], 1);
      if (lane == 31) e = INT_MAX;
      ex[f] = min(e, wt);
    }
  }
  for (int i = lo; i < hi; ++i) {
    const int4 x = all[i];
    ex[0] = max(ex[0], x.x); ex[1] = max(ex[1], x.y); ex[2] = max(ex[2], x.w);
    out[0][i] = ex[0]; out[1][i] = ex[1]; out[2][i] = ex[2];
  }
  for (int i = hi - 1; i >= lo; --i) {
    const int4 x = all[i];
    ex[3] = min(ex[3], x.x); ex[4] = min(ex[4], x.y); ex[5] = min(ex[5], x.z);
    out[3][i] = ex[3]; out[4][i] = ex[4]; out[5][i] = ex[5];
  }
  __syncthreads();
}

// First index i in [0, n) with pred(i) true, for a predicate that is false then true
// along i (n if it never holds).
template <typename P>
__device__ __forceinline__ int first_true(int n, P pred) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pred(mid)) hi = mid; else lo = mid + 1;
  }
  return lo;
}

template <bool kQueryOuter>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kCThreads, 4)
sparse_mask_cluster_kernel(Side outer, Side inner, int causal, int window_left, int window_right,
                           int pad_id, int pad_remap, int* __restrict__ lower,
                           int* __restrict__ upper, int* __restrict__ lower_full,
                           int* __restrict__ upper_full, int vec_outer, int vec_inner) {
  extern __shared__ int4 csm[];
  __shared__ int scan_tmp[6 * kCWarps];
  cg::cluster_group cluster = cg::this_cluster();
  const int r = static_cast<int>(cluster.block_rank());
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int nbi = inner.nb, nbo = outer.nb;
  const int islice = (nbi + kCluster - 1) / kCluster;
  const int oslice = (nbo + kCluster - 1) / kCluster;
  int4* own_inner = csm;                  // [islice]: read by the whole cluster
  int4* all_inner = own_inner + islice;   // [nbi]
  int4* own_outer = all_inner + nbi;      // [oslice]
  int* pmx_pmin = reinterpret_cast<int*>(own_outer + oslice);  // prefix max of pos_min
  int* pmx_pmax = pmx_pmin + nbi;                               // prefix max of pos_max
  int* pmx_smax = pmx_pmax + nbi;                               // prefix max of seg_max
  int* smn_pmin = pmx_smax + nbi;                               // suffix min of pos_min
  int* smn_pmax = smn_pmin + nbi;                               // suffix min of pos_max
  int* smn_smin = smn_pmax + nbi;                               // suffix min of seg_min

  // 1. this CTA's slices of the row, each block summarised once: the inner slice, then
  // (while the cluster's other CTAs finish theirs) the outer slice
  const int i0 = r * islice, ni = max(0, min(islice, nbi - i0));
  const int o0 = r * oslice, no = max(0, min(oslice, nbo - o0));
  summarize_slice(inner.pos + (long long)b * inner.T, inner.seg + (long long)b * inner.T, inner,
                  i0, ni, vec_inner != 0, pad_id, pad_remap, own_inner);
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  summarize_slice(outer.pos + (long long)b * outer.T, outer.seg + (long long)b * outer.T, outer,
                  o0, no, vec_outer != 0, pad_id, pad_remap, own_outer);
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");

  // 2. the whole row of inner summaries from the cluster's shared memory, scanned on the
  // way in.  This CTA's slice must stay in place until every peer has copied it: arrive
  // once the copies are done, wait at the very end of the kernel.
  {
    int* const arrays[6] = {pmx_pmin, pmx_pmax, pmx_smax, smn_pmin, smn_pmax, smn_smin};
    gather_scans(cluster, own_inner, islice, all_inner, nbi, arrays, scan_tmp);
  }
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");

  // 3. candidate ranges with one lane pair per outer block (the binary searches run in
  // parallel across lanes: the even lane finds the lower end, the odd lane the upper
  // end), then per outer block the exact predicates on its candidates, split between
  // the pair.  Outer block jl goes to warp jl % kCWarps, pair (jl / kCWarps) % 16, so
  // every warp gets work.
  const int pair = lane >> 1, half = lane & 1;
  // the page's predicates on the candidates i_begin, i_begin + i_step, ... of one outer
  // block, folded into the four bounds
  auto eval_range = [&](const int4& ob, int i_begin, int i_end, int i_step, int& lo, int& up,
                        int& lo_full, int& up_full) {
    const long long o_min = ob.x, o_max = ob.y;
    for (int i = i_begin; i < i_end; i += i_step) {
      const int4 in = all_inner[i];
      const bool attend_seg = (in.z <= ob.w) && (ob.z <= in.w);
      const bool full_seg = (ob.z == ob.w) && (in.z == in.w);
      bool attend_pos, full_pos;
      position_tests<kQueryOuter>(causal != 0, window_left, window_right, o_min, o_max, in.x,
                                  in.y, attend_pos, full_pos);
      const bool attend = attend_pos && attend_seg && !(in.z == pad_remap);
      const bool full = full_seg && full_pos && attend;
      if (attend) { up = max(up, i + 1); lo = min(lo, i); }
      if (full) { up_full = max(up_full, i + 1); lo_full = min(lo_full, i); }
    }
  };
  // clipped as the fix-up does; `which` 0 stores lower / upper, 1 lower_full /
  // upper_full, 2 all four
  auto store = [&](long long out, bool all_pad, int lo, int up, int lo_full, int up_full, int which) {
    if (all_pad) {  // query / key block made only of padding
      lo = up = lo_full = up_full = 0;
    } else {
      lo = min(max(lo, 0), nbi);
      up = min(max(up, 0), nbi);
      lo = min(lo, up);
      lo_full = max(min(max(lo_full, 0), nbi), lo);
      up_full = min(max(min(max(up_full, 0), nbi), lo_full), up);
    }
    if (which != 1) { lower[out] = lo; upper[out] = up; }
    if (which != 0) { lower_full[out] = lo_full; upper_full[out] = up_full; }
  };
  for (int g0 = 0; g0 < no; g0 += kCWarps * 16) {
    const int jl = g0 + pair * kCWarps + warp;
    const bool mine = jl < no;
    int4 o = make_int4(0, 0, 0, 0);
    int bound = 0;
    if (mine) {
      o = own_outer[jl];
      const long long o_max = o.y;
      // lower end: the first block from which every necessary "inner >= threshold"
      // condition can hold (prefix maxima: each condition, and so their conjunction, is
      // false then true along the row); upper end: the first block from which some
      // necessary "inner <= threshold" condition fails for it and every later block
      // (suffix minima: the disjunction is false then true as well)
      const bool wl_on = window_left >= 0, wr_on = window_right >= 0, causal_on = causal != 0;
      const long long thr_l = (long long)o.x - window_left, thr_r = o_max + window_right;
      if (kQueryOuter) {
        if (half == 0)
          bound = first_true(nbi, [&](int i) {
            return pmx_smax[i] >= o.z && (!wl_on || (long long)pmx_pmin[i] >= thr_l);
          });
        else
          bound = first_true(nbi, [&](int i) {
            return smn_smin[i] > o.w || (causal_on && (long long)smn_pmin[i] > o_max) ||
                   (wr_on && (long long)smn_pmax[i] > thr_r);
          });
      } else {
        if (half == 0)
          bound = first_true(nbi, [&](int i) {
            return pmx_smax[i] >= o.z && (!causal_on || (long long)pmx_pmax[i] >= o.x) &&
                   (!wl_on || (long long)pmx_pmax[i] >= thr_l);
          });
        else
          bound = first_true(nbi, [&](int i) {
            return smn_smin[i] > o.w || (wr_on && (long long)smn_pmin[i] > thr_r);
          });
      }
    }
    const int other = __shfl_xor_sync(0xffffffffu, bound, 1);
    const int clo = half ? other : bound, cup = half ? bound : other;
    const bool pad_blk = mine && (o.z == o.w) && (o.z == pad_remap);
    const int ncand = mine && !pad_blk ? max(cup - clo, 0) : 0;
    if (__reduce_max_sync(0xffffffffu, ncand) <= 64) {
      // short ranges: the pair evaluates its own outer block, alternate candidates each
      int up = 0, lo = nbi, up_full = 0, lo_full = nbi;
      if (mine && !pad_blk) eval_range(o, clo + half, cup, 2, lo, up, lo_full, up_full);
      up = max(up, __shfl_xor_sync(0xffffffffu, up, 1));
      lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, 1));
      up_full = max(up_full, __shfl_xor_sync(0xffffffffu, up_full, 1));
      lo_full = min(lo_full, __shfl_xor_sync(0xffffffffu, lo_full, 1));
      if (mine) store((long long)b * nbo + o0 + jl, pad_blk, lo, up, lo_full, up_full, half);
      continue;
    }
    // long ranges: the warp evaluates one outer block at a time, one inner block per lane
    for (int k = 0; k < 16; ++k) {
      const int jk = g0 + k * kCWarps + warp;
      if (jk >= no) break;  // warp-uniform
      const int src = 2 * k;
      const int4 ok4 = make_int4(__shfl_sync(0xffffffffu, o.x, src), __shfl_sync(0xffffffffu, o.y, src),
                                 __shfl_sync(0xffffffffu, o.z, src), __shfl_sync(0xffffffffu, o.w, src));
      const int klo = __shfl_sync(0xffffffffu, clo, src), kup = __shfl_sync(0xffffffffu, cup, src);
      const bool kpad = (ok4.z == ok4.w) && (ok4.z == pad_remap);
      int up = 0, lo = nbi, up_full = 0, lo_full = nbi;
      if (!kpad) eval_range(ok4, klo + lane, kup, 32, lo, up, lo_full, up_full);
      up = __reduce_max_sync(0xffffffffu, up);
      lo = __reduce_min_sync(0xffffffffu, lo);
      up_full = __reduce_max_sync(0xffffffffu, up_full);
      lo_full = __reduce_min_sync(0xffffffffu, lo_full);
      if (lane == 0) store((long long)b * nbo + o0 + jk, kpad, lo, up, lo_full, up_full, 2);
    }
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

size_t cluster_smem_bytes(int nbi, int nbo) {
  const size_t islice = (nbi + kCluster - 1) / kCluster, oslice = (nbo + kCluster - 1) / kCluster;
  return 16 * (islice + nbi + oslice) + 6 * 4 * static_cast<size_t>(nbi);
}

}  // namespace

unsigned read_and_clear_error_mask(cudaStream_t, std::string*) {
  unsigned w = 0, zero = 0;
  cudaMemcpyFromSymbol(&w, g_err_mask, sizeof(w));
  if (w) cudaMemcpyToSymbol(g_err_mask, &zero, sizeof(zero));
  return w;
}

int launch_sparse_mask_bounds(const int32_t* q_pos, const int32_t* q_seg, const int32_t* kv_pos,
                              const int32_t* kv_seg, int B, int Tq, int Tkv, int q_block,
                              int kv_block, int causal, int window_left, int window_right,
                              int pad_id, int32_t* lower, int32_t* upper, int32_t* lower_full,
                              int32_t* upper_full, int dkdv, cudaStream_t stream) {
  const int nbq = (Tq + q_block - 1) / q_block;
  const int nbkv = (Tkv + kv_block - 1) / kv_block;
  auto al16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  const int vec_q = (Tq % 4 == 0) && (q_block % 4 == 0) && al16(q_pos) && al16(q_seg);
  const int vec_kv = (Tkv % 4 == 0) && (kv_block % 4 == 0) && al16(kv_pos) && al16(kv_seg);
  const Side qside{q_pos, q_seg, Tq, q_block, nbq, -1};
  const Side kvside{kv_pos, kv_seg, Tkv, kv_block, nbkv, INT_MAX};
  const int pad_remap = nbkv * kv_block + 1;  // padded Tkv + 1
  const Side& outer = dkdv ? kvside : qside;
  const Side& inner = dkdv ? qside : kvside;
  const int vec_o = dkdv ? vec_kv : vec_q, vec_i = dkdv ? vec_q : vec_kv;
  const int oslice = (outer.nb + kCluster - 1) / kCluster;
  if (inner.nb <= kMaxInner && oslice <= kMaxOuterSlice) {
    // one cluster per batch row, each block summarised once
    const size_t smem = cluster_smem_bytes(inner.nb, outer.nb);
    // the largest request (kMaxInner inner blocks, kMaxOuterSlice outer blocks per CTA)
    static const size_t kSmemMax = cluster_smem_bytes(kMaxInner, kMaxOuterSlice * kCluster);
    static bool attr_done[2] = {false, false};
    if (!attr_done[dkdv]) {
      cudaError_t e = dkdv ? cudaFuncSetAttribute(sparse_mask_cluster_kernel<false>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(kSmemMax))
                           : cudaFuncSetAttribute(sparse_mask_cluster_kernel<true>,
                                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>(kSmemMax));
      if (e != cudaSuccess) return cuda_error(e, "sparse_mask_bounds: set smem attribute");
      attr_done[dkdv] = true;
    }
    dim3 grid(kCluster, B);
    if (dkdv)
      sparse_mask_cluster_kernel<false><<<grid, kCThreads, smem, stream>>>(
          outer, inner, causal, window_left, window_right, pad_id, pad_remap, lower, upper,
          lower_full, upper_full, vec_o, vec_i);
    else
      sparse_mask_cluster_kernel<true><<<grid, kCThreads, smem, stream>>>(
          outer, inner, causal, window_left, window_right, pad_id, pad_remap, lower, upper,
          lower_full, upper_full, vec_o, vec_i);
  } else {
    dim3 grid((outer.nb + kWarps - 1) / kWarps, B);
    if (dkdv)
      sparse_mask_bounds_kernel<false><<<grid, kThreads, 0, stream>>>(
          outer, inner, causal, window_left, window_right, pad_id, pad_remap, lower, upper,
          lower_full, upper_full, vec_o, vec_i);
    else
      sparse_mask_bounds_kernel<true><<<grid, kThreads, 0, stream>>>(
          outer, inner, causal, window_left, window_right, pad_id, pad_remap, lower, upper,
          lower_full, upper_full, vec_o, vec_i);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "sparse_mask_bounds launch");
  return SBA_OK;
}

}  // namespace sba
