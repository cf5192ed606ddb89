// SparseMask block bounds: forward / dQ (query blocks outer) and dK/dV (key/value blocks
// outer).
//
// Follows "ejkernel.kernels._triton.blocksparse_attention._mask" (module source page):
// kernel _compute_sparse_mask (both choices of outer operand) and the padding /
// padding-segment remap / clip fix-up of define_sparse_mask_fn, fused into one launch.
//
// Layout of the work: grid (ceil(NB_outer / kWarps), B); warp w of a CTA owns one
// outer block.  The CTA sweeps the inner blocks of its batch row in chunks: every warp
// summarises inner blocks (min/max of positions and remapped segment ids) with
// coalesced 16-byte loads and warp min/max reductions into shared memory, then each
// warp tests its outer block against the chunk with one inner block per lane and
// folds the lane results with warp min/max reductions.  Integer results are exact.
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
  if (dkdv) {
    dim3 grid((nbkv + kWarps - 1) / kWarps, B);
    sparse_mask_bounds_kernel<false><<<grid, kThreads, 0, stream>>>(
        kvside, qside, causal, window_left, window_right, pad_id, pad_remap, lower, upper,
        lower_full, upper_full, vec_kv, vec_q);
  } else {
    dim3 grid((nbq + kWarps - 1) / kWarps, B);
    sparse_mask_bounds_kernel<true><<<grid, kThreads, 0, stream>>>(
        qside, kvside, causal, window_left, window_right, pad_id, pad_remap, lower, upper,
        lower_full, upper_full, vec_q, vec_kv);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "sparse_mask_bounds launch");
  return SBA_OK;
}

}  // namespace sba
