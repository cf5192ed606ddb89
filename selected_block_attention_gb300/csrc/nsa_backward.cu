// Native-sparse-attention backward, selection branch, for sm_103a: dQ, dK, dV.
//
// Follows "ejkernel.modules.operations.native_sparse_attention" (operation API page),
// NativeSparseAttention.run / native_sparse_attention, which is differentiable in
// q, k and v.  The page prints no gradient algorithm; the gradient of the forward is
// the softmax backward over each row's explicit key set:
//   P = exp(scale * Q K^T - LSE) on the selected keys, dP = dO V^T,
//   Delta = rowsum(dO * O), dS = P * (dP - Delta),
//   dQ = scale * dS K,  dK = scale * dS^T Q,  dV = P^T dO,
// where a key of a block the row's token did not select (or past its causal /
// sequence limit) has P = 0.
//
// Launch sequence (all on the caller's stream, scratch in the caller's workspace):
//   1. prep (count): Delta per (token, query head); for every (token, KV head) its
//      filtered, de-duplicated selected blocks are counted per key-block slot;
//   2. scan: offsets of each slot's token list;
//   3. prep (fill): the token lists (the reverse of block_indices: which tokens chose a
//      key block of a KV head);
//   4. dQ kernel (query-centric, tensor cores): a work item is NT = 128 / G consecutive
//      tokens and one KV head, 128 query rows; the union of the tokens' selected blocks
//      is walked in 64-key tiles gathered by TMA.  Per tile: S = Q K^T and dP = dO V^T
//      (both operands in shared memory, fp32 in tensor memory), then a softmax
//      warpgroup (one row per thread) forms dS in bf16 into tensor memory, and
//      dQ += dS K accumulates in tensor memory (A = dS from TMEM).  S/dP and dS are
//      double-buffered and two softmax warpgroups take alternate tiles, so one tile's
//      MMAs run while the other tile's softmax works;
//   5. dK/dV kernel (key-centric, tensor cores): a work item is one key block of one KV
//      head; the tokens that selected it are processed in chunks of NT tokens (their Q
//      and dO rows gathered by TMA, one box of G heads per token).  Per chunk: S and dP
//      as above, the softmax warps write P and dS (bf16) to shared memory, and
//      dV^T += dO^T P, dK^T += Q^T dS accumulate in tensor memory (M = head dim,
//      N = the block's 64 keys); the block's dK and dV are written once at the end.
// No atomics touch the gradients; the order of a list's tokens (filled with atomics)
// decides the fp32 summation order of dK/dV, so results may differ in the last bits
// between runs.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "common.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace sba {

static __device__ DevError g_err_nsab = {0u, 0u, 0};

namespace {

using namespace ptx;

constexpr int kD = 128;                     // head dimension of the tensor-core path
constexpr int kBS = 64;                     // selection block = key tile
constexpr int kRows = 128;                  // MMA M: NT tokens x G query heads
constexpr int kMaxNT = 16;
constexpr int kMaxSel = 32;
constexpr int kMaxG = 16;                   // query heads per KV head
constexpr int kMaxUnion = kMaxNT * kMaxSel;
constexpr int kThreads = 256;               // dK/dV: warps 0-3 loader, 2 MMA, spare; 4-7 softmax
constexpr int kDqThreads = 384;             // dQ: warps 0-3 loader, MMA, builder, spare; 4-11 softmax
constexpr float kLog2e = 1.4426950408889634f;

enum Role : unsigned { kRoleLoader = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleBuilder = 4 };
enum BarId : unsigned {
  kBarItemFull = 1, kBarItemEmpty, kBarQdoFull, kBarQdoEmpty, kBarKvFull, kBarKvEmpty,
  kBarSdpFull, kBarSdpEmpty, kBarDsFull, kBarDsEmpty, kBarAccFull, kBarAccEmpty
};

struct Params {
  const __nv_bfloat16* out;
  const __nv_bfloat16* dout;
  const float* lse;
  float* delta;                 // [n_tok, Hq]
  const int* block_indices;
  const int* block_counts;
  const int* cu_seqlens;
  int count_scalar, S, num_seqs;
  int B, T, Hq, Hkv, G, causal;
  int NT;                       // tokens per item / chunk (128 / G)
  float scale, scale_log2;
  int n_tok;                    // B * T
  int nbr;                      // key-block slots per (batch row, KV head)
  int n_slots;                  // B * Hkv * nbr
  int* slot_cnt;
  int* slot_off;
  int* slot_cur;
  int* slot_tok;
  int* kv_next;                 // next dK/dV work item (zeroed by the scan kernel)
  int* dq_next;                 // next dQ work item (zeroed by the scan kernel)
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int n_items_dq;
  long long wait_limit;
};

// ------------------------------------------------------------------ token / slot helpers
// Sequence of token t of batch row b: first row (absolute), length, position inside.
__device__ __forceinline__ bool locate(const Params& p, int b, int t, int& seq, int& seq0, int& slen,
                                       int& trel) {
  seq = 0;
  seq0 = b * p.T;
  slen = p.T;
  trel = t;
  if (p.cu_seqlens == nullptr) return true;
  int lo = 0, hi = p.num_seqs;  // largest s with cu[s] <= t
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (p.cu_seqlens[mid] <= t) lo = mid; else hi = mid;
  }
  const int c0 = p.cu_seqlens[lo], c1 = p.cu_seqlens[lo + 1];
  if (!(c0 <= t && t < c1) || p.cu_seqlens[0] != 0 || p.cu_seqlens[p.num_seqs] != p.T) {
    atomicOr(&g_err_nsab.flags, kDevErrInput);
    return false;
  }
  seq = lo;
  seq0 = c0;
  slen = c1 - c0;
  trel = t - c0;
  return true;
}

// First slot of a sequence inside its (batch row, KV head) range: sequence s starting
// at row c0 gets slots [c0 / 64 + s, ...), one per key block; consecutive sequences
// never overlap since floor((c0 + L) / 64) - floor(c0 / 64) + 1 >= ceil(L / 64).
__device__ __forceinline__ int seq_slot_base(int seq, int seq0_in_row) { return seq0_in_row / kBS + seq; }

// Key block of slot (b, hkv, sidx): absolute first key row and number of keys; false
// when the slot holds no block (a gap between packed sequences or past the row).
__device__ __forceinline__ bool decode_slot(const Params& p, int b, int sidx, int& row0, int& nkeys) {
  if (p.cu_seqlens == nullptr) {
    const int nb = (p.T + kBS - 1) / kBS;
    if (sidx >= nb) return false;
    row0 = b * p.T + sidx * kBS;
    nkeys = min(kBS, p.T - sidx * kBS);
    return true;
  }
  int lo = 0, hi = p.num_seqs;  // largest s with base(s) <= sidx
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (seq_slot_base(mid, p.cu_seqlens[mid]) <= sidx) lo = mid; else hi = mid;
  }
  const int c0 = p.cu_seqlens[lo], len = p.cu_seqlens[lo + 1] - c0;
  const int j = sidx - seq_slot_base(lo, c0);
  if (j < 0 || len <= 0 || j * kBS >= len) return false;
  row0 = c0 + j * kBS;
  nkeys = min(kBS, len - j * kBS);
  return true;
}

// ------------------------------------------------------------------ 1/3. prep
// One warp per (token, KV head).  kFill == false: Delta of the token's G query heads and
// the count of each selected block's slot; kFill == true: the token into each slot's list.
template <bool kFill>
__global__ void __launch_bounds__(256) nsa_bwd_prep_kernel(const Params p) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < (long long)p.n_tok * p.Hkv;
       w += warps) {
    const int tok = static_cast<int>(w / p.Hkv), hkv = static_cast<int>(w - (long long)tok * p.Hkv);
    if (!kFill) {
      // Delta[tok, hq] = <dO, O> in fp32.  The G heads of one KV head are contiguous
      // (G x 128 bf16): each lane loads 16 B per step, so one step covers two heads
      // (lanes 0-15 head 2i, lanes 16-31 head 2i+1); all loads are issued before the
      // half-warp reductions.
      const long long base = ((long long)tok * p.Hq + hkv * p.G) * kD;
      const uint4* o4 = reinterpret_cast<const uint4*>(p.out + base) + lane;
      const uint4* d4 = reinterpret_cast<const uint4*>(p.dout + base) + lane;
      const int steps = p.G >> 1;
      uint4 ov[kMaxG / 2], dv[kMaxG / 2];
#pragma unroll
      for (int i = 0; i < kMaxG / 2; ++i) {
        if (i < steps) {
          ov[i] = o4[i * 32];
          dv[i] = d4[i * 32];
        }
      }
      float mine = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxG / 2; ++i) {
        if (i < steps) {
          const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov[i]);
          const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv[i]);
          float acc = 0.f;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float2 a = __bfloat1622float2(o2[u]), c = __bfloat1622float2(d2[u]);
            acc = fmaf(a.x, c.x, fmaf(a.y, c.y, acc));
          }
#pragma unroll
          for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
          if ((lane & 15) == i) mine = acc;
        }
      }
      if ((lane & 15) < steps)
        p.delta[(long long)tok * p.Hq + hkv * p.G + 2 * (lane & 15) + (lane >> 4)] = mine;
    }
    const int b = p.cu_seqlens ? 0 : tok / p.T;
    const int t = p.cu_seqlens ? tok : tok - b * p.T;
    int seq, seq0, slen, trel;
    if (!locate(p, b, t, seq, seq0, slen, trel)) continue;
    int cnt = p.block_counts ? p.block_counts[(long long)tok * p.Hkv + hkv] : p.count_scalar;
    cnt = min(max(cnt, 0), p.S);
    const int nb = (slen + kBS - 1) / kBS;
    int e = -1;
    if (lane < cnt) e = p.block_indices[((long long)tok * p.Hkv + hkv) * p.S + lane];
    const bool valid = lane < cnt && e >= 0 && e < nb && (!p.causal || e * kBS <= trel);
    bool dup = false;
    for (int j = 0; j < kMaxSel; ++j) {
      const int ej = __shfl_sync(0xffffffffu, e, j);
      const bool vj = __shfl_sync(0xffffffffu, valid, j);
      if (j < lane && vj && ej == e) dup = true;
    }
    if (valid && !dup) {
      const int base = seq_slot_base(seq, seq0 - b * p.T);
      const long long slot = ((long long)b * p.Hkv + hkv) * p.nbr + base + e;
      if (!kFill) {
        atomicAdd(&p.slot_cnt[slot], 1);
      } else {
        const int pos = p.slot_off[slot] + atomicAdd(&p.slot_cur[slot], 1);
        p.slot_tok[pos] = tok;
      }
    }
  }
}

// ------------------------------------------------------------------ 2. scan
// Exclusive prefix sum of the slot counts (one CTA of 1024 threads, chunks of 1024),
// and the fill cursors reset to zero.
__global__ void __launch_bounds__(1024) nsa_bwd_scan_kernel(const Params p) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int c0 = 0; c0 < p.n_slots; c0 += 1024) {
    const int i = c0 + tid;
    const int v = i < p.n_slots ? p.slot_cnt[i] : 0;
    int incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      int ws = warp_sums[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, ws, d);
        if (lane >= d) ws += o;
      }
      warp_sums[lane] = ws;  // inclusive over warps
    }
    __syncthreads();
    const int before = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + incl - v;
    if (i < p.n_slots) {
      p.slot_off[i] = before;
      p.slot_cur[i] = 0;
    }
    if (c0 == 0 && tid == 0) {
      *p.kv_next = 0;
      *p.dq_next = 0;
    }
    __syncthreads();
    if (tid == 0) carry += warp_sums[31];
    __syncthreads();
  }
}

// ------------------------------------------------------------------ shared pieces
// K-major 128-byte-swizzled operand of `rows` rows: byte offset of K-step kk (16 elements)
__device__ __forceinline__ uint64_t kmajor_step(int kk, int panel_bytes) {
  return static_cast<uint64_t>(((kk / 4) * panel_bytes + (kk % 4) * 32) >> 4);
}

// 64 columns at each of two TMEM addresses of the lane row (four loads, one wait)
__device__ __forceinline__ void tmem_ld64x2(uint32_t ta, float* x, uint32_t tb, float* y) {
  tmem_ld_32x32b_x32_nw(ta, x);
  tmem_ld_32x32b_x32_nw(ta + 32, x + 32);
  tmem_ld_32x32b_x32_nw(tb, y);
  tmem_ld_32x32b_x32_nw(tb + 32, y + 32);
  tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < 64; ++j) {
    tmem_ld_ready(x[j]);
    tmem_ld_ready(y[j]);
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h2 = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h2);
}

// P and dS of one row from its S and dP columns: the first nvalid keys are admissible.
// P = 2^(s scale log2(e) - lse log2(e)), dS = P (dP - Delta); two keys per instruction.
__device__ __forceinline__ void row_grads(const float* s, const float* dp, int nvalid, float scale_log2,
                                          float lse2, float delta, uint32_t* p_pk, uint32_t* ds_pk) {
  const uint64_t scale2 = pack_f32x2(scale_log2, scale_log2);
  const uint64_t neglse2 = pack_f32x2(-lse2, -lse2);
  const uint64_t negdelta2 = pack_f32x2(-delta, -delta);
#pragma unroll
  for (int j = 0; j < 64; j += 2) {
    float a0, a1;
    unpack_f32x2(fma_f32x2(pack_f32x2(s[j], s[j + 1]), scale2, neglse2), a0, a1);
    const float p0 = j < nvalid ? ex2(a0) : 0.f;
    const float p1 = j + 1 < nvalid ? ex2(a1) : 0.f;
    if (p_pk != nullptr) p_pk[j >> 1] = pack_bf16(p0, p1);
    float d0, d1;
    unpack_f32x2(mul_f32x2(add_f32x2(pack_f32x2(dp[j], dp[j + 1]), negdelta2), pack_f32x2(p0, p1)), d0, d1);
    ds_pk[j >> 1] = pack_bf16(d0, d1);
  }
}

// ------------------------------------------------------------------ 4. dQ kernel
struct DqItem {
  int n_union;                      // -1: no more items (the builder's last publication)
  int item;                         // item index: g * Hkv + hkv
  unsigned tok_valid;
  int tok[kMaxNT];                  // token of slot i (-1: none)
  int limit[kMaxNT];                // last key row (absolute) token i may see; -1 if none
  int ux[kMaxUnion];                // first key row (absolute) of each union block
  unsigned short ubits[kMaxUnion];  // tokens of the item that selected it
};

struct DqCfg {
  static constexpr int kQBytes = kRows * kD * 2;           // 32 KB: 2 panels of 128 rows x 128 B
  static constexpr int kQPanel = kRows * 128;
  static constexpr int kTileBytes = kBS * kD * 2;          // 16 KB: K (or V) of one 64-key tile
  static constexpr int kTilePanel = kBS * 128;
  static constexpr int kStages = 3;
  static constexpr int kItemSlots = 2;
  static constexpr int kItemBytes = (static_cast<int>(sizeof(DqItem)) + 127) & ~127;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kQBytes;
  static constexpr int kOffRing = 2 * kQBytes;             // stage s: K at s * 32 KB, V + 16 KB
  static constexpr int kOffItems = kOffRing + kStages * 2 * kTileBytes;
  static constexpr int kOffSort = kOffItems + kItemSlots * kItemBytes;
  static constexpr int kOffBars = kOffSort + kMaxUnion * 8;
  static constexpr int kNumBars = 2 * kItemSlots + 2 + 2 * kStages + 8 + 2 + 2;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  // tensor memory: S[2], dP[2] (64 fp32 each), dS[2] (64 bf16 = 32 columns each), dQ (128)
  static constexpr int kSCol = 0, kDpCol = 128, kDsCol = 256, kDqCol = 320;
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kIdescS = make_idesc(128, kBS, 1u, false, false);
  static constexpr uint32_t kIdescDq = make_idesc(128, kD, 1u, false, true);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Union of the selected blocks of the item's tokens for one KV head (one warp): entries
// (first key row << 16 | token bit) sorted with a bitonic network in shared memory, equal
// rows merged by OR-ing their token bits.
__device__ void build_dq_item(const Params& p, int g, int hkv, int lane, DqItem& it, uint64_t* keys) {
  const unsigned kFull = 0xffffffffu;
  const unsigned lt_mask = (1u << lane) - 1u;
  const int tok = (lane < p.NT && g * p.NT + lane < p.n_tok) ? g * p.NT + lane : -1;
  int seq = 0, seq0 = 0, slen = 0, trel = 0, cnt = 0, limit = -1;
  if (tok >= 0) {
    const int b = p.cu_seqlens ? 0 : tok / p.T;
    const int t = p.cu_seqlens ? tok : tok - b * p.T;
    if (locate(p, b, t, seq, seq0, slen, trel)) {
      cnt = p.block_counts ? p.block_counts[(long long)tok * p.Hkv + hkv] : p.count_scalar;
      cnt = min(max(cnt, 0), p.S);
      limit = p.causal ? tok : seq0 + slen - 1;
    }
  }
  const int total = p.NT * p.S;
  int n = 0;
  for (int c0 = 0; c0 < total; c0 += 32) {
    const int idx = c0 + lane;
    const int i = idx < total ? idx / p.S : 0, j = idx - i * p.S;
    const int trow = __shfl_sync(kFull, tok, i);
    const int cnt_i = __shfl_sync(kFull, cnt, i);
    const int seq0_i = __shfl_sync(kFull, seq0, i);
    const int slen_i = __shfl_sync(kFull, slen, i);
    const int trel_i = __shfl_sync(kFull, trel, i);
    int e = -1;
    if (idx < total && trow >= 0 && j < cnt_i) e = p.block_indices[((long long)trow * p.Hkv + hkv) * p.S + j];
    const int nb = (slen_i + kBS - 1) / kBS;
    const bool valid = idx < total && trow >= 0 && j < cnt_i && e >= 0 && e < nb &&
                       (!p.causal || e * kBS <= trel_i);
    const unsigned bal = __ballot_sync(kFull, valid);
    if (valid)
      keys[n + __popc(bal & lt_mask)] =
          (static_cast<uint64_t>(static_cast<uint32_t>(seq0_i + e * kBS)) << 16) | (1u << i);
    n += __popc(bal);
  }
  int N = 32;
  while (N < n) N <<= 1;
  for (int idx = n + lane; idx < N; idx += 32) keys[idx] = ~0ull;
  __syncwarp();
  for (int k = 2; k <= N; k <<= 1) {
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      for (int idx = lane; idx < N; idx += 32) {
        const int ixj = idx ^ jj;
        if (ixj > idx) {
          const uint64_t a = keys[idx], b = keys[ixj];
          if ((a > b) == ((idx & k) == 0)) {
            keys[idx] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncwarp();
    }
  }
  int nu = 0;
  for (int base = 0; base < n; base += 32) {
    const int idx = base + lane;
    bool head = false;
    uint32_t x = 0;
    unsigned bits = 0;
    if (idx < n) {
      const uint64_t key = keys[idx];
      x = static_cast<uint32_t>(key >> 16);
      head = idx == 0 || static_cast<uint32_t>(keys[idx - 1] >> 16) != x;
      if (head) {
        bits = static_cast<unsigned>(key & 0xFFFFu);
        for (int u = idx + 1; u < n; ++u) {
          const uint64_t k2 = keys[u];
          if (static_cast<uint32_t>(k2 >> 16) != x) break;
          bits |= static_cast<unsigned>(k2 & 0xFFFFu);
        }
      }
    }
    const unsigned bal = __ballot_sync(kFull, head);
    if (head) {
      const int pos = nu + __popc(bal & lt_mask);
      it.ux[pos] = static_cast<int>(x);
      it.ubits[pos] = static_cast<unsigned short>(bits);
    }
    nu += __popc(bal);
  }
  if (lane < kMaxNT) {
    it.tok[lane] = tok;
    it.limit[lane] = limit;
  }
  const unsigned tv_bits = __ballot_sync(kFull, tok >= 0);
  if (lane == 0) {
    it.n_union = nu;
    it.tok_valid = tv_bits;
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kDqThreads, 1)
nsa_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const Params p) {
  using C = DqCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem + C::kOffSort);
  uint64_t* bb = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* item_full = bb;  bb += C::kItemSlots;
  uint64_t* item_empty = bb; bb += C::kItemSlots;
  uint64_t* qdo_full = bb;   bb += 1;
  uint64_t* qdo_empty = bb;  bb += 1;
  uint64_t* kv_full = bb;    bb += C::kStages;
  uint64_t* kv_empty = bb;   bb += C::kStages;
  uint64_t* sdp_full = bb;   bb += 2;
  uint64_t* sdp_empty = bb;  bb += 2;
  uint64_t* ds_full = bb;    bb += 2;
  uint64_t* ds_empty = bb;   bb += 2;
  uint64_t* dq_full = bb;    bb += 1;
  uint64_t* dq_empty = bb;   bb += 1;
  uint64_t* mma_done = bb;   // [2]: per issuing thread
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const Abort ab{abort_flag, &g_err_nsab, 3u, p.wait_limit};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto item_at = [&](int slot) -> DqItem& {
    return *reinterpret_cast<DqItem*>(smem + C::kOffItems + slot * C::kItemBytes);
  };

  if (threadIdx.x == 0) {
    // an item slot is released by the loader, the two MMA threads and the 8 softmax warps
    for (int i = 0; i < C::kItemSlots; ++i) { mbar_init(&item_full[i], 1); mbar_init(&item_empty[i], 11); }
    mbar_init(qdo_full, 1); mbar_init(qdo_empty, 1);
    for (int i = 0; i < C::kStages; ++i) { mbar_init(&kv_full[i], 1); mbar_init(&kv_empty[i], 1); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sdp_full[i], 1); mbar_init(&sdp_empty[i], 4);
      mbar_init(&ds_full[i], 4); mbar_init(&ds_empty[i], 1);
    }
    mbar_init(dq_full, 1); mbar_init(dq_empty, 8);
    mbar_init(&mma_done[0], 1); mbar_init(&mma_done[1], 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 2) {
    // ------------------------------------------------------------------ item builder
    int islot = 0; uint32_t iphase = 0;
    // items are handed out one at a time from a counter once a slot is free, so a CTA
    // that drew small unions takes more; from the last token group down, since under
    // causal masking later tokens choose among more blocks and have the larger unions
    while (true) {
      if (!warp_wait(&item_empty[islot], iphase ^ 1, ab, kRoleBuilder, kBarItemEmpty, -1)) break;
      int item = 0;
      if (lane == 0) item = p.n_items_dq - 1 - atomicAdd(p.dq_next, 1);
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item < 0) {
        // no more items: publish the end marker
        if (lane == 0) {
          item_at(islot).n_union = -1;
          mbar_arrive(&item_full[islot]);
        }
        __syncwarp();
        break;
      }
      const int g = item / p.Hkv, hkv = item - g * p.Hkv;
      build_dq_item(p, g, hkv, lane, item_at(islot), keys);
      if (lane == 0) {
        item_at(islot).item = item;
        mbar_arrive(&item_full[islot]);
      }
      if (++islot == C::kItemSlots) { islot = 0; iphase ^= 1; }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------------ loader
    int islot = 0; uint32_t iphase = 0;
    uint32_t qph = 0;
    int stage = 0; uint32_t kph = 0;
    uint32_t issued = 0u, last = 0u;  // stage i issued / parity of its last load in bit i
    bool q_issued = false; uint32_t q_last = 0;
    bool ok = true;
    while (ok) {
      if (!warp_wait(&item_full[islot], iphase, ab, kRoleLoader, kBarItemFull, -1)) break;
      const DqItem& it = item_at(islot);
      const int nu = it.n_union;
      if (nu < 0) break;  // no more items
      const int item = it.item;
      const int g = item / p.Hkv, hkv = item - g * p.Hkv;
      if (nu > 0) {
        if (!warp_wait(qdo_empty, qph ^ 1, ab, kRoleLoader, kBarQdoEmpty, item)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(qdo_full, 2 * C::kQBytes);
#pragma unroll
          for (int pn = 0; pn < kD / 64; ++pn) {
            tma_load_3d(smem + C::kOffQ + pn * C::kQPanel, &tm_q, qdo_full, pn * 64, hkv * p.G, g * p.NT);
            tma_load_3d(smem + C::kOffDO + pn * C::kQPanel, &tm_do, qdo_full, pn * 64, hkv * p.G, g * p.NT);
          }
        }
        q_issued = true; q_last = qph; qph ^= 1;
        for (int u = 0; u < nu; ++u) {
          if (!warp_wait(&kv_empty[stage], kph ^ 1, ab, kRoleLoader, kBarKvEmpty, item)) { ok = false; break; }
          if (lane == 0) {
            uint8_t* kdst = smem + C::kOffRing + stage * 2 * C::kTileBytes;
            mbar_arrive_expect_tx(&kv_full[stage], 2 * C::kTileBytes);
#pragma unroll
            for (int pn = 0; pn < kD / 64; ++pn) {
              tma_load_3d(kdst + pn * C::kTilePanel, &tm_k, &kv_full[stage], pn * 64, hkv, it.ux[u]);
              tma_load_3d(kdst + C::kTileBytes + pn * C::kTilePanel, &tm_v, &kv_full[stage], pn * 64, hkv,
                          it.ux[u]);
            }
          }
          issued |= 1u << stage; last = (last & ~(1u << stage)) | (kph << stage);
          if (++stage == C::kStages) { stage = 0; kph ^= 1; }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[islot]);
      if (++islot == C::kItemSlots) { islot = 0; iphase ^= 1; }
    }
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s)
        if ((issued >> s) & 1u) drain_wait(&kv_full[s], (last >> s) & 1u);
      if (q_issued) drain_wait(qdo_full, q_last);
    }
  } else if (warp == 1 || warp == 3) {
    // ------------------------------------------------------------------ MMA issuers
    // Two threads issue MMAs: warp 1 S = Q K^T and dP = dO V^T of each tile, warp 3
    // dQ += dS K.  A warp's barrier wait then stalls only its own stream while the
    // tensor core runs the other's MMAs.  Each warp runs its loop converged; one elected
    // lane issues the tcgen05 operations, lane 0 the plain arrivals.  A tile's K/V stage is released by the dQ
    // thread: its dQ MMA follows the tile's softmax, which followed the S/dP MMAs.
    const bool sdp_role = warp == 1;
    {
      const uint32_t leader = elect_one();
      int islot = 0; uint32_t iphase = 0;
      uint32_t qph = 0, dqph = 0;
      int stage = 0; uint32_t kph = 0;
      uint32_t sdp_ph = 0u, ds_ph = 0u;  // phase of buffer i in bit i (bit sets: no local memory)
      int buf = 0;  // S/dP (sdp_role) or dS buffer of the next tile
      bool ok = true;
      const uint64_t q_desc = make_sdesc(smem_base + C::kOffQ, 16, 1024, kLayoutSW128);
      const uint64_t do_desc = make_sdesc(smem_base + C::kOffDO, 16, 1024, kLayoutSW128);
      const uint64_t ring_k = make_sdesc(smem_base + C::kOffRing, 16, 1024, kLayoutSW128);
      const uint64_t ring_kmn = make_sdesc(smem_base + C::kOffRing, C::kTilePanel, 1024, kLayoutSW128);
      while (ok) {
        if (!warp_wait(&item_full[islot], iphase, ab, kRoleMma, kBarItemFull, -1)) break;
        const int nu = item_at(islot).n_union;
        if (nu < 0) break;  // no more items
        const int item = item_at(islot).item;
        if (lane == 0) mbar_arrive(&item_empty[islot]);
        if (++islot == C::kItemSlots) { islot = 0; iphase ^= 1; }
        if (nu == 0) continue;
        if (sdp_role) {
          if (!warp_wait(qdo_full, qph, ab, kRoleMma, kBarQdoFull, item)) break;
          qph ^= 1;
          for (int u = 0; u < nu; ++u) {
            if (!warp_wait(&kv_full[stage], kph, ab, kRoleMma, kBarKvFull, item) ||
                !warp_wait(&sdp_empty[buf], ((sdp_ph >> buf) & 1u) ^ 1u, ab, kRoleMma, kBarSdpEmpty, item)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t kd = ring_k + static_cast<uint64_t>((stage * 2 * C::kTileBytes) >> 4);
            const uint64_t vd = kd + static_cast<uint64_t>(C::kTileBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_f16_ss_by(leader, tmem + C::kSCol + buf * kBS, q_desc + kmajor_step(kk, C::kQPanel),
                         kd + kmajor_step(kk, C::kTilePanel), C::kIdescS, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_f16_ss_by(leader, tmem + C::kDpCol + buf * kBS, do_desc + kmajor_step(kk, C::kQPanel),
                         vd + kmajor_step(kk, C::kTilePanel), C::kIdescS, kk > 0 ? 1u : 0u);
            mma_commit_by(leader, &sdp_full[buf]);
            if (u == nu - 1) mma_commit_by(leader, qdo_empty);
            sdp_ph ^= 1u << buf;
            buf ^= 1;
            if (++stage == C::kStages) { stage = 0; kph ^= 1; }
          }
        } else {
          for (int u = 0; u < nu; ++u) {
            // dQ += dS(u) K(u)
            if (!warp_wait(&ds_full[buf], (ds_ph >> buf) & 1u, ab, kRoleMma, kBarDsFull, item)) { ok = false; break; }
            ds_ph ^= 1u << buf;
            if (u == 0) {
              if (!warp_wait(dq_empty, dqph ^ 1, ab, kRoleMma, kBarAccEmpty, item)) { ok = false; break; }
              dqph ^= 1;
            }
            tc_fence_after();
            const uint64_t kmn = ring_kmn + static_cast<uint64_t>((stage * 2 * C::kTileBytes) >> 4);
#pragma unroll
            for (int kk = 0; kk < kBS / 16; ++kk)
              mma_f16_ts_by(leader, tmem + C::kDqCol, tmem + C::kDsCol + buf * (kBS / 2) + kk * 8,
                         kmn + static_cast<uint64_t>((kk * 16 * 128) >> 4), C::kIdescDq,
                         (u == 0 && kk == 0) ? 0u : 1u);
            mma_commit_by(leader, &kv_empty[stage]);
            mma_commit_by(leader, &ds_empty[buf]);
            buf ^= 1;
            if (++stage == C::kStages) stage = 0;
          }
          if (ok) mma_commit_by(leader, dq_full);
        }
      }
      // every tcgen05 op issued by this thread has finished once its mma_done fires
      mma_commit_by(leader, &mma_done[sdp_role ? 0 : 1]);
      drain_wait(&mma_done[sdp_role ? 0 : 1], 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    // Two warpgroups: warpgroup w takes the tiles that land in S/dP and dS buffer w (the
    // MMA thread alternates buffers tile by tile, across items), and in the epilogue
    // head-dim columns 64 w .. 64 w + 63 of dQ.
    const int w = (warp - 4) >> 2;
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;          // row of the item = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int ti = r / p.G, h = r - (r / p.G) * p.G;
    int islot = 0; uint32_t iphase = 0;
    uint32_t sdp_ph = 0, ds_ph = 0, dqph = 0;
    int tiles_before = 0;                  // tiles of earlier items of this CTA
    while (true) {
      if (!warp_wait(&item_full[islot], iphase, ab, kRoleSoftmax, kBarItemFull, -1)) break;
      const DqItem& it = item_at(islot);
      const int nu = it.n_union;
      if (nu < 0) break;  // no more items
      const int item = it.item;
      const int hkv = item % p.Hkv;
      const int tok = ti < p.NT ? it.tok[ti] : -1;
      const int limit = ti < p.NT ? it.limit[ti] : -1;
      const long long hrow = (long long)(tok >= 0 ? tok : 0) * p.Hq + hkv * p.G + h;
      float lse2 = -INFINITY, delta = 0.f;
      if (tok >= 0) {
        lse2 = p.lse[hrow] * kLog2e;
        delta = p.delta[hrow];
      }
      // the LSE / Delta loads above are first used after the first tile's wait and score
      // loads, so their latency overlaps that wait
      const unsigned tbit = 1u << ti;
      bool ok = true;
      for (int u = ((tiles_before & 1) == w) ? 0 : 1; u < nu; u += 2) {
        const int x0 = it.ux[u];
        const bool sel = tok >= 0 && (it.ubits[u] & tbit) != 0u;
        int nvalid = sel ? min(max(limit - x0 + 1, 0), kBS) : 0;
        if (!warp_wait(&sdp_full[w], sdp_ph, ab, kRoleSoftmax, kBarSdpFull, item)) { ok = false; break; }
        sdp_ph ^= 1;
        tc_fence_after();
        float s[64], dp[64];
        tmem_ld64x2(tmem + lane_off + C::kSCol + w * kBS, s, tmem + lane_off + C::kDpCol + w * kBS, dp);
        if (lse2 == -INFINITY) nvalid = 0;  // a row with no attended key: P = dS = 0
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sdp_empty[w]);
        uint32_t ds_pk[32];
        row_grads(s, dp, nvalid, p.scale_log2, lse2, delta, nullptr, ds_pk);
        // the dQ MMA that read this dS buffer two tiles ago must be done
        if (!warp_wait(&ds_empty[w], ds_ph ^ 1, ab, kRoleSoftmax, kBarDsEmpty, item)) { ok = false; break; }
        ds_ph ^= 1;
        tc_fence_after();
        tmem_st_32x32b_x32_u(tmem + lane_off + C::kDsCol + w * (kBS / 2), ds_pk);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ds_full[w]);
      }
      if (!ok) break;
      tiles_before += nu;
      __nv_bfloat16* drow = p.dq + hrow * kD + w * (kD / 2);
      if (nu > 0) {
        if (!warp_wait(dq_full, dqph, ab, kRoleSoftmax, kBarAccFull, item)) break;
        dqph ^= 1;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kD / 64; ++c) {
          float v[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::kDqCol + w * (kD / 2) + c * 32, v);
          if (tok >= 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint4 w4;
              w4.x = pack_bf16(v[j] * p.scale, v[j + 1] * p.scale);
              w4.y = pack_bf16(v[j + 2] * p.scale, v[j + 3] * p.scale);
              w4.z = pack_bf16(v[j + 4] * p.scale, v[j + 5] * p.scale);
              w4.w = pack_bf16(v[j + 6] * p.scale, v[j + 7] * p.scale);
              *reinterpret_cast<uint4*>(drow + c * 32 + j) = w4;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dq_empty);
      } else if (tok >= 0) {
#pragma unroll
        for (int j = 0; j < kD / 2; j += 8) *reinterpret_cast<uint4*>(drow + j) = make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[islot]);
      if (++islot == C::kItemSlots) { islot = 0; iphase ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------ 5. dK/dV kernel
struct KvCfg {
  static constexpr int kQBytes = kRows * kD * 2;           // 32 KB (Q or dO of a chunk)
  static constexpr int kQPanel = kRows * 128;
  static constexpr int kTileBytes = kBS * kD * 2;          // 16 KB
  static constexpr int kTilePanel = kBS * 128;
  static constexpr int kPBytes = kRows * kBS * 2;          // 16 KB: P (or dS), 128 rows x 128 B
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQ = 2 * kTileBytes;             // buffer b: Q at + b * 64 KB, dO + 32 KB
  static constexpr int kOffP = kOffQ + 4 * kQBytes;
  static constexpr int kOffDs = kOffP + kPBytes;
  static constexpr int kOffBars = kOffDs + kPBytes;
  static constexpr int kNumBars = 2 + 4 + 2 + 2 + 2 + 2 + 4;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  // tensor memory: S, dP (64 fp32 each), dV^T, dK^T (lanes = head dim, 64 key columns)
  static constexpr int kSCol = 0, kDpCol = 64, kDvCol = 128, kDkCol = 192;
  static constexpr int kTmemCols = 256;
  static constexpr uint32_t kIdescS = make_idesc(128, kBS, 1u, false, false);
  static constexpr uint32_t kIdescAcc = make_idesc(128, kBS, 1u, true, true);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// Work items: the (KV head, batch row) groups in windows of kGroupWindow, and inside a
// window key block by key block across its groups.  Under causal masking the early key
// blocks are chosen by the most tokens, so each window's largest items go out first and
// its small ones fill the end (handed out group by group, the last group's largest items
// started late and set the end of the launch); a window bounds the Q / dO rows the items
// running at once gather (four groups measured faster than one or all eight on the
// prefill workload).  The slot arrays are indexed (batch row, KV head, key block).
constexpr int kGroupWindow = 4;
__device__ __forceinline__ void kv_item(const Params& p, int item, int& b, int& hkv, int& sidx,
                                        int& slot) {
  const int ng = p.B * p.Hkv;
  const int win = item / (kGroupWindow * p.nbr);
  const int rem = item - win * kGroupWindow * p.nbr;
  const int wsz = min(kGroupWindow, ng - win * kGroupWindow);  // the last window may be short
  sidx = rem / wsz;
  const int r = win * kGroupWindow + rem % wsz;
  b = r % p.B;
  hkv = r / p.B;
  slot = (b * p.Hkv + hkv) * p.nbr + sidx;
}

__global__ void __launch_bounds__(kThreads, 1)
nsa_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const Params p) {
  using C = KvCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bb = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* kv_full = bb;    bb += 1;
  uint64_t* kv_empty = bb;   bb += 1;
  uint64_t* qdo_full = bb;   bb += 2;
  uint64_t* qdo_empty = bb;  bb += 2;
  uint64_t* sdp_full = bb;   bb += 1;
  uint64_t* sdp_empty = bb;  bb += 1;
  uint64_t* pds_full = bb;   bb += 1;
  uint64_t* pds_empty = bb;  bb += 1;
  uint64_t* acc_full = bb;   bb += 1;
  uint64_t* acc_empty = bb;  bb += 1;
  uint64_t* mma_done = bb;   bb += 2;   // per issuing thread
  uint64_t* item_full = bb;  bb += 2;   // work item published in slot i
  uint64_t* item_empty = bb;            // [2]: slot i read by every consumer
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  volatile int* slot_item = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);  // [2]
  const Abort ab{abort_flag, &g_err_nsab, 4u, p.wait_limit};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = p.n_slots;
  // Work items are handed out dynamically (a global counter, in item order): the CTAs
  // then work on neighbouring items, i.e. on one (KV head, batch row) group at a time,
  // whose Q / dO rows stay in L2 across the groups' token lists.  The loader fetches an
  // item and publishes it in a two-slot ring that the MMA threads and the softmax warps
  // read (-1: no more items).
  // (called by whole warps: the MMA warps and the softmax warps)
  auto take_item = [&](int& islot, uint32_t& iph, unsigned role) -> int {
    const bool ok = warp_wait(&item_full[islot], iph, ab, role, kBarItemFull, -1);
    int item = ok ? slot_item[islot] : -1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&item_empty[islot]);
    if (++islot == 2) { islot = 0; iph ^= 1; }
    return item;
  };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1); mbar_init(kv_empty, 1);
    for (int i = 0; i < 2; ++i) { mbar_init(&qdo_full[i], 1); mbar_init(&qdo_empty[i], 1); }
    mbar_init(sdp_full, 1); mbar_init(sdp_empty, 4);
    mbar_init(pds_full, 4); mbar_init(pds_empty, 1);
    mbar_init(acc_full, 1); mbar_init(acc_empty, 4);
    mbar_init(&mma_done[0], 1); mbar_init(&mma_done[1], 1);
    // an item slot is read by the two MMA warps and the four softmax warps
    for (int i = 0; i < 2; ++i) { mbar_init(&item_full[i], 1); mbar_init(&item_empty[i], 6); }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const uint32_t smem_base = smem_u32(smem);

  if (warp == 0) {
    // ------------------------------------------------------------------ loader
    int pslot = 0; uint32_t pph = 0;
    uint32_t kvph = 0;
    uint32_t qph = 0u;  // phase of Q / dO buffer i in bit i (bit sets: no local memory)
    int qb = 0;
    bool kv_issued = false; uint32_t kv_last = 0;
    uint32_t q_issued = 0u, q_last = 0u;
    bool ok = true;
    while (ok) {
      // fetch the next item and publish it
      if (!warp_wait(&item_empty[pslot], pph ^ 1, ab, kRoleLoader, kBarItemEmpty, -1)) break;
      int item = 0;
      if (lane == 0) {
        item = atomicAdd(p.kv_next, 1);
        if (item >= n_items) item = -1;
        slot_item[pslot] = item;
        mbar_arrive(&item_full[pslot]);
      }
      item = __shfl_sync(0xffffffffu, item, 0);
      if (++pslot == 2) { pslot = 0; pph ^= 1; }
      if (item < 0) break;
      int b, hkv, sidx, slot, row0 = 0, nkeys = 0;
      kv_item(p, item, b, hkv, sidx, slot);
      if (!decode_slot(p, b, sidx, row0, nkeys)) continue;
      const int cnt = p.slot_cnt[slot], off = p.slot_off[slot];
      if (cnt == 0) continue;
      if (!warp_wait(kv_empty, kvph ^ 1, ab, kRoleLoader, kBarKvEmpty, item)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
#pragma unroll
        for (int pn = 0; pn < kD / 64; ++pn) {
          tma_load_3d(smem + C::kOffK + pn * C::kTilePanel, &tm_k, kv_full, pn * 64, hkv, row0);
          tma_load_3d(smem + C::kOffV + pn * C::kTilePanel, &tm_v, kv_full, pn * 64, hkv, row0);
        }
      }
      kv_issued = true; kv_last = kvph; kvph ^= 1;
      const int nch = (cnt + p.NT - 1) / p.NT;
      // lane i < NT: token of slot i of a chunk (past the list: a row past the end, which
      // the TMA fills with zeros); loaded one chunk ahead of its TMA loads
      auto chunk_tok = [&](int c) -> int {
        const int k = c * p.NT + lane;
        return (c < nch && lane < p.NT && k < cnt) ? p.slot_tok[off + k] : p.n_tok;
      };
      int tk_n = chunk_tok(0);
      for (int c = 0; c < nch; ++c) {
        const int tk = tk_n;
        tk_n = chunk_tok(c + 1);
        if (!warp_wait(&qdo_empty[qb], ((qph >> qb) & 1u) ^ 1u, ab, kRoleLoader, kBarQdoEmpty, item)) { ok = false; break; }
        if (lane == 0) mbar_arrive_expect_tx(&qdo_full[qb], 2 * C::kQBytes);
        __syncwarp();
        uint8_t* qdst = smem + C::kOffQ + qb * 2 * C::kQBytes;
        for (int i = 0; i < p.NT; ++i) {
          const int ti = __shfl_sync(0xffffffffu, tk, i);
          if (lane == 0) {
#pragma unroll
            for (int pn = 0; pn < kD / 64; ++pn) {
              tma_load_3d(qdst + pn * C::kQPanel + i * p.G * 128, &tm_q, &qdo_full[qb], pn * 64, hkv * p.G, ti);
              tma_load_3d(qdst + C::kQBytes + pn * C::kQPanel + i * p.G * 128, &tm_do, &qdo_full[qb], pn * 64,
                          hkv * p.G, ti);
            }
          }
        }
        q_issued |= 1u << qb; q_last = (q_last & ~(1u << qb)) | (qph & (1u << qb)); qph ^= 1u << qb;
        qb ^= 1;
      }
    }
    if (lane == 0) {
      if (kv_issued) drain_wait(kv_full, kv_last);
      for (int i = 0; i < 2; ++i)
        if ((q_issued >> i) & 1u) drain_wait(&qdo_full[i], (q_last >> i) & 1u);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------------ MMA issuers
    // Warp 1 issues S = Q K^T and dP = dO V^T of each chunk (running one chunk ahead of
    // the softmax warps, which release S / dP as soon as they have loaded them); warp 2
    // issues dV^T += dO^T P and dK^T += Q^T dS and releases the chunk's Q / dO buffer,
    // and at the end of an item the K / V tile (its MMAs follow the item's last S / dP).
    // Each warp runs its loop converged; one elected lane issues the tcgen05 operations.
    const bool sdp_role = warp == 1;
    {
      const uint32_t leader = elect_one();
      uint32_t kvph = 0, sdph = 0, pdph = 0, accph = 0;
      uint32_t qph = 0u;  // phase of Q / dO buffer i in bit i
      int qb = 0;
      bool ok = true;
      const uint64_t k_desc = make_sdesc(smem_base + C::kOffK, 16, 1024, kLayoutSW128);
      const uint64_t v_desc = make_sdesc(smem_base + C::kOffV, 16, 1024, kLayoutSW128);
      const uint64_t qk_desc = make_sdesc(smem_base + C::kOffQ, 16, 1024, kLayoutSW128);
      const uint64_t qmn_desc = make_sdesc(smem_base + C::kOffQ, C::kQPanel, 1024, kLayoutSW128);
      const uint64_t p_desc = make_sdesc(smem_base + C::kOffP, C::kPBytes, 1024, kLayoutSW128);
      const uint64_t ds_desc = make_sdesc(smem_base + C::kOffDs, C::kPBytes, 1024, kLayoutSW128);
      int islot = 0; uint32_t iph = 0;
      while (ok) {
        const int item = take_item(islot, iph, kRoleMma);
        if (item < 0) break;
        int b, hkv, sidx, slot, row0 = 0, nkeys = 0;
        kv_item(p, item, b, hkv, sidx, slot);
        if (!decode_slot(p, b, sidx, row0, nkeys)) continue;
        const int cnt = p.slot_cnt[slot];
        if (cnt == 0) continue;
        const int nch = (cnt + p.NT - 1) / p.NT;
        if (sdp_role) {
          if (!warp_wait(kv_full, kvph, ab, kRoleMma, kBarKvFull, item)) break;
          kvph ^= 1;
          for (int c = 0; c < nch; ++c) {
            if (!warp_wait(&qdo_full[qb], (qph >> qb) & 1u, ab, kRoleMma, kBarQdoFull, item) ||
                !warp_wait(sdp_empty, sdph ^ 1, ab, kRoleMma, kBarSdpEmpty, item)) { ok = false; break; }
            qph ^= 1u << qb;
            sdph ^= 1;
            tc_fence_after();
            const uint64_t qo = static_cast<uint64_t>((qb * 2 * C::kQBytes) >> 4);
            const uint64_t doo = qo + static_cast<uint64_t>(C::kQBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_f16_ss_by(leader, tmem + C::kSCol, qk_desc + qo + kmajor_step(kk, C::kQPanel),
                         k_desc + kmajor_step(kk, C::kTilePanel), C::kIdescS, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_f16_ss_by(leader, tmem + C::kDpCol, qk_desc + doo + kmajor_step(kk, C::kQPanel),
                         v_desc + kmajor_step(kk, C::kTilePanel), C::kIdescS, kk > 0 ? 1u : 0u);
            mma_commit_by(leader, sdp_full);
            qb ^= 1;
          }
        } else {
          for (int c = 0; c < nch; ++c) {
            // dV^T += dO^T P and dK^T += Q^T dS over the chunk's 128 rows (K = rows)
            if (!warp_wait(pds_full, pdph, ab, kRoleMma, kBarDsFull, item)) { ok = false; break; }
            pdph ^= 1;
            if (c == 0) {
              if (!warp_wait(acc_empty, accph ^ 1, ab, kRoleMma, kBarAccEmpty, item)) { ok = false; break; }
              accph ^= 1;
            }
            tc_fence_after();
            const uint64_t qo = static_cast<uint64_t>((qb * 2 * C::kQBytes) >> 4);
            const uint64_t doo = qo + static_cast<uint64_t>(C::kQBytes >> 4);
#pragma unroll
            for (int kk = 0; kk < kRows / 16; ++kk) {
              const uint64_t step = static_cast<uint64_t>((kk * 16 * 128) >> 4);
              mma_f16_ss_by(leader, tmem + C::kDvCol, qmn_desc + doo + step, p_desc + step, C::kIdescAcc,
                         (c == 0 && kk == 0) ? 0u : 1u);
            }
#pragma unroll
            for (int kk = 0; kk < kRows / 16; ++kk) {
              const uint64_t step = static_cast<uint64_t>((kk * 16 * 128) >> 4);
              mma_f16_ss_by(leader, tmem + C::kDkCol, qmn_desc + qo + step, ds_desc + step, C::kIdescAcc,
                         (c == 0 && kk == 0) ? 0u : 1u);
            }
            mma_commit_by(leader, &qdo_empty[qb]);
            mma_commit_by(leader, pds_empty);
            qb ^= 1;
          }
          if (!ok) break;
          mma_commit_by(leader, kv_empty);
          mma_commit_by(leader, acc_full);
        }
      }
      // every tcgen05 op issued by this thread has finished once its mma_done fires
      mma_commit_by(leader, &mma_done[sdp_role ? 0 : 1]);
      drain_wait(&mma_done[sdp_role ? 0 : 1], 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;          // row of the chunk = TMEM lane; head-dim row in the epilogue
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int ti = r / p.G, h = r - (r / p.G) * p.G;
    uint32_t sdph = 0, pdph = 0, accph = 0;
    uint8_t* prow = smem + C::kOffP + r * 128;
    uint8_t* dsrow = smem + C::kOffDs + r * 128;
    int islot = 0; uint32_t iph = 0;
    while (true) {
      const int item = take_item(islot, iph, kRoleSoftmax);
      if (item < 0) break;
      int b, hkv, sidx, slot, row0 = 0, nkeys = 0;
      kv_item(p, item, b, hkv, sidx, slot);
      if (!decode_slot(p, b, sidx, row0, nkeys)) continue;
      const int cnt = p.slot_cnt[slot], off = p.slot_off[slot];
      if (cnt == 0) {
        // no token chose this block: its keys get zero gradients
        for (int i = r; i < nkeys * (kD / 8); i += kRows) {
          const long long o = ((long long)(row0 + i / (kD / 8)) * p.Hkv + hkv) * kD + (i % (kD / 8)) * 8;
          *reinterpret_cast<uint4*>(p.dk + o) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(p.dv + o) = make_uint4(0u, 0u, 0u, 0u);
        }
        continue;
      }
      const int nch = (cnt + p.NT - 1) / p.NT;
      bool ok = true;
      // This row's token of a chunk (-1: none), and its LSE (log2 units) and Delta.  The
      // loads run ahead of their use: a chunk's token two chunks early, its LSE / Delta
      // one chunk early, so neither global latency sits between two chunks.
      auto chunk_tok = [&](int c) -> int {
        const int k = c * p.NT + ti;
        return (c < nch && k < cnt) ? p.slot_tok[off + k] : -1;
      };
      auto tok_lse = [&](int tk, float& l2, float& dl) {
        l2 = -INFINITY;
        dl = 0.f;
        if (tk >= 0) {
          const long long hrow = (long long)tk * p.Hq + hkv * p.G + h;
          l2 = p.lse[hrow] * kLog2e;
          dl = p.delta[hrow];
        }
      };
      int tok_n = chunk_tok(0);      // chunk c + 1 at the top of chunk c
      float lse2_n, delta_n;
      tok_lse(tok_n, lse2_n, delta_n);
      int tok_nn = chunk_tok(1);     // chunk c + 2
      for (int c = 0; c < nch; ++c) {
        const int tok = tok_n;
        const float lse2 = lse2_n, delta = delta_n;
        tok_n = tok_nn;
        tok_lse(tok_n, lse2_n, delta_n);
        tok_nn = chunk_tok(c + 2);
        // keys of the block this row may see: causal limit of its token, the block's end
        int nvalid = 0;
        if (tok >= 0 && lse2 != -INFINITY) nvalid = p.causal ? min(max(tok - row0 + 1, 0), nkeys) : nkeys;
        if (!warp_wait(sdp_full, sdph, ab, kRoleSoftmax, kBarSdpFull, item)) { ok = false; break; }
        sdph ^= 1;
        tc_fence_after();
        float s[64], dp[64];
        tmem_ld64x2(tmem + lane_off + C::kSCol, s, tmem + lane_off + C::kDpCol, dp);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sdp_empty);
        uint32_t p_pk[32], ds_pk[32];
        row_grads(s, dp, nvalid, p.scale_log2, lse2, delta, p_pk, ds_pk);
        // the previous chunk's dV/dK MMAs must be done with the P / dS buffers
        if (!warp_wait(pds_empty, pdph ^ 1, ab, kRoleSoftmax, kBarDsEmpty, item)) { ok = false; break; }
        pdph ^= 1;
        // row r of P and dS, 128-byte swizzle: 16-byte chunk j at position j ^ (r & 7)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int pos = (j ^ (r & 7)) * 16;
          *reinterpret_cast<uint4*>(prow + pos) = make_uint4(p_pk[4 * j], p_pk[4 * j + 1], p_pk[4 * j + 2], p_pk[4 * j + 3]);
          *reinterpret_cast<uint4*>(dsrow + pos) =
              make_uint4(ds_pk[4 * j], ds_pk[4 * j + 1], ds_pk[4 * j + 2], ds_pk[4 * j + 3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(pds_full);
      }
      if (!ok) break;
      // epilogue: lane r of dV^T / dK^T is head-dim index r; 64 key columns each
      if (!warp_wait(acc_full, accph, ab, kRoleSoftmax, kBarAccFull, item)) break;
      accph ^= 1;
      tc_fence_after();
      float av[64], ak[64];
      tmem_ld64x2(tmem + lane_off + C::kDvCol, av, tmem + lane_off + C::kDkCol, ak);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
#pragma unroll
      for (int key = 0; key < 64; ++key) {
        if (key < nkeys) {
          const long long o = ((long long)(row0 + key) * p.Hkv + hkv) * kD + r;
          p.dv[o] = __float2bfloat16_rn(av[key]);
          p.dk[o] = __float2bfloat16_rn(ak[key] * p.scale);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

struct BwdLayout {
  size_t delta, cnt, off, cur, tok, next, total;
};
size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
BwdLayout bwd_layout(int B, int T, int Hq, int Hkv, int S, int num_seqs) {
  BwdLayout L{};
  const size_t nbr = static_cast<size_t>((T + kBS - 1) / kBS) + static_cast<size_t>(num_seqs) + 1;
  const size_t n_slots = static_cast<size_t>(B) * Hkv * nbr;
  size_t o = 0;
  L.delta = o; o += round256(static_cast<size_t>(B) * T * Hq * 4);
  L.cnt = o;   o += round256(n_slots * 4);
  L.off = o;   o += round256(n_slots * 4);
  L.cur = o;   o += round256(n_slots * 4);
  L.tok = o;   o += round256(static_cast<size_t>(B) * T * Hkv * std::min(S, kMaxSel) * 4);
  L.next = o;  o += 256;
  L.total = o;
  return L;
}

}  // namespace

unsigned read_and_clear_error_nsa_bwd(cudaStream_t, std::string* where) {
  DevError w{0u, 0u, 0}, zero{0u, 0u, 0};
  cudaMemcpyFromSymbol(&w, g_err_nsab, sizeof(w));
  if (w.flags) {
    cudaMemcpyToSymbol(g_err_nsab, &zero, sizeof(zero));
    if (where && w.where) {
      char buf[96];
      snprintf(buf, sizeof(buf), " [nsa_select_bwd %s role %u barrier %u item %d]",
               ((w.where >> 24) & 0xFFu) == 3u ? "dq" : "dkdv", (w.where >> 16) & 0xFFu,
               w.where & 0xFFFFu, w.item);
      *where += buf;
    }
  }
  return w.flags;
}

size_t nsa_bwd_workspace_bytes(int B, int T, int Hq, int Hkv, int S, int num_seqs) {
  return bwd_layout(B, T, Hq, Hkv, S, num_seqs).total;
}

int launch_nsa_select_bwd(const void* q, const void* k, const void* v, const void* out,
                          const float* lse, const void* d_out, const int32_t* block_indices,
                          const int32_t* block_counts, int block_count_scalar, int S,
                          const int32_t* cu_seqlens, int num_seqs, int B, int T, int Hq, int Hkv,
                          int causal, float scale, void* dq, void* dk, void* dv, void* workspace,
                          cudaStream_t stream) {
  const BwdLayout L = bwd_layout(B, T, Hq, Hkv, S, num_seqs);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  Params p{};
  p.out = static_cast<const __nv_bfloat16*>(out);
  p.dout = static_cast<const __nv_bfloat16*>(d_out);
  p.lse = lse;
  p.delta = reinterpret_cast<float*>(ws + L.delta);
  p.block_indices = block_indices;
  p.block_counts = block_counts;
  p.cu_seqlens = cu_seqlens;
  p.count_scalar = block_count_scalar;
  p.S = S;
  p.num_seqs = num_seqs;
  p.B = B; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv;
  p.causal = causal;
  p.NT = kRows / p.G;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.n_tok = B * T;
  p.nbr = (T + kBS - 1) / kBS + num_seqs + 1;
  p.n_slots = B * Hkv * p.nbr;
  p.slot_cnt = reinterpret_cast<int*>(ws + L.cnt);
  p.slot_off = reinterpret_cast<int*>(ws + L.off);
  p.slot_cur = reinterpret_cast<int*>(ws + L.cur);
  p.slot_tok = reinterpret_cast<int*>(ws + L.tok);
  p.kv_next = reinterpret_cast<int*>(ws + L.next);
  p.dq_next = p.kv_next + 1;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.n_items_dq = ((p.n_tok + p.NT - 1) / p.NT) * Hkv;
  p.wait_limit = wait_timeout_cycles();

  // tensor maps: Q and dO [n_tok, Hq, D] (boxes of G heads x NT tokens, or x 1 token for
  // the per-token gather), K and V [n_tok, Hkv, D] (boxes of 64 keys)
  CUtensorMap tq_dq, tdo_dq, tq_kv, tdo_kv, tk, tv;
  {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)Hq, (cuuint64_t)p.n_tok};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)Hq * kD * 2};
    cuuint32_t box_dq[3] = {64, (cuuint32_t)p.G, (cuuint32_t)p.NT};
    cuuint32_t box_kv[3] = {64, (cuuint32_t)p.G, 1};
    if (encode_tensor_map(&tq_dq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                          box_dq, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&tdo_dq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(d_out), dims,
                          strides, box_dq, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&tq_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                          box_kv, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&tdo_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(d_out), dims,
                          strides, box_kv, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "nsa_select_bwd: tensor map (q / d_out) failed");
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)Hkv, (cuuint64_t)p.n_tok};
    cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)Hkv * kD * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kBS};
    if (encode_tensor_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "nsa_select_bwd: tensor map (k / v) failed");
  }
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(nsa_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DqCfg::kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(nsa_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               KvCfg::kSmemBytes);
    if (e != cudaSuccess) return cuda_error(e, "nsa_select_bwd: set smem attribute");
    attr_done = true;
  }
  cudaError_t e = cudaMemsetAsync(p.slot_cnt, 0, static_cast<size_t>(p.n_slots) * 4, stream);
  if (e != cudaSuccess) return cuda_error(e, "nsa_select_bwd: clear slot counts");
  const int prep_blocks = std::min<long long>(((long long)p.n_tok * Hkv + 7) / 8, 8LL * num_sms());
  nsa_bwd_prep_kernel<false><<<prep_blocks, 256, 0, stream>>>(p);
  nsa_bwd_scan_kernel<<<1, 1024, 0, stream>>>(p);
  nsa_bwd_prep_kernel<true><<<prep_blocks, 256, 0, stream>>>(p);
  nsa_bwd_dq_kernel<<<std::min(p.n_items_dq, num_sms()), kDqThreads, DqCfg::kSmemBytes, stream>>>(
      tq_dq, tdo_dq, tk, tv, p);
  nsa_bwd_dkdv_kernel<<<std::min(p.n_slots, num_sms()), kThreads, KvCfg::kSmemBytes, stream>>>(
      tq_kv, tdo_kv, tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "nsa_select_bwd launch");
  return SBA_OK;
}

}  // namespace sba
