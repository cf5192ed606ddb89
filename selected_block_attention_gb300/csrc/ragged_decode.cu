// Ragged decode attention, one or several query tokens per batch row: split-KV kernel
// whose last split of each row tile combines the partials.
//
// Follows "ejkernel.kernels._xla.ragged_decode_attention._xla_impl_fwd" (API page):
// ragged_decode_mqa_xla / inner_decode_xla (one query per row) and
// ragged_flash_attention_xla (Q queries per row) over the per-row key range
// [sequence_start, sequence_end) with sliding window, logits soft cap and softmax_aux
// sinks; create_attention_mask (sinks always attendable), apply_logits_soft_cap,
// apply_attention_sinks_block, and the online-softmax carry of flash_attention_block.
//
// Query i of a row sits at position end - Q + i (Q = 1: the decode query at end - 1).
// Key k is attendable by it iff start <= k < end and k is inside the query's inclusive
// window or k < num_sinks.  Logit: scale * <q, k>, then cap * tanh(. / cap) when
// cap > 0, then + sink bias for k < num_sinks.
//
// Rows: the Q * G (query, head) pairs of one KV head, query-major; a row tile is 16
// consecutive pairs, the 16 rows of an m16n8k16 MMA (the G heads of one query when
// Q = 1; rows past the end are zero).  Work split: CTA (split s, KV head h, row tile
// rt of batch row b) covers kKeysPerCta keys of the union [lo, hi) of its rows'
// windows; its four warps each stream kKeysPerWarp of them as 16-key K/V tiles with
// 16-byte cp.async (each key row of one head is 256 contiguous bytes) through a
// 2-stage shared-memory ring, and keep the online-softmax state in registers.  Tiles
// inside every row's window skip the per-element mask; edge tiles mask each element
// with its own row's window.  Sink keys outside [lo, hi) go through an extra sink tile
// of split 0.  The four warps merge through shared memory and write one fp32 partial
// (o * exp(-m), m, l) per (row, split, query, head).  The CTA that completes the last
// split of a row tile (a counter per tile in the workspace, cleared by a small kernel
// launched just before, which the split kernel overlaps and waits for only at its first
// counter use) merges the tile's partials with max / exp weights and writes the bf16
// output and the natural-log LSE.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>
#include <mutex>
#include <string>

#include "common.cuh"
#include "ptx.cuh"

namespace sba {

static __device__ unsigned g_err_decode = 0;

namespace {

constexpr int kD = 128;
constexpr int kWarps = 4;
constexpr int kKeysPerWarp = 256;
constexpr int kKeysPerCta = kWarps * kKeysPerWarp;
constexpr int kTileKeys = 16;
constexpr int kStages = 2;  // 70 KB of ring per CTA: three CTAs (12 warps) per SM
constexpr int kRowBytes = kD * 2 + 16;  // padded shared-memory row (ldmatrix without conflicts)
constexpr int kTileBytes = kTileKeys * kRowBytes;
constexpr int kWarpSmem = kStages * 2 * kTileBytes;
constexpr int kSmemBytes = kWarps * kWarpSmem;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Issue the cp.async copies of one 16-key K/V tile of KV head h.  Keys are clamped into
// the row's own range [start, end) (end > start), so no copy reads a cache slot the row
// does not own (never written, possibly NaN: its V row would reach P V, where 0 * NaN is
// NaN); the clamped duplicates are masked later.
__device__ __forceinline__ void load_tile(const __nv_bfloat16* k, const __nv_bfloat16* v, int S,
                                          int Hkv, int b, int h, int key0, int start, int end,
                                          uint32_t k_dst, uint32_t v_dst, int lane) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int u = lane + 32 * i;  // 256 chunks of 16 bytes per tensor
    const int key = u >> 4, part = u & 15;
    const int kk = min(max(key0 + key, start), end - 1);
    const long long row = ((long long)b * S + kk) * Hkv + h;
    const uint32_t off = key * kRowBytes + part * 16;
    cp_async16(k_dst + off, k + row * kD + part * 8);
    cp_async16(v_dst + off, v + row * kD + part * 8);
  }
}

struct MqParams {
  const __nv_bfloat16* q;  // [B, Q, Hq, D]
  const __nv_bfloat16* k;  // [B, S, Hkv, D]
  const __nv_bfloat16* v;
  const int* seq_start;
  const int* seq_end;
  const float* sink_bias;
  float* o_part;   // [B][max_splits][Q][Hq][D]
  float* ml_part;  // [B][max_splits][Q][Hq][2]
  int* tile_count; // [B][Hkv][row_tiles]: splits of a row tile done (zero between calls)
  __nv_bfloat16* out;
  float* lse;
  int B, Qn, Hq, Hkv, S, G, max_splits, row_tiles;
  float scale, cap;
  int window_left, window_right, num_sinks, sink_per_head;
};

struct MqRange {
  int start, end;  // the row's clamped range [start, end)
  int lo, hi;      // union of the tile's windows inside it
  int sink_end;    // sink keys are [start, sink_end)
  bool sink_tile;  // some sink key lies outside [lo, hi)
  int n_split;
};

// Key range of row tile rt of batch row b: every CTA of the tile derives the same number
// of splits from it (the last one to finish combines).
__device__ __forceinline__ MqRange mq_tile_range(const MqParams& p, int b, int rt) {
  MqRange R;
  R.start = max(p.seq_start[b], 0);
  R.end = min(p.seq_end[b], p.S);
  R.n_split = 0;
  R.sink_tile = false;
  if (R.end <= R.start) {
    R.start = R.lo = R.hi = R.sink_end = R.end;
    return R;
  }
  const int nrows = p.Qn * p.G;
  const int r0 = rt * 16, r1 = min(r0 + 15, nrows - 1);
  const long long p_lo = (long long)R.end - p.Qn + r0 / p.G;
  const long long p_hi = (long long)R.end - p.Qn + r1 / p.G;
  long long lo = R.start, hi = R.end;
  if (p.window_left >= 0) lo = max(lo, p_lo - p.window_left);
  if (p.window_right >= 0) hi = min(hi, p_hi + p.window_right + 1);
  if (hi <= lo) lo = hi = R.end;  // no window key: only sinks can remain
  R.lo = static_cast<int>(lo);
  R.hi = static_cast<int>(hi);
  R.sink_end = min(p.num_sinks, R.end);
  R.sink_tile = min(R.sink_end, R.lo) > R.start || R.sink_end > max(R.hi, R.start);
  int n = (R.hi - R.lo + kKeysPerCta - 1) / kKeysPerCta;
  if (n == 0 && R.sink_tile) n = 1;
  R.n_split = min(n, p.max_splits);  // the host's bound already covers n; never read past it
  return R;
}

// kHiRows: Q * G > 8, so the rows g + 8 of the m16n8k16 tiles are used.  kCap: logits
// soft cap on.
template <bool kHiRows, bool kCap>
__global__ void __launch_bounds__(kWarps * 32, 3)
ragged_mq_split_kernel(const MqParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int s = blockIdx.x, h = blockIdx.y;
  const int b = blockIdx.z / p.row_tiles, rt = blockIdx.z % p.row_tiles;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;

  const MqRange R = mq_tile_range(p, b, rt);
  if (R.n_split == 0) {
    // no attendable key for any row of the tile: output 0 and LSE -inf, once
    if (s == 0) {
      const int nr = p.Qn * p.G, tile_rows = min(16, nr - rt * 16);
      for (int r = 0; r < tile_rows; ++r) {
        const int rr = rt * 16 + r;
        const long long orow = ((long long)b * p.Qn + rr / p.G) * p.Hq + h * p.G + rr % p.G;
        p.out[orow * kD + threadIdx.x] = __float2bfloat16_rn(0.f);
        if (p.lse != nullptr && threadIdx.x == 0) p.lse[orow] = -INFINITY;
      }
    }
    return;
  }
  if (s >= R.n_split) return;
  const bool do_sinks = (s == 0) && (warp == 0) && R.sink_tile;
  const int key_lo = R.lo + s * kKeysPerCta + warp * kKeysPerWarp;
  const int key_hi = min(key_lo + kKeysPerWarp, R.hi);
  const int n_tiles = key_hi > key_lo ? (key_hi - key_lo + kTileKeys - 1) / kTileKeys : 0;
  const int first_tile = do_sinks ? -1 : 0;  // tile -1 = sink tile at keys [0, 16)

  // This thread's two rows (g and g + 8 of the tile): query, head, window.
  const int nrows = p.Qn * p.G;
  const int rr0 = rt * 16 + g, rr1 = rr0 + 8;
  const bool ok0 = rr0 < nrows, ok1 = kHiRows && rr1 < nrows;
  const int i0 = ok0 ? rr0 / p.G : 0, i1 = ok1 ? rr1 / p.G : 0;
  const int hq0 = h * p.G + (rr0 - i0 * p.G) * ok0, hq1 = h * p.G + (rr1 - i1 * p.G) * ok1;
  auto win_lo = [&](int i) -> int {  // smallest window key of query i (keys are >= 0)
    if (p.window_left < 0) return -1;
    return static_cast<int>(max((long long)R.end - p.Qn + i - p.window_left, -1LL));
  };
  auto win_hi = [&](int i) -> int {  // largest window key of query i
    if (p.window_right < 0) return INT_MAX;
    return static_cast<int>(min((long long)R.end - p.Qn + i + p.window_right, (long long)INT_MAX));
  };
  const int wlo0 = win_lo(i0), whi0 = ok0 ? win_hi(i0) : -1;
  const int wlo1 = win_lo(i1), whi1 = ok1 ? win_hi(i1) : -1;
  // The part of the window that every row of the tile shares (rows past the end do not
  // count): a key tile inside it, holding no sink, needs no per-element mask.
  int all_lo = max(ok0 ? wlo0 : INT_MIN, ok1 ? wlo1 : INT_MIN);
  int all_hi = min(ok0 ? whi0 : INT_MAX, ok1 ? whi1 : INT_MAX);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    all_lo = max(all_lo, __shfl_xor_sync(0xffffffffu, all_lo, off));
    all_hi = min(all_hi, __shfl_xor_sync(0xffffffffu, all_hi, off));
  }

  // Query fragments (A operand): row r of the tile is (query, head) pair rt * 16 + r.
  uint32_t qa[8][4];
  {
    const __nv_bfloat16* qr0 = ok0 ? p.q + ((long long)(b * p.Qn + i0) * p.Hq + hq0) * kD : nullptr;
    const __nv_bfloat16* qr1 = ok1 ? p.q + ((long long)(b * p.Qn + i1) * p.Hq + hq1) * kD : nullptr;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int d0 = ks * 16 + 2 * c;
      auto ld = [&](const __nv_bfloat16* r, int d) -> uint32_t {
        return r != nullptr ? *reinterpret_cast<const uint32_t*>(r + d) : 0u;
      };
      qa[ks][0] = ld(qr0, d0);
      qa[ks][1] = ld(qr1, d0);
      qa[ks][2] = ld(qr0, d0 + 8);
      qa[ks][3] = ld(qr1, d0 + 8);
    }
  }
  const float* bias_row0 = nullptr;
  const float* bias_row1 = nullptr;
  if (p.num_sinks > 0) {
    bias_row0 = p.sink_bias + (p.sink_per_head ? (long long)hq0 * p.num_sinks : 0);
    bias_row1 = p.sink_bias + (p.sink_per_head ? (long long)hq1 * p.num_sinks : 0);
  }

  const uint32_t wbase = ptx::smem_u32(smem) + warp * kWarpSmem;
  auto k_stage = [&](int st) { return wbase + st * 2 * kTileBytes; };
  auto v_stage = [&](int st) { return wbase + st * 2 * kTileBytes + kTileBytes; };
  auto tile_key0 = [&](int t) { return t < 0 ? 0 : key_lo + t * kTileKeys; };
  // Copies of one tile: lane copies 16-byte part (lane & 15) of keys 2 i + (lane >> 4).
  // Tiles inside the row's range [start, end) step one pointer; the rare edge tile clamps
  // key by key into that range.
  const long long key_stride = (long long)p.Hkv * kD;
  const long long lane_off = ((long long)b * p.S * p.Hkv + h) * kD + (lane & 15) * 8;
  const uint32_t lane_dst = (lane >> 4) * kRowBytes + (lane & 15) * 16;
  auto issue_tile = [&](int key0, uint32_t k_dst, uint32_t v_dst) {
    if (key0 >= R.start && key0 + kTileKeys <= R.end) {
      const long long off = lane_off + (long long)(key0 + (lane >> 4)) * key_stride;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        cp_async16(k_dst + lane_dst + 2 * i * kRowBytes, p.k + off + 2 * i * key_stride);
        cp_async16(v_dst + lane_dst + 2 * i * kRowBytes, p.v + off + 2 * i * key_stride);
      }
    } else {
      load_tile(p.k, p.v, p.S, p.Hkv, b, h, key0, R.start, R.end, k_dst, v_dst, lane);
    }
  };
  // Logits in log2 units: s * scale * log2(e), or with the cap
  // log2(e) * cap * tanh(s * scale / cap) = c3 - c2 / (1 + 2^(s * c1)).
  const float c0 = p.scale * kLog2e;
  const float c1 = kCap ? p.scale * 2.f * kLog2e / p.cap : 0.f;
  const float c2 = kCap ? 2.f * p.cap * kLog2e : 0.f;
  const float c3 = kCap ? p.cap * kLog2e : 0.f;
  auto logit = [&](float x) -> float {
    if constexpr (kCap) {
      const float e = ptx::ex2(x * c1);
      float r;
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.f + e));
      return fmaf(-c2, r, c3);
    } else {
      return x * c0;
    }
  };

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  const int last_tile = n_tiles - 1;
#pragma unroll
  for (int i = 0; i < kStages - 1; ++i) {
    const int t = first_tile + i;
    if (t <= last_tile) issue_tile(tile_key0(t), k_stage(i), v_stage(i));
    cp_async_commit();
  }
  int stage = 0;
  for (int t = first_tile; t <= last_tile; ++t) {
    {
      const int tn = t + kStages - 1;
      const int sn = (stage + kStages - 1) % kStages;
      if (tn <= last_tile) issue_tile(tile_key0(tn), k_stage(sn), v_stage(sn));
      cp_async_commit();
    }
    cp_async_wait<kStages - 1>();
    __syncwarp();
    const uint32_t ks_base = k_stage(stage), vs_base = v_stage(stage);
    const int key0 = tile_key0(t);

    float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    {
      const int mi = lane >> 3, ri = lane & 7;
      const uint32_t row_addr = ks_base + ((mi >> 1) * 8 + ri) * kRowBytes + (mi & 1) * 16;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        uint32_t b00, b01, b10, b11;
        ldsm_x4(row_addr + kk * 32, b00, b01, b10, b11);
        mma_bf16(sc[0], qa[kk], b00, b01);
        mma_bf16(sc[1], qa[kk], b10, b11);
      }
    }
    float tmax0 = -INFINITY, tmax1 = -INFINITY;
    const bool plain = t >= 0 && key0 >= p.num_sinks && key0 >= key_lo &&
                       key0 + kTileKeys <= key_hi && key0 >= all_lo &&
                       key0 + kTileKeys - 1 <= all_hi;  // warp-uniform
    if (plain) {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sc[nt][e] = logit(sc[nt][e]);
          tmax0 = fmaxf(tmax0, sc[nt][e]);
          if constexpr (kHiRows) {
            sc[nt][2 + e] = logit(sc[nt][2 + e]);
            tmax1 = fmaxf(tmax1, sc[nt][2 + e]);
          } else {
            sc[nt][2 + e] = -INFINITY;
          }
        }
      }
    } else {
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key0 + nt * 8 + 2 * c + e;
          const bool sink = key < p.num_sinks;
          bool in0, in1;
          if (t < 0) {  // sink tile: in-range sink keys outside the union window, every row
            const bool outside = key >= R.start && key < R.sink_end && (key < R.lo || key >= R.hi);
            in0 = ok0 && outside;
            in1 = ok1 && outside;
          } else {
            const bool in_tile = key >= key_lo && key < key_hi;
            in0 = ok0 && in_tile && ((key >= wlo0 && key <= whi0) || sink);
            in1 = ok1 && in_tile && ((key >= wlo1 && key <= whi1) || sink);
          }
          float y0 = logit(sc[nt][e]);
          if (sink) y0 = fmaf(bias_row0[key], kLog2e, y0);
          sc[nt][e] = in0 ? y0 : -INFINITY;
          tmax0 = fmaxf(tmax0, sc[nt][e]);
          if constexpr (kHiRows) {
            float y1 = logit(sc[nt][2 + e]);
            if (sink) y1 = fmaf(bias_row1[key], kLog2e, y1);
            sc[nt][2 + e] = in1 ? y1 : -INFINITY;
            tmax1 = fmaxf(tmax1, sc[nt][2 + e]);
          } else {
            sc[nt][2 + e] = -INFINITY;
          }
        }
      }
    }
    tmax0 = fmaxf(tmax0, __shfl_xor_sync(0xffffffffu, tmax0, 1));
    tmax0 = fmaxf(tmax0, __shfl_xor_sync(0xffffffffu, tmax0, 2));
    if constexpr (kHiRows) {
      tmax1 = fmaxf(tmax1, __shfl_xor_sync(0xffffffffu, tmax1, 1));
      tmax1 = fmaxf(tmax1, __shfl_xor_sync(0xffffffffu, tmax1, 2));
    }
    const float mn0 = (tmax0 > m0 + kRescaleThreshold || (m0 == -INFINITY && tmax0 != -INFINITY)) ? tmax0 : m0;
    const float mn1 = (tmax1 > m1 + kRescaleThreshold || (m1 == -INFINITY && tmax1 != -INFINITY)) ? tmax1 : m1;
    const bool mv0 = mn0 != m0, mv1 = mn1 != m1;
    const float alpha0 = (mv0 && m0 != -INFINITY) ? ptx::ex2(m0 - mn0) : 1.f;
    const float alpha1 = (mv1 && m1 != -INFINITY) ? ptx::ex2(m1 - mn1) : 1.f;
    m0 = mn0;
    m1 = mn1;
    float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float p0 = mn0 == -INFINITY ? 0.f : ptx::ex2(sc[nt][e] - mn0);
        sc[nt][e] = p0;
        ps0 += p0;
        if constexpr (kHiRows) {
          const float p1 = mn1 == -INFINITY ? 0.f : ptx::ex2(sc[nt][2 + e] - mn1);
          sc[nt][2 + e] = p1;
          ps1 += p1;
        } else {
          sc[nt][2 + e] = 0.f;
        }
      }
    }
    l0 = l0 * alpha0 + ps0;
    l1 = l1 * alpha1 + ps1;
    if (__any_sync(0xffffffffu, mv0 || mv1)) {
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        o[dn][0] *= alpha0; o[dn][1] *= alpha0; o[dn][2] *= alpha1; o[dn][3] *= alpha1;
      }
    }
    uint32_t pa[4];
    pa[0] = pack_bf16(sc[0][0], sc[0][1]);
    pa[1] = pack_bf16(sc[0][2], sc[0][3]);
    pa[2] = pack_bf16(sc[1][0], sc[1][1]);
    pa[3] = pack_bf16(sc[1][2], sc[1][3]);
    {
      const int mi = lane >> 3, ri = lane & 7;
      const uint32_t row_addr = vs_base + ((mi & 1) * 8 + ri) * kRowBytes + (mi >> 1) * 16;
#pragma unroll
      for (int dn = 0; dn < 16; dn += 2) {
        uint32_t b00, b01, b10, b11;
        ldsm_x4_t(row_addr + dn * 16, b00, b01, b10, b11);
        mma_bf16(o[dn], pa, b00, b01);
        mma_bf16(o[dn + 1], pa, b10, b11);
      }
    }
    __syncwarp();
    stage = (stage + 1) % kStages;
  }
  cp_async_wait<0>();
  __syncthreads();

  m0 = m0 == -INFINITY ? m0 : m0 * kLn2;
  m1 = m1 == -INFINITY ? m1 : m1 * kLn2;
  float* s_o = reinterpret_cast<float*>(smem);  // [kWarps][16][kD]
  float* s_ml = s_o + kWarps * 16 * kD;          // [kWarps][16][2]
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
  for (int dn = 0; dn < 16; ++dn) {
    const int d = dn * 8 + 2 * c;
    s_o[(warp * 16 + g) * kD + d] = o[dn][0];
    s_o[(warp * 16 + g) * kD + d + 1] = o[dn][1];
    s_o[(warp * 16 + g + 8) * kD + d] = o[dn][2];
    s_o[(warp * 16 + g + 8) * kD + d + 1] = o[dn][3];
  }
  if (c == 0) {
    s_ml[(warp * 16 + g) * 2 + 0] = m0;
    s_ml[(warp * 16 + g) * 2 + 1] = l0;
    s_ml[(warp * 16 + g + 8) * 2 + 0] = m1;
    s_ml[(warp * 16 + g + 8) * 2 + 1] = l1;
  }
  __syncthreads();
  // Per row: the merged max and sum and each warp's weight, once (16 threads).
  float* s_f = s_ml + kWarps * 16 * 2;  // [16][kWarps] weights
  float* s_m = s_f + 16 * kWarps;       // [16] merged max
  float* s_l = s_m + 16;                // [16] merged sum
  if (threadIdx.x < 16) {
    const int r = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_ml[(w * 16 + r) * 2]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = s_ml[(w * 16 + r) * 2];
      const float f = (M == -INFINITY || mw == -INFINITY) ? 0.f : ptx::ex2((mw - M) * kLog2e);
      s_f[r * kWarps + w] = f;
      L += f * s_ml[(w * 16 + r) * 2 + 1];
    }
    s_m[r] = M;
    s_l[r] = L;
  }
  __syncthreads();
  const int d = threadIdx.x;  // kD == blockDim.x
  const int tile_rows = min(16, nrows - rt * 16);
  for (int r = 0; r < tile_rows; ++r) {
    const float M = s_m[r], L = s_l[r];
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) O = fmaf(s_f[r * kWarps + w], s_o[(w * 16 + r) * kD + d], O);
    const int rr = rt * 16 + r;
    const int qi = rr / p.G, hq = h * p.G + rr % p.G;
    const long long slot = (((long long)b * p.max_splits + s) * p.Qn + qi) * p.Hq + hq;
    p.o_part[slot * kD + d] = O;
    if (d == 0) {
      p.ml_part[slot * 2 + 0] = M;
      p.ml_part[slot * 2 + 1] = L;
    }
  }
  // Combine: the CTA that finishes a row tile's last split merges the tile's partials
  // (max / exp weights over the splits) and writes the bf16 output and the LSE.  Each
  // thread's partial stores are made visible before the count (fence, barrier, atomic);
  // the last CTA fences again before it reads the others' partials.
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int* cnt = p.tile_count + ((long long)b * p.Hkv + h) * p.row_tiles + rt;
    // the counters were cleared by the launch before this one, which may still be running
    // (programmatic dependent launch): wait for it to finish before the first use
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int done = atomicAdd(cnt, 1) + 1;
    s_last = done == R.n_split;
    if (s_last) *cnt = 0;  // every split has counted: ready for the next call
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // weights of each (row, split): (m, l) of all splits into shared memory, then one
  // thread per row; then every thread sums its head-dim column over rows and splits
  const long long split_stride = (long long)p.Qn * p.Hq;
  // shared memory after the merge buffers holds 16 rows x kComboSplits splits of weights
  constexpr int kComboFloats = (kSmemBytes / 4) - (kWarps * 16 * kD + kWarps * 16 * 2 + 16 * kWarps + 32);
  constexpr int kComboSplits = (kComboFloats - 32) / (16 * 3);
  if (R.n_split > kComboSplits) {
    // very long rows: one (row, split) at a time
    for (int r = 0; r < tile_rows; ++r) {
      const int rr = rt * 16 + r;
      const int qi = rr / p.G, hq = h * p.G + rr % p.G;
      const long long base = ((long long)b * p.max_splits * p.Qn + qi) * p.Hq + hq;
      float M = -INFINITY;
      for (int sp = 0; sp < R.n_split; ++sp) M = fmaxf(M, __ldcg(&p.ml_part[(base + sp * split_stride) * 2]));
      float L = 0.f, O = 0.f;
      if (M != -INFINITY) {
        for (int sp = 0; sp < R.n_split; ++sp) {
          const long long slot = base + sp * split_stride;
          const float ms = __ldcg(&p.ml_part[slot * 2]);
          const float f = ms == -INFINITY ? 0.f : ptx::ex2((ms - M) * kLog2e);
          L += f * __ldcg(&p.ml_part[slot * 2 + 1]);
          O += f * __ldcg(&p.o_part[slot * kD + d]);
        }
      }
      const long long orow = ((long long)b * p.Qn + qi) * p.Hq + hq;
      p.out[orow * kD + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
      if (p.lse != nullptr && d == 0) p.lse[orow] = L > 0.f ? M + logf(L) : -INFINITY;
    }
    return;
  }
  float* c_ml = s_l + 16;                       // [16][kComboSplits][2]
  float* c_w = c_ml + 16 * kComboSplits * 2;    // [16][kComboSplits] weights
  float* c_ml_row = c_w + 16 * kComboSplits;    // [16][2] merged max and sum
  for (int i = threadIdx.x; i < tile_rows * R.n_split; i += blockDim.x) {
    const int r = i / R.n_split, sp = i - r * R.n_split;
    const int rr = rt * 16 + r;
    const long long slot = ((long long)b * p.max_splits * p.Qn + rr / p.G) * p.Hq + h * p.G + rr % p.G +
                           sp * split_stride;
    c_ml[(r * kComboSplits + sp) * 2] = __ldcg(&p.ml_part[slot * 2]);
    c_ml[(r * kComboSplits + sp) * 2 + 1] = __ldcg(&p.ml_part[slot * 2 + 1]);
  }
  __syncthreads();
  if (threadIdx.x < tile_rows) {
    const int r = threadIdx.x;
    float M = -INFINITY;
    for (int sp = 0; sp < R.n_split; ++sp) M = fmaxf(M, c_ml[(r * kComboSplits + sp) * 2]);
    float L = 0.f;
    for (int sp = 0; sp < R.n_split; ++sp) {
      const float ms = c_ml[(r * kComboSplits + sp) * 2];
      const float f = (M == -INFINITY || ms == -INFINITY) ? 0.f : ptx::ex2((ms - M) * kLog2e);
      c_w[r * kComboSplits + sp] = f;
      L += f * c_ml[(r * kComboSplits + sp) * 2 + 1];
    }
    c_ml_row[r * 2] = M;
    c_ml_row[r * 2 + 1] = L;
  }
  __syncthreads();
#pragma unroll 4
  for (int r = 0; r < tile_rows; ++r) {
    const int rr = rt * 16 + r;
    const int qi = rr / p.G, hq = h * p.G + rr % p.G;
    const long long base = ((long long)b * p.max_splits * p.Qn + qi) * p.Hq + hq;
    float O = 0.f;
    for (int sp = 0; sp < R.n_split; ++sp)
      O = fmaf(c_w[r * kComboSplits + sp], __ldcg(&p.o_part[(base + sp * split_stride) * kD + d]), O);
    const float M = c_ml_row[r * 2], L = c_ml_row[r * 2 + 1];
    const long long orow = ((long long)b * p.Qn + qi) * p.Hq + hq;
    p.out[orow * kD + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
    if (p.lse != nullptr && d == 0) p.lse[orow] = L > 0.f ? M + logf(L) : -INFINITY;
  }
}

}  // namespace

// Clears the split counters of a call.  It lets the split kernel launch at once
// (programmatic dependent launch): that kernel waits for this one only where it first
// touches a counter, after its loads and arithmetic.
__global__ void clear_counters_kernel(int* cnt, long long n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (long long i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    cnt[i] = 0;
}

unsigned read_and_clear_error_decode(cudaStream_t, std::string*) {
  unsigned w = 0, zero = 0;
  cudaMemcpyFromSymbol(&w, g_err_decode, sizeof(w));
  if (w) cudaMemcpyToSymbol(g_err_decode, &zero, sizeof(zero));
  return w;
}

static int mq_max_splits(int Qn, int S, int window_left, int window_right) {
  // Longest union window of a 16-row tile.  Its rows belong to queries i_lo..i_hi
  // (i_hi - i_lo <= 15), so hi - lo <= window_left + min(Q - i_lo, i_hi - i_lo + 1 +
  // window_right) <= window_left + min(Q, window_right + 16); window_left + 1 when Q = 1.
  long long win = S;
  if (window_left >= 0) {
    const long long span = (long long)window_left +
                           (window_right >= 0 ? std::min<long long>(Qn, (long long)window_right + 16) : Qn);
    win = std::min<long long>(win, span);
  }
  return static_cast<int>(std::max<long long>(1, (win + kKeysPerCta - 1) / kKeysPerCta));
}

// Workspace: fp32 partials o [B][splits][Q][Hq][D] and (m, l) [..][2], then the row
// tiles' split counters [B][Hkv][row_tiles], cleared on the stream by each call.
static size_t mq_partials_bytes(int B, int Qn, int Hq, int S, int window_left, int window_right) {
  const size_t splits = mq_max_splits(Qn, S, window_left, window_right);
  return ((size_t)B * splits * Qn * Hq * (kD + 2) * sizeof(float) + 255) & ~static_cast<size_t>(255);
}
static size_t mq_counter_bytes(int B, int Qn, int Hq) {
  // Hkv * ceil(Q * G / 16) <= Q * Hq / 16 + Hkv <= ceil(Q * Hq / 16) + Hq
  return (size_t)B * (((size_t)Qn * Hq + 15) / 16 + Hq) * sizeof(int);
}

size_t ragged_mq_workspace_bytes(int B, int Qn, int Hq, int S, int window_left,
                                 int window_right) {
  return mq_partials_bytes(B, Qn, Hq, S, window_left, window_right) + mq_counter_bytes(B, Qn, Hq);
}

int launch_ragged_mq(const void* q, const void* k, const void* v, const int32_t* seq_start,
                     const int32_t* seq_end, int B, int Qn, int Hq, int Hkv, int S, float scale,
                     int window_left, int window_right, float cap, const float* sink_bias,
                     int num_sinks, int sink_per_head, void* out, float* lse, void* workspace,
                     cudaStream_t stream) {
  // Long chunks without a soft cap or sinks run on the tensor-memory block pipeline
  // (query blocks of 128 rows, two heads of a KV head per item, key blocks of 128).
  if (Qn >= 128 && cap <= 0.f && num_sinks == 0)
    return launch_ragged_chunk(q, k, v, seq_start, seq_end, B, Qn, Hq, Hkv, S, scale, window_left,
                               window_right, out, lse, stream);
  MqParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.seq_start = seq_start;
  p.seq_end = seq_end;
  p.sink_bias = sink_bias;
  p.B = B; p.Qn = Qn; p.Hq = Hq; p.Hkv = Hkv; p.S = S; p.G = Hq / Hkv;
  p.row_tiles = (Qn * p.G + 15) / 16;
  p.max_splits = mq_max_splits(Qn, S, window_left, window_right);
  if ((long long)B * p.row_tiles > 65535 || Hkv > 65535 || Qn > 65535)
    return set_error(SBA_ERR_UNSUPPORTED,
                     "ragged attention: B * ceil(Q * Hq / Hkv / 16), Hkv and Q must be <= 65535");
  p.o_part = static_cast<float*>(workspace);
  p.ml_part = p.o_part + (size_t)B * p.max_splits * Qn * Hq * kD;
  p.tile_count = reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) +
                                        mq_partials_bytes(B, Qn, Hq, S, window_left, window_right));
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.scale = scale;
  p.cap = cap > 0.f ? cap : 0.f;
  p.window_left = window_left;
  p.window_right = window_right;
  p.num_sinks = num_sinks;
  p.sink_per_head = sink_per_head;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaSuccess;
    for (auto fn : {ragged_mq_split_kernel<false, false>, ragged_mq_split_kernel<false, true>,
                    ragged_mq_split_kernel<true, false>, ragged_mq_split_kernel<true, true>})
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return cuda_error(e, "ragged attention: set smem attribute");
    attr_done = true;
  }
  const long long n_cnt = (long long)B * Hkv * p.row_tiles;
  clear_counters_kernel<<<(int)std::min<long long>((n_cnt + 255) / 256, 64), 256, 0, stream>>>(p.tile_count, n_cnt);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "ragged attention: clear split counters");
  dim3 grid(p.max_splits, Hkv, B * p.row_tiles);
  const bool hi_rows = Qn * p.G > 8, capped = p.cap > 0.f;
  auto kernel = hi_rows ? (capped ? ragged_mq_split_kernel<true, true> : ragged_mq_split_kernel<true, false>)
                        : (capped ? ragged_mq_split_kernel<false, true> : ragged_mq_split_kernel<false, false>);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kWarps * 32);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, p);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "ragged attention split launch");
  return SBA_OK;
}


// Single-token decode: the Q = 1 case (the query at end - 1; a right window never cuts).
size_t decode_workspace_bytes(int B, int Hq, int S, int D, int window_left) {
  (void)D;
  return ragged_mq_workspace_bytes(B, 1, Hq, S, window_left, -1);
}

int launch_ragged_decode(const void* q, const void* k, const void* v, const int32_t* seq_start,
                         const int32_t* seq_end, int B, int Hq, int Hkv, int S, int D,
                         float scale, int window_left, int window_right, float cap,
                         const float* sink_bias, int num_sinks, int sink_per_head, void* out,
                         float* lse, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
  (void)D;
  (void)workspace_bytes;
  return launch_ragged_mq(q, k, v, seq_start, seq_end, B, 1, Hq, Hkv, S, scale, window_left,
                          window_right, cap, sink_bias, num_sinks, sink_per_head, out, lse,
                          workspace, stream);
}

}  // namespace sba

// ---------------------------------------------------------------------------------------
// Decode without caller-provided workspace.
//
// Some callers cannot allocate device memory at call time: a host application whose
// device memory is owned by another allocator with a fixed budget, a plugin interface
// that hands the library nothing but its input and output buffers, or a serving loop
// that must not take the device-wide synchronisation a cudaMalloc/cudaFree can cause.
// For them the split partials live in a fixed array inside the library.  Every GPU that
// loads the library reserves this array until the process exits, and every call on a
// device shares it.
namespace sba {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB of fp32 partials
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The array's name in host
// code is only a host-side stand-in, so the address is looked up once per device (with
// that device current) and cached.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "sba_ragged_decode_fwd_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(SBA_ERR_UNSUPPORTED, "sba_ragged_decode_fwd_noalloc: device ordinal >= 64");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return cuda_error(e, "sba_ragged_decode_fwd_noalloc: cudaGetSymbolAddress(scratch)");
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return SBA_OK;
}

}  // namespace
}  // namespace sba

extern "C" SBA_API int sba_ragged_decode_fwd_noalloc(
    const void* q, const void* k, const void* v, const int32_t* seq_start, const int32_t* seq_end,
    int B, int Hq, int Hkv, int S, int D, float softmax_scale, int window_left, int window_right,
    float logits_soft_cap, const float* sink_bias, int num_sinks, int sink_bias_per_head,
    void* out, float* lse, sba_stream_t stream) {
  using namespace sba;
  const size_t need = sba_ragged_decode_workspace_size(B, Hq, S, D, window_left);
  if (need > kNoAllocScratchBytes)
    return set_error(SBA_ERR_INVALID_ARG,
                     "sba_ragged_decode_fwd_noalloc: these sizes need " + std::to_string(need) +
                         " bytes of split partials, more than the built-in " +
                         std::to_string(kNoAllocScratchBytes) +
                         " bytes; use sba_ragged_decode_fwd with a workspace");
  void* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != SBA_OK) return rc;
  // The partials need no initialisation: every slot the combining CTA reads is written
  // by the same call, and the call clears the split counters itself (a kernel on the
  // stream, no allocation).
  return sba_ragged_decode_fwd(q, k, v, seq_start, seq_end, B, Hq, Hkv, S, D, softmax_scale,
                               window_left, window_right, logits_soft_cap, sink_bias, num_sinks,
                               sink_bias_per_head, out, lse, scratch, kNoAllocScratchBytes, stream);
}
