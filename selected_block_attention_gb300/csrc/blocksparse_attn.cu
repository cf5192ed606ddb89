// Attention over SparseMask block bounds, for sm_103a.
//
// Follows "ejkernel.kernels._triton.blocksparse_attention._mask" (module source page),
// module docstring and SparseMask docstring: for each query block only the key blocks
// in [lower, upper) are computed, and blocks in [lower_full, upper_full) need no
// per-token mask.  The token mask used elsewhere (same segment, neither padding,
// causal and inclusive window on positions) is applied to every other block.
//
// Work item = (batch row, query block of 128 tokens, query head).  A persistent CTA
// per SM runs a warp-specialised pipeline:
//   warp 0      producer: TMA loads of the Q tile, then per key block of the item's
//               range the K and V tiles plus the block's positions / segment ids
//               (bulk copy) into a shared-memory ring;
//   warp 1      MMA issuer (one thread): S = Q K^T (M = 128 queries, N = key block,
//               fp32 in TMEM, double-buffered), O += P V (N = head dim, O kept in
//               TMEM for the whole item);
//   warps 4..7  softmax warpgroup, one thread per query row: mask, online softmax
//               with a lazy rescale (O in TMEM is rescaled only when the running max
//               grows by more than 2^8), P to shared memory in the 128-byte-swizzled
//               K-major layout the MMA reads, and the epilogue O / l, LSE.
#include <cuda_bf16.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace sba {

static __device__ DevError g_err_bsa = {0u, 0u, 0};

namespace {

using namespace ptx;

constexpr int kThreads = 256;
constexpr int kM = 128;  // query rows per tile
constexpr int kItemSlots = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Item {
  int b, hq, qblk;
  int lo, up, lof, upf;
};

struct Params {
  const int* q_pos;
  const int* q_seg;
  const int* kv_pos;
  const int* kv_seg;
  const int* lower;
  const int* upper;
  const int* lower_full;
  const int* upper_full;
  __nv_bfloat16* out;
  float* lse;
  int B, T, Hq, Hkv, G, nbq, causal, window_left, window_right, pad_id;
  float scale_log2;
  int n_items;
};

template <int D, int KB>
struct Cfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kQPanelBytes = kM * 128;
  static constexpr int kQBytes = kPanels * kQPanelBytes;
  static constexpr int kKVPanelBytes = KB * 128;
  static constexpr int kKVTileBytes = kPanels * kKVPanelBytes;
  static constexpr int kPosSegBytes = 2 * KB * 4;
  static constexpr int kStageBytes = 2 * kKVTileBytes + 1024;  // K, V, positions/segments (1024-padded)
  static constexpr int kStages = (kStageBytes <= 40 * 1024) ? 3 : 2;
  static constexpr int kPPanels = KB / 64;
  static constexpr int kPBytes = kPPanels * kM * 128;
  static constexpr int kTmemCols = (2 * KB + D <= 256) ? 256 : 512;
  static constexpr int kOCol = 2 * KB;
  static constexpr uint32_t kIdescQK = make_idesc(128, KB, 1u, false, false);
  static constexpr uint32_t kIdescPV = make_idesc(128, D, 1u, false, true);
  static constexpr int kOffQ = 0;
  static constexpr int kOffStages = kOffQ + kQBytes;
  static constexpr int kOffP = kOffStages + kStages * kStageBytes;
  static constexpr int kOffItems = kOffP + kPBytes;
  static constexpr int kOffBars = kOffItems + kItemSlots * (int)sizeof(Item) + 64;
  static constexpr int kNumBars = 2 * kItemSlots + 2 + 2 * kStages + 4 + 3 + 2;
  static constexpr int kOffMisc = ((kOffBars + kNumBars * 8) + 15) & ~15;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

enum Role : unsigned { kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3 };
enum BarId : unsigned {
  kBarItemFull = 1, kBarItemEmpty, kBarQFull, kBarQEmpty, kBarKvFull, kBarKvEmpty, kBarSFull,
  kBarSEmpty, kBarPFull, kBarPvDone, kBarOEmpty, kBarWg
};

__device__ __forceinline__ void decode_item(const Params& p, int item, int& b, int& hq, int& qblk) {
  const int g = item % p.G;
  int r = item / p.G;
  qblk = r % p.nbq;
  r /= p.nbq;
  const int hkv = r % p.Hkv;
  b = r / p.Hkv;
  hq = hkv * p.G + g;
}

template <int D, int KB>
__global__ void __launch_bounds__(kThreads, 1)
blocksparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<D, KB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Item* items = reinterpret_cast<Item*>(smem + C::kOffItems);
  uint64_t* bb = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* item_full = bb;            bb += kItemSlots;
  uint64_t* item_empty = bb;           bb += kItemSlots;
  uint64_t* q_full = bb;               bb += 1;
  uint64_t* q_empty = bb;              bb += 1;
  uint64_t* kv_full = bb;              bb += C::kStages;
  uint64_t* kv_empty = bb;             bb += C::kStages;
  uint64_t* s_full = bb;               bb += 2;
  uint64_t* s_empty = bb;              bb += 2;
  uint64_t* p_full = bb;               bb += 1;
  uint64_t* pv_done = bb;              bb += 1;
  uint64_t* o_empty = bb;              bb += 1;
  uint64_t* mma_done = bb;             bb += 1;
  uint64_t* wg_bar = bb;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const Abort ab{abort_flag, &g_err_bsa, 2u};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kItemSlots; ++i) { mbar_init(&item_full[i], 1); mbar_init(&item_empty[i], 2); }
    mbar_init(q_full, 1); mbar_init(q_empty, 1);
    for (int i = 0; i < C::kStages; ++i) { mbar_init(&kv_full[i], 1); mbar_init(&kv_empty[i], 1); }
    for (int i = 0; i < 2; ++i) { mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], 4); }
    mbar_init(p_full, 4); mbar_init(pv_done, 1); mbar_init(o_empty, 4); mbar_init(mma_done, 1);
    mbar_init(wg_bar, 4);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
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
    // ------------------------------------------------------------------ producer
    int islot = 0; uint32_t iphase = 0;
    uint32_t qphase = 0;
    int stage = 0; uint32_t kvphase = 0;
    bool kv_issued[4] = {false, false, false, false};
    uint32_t last_kv_parity[4] = {0, 0, 0, 0};
    bool q_issued = false;
    uint32_t last_q_parity = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
      int b, hq, qblk;
      decode_item(p, item, b, hq, qblk);
      const long long brow = (long long)b * p.nbq + qblk;
      int lo = p.lower[brow], up = p.upper[brow], lof = p.lower_full[brow], upf = p.upper_full[brow];
      const int nbkv = p.T / KB;
      lo = max(lo, 0);
      up = min(up, nbkv);
      if (!warp_wait(&item_empty[islot], iphase ^ 1, ab, kRoleProducer, kBarItemEmpty, item)) break;
      if (lane == 0) {
        Item& it = items[islot];
        it.b = b; it.hq = hq; it.qblk = qblk; it.lo = lo; it.up = up; it.lof = lof; it.upf = upf;
        mbar_arrive(&item_full[islot]);
      }
      __syncwarp();
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
      if (up <= lo) continue;
      const int hkv = hq / p.G;
      if (!warp_wait(q_empty, qphase ^ 1, ab, kRoleProducer, kBarQEmpty, item)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, C::kQBytes);
#pragma unroll
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_3d(smem + C::kOffQ + pn * C::kQPanelBytes, &tm_q, q_full, pn * 64, hq,
                      b * p.T + qblk * kM);
      }
      q_issued = true;
      last_q_parity = qphase;
      qphase ^= 1;
      for (int blk = lo; blk < up; ++blk) {
        if (!warp_wait(&kv_empty[stage], kvphase ^ 1, ab, kRoleProducer, kBarKvEmpty, item)) { ok = false; break; }
        if (lane == 0) {
          uint64_t* fb = &kv_full[stage];
          mbar_arrive_expect_tx(fb, 2 * C::kKVTileBytes + C::kPosSegBytes);
          uint8_t* kdst = smem + C::kOffStages + stage * C::kStageBytes;
          uint8_t* vdst = kdst + C::kKVTileBytes;
          uint8_t* ps = vdst + C::kKVTileBytes;
          const int tok0 = b * p.T + blk * KB;
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn) {
            tma_load_3d(kdst + pn * C::kKVPanelBytes, &tm_k, fb, pn * 64, hkv, tok0);
            tma_load_3d(vdst + pn * C::kKVPanelBytes, &tm_v, fb, pn * 64, hkv, tok0);
          }
          bulk_load(ps, p.kv_pos + tok0, KB * 4, fb);
          bulk_load(ps + KB * 4, p.kv_seg + tok0, KB * 4, fb);
        }
        kv_issued[stage] = true;
        last_kv_parity[stage] = kvphase;
        if (++stage == C::kStages) { stage = 0; kvphase ^= 1; }
      }
    }
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s)
        if (kv_issued[s]) drain_wait(&kv_full[s], last_kv_parity[s]);
      if (q_issued) drain_wait(q_full, last_q_parity);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int islot = 0; uint32_t iphase = 0;
      uint32_t qphase = 0;
      int stage = 0; uint32_t kvphase = 0;
      int sbuf = 0; uint32_t sphase = 0;
      uint32_t pphase = 0, ophase = 0;
      int pending_stage = -1;
      bool pending_first = false;
      int cur_item = -1;
      bool ok = true;
      auto issue_pv = [&](int st, bool first) -> bool {
        if (!bounded_wait(p_full, pphase, ab, kRoleMma, kBarPFull, cur_item)) return false;
        pphase ^= 1;
        if (first) {
          if (!bounded_wait(o_empty, ophase ^ 1, ab, kRoleMma, kBarOEmpty, cur_item)) return false;
          ophase ^= 1;
        }
        tc_fence_after();
        const uint32_t v_addr = smem_base + C::kOffStages + st * C::kStageBytes + C::kKVTileBytes;
        const uint32_t p_addr = smem_base + C::kOffP;
#pragma unroll
        for (int k = 0; k < KB / 16; ++k) {
          const uint64_t a = make_sdesc(p_addr + (k / 4) * (kM * 128) + (k % 4) * 32, 16, 1024, kLayoutSW128);
          const uint64_t bd = make_sdesc(v_addr + k * 16 * 128, C::kKVPanelBytes, 1024, kLayoutSW128);
          mma_f16_ss(tmem + C::kOCol, a, bd, C::kIdescPV, (first && k == 0) ? 0u : 1u);
        }
        mma_commit(&kv_empty[st]);
        mma_commit(pv_done);
        return true;
      };
      for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        cur_item = item;
        if (!bounded_wait(&item_full[islot], iphase, ab, kRoleMma, kBarItemFull, item)) break;
        const int n = items[islot].up - items[islot].lo;
        if (n <= 0 && pending_stage >= 0) {
          // nothing to compute: release the deferred PV now so the softmax group, which
          // waits for it before finishing the previous item, never starves
          if (!issue_pv(pending_stage, pending_first)) break;
          pending_stage = -1;
        }
        if (n > 0) {
          if (!bounded_wait(q_full, qphase, ab, kRoleMma, kBarQFull, item)) break;
          qphase ^= 1;
        }
        for (int i = 0; i < n; ++i) {
          if (!bounded_wait(&kv_full[stage], kvphase, ab, kRoleMma, kBarKvFull, item) ||
              !bounded_wait(&s_empty[sbuf], sphase ^ 1, ab, kRoleMma, kBarSEmpty, item)) { ok = false; break; }
          tc_fence_after();
          const uint32_t k_addr = smem_base + C::kOffStages + stage * C::kStageBytes;
          const uint32_t q_addr = smem_base + C::kOffQ;
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const int pn = k / 4, kk = k % 4;
            const uint64_t a = make_sdesc(q_addr + pn * C::kQPanelBytes + kk * 32, 16, 1024, kLayoutSW128);
            const uint64_t bd = make_sdesc(k_addr + pn * C::kKVPanelBytes + kk * 32, 16, 1024, kLayoutSW128);
            mma_f16_ss(tmem + sbuf * KB, a, bd, C::kIdescQK, k > 0);
          }
          mma_commit(&s_full[sbuf]);
          if (i == n - 1) mma_commit(q_empty);
          if (pending_stage >= 0 && !issue_pv(pending_stage, pending_first)) { ok = false; break; }
          pending_stage = stage;
          pending_first = (i == 0);
          if (++stage == C::kStages) { stage = 0; kvphase ^= 1; }
          if (++sbuf == 2) { sbuf = 0; sphase ^= 1; }
        }
        if (!ok) break;
        mbar_arrive(&item_empty[islot]);
        if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
      }
      if (ok && pending_stage >= 0) issue_pv(pending_stage, pending_first);
      mma_commit(mma_done);
      drain_wait(mma_done, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    const int q4 = warp - 4;
    const int r = q4 * 32 + lane;  // query row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    int islot = 0; uint32_t iphase = 0;
    int stage = 0; uint32_t kvphase = 0;
    int sbuf = 0; uint32_t sphase = 0;
    uint32_t pvphase = 0;
    uint32_t wg_phase = 0;
    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
      if (!warp_wait(&item_full[islot], iphase, ab, kRoleSoftmax, kBarItemFull, item)) break;
      const Item it = items[islot];
      const int n = it.up - it.lo;
      const int t = it.qblk * kM + r;
      const long long orow = ((long long)it.b * p.T + t) * p.Hq + it.hq;
      const int qp = p.q_pos[(long long)it.b * p.T + t];
      const int qs = p.q_seg[(long long)it.b * p.T + t];
      const bool q_pad = qs == p.pad_id;
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      for (int i = 0; i < n; ++i) {
        const int blk = it.lo + i;
        if (!warp_wait(&s_full[sbuf], sphase, ab, kRoleSoftmax, kBarSFull, item)) { ok = false; break; }
        tc_fence_after();
        float x[KB];
#pragma unroll
        for (int c = 0; c < KB / 32; ++c) tmem_ld_32x32b_x32(tmem + lane_off + sbuf * KB + c * 32, x + c * 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[sbuf]);
        if (++sbuf == 2) { sbuf = 0; sphase ^= 1; }
        const bool full = blk >= it.lof && blk < it.upf;
        // the block's positions / segment ids arrived with the K/V tiles of this stage
        if (!warp_wait(&kv_full[stage], kvphase, ab, kRoleSoftmax, kBarKvFull, item)) { ok = false; break; }
        float tmax = -INFINITY;
        if (full) {
#pragma unroll
          for (int j = 0; j < KB; ++j) { x[j] *= p.scale_log2; tmax = fmaxf(tmax, x[j]); }
        } else {
          const int* ps = reinterpret_cast<const int*>(smem + C::kOffStages + stage * C::kStageBytes + 2 * C::kKVTileBytes);
#pragma unroll
          for (int j = 0; j < KB; j += 4) {
            const int4 kp4 = *reinterpret_cast<const int4*>(ps + j);
            const int4 ks4 = *reinterpret_cast<const int4*>(ps + KB + j);
            const int kp[4] = {kp4.x, kp4.y, kp4.z, kp4.w};
            const int ks[4] = {ks4.x, ks4.y, ks4.z, ks4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              bool ok_k = !q_pad && ks[u] == qs;
              if (p.causal) ok_k = ok_k && kp[u] <= qp;
              if (p.window_left >= 0) ok_k = ok_k && (long long)qp - kp[u] <= p.window_left;
              if (p.window_right >= 0) ok_k = ok_k && (long long)kp[u] - qp <= p.window_right;
              x[j + u] = ok_k ? x[j + u] * p.scale_log2 : -INFINITY;
              tmax = fmaxf(tmax, x[j + u]);
            }
          }
        }
        if (++stage == C::kStages) { stage = 0; kvphase ^= 1; }
        // lazy online softmax: move the reference max only when it grows by > 2^8
        float m_new = m;
        if (tmax > m + kRescaleThreshold || (m == -INFINITY && tmax != -INFINITY)) m_new = tmax;
        const float alpha = (m == -INFINITY || m_new == m) ? (m_new == m ? 1.f : 0.f) : ex2(m - m_new);
        float psum = 0.f;
        if (m_new == -INFINITY) {
#pragma unroll
          for (int j = 0; j < KB; ++j) x[j] = 0.f;
        } else {
#pragma unroll
          for (int j = 0; j < KB; ++j) { x[j] = ex2(x[j] - m_new); psum += x[j]; }
        }
        l = l * alpha + psum;
        // previous PV must be done: P buffer reusable and O stable
        if (i > 0) {
          if (!warp_wait(pv_done, pvphase, ab, kRoleSoftmax, kBarPvDone, item)) { ok = false; break; }
          pvphase ^= 1;
          tc_fence_after();
          // TMEM loads/stores are warp-collective (.sync.aligned): the whole warp rescales
          // together when any of its rows moved its reference max; other rows use 1.
          const bool my_rescale = m_new != m && m != -INFINITY;
          if (__any_sync(0xffffffffu, my_rescale)) {
            const float f = my_rescale ? alpha : 1.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              float ov[32];
              tmem_ld_32x32b_x32(tmem + lane_off + C::kOCol + c * 32, ov);
#pragma unroll
              for (int j = 0; j < 32; ++j) ov[j] *= f;
              tmem_st_32x32b_x32(tmem + lane_off + C::kOCol + c * 32, ov);
            }
          }
        }
        m = m_new;
        // P row (bf16) -> shared memory, 128-byte swizzled K-major panels of 64 keys
        const uint32_t prow = smem_base + C::kOffP + r * 128;
#pragma unroll
        for (int pp = 0; pp < C::kPPanels; ++pp) {
#pragma unroll
          for (int cchunk = 0; cchunk < 8; ++cchunk) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(x[pp * 64 + cchunk * 8 + 2 * u],
                                                        x[pp * 64 + cchunk * 8 + 2 * u + 1]);
              w[u] = *reinterpret_cast<uint32_t*>(&h2);
            }
            st_shared_v4(prow + pp * (kM * 128) + ((cchunk ^ (r & 7)) * 16), w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full);
      }
      if (!ok) break;
      __nv_bfloat16* orow_ptr = p.out + orow * D;
      if (n > 0) {
        if (!warp_wait(pv_done, pvphase, ab, kRoleSoftmax, kBarPvDone, item)) break;
        pvphase ^= 1;
        tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::kOCol + c * 32, ov);
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              __nv_bfloat162 h2 = __floats2bfloat162_rn(ov[j + 2 * u] * inv, ov[j + 2 * u + 1] * inv);
              w[u] = *reinterpret_cast<uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(orow_ptr + c * 32 + j) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_empty);
        if (p.lse != nullptr) p.lse[orow] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      } else {
#pragma unroll
        for (int j = 0; j < D; j += 8)
          *reinterpret_cast<uint4*>(orow_ptr + j) = make_uint4(0u, 0u, 0u, 0u);
        if (p.lse != nullptr) p.lse[orow] = -INFINITY;
      }
      if (!warps_barrier(wg_bar, wg_phase, ab, kRoleSoftmax, kBarWg, item)) break;
      if (r == 0) mbar_arrive(&item_empty[islot]);
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <int D, int KB>
int launch_impl(const void* q, const void* k, const void* v, const Params& p, cudaStream_t stream) {
  using C = Cfg<D, KB>;
  CUtensorMap tq, tk, tv;
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.B * p.T};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hq * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kM};
    if (encode_tensor_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "blocksparse_attn: tensor map (q) failed");
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hkv, (cuuint64_t)p.B * p.T};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hkv * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)KB};
    if (encode_tensor_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "blocksparse_attn: tensor map (k/v) failed");
  }
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(blocksparse_attn_kernel<D, KB>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return cuda_error(e, "blocksparse_attn: set smem attribute");
    attr_done = true;
  }
  const int grid = std::min(p.n_items, num_sms());
  blocksparse_attn_kernel<D, KB><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "blocksparse_attn launch");
  return SBA_OK;
}

}  // namespace

unsigned read_and_clear_error_blocksparse(cudaStream_t, std::string* where) {
  DevError w{0u, 0u, 0}, zero{0u, 0u, 0};
  cudaMemcpyFromSymbol(&w, g_err_bsa, sizeof(w));
  if (w.flags) {
    cudaMemcpyToSymbol(g_err_bsa, &zero, sizeof(zero));
    if (where && w.where) {
      char buf[96];
      snprintf(buf, sizeof(buf), " [blocksparse_attn role %u barrier %u item %d]",
               (w.where >> 16) & 0xFFu, w.where & 0xFFFFu, w.item);
      *where += buf;
    }
  }
  return w.flags;
}

int launch_blocksparse_attn(const void* q, const void* k, const void* v, const int32_t* q_pos,
                            const int32_t* q_seg, const int32_t* kv_pos, const int32_t* kv_seg,
                            const int32_t* lower, const int32_t* upper, const int32_t* lower_full,
                            const int32_t* upper_full, int B, int T, int Hq, int Hkv, int D,
                            int q_block, int kv_block, int causal, int window_left,
                            int window_right, int pad_id, float scale, void* out, float* lse,
                            cudaStream_t stream) {
  (void)q_block;
  Params p;
  p.q_pos = q_pos; p.q_seg = q_seg; p.kv_pos = kv_pos; p.kv_seg = kv_seg;
  p.lower = lower; p.upper = upper; p.lower_full = lower_full; p.upper_full = upper_full;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.B = B; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv;
  p.nbq = T / kM;
  p.causal = causal;
  p.window_left = window_left;
  p.window_right = window_right;
  p.pad_id = pad_id;
  p.scale_log2 = scale * kLog2e;
  const long long n_items = (long long)B * Hq * p.nbq;
  if (n_items >= (1LL << 31)) return set_error(SBA_ERR_UNSUPPORTED, "blocksparse_attn: too many items");
  p.n_items = static_cast<int>(n_items);
  if (D == 128 && kv_block == 128) return launch_impl<128, 128>(q, k, v, p, stream);
  if (D == 128 && kv_block == 64) return launch_impl<128, 64>(q, k, v, p, stream);
  if (D == 64 && kv_block == 128) return launch_impl<64, 128>(q, k, v, p, stream);
  return launch_impl<64, 64>(q, k, v, p, stream);
}

}  // namespace sba
