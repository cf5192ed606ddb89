// Attention over SparseMask block bounds, for sm_103a.
//
// Follows "ejkernel.kernels._triton.blocksparse_attention._mask" (module source page),
// module docstring and SparseMask docstring: for each query block only the key blocks
// in [lower, upper) are computed, and blocks in [lower_full, upper_full) need no
// per-token mask.  The token mask used elsewhere (same segment, neither padding,
// causal and inclusive window on positions) is applied to every other block.
//
// Work item = (batch row, query block of 128 tokens, query head): 128 rows of one
// head.  Its key blocks are walked in tiles of 64 keys.  A persistent CTA per SM runs
// the same warp-specialised pipeline as the NSA selection kernel:
//   warp 0      loader: publishes the item (bounds of its query block), then TMA loads
//               the Q rows (staging buffer) and per tile the K / V boxes plus the tile's
//               key positions and segment ids (bulk copy) into a shared-memory ring;
//   warp 1      QK issuer (one thread): copies Q into tensor memory (tcgen05.cp, in
//               order with its MMAs), S = Q K^T (M = 128, N = 64, A from TMEM);
//   warp 3      PV issuer (one thread): O_w += P_w V (A = P from TMEM);
//   warps 4..11 two softmax warpgroups on alternate tiles, each with its own S buffer,
//               P columns, O accumulator and running (m, l): token mask outside the
//               full block range, lazy online softmax (O rescaled only when the max
//               grows by > 2^8); the epilogue merges the two partial results.
#include <cuda_bf16.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace sba {

static __device__ DevError g_err_bsa = {0u, 0u, 0};

namespace {

using namespace ptx;

constexpr int kThreads = 384;   // warps 0-3: loader, QK issuer, spare, PV issuer; 4-11: softmax
constexpr int kM = 128;         // query rows per item
constexpr int kTileKeys = 64;   // keys per pipeline tile
constexpr int kItemSlots = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Item {
  int b, hq, qblk;
  int lo, up, lof, upf;  // kv blocks [lo, up); [lof, upf) need no token mask
  int n_tiles;
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

enum Role : unsigned { kRoleLoader = 1, kRoleMma = 2, kRoleSoftmax = 3 };
enum BarId : unsigned {
  kBarItemFull = 1, kBarItemEmpty, kBarQFull, kBarQEmpty, kBarKvFull, kBarKvEmpty, kBarSFull,
  kBarSEmpty, kBarPFull, kBarPvDone, kBarOEmpty, kBarXch
};

template <int D, int KB>
struct Cfg {
  static constexpr int kPanels = D / 64;
  static constexpr int kTilesPerBlock = KB / kTileKeys;
  static constexpr int kKVPanelBytes = kTileKeys * 128;    // 8 KB
  static constexpr int kKTileBytes = kPanels * kKVPanelBytes;
  static constexpr int kPosSegBytes = 2 * kTileKeys * 4;
  static constexpr int kLoadBytes = 2 * kKTileBytes + kPosSegBytes;
  static constexpr int kStageBytes = (kLoadBytes + 1023) & ~1023;  // [K][V][positions, segments]
  static constexpr int kQPanelBytes = kM * 128;
  static constexpr int kQBytes = kPanels * kQPanelBytes;
  static constexpr int kItemBytes = (static_cast<int>(sizeof(Item)) + 15) & ~15;
  static constexpr int kMlBytes = 2 * 2 * kM * 8;           // (m, l) per row: [item parity][wg]
  static constexpr int kOffQ = 0;
  static constexpr int kOffStages = kQBytes;
  static constexpr int kFixed = kQBytes + kItemSlots * kItemBytes + kMlBytes + 1024 + 1024;
  static constexpr int kStagesFit = (232448 - kFixed) / kStageBytes;
  static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
  static constexpr int kOffItems = kOffStages + kStages * kStageBytes;
  static constexpr int kOffMl = kOffItems + kItemSlots * kItemBytes;
  static constexpr int kOffBars = (kOffMl + kMlBytes + 7) & ~7;
  static constexpr int kNumBars = 2 * kItemSlots + 3 + 2 * kStages + 8 + 4;
  static constexpr int kOffMisc = ((kOffBars + kNumBars * 8) + 15) & ~15;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;
  // tensor memory columns: S, P and O per warpgroup, Q of the item
  static constexpr int kSCol = 0;                    // S of wg w: 64 fp32 at w * 64
  static constexpr int kOCol = 2 * kTileKeys;        // O of wg w: D fp32 at kOCol + w * D
  static constexpr int kPCol = kOCol + 2 * D;        // P of wg w: 64 bf16 (32 cols) at kPCol + w * 32
  static constexpr int kQCol = kPCol + kTileKeys;    // Q: D bf16 (D / 2 cols)
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kIdescQK = make_idesc(128, kTileKeys, 1u, false, false);
  static constexpr uint32_t kIdescPV = make_idesc(128, D, 1u, false, true);
  static_assert(kStages >= 3, "pipeline depth");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kQCol + D / 2 <= kTmemCols, "tensor memory budget");
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
  float2* ml = reinterpret_cast<float2*>(smem + C::kOffMl);
  uint64_t* bb = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* item_full = bb;   bb += kItemSlots;
  uint64_t* item_empty = bb;  bb += kItemSlots;
  uint64_t* q_full = bb;      bb += 1;   // Q staging loaded
  uint64_t* q_empty = bb;     bb += 1;   // Q staging copied into TMEM
  uint64_t* q_used = bb;      bb += 1;   // last QK of an item done: TMEM Q may be replaced
  uint64_t* kv_full = bb;     bb += C::kStages;
  uint64_t* kv_empty = bb;    bb += C::kStages;
  uint64_t* s_full = bb;      bb += 2;   // per warpgroup
  uint64_t* s_empty = bb;     bb += 2;
  uint64_t* p_full = bb;      bb += 2;
  uint64_t* pv_done = bb;     bb += 2;
  uint64_t* o_empty = bb;     bb += 1;
  uint64_t* mma_done = bb;    bb += 2;   // per issuing thread
  uint64_t* xch = bb;                    // (m, l) exchange between the two warpgroups
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const Abort ab{abort_flag, &g_err_bsa, 2u};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto item_at = [&](int slot) -> Item& {
    return *reinterpret_cast<Item*>(smem + C::kOffItems + slot * C::kItemBytes);
  };

  if (threadIdx.x == 0) {
    // item slots are released by the two MMA threads and the 8 softmax warps
    for (int i = 0; i < kItemSlots; ++i) { mbar_init(&item_full[i], 1); mbar_init(&item_empty[i], 10); }
    mbar_init(q_full, 1); mbar_init(q_empty, 1); mbar_init(q_used, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1); mbar_init(&s_empty[i], 4);
      mbar_init(&p_full[i], 4); mbar_init(&pv_done[i], 1);
    }
    for (int i = 0; i < C::kStages; ++i) { mbar_init(&kv_full[i], 1); mbar_init(&kv_empty[i], 1); }
    mbar_init(o_empty, 8); mbar_init(&mma_done[0], 1); mbar_init(&mma_done[1], 1); mbar_init(xch, 8);
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
    // ------------------------------------------------------------------ loader
    int islot = 0; uint32_t iphase = 0;
    uint32_t qphase = 0;
    int stage = 0; uint32_t kvphase = 0;
    bool kv_issued[8];
    uint32_t last_kv_parity[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) { kv_issued[i] = false; last_kv_parity[i] = 0; }
    bool q_issued = false;
    uint32_t last_q_parity = 0;
    const int nbkv = p.T / KB;
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
      int b, hq, qblk;
      decode_item(p, item, b, hq, qblk);
      const long long brow = (long long)b * p.nbq + qblk;
      const int lo = max(p.lower[brow], 0), up = min(p.upper[brow], nbkv);
      const int lof = p.lower_full[brow], upf = p.upper_full[brow];
      const int nt = up > lo ? (up - lo) * C::kTilesPerBlock : 0;
      if (!warp_wait(&item_empty[islot], iphase ^ 1, ab, kRoleLoader, kBarItemEmpty, item)) break;
      if (lane == 0) {
        Item& it = item_at(islot);
        it.b = b; it.hq = hq; it.qblk = qblk;
        it.lo = lo; it.up = up; it.lof = lof; it.upf = upf; it.n_tiles = nt;
        mbar_arrive(&item_full[islot]);
      }
      __syncwarp();
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
      if (nt == 0) continue;
      const int hkv = hq / p.G;
      if (!warp_wait(q_empty, qphase ^ 1, ab, kRoleLoader, kBarQEmpty, item)) break;
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
      for (int t = 0; t < nt; ++t) {
        if (!warp_wait(&kv_empty[stage], kvphase ^ 1, ab, kRoleLoader, kBarKvEmpty, item)) { ok = false; break; }
        if (lane == 0) {
          uint64_t* fb = &kv_full[stage];
          mbar_arrive_expect_tx(fb, C::kLoadBytes);
          uint8_t* kdst = smem + C::kOffStages + stage * C::kStageBytes;
          uint8_t* vdst = kdst + C::kKTileBytes;
          uint8_t* ps = vdst + C::kKTileBytes;
          const int tok0 = b * p.T + lo * KB + t * kTileKeys;
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn) {
            tma_load_3d(kdst + pn * C::kKVPanelBytes, &tm_k, fb, pn * 64, hkv, tok0);
            tma_load_3d(vdst + pn * C::kKVPanelBytes, &tm_v, fb, pn * 64, hkv, tok0);
          }
          bulk_load(ps, p.kv_pos + tok0, kTileKeys * 4, fb);
          bulk_load(ps + kTileKeys * 4, p.kv_seg + tok0, kTileKeys * 4, fb);
        }
        kv_issued[stage] = true;
        last_kv_parity[stage] = kvphase;
        if (++stage == C::kStages) { stage = 0; kvphase ^= 1; }
      }
    }
    // Drain: wait (bounded) for every copy this warp issued before the CTA exits.
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s)
        if (kv_issued[s]) drain_wait(&kv_full[s], last_kv_parity[s]);
      if (q_issued) drain_wait(q_full, last_q_parity);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ QK issuer
    // Two threads issue the MMAs (QK here, PV in warp 3): a thread's wait on a barrier
    // stalls only its own stream while the tensor core runs the other's MMAs.
    if (lane == 0) {
      int islot = 0; uint32_t iphase = 0;
      uint32_t qphase = 0, quphase = 0;
      bool q_in_use = false;  // a QK of an earlier item may still read the TMEM copy of Q
      int stage = 0; uint32_t kvphase = 0;
      uint32_t sph[2] = {0u, 0u};
      bool ok = true;
      const uint64_t q_desc0 = make_sdesc(smem_base + C::kOffQ, 16, 1024, kLayoutSW128);
      const uint64_t k_desc0 = make_sdesc(smem_base + C::kOffStages, 16, 1024, kLayoutSW128);
      for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        if (!bounded_wait(&item_full[islot], iphase, ab, kRoleMma, kBarItemFull, item)) break;
        const int nt = item_at(islot).n_tiles;
        mbar_arrive(&item_empty[islot]);
        if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
        if (nt == 0) continue;
        if (!bounded_wait(q_full, qphase, ab, kRoleMma, kBarQFull, item)) break;
        qphase ^= 1;
        if (q_in_use) {
          if (!bounded_wait(q_used, quphase, ab, kRoleMma, kBarQEmpty, item)) break;
          quphase ^= 1;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tmem_cp_128x256b(tmem + C::kQCol + kk * 8,
                           q_desc0 + static_cast<uint64_t>(((kk / 4) * C::kQPanelBytes + (kk % 4) * 32) >> 4));
        mma_commit(q_empty);
        for (int t = 0; t < nt; ++t) {
          const int w = t & 1;
          if (!bounded_wait(&kv_full[stage], kvphase, ab, kRoleMma, kBarKvFull, item) ||
              !bounded_wait(&s_empty[w], sph[w] ^ 1, ab, kRoleMma, kBarSEmpty, item)) { ok = false; break; }
          sph[w] ^= 1;
          tc_fence_after();
          const uint64_t kd = k_desc0 + static_cast<uint64_t>((stage * C::kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_f16_ts(tmem + C::kSCol + w * kTileKeys, tmem + C::kQCol + kk * 8,
                       kd + static_cast<uint64_t>(((kk / 4) * C::kKVPanelBytes + (kk % 4) * 32) >> 4),
                       C::kIdescQK, kk > 0);
          mma_commit(&s_full[w]);
          if (t == nt - 1) {
            mma_commit(q_used);
            q_in_use = true;
          }
          if (++stage == C::kStages) { stage = 0; kvphase ^= 1; }
        }
      }
      mma_commit(&mma_done[0]);
      drain_wait(&mma_done[0], 0);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------------ PV issuer
    if (lane == 0) {
      int islot = 0; uint32_t iphase = 0;
      int stage = 0;
      uint32_t pph[2] = {0u, 0u};
      uint32_t ophase = 0;
      bool ok = true;
      const uint64_t v_desc0 =
          make_sdesc(smem_base + C::kOffStages + C::kKTileBytes, C::kKVPanelBytes, 1024, kLayoutSW128);
      for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        if (!bounded_wait(&item_full[islot], iphase, ab, kRoleMma, kBarItemFull, item)) break;
        const int nt = item_at(islot).n_tiles;
        mbar_arrive(&item_empty[islot]);
        if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
        // PV of tile t (A = P of warpgroup t & 1 in TMEM, B = V tile) goes to the O
        // accumulator of warpgroup t & 1; each warpgroup's first tile of an item
        // overwrites it.  A PV follows its tile's softmax, which follows the tile's QK,
        // so the stage is free once the PV is done.
        for (int t = 0; t < nt; ++t) {
          const int w = t & 1;
          if (!bounded_wait(&p_full[w], pph[w], ab, kRoleMma, kBarPFull, item)) { ok = false; break; }
          pph[w] ^= 1;
          if (t == 0) {
            if (!bounded_wait(o_empty, ophase ^ 1, ab, kRoleMma, kBarOEmpty, item)) { ok = false; break; }
            ophase ^= 1;
          }
          tc_fence_after();
          const uint64_t vd = v_desc0 + static_cast<uint64_t>((stage * C::kStageBytes) >> 4);
#pragma unroll
          for (int k = 0; k < kTileKeys / 16; ++k)
            mma_f16_ts(tmem + C::kOCol + w * D, tmem + C::kPCol + w * (kTileKeys / 2) + k * 8,
                       vd + static_cast<uint64_t>((k * 16 * 128) >> 4), C::kIdescPV,
                       (t < 2 && k == 0) ? 0u : 1u);
          mma_commit(&kv_empty[stage]);
          mma_commit(&pv_done[w]);
          if (++stage == C::kStages) stage = 0;
        }
      }
      mma_commit(&mma_done[1]);
      drain_wait(&mma_done[1], 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    const int w = (warp - 4) >> 2;   // warpgroup: tiles t with t & 1 == w
    const int q4 = warp & 3;         // TMEM lane quadrant of this warp
    const int r = q4 * 32 + lane;    // query row of the item = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t s_col = tmem + lane_off + C::kSCol + w * kTileKeys;
    const uint32_t o_col = tmem + lane_off + C::kOCol + w * D;
    const uint32_t p_col = tmem + lane_off + C::kPCol + w * (kTileKeys / 2);
    int islot = 0; uint32_t iphase = 0;
    int stage = 0; uint32_t kvphase = 0;
    uint32_t sph = 0, pvph = 0, xph = 0;
    int par = 0;
    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
      if (!warp_wait(&item_full[islot], iphase, ab, kRoleSoftmax, kBarItemFull, item)) break;
      const Item it = item_at(islot);
      const int nt = it.n_tiles;
      const long long tok = (long long)it.b * p.T + it.qblk * kM + r;
      const int qp = p.q_pos[tok];
      const int qs = p.q_seg[tok];
      const bool q_pad = qs == p.pad_id;
      float m = -INFINITY, l = 0.f;  // log2 units, lazily moved reference max
      int mine = 0;                  // tiles of this item handled by this warpgroup so far
      bool ok = true;
      for (int t = 0; t < nt; ++t) {
        if ((t & 1) != w) {
          if (++stage == C::kStages) { stage = 0; kvphase ^= 1; }
          continue;
        }
        const int blk = it.lo + t / C::kTilesPerBlock;
        const bool full = blk >= it.lof && blk < it.upf;
        if (!warp_wait(&s_full[w], sph, ab, kRoleSoftmax, kBarSFull, item)) { ok = false; break; }
        sph ^= 1;
        float x[kTileKeys];
        tc_fence_after();
        tmem_ld_32x32b_x32(s_col, x);
        tmem_ld_32x32b_x32(s_col + 32, x + 32);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[w]);
        if (!full) {
          // the tile's key positions / segment ids arrived with its K / V
          if (!warp_wait(&kv_full[stage], kvphase, ab, kRoleSoftmax, kBarKvFull, item)) { ok = false; break; }
          const int* ps = reinterpret_cast<const int*>(smem + C::kOffStages + stage * C::kStageBytes +
                                                       2 * C::kKTileBytes);
#pragma unroll
          for (int j = 0; j < kTileKeys; j += 4) {
            const int4 kp4 = *reinterpret_cast<const int4*>(ps + j);
            const int4 ks4 = *reinterpret_cast<const int4*>(ps + kTileKeys + j);
            const int kp[4] = {kp4.x, kp4.y, kp4.z, kp4.w};
            const int ks[4] = {ks4.x, ks4.y, ks4.z, ks4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              bool ok_k = !q_pad && ks[u] == qs;
              if (p.causal) ok_k = ok_k && kp[u] <= qp;
              if (p.window_left >= 0) ok_k = ok_k && (long long)qp - kp[u] <= p.window_left;
              if (p.window_right >= 0) ok_k = ok_k && (long long)kp[u] - qp <= p.window_right;
              if (!ok_k) x[j + u] = -INFINITY;
            }
          }
        }
        if (++stage == C::kStages) { stage = 0; kvphase ^= 1; }
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < kTileKeys; ++j) mx[j & 3] = fmaxf(mx[j & 3], x[j]);
        const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.scale_log2;
        // lazy online softmax: move the reference max only when it grows by > 2^8
        float m_new = m;
        if (tmax > m + kRescaleThreshold || (m == -INFINITY && tmax != -INFINITY)) m_new = tmax;
        const float alpha = (m == -INFINITY || m_new == m) ? (m_new == m ? 1.f : 0.f) : ex2(m - m_new);
        float psum = 0.f;
        if (m_new == -INFINITY) {
#pragma unroll
          for (int j = 0; j < kTileKeys; ++j) x[j] = 0.f;
        } else {
          float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < kTileKeys; ++j) {
            x[j] = ex2(fmaf(x[j], p.scale_log2, -m_new));
            ps4[j & 3] += x[j];
          }
          psum = (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
        }
        l = l * alpha + psum;
        uint32_t pk[kTileKeys / 2];
#pragma unroll
        for (int j = 0; j < kTileKeys / 2; ++j) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(x[2 * j], x[2 * j + 1]);
          pk[j] = *reinterpret_cast<uint32_t*>(&h2);
        }
        // this warpgroup's previous PV must be done before its P is replaced and its O
        // rescaled
        if (mine > 0) {
          if (!warp_wait(&pv_done[w], pvph, ab, kRoleSoftmax, kBarPvDone, item)) { ok = false; break; }
          pvph ^= 1;
          tc_fence_after();
        }
        tmem_st_32x32b_x32_u(p_col, pk);
        if (mine > 0) {
          // TMEM loads/stores are warp-collective (.sync.aligned): the whole warp rescales
          // together when any of its rows moved its reference max; other rows use 1.
          const bool my_rescale = m_new != m && m != -INFINITY;
          if (__any_sync(0xffffffffu, my_rescale)) {
            const float f = my_rescale ? alpha : 1.f;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              float ov[32];
              tmem_ld_32x32b_x32(o_col + c * 32, ov);
#pragma unroll
              for (int j = 0; j < 32; ++j) ov[j] *= f;
              tmem_st_32x32b_x32(o_col + c * 32, ov);
            }
          }
        }
        m = m_new;
        ++mine;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[w]);
      }
      if (!ok) break;
      if (mine > 0) {
        if (!warp_wait(&pv_done[w], pvph, ab, kRoleSoftmax, kBarPvDone, item)) break;
        pvph ^= 1;
      }
      // merge the two warpgroups' partial results row by row
      ml[(par * 2 + w) * kM + r] = make_float2(m, l);
      __syncwarp();
      if (lane == 0) mbar_arrive(xch);
      if (!warp_wait(xch, xph, ab, kRoleSoftmax, kBarXch, item)) break;
      xph ^= 1;
      const float2 oth = ml[(par * 2 + (w ^ 1)) * kM + r];
      const float mxr = fmaxf(m, oth.x);
      const float a_me = l > 0.f ? ex2(m - mxr) : 0.f;
      const float a_ot = oth.y > 0.f ? ex2(oth.x - mxr) : 0.f;
      const float L = l * a_me + oth.y * a_ot;
      const float a0 = w == 0 ? a_me : a_ot, a1 = w == 0 ? a_ot : a_me;
      const float inv = L > 0.f ? 1.f / L : 0.f;
      constexpr int kOutHalf = D / 2;
      __nv_bfloat16* orow = p.out + (tok * p.Hq + it.hq) * D;
      if (nt > 0) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kOutHalf / 32; ++c) {
          const int col = w * kOutHalf + c * 32;
          float o0[32], o1[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::kOCol + col, o0);
          tmem_ld_32x32b_x32(tmem + lane_off + C::kOCol + D + col, o1);
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint32_t wv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              // an accumulator that received no PV this item holds stale data: select
              const int j0 = j + 2 * u;
              const float v0 = ((a0 > 0.f) ? o0[j0] * a0 : 0.f) + ((a1 > 0.f) ? o1[j0] * a1 : 0.f);
              const float v1 = ((a0 > 0.f) ? o0[j0 + 1] * a0 : 0.f) + ((a1 > 0.f) ? o1[j0 + 1] * a1 : 0.f);
              __nv_bfloat162 h2 = __floats2bfloat162_rn(v0 * inv, v1 * inv);
              wv[u] = *reinterpret_cast<uint32_t*>(&h2);
            }
            *reinterpret_cast<uint4*>(orow + col + j) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_empty);
      } else {
#pragma unroll
        for (int j = 0; j < kOutHalf; j += 8)
          *reinterpret_cast<uint4*>(orow + w * kOutHalf + j) = make_uint4(0u, 0u, 0u, 0u);
      }
      if (w == 0 && p.lse != nullptr) p.lse[tok * p.Hq + it.hq] = L > 0.f ? (mxr + log2f(L)) * kLn2 : -INFINITY;
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[islot]);
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
      par ^= 1;
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
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kTileKeys};
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
