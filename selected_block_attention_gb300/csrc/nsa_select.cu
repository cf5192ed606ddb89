// Native-sparse-attention forward, selection branch, for sm_103a.
//
// Follows "ejkernel.modules.operations.native_sparse_attention" (operation API page),
// NativeSparseAttention.run / native_sparse_attention: each query token attends, per
// KV head, only to the key blocks named by block_indices[b, t, h_kv, :count]; the G
// query heads of a KV head share its keys (GQA); cu_seqlens packs sequences.
//
// bf16 path (tensor cores).  Work item = one (token, KV head) "token group".  A
// persistent CTA per SM walks the items with a warp-specialised pipeline:
//   warp 0      producer: filters/deduplicates the token's block list (one index per
//               lane), then TMA-gathers the selected K and V blocks into a shared-memory
//               ring (128 keys per tile = 128 / block_size blocks; a missing block is
//               fetched from beyond the last token, which TMA fills with zeros) and the
//               token's G query rows;
//   warp 1      MMA issuer (one thread): S^T = K_tile * Q^T with tcgen05
//               (M = 128 keys, N = 16 query heads, fp32 accumulator in TMEM), then
//               O_tile^T = V_tile^T * P^T (M = 128 head-dim rows, N = 16);
//   warps 4..7  softmax warpgroup: one thread per key lane reads its 16 head scores
//               from TMEM, masks (causal, sequence end, padding block), finds per-head
//               tile maxima by a warp reduce-scatter plus a shared-memory exchange,
//               writes P^T (bf16) for the PV MMA, and folds each O_tile (one thread per
//               head-dim lane) into a register accumulator with the online-softmax
//               rescale; finally writes O / l and the natural-log LSE.
// Keys sit on the MMA M dimension and the query heads of one KV head on N, so every
// gathered block feeds a dense MMA with no padded rows.
//
// fp32 path (CUDA cores, exact fp32 products and sums): one CTA per token group.
// Tensor cores would round fp32 inputs to tf32, which is not accurate enough for the
// float32 contract, and the fp32 workloads are small.
#include <cuda_bf16.h>

#include <cmath>

#include "common.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace sba {

static __device__ DevError g_err_nsa = {0u, 0u, 0};

namespace {

using namespace ptx;

constexpr int kThreads = 256;
constexpr int kTileKeys = 128;  // MMA M of the S^T product (keys)
constexpr int kNH = 16;         // MMA N (query heads of one KV head, padded)
constexpr int kMaxSel = 32;
constexpr int kItemSlots = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

enum Role : unsigned { kRoleProducer = 1, kRoleMma = 2, kRoleSoftmax = 3 };
enum BarId : unsigned {
  kBarItemFull = 1, kBarItemEmpty, kBarQFull, kBarQEmpty, kBarKvFull, kBarKvEmpty, kBarSFull,
  kBarSEmpty, kBarPFull, kBarPEmpty, kBarOFull, kBarOEmpty, kBarWg
};

struct Item {
  int tok;       // global token row b * T + t
  int hkv;
  int t_rel;     // position inside the token's sequence
  int seq_len;
  int seq_tok0;  // global token row of the sequence start
  int n_blocks;  // selected blocks after filtering
  int blocks[kMaxSel];
};

struct Params {
  const int* block_indices;
  const int* block_counts;
  const int* cu_seqlens;
  void* out;
  float* lse;
  int count_scalar, S, num_seqs;
  int B, T, Hq, Hkv, G, causal, bs;
  float scale, scale_log2;
  int n_items, n_tok;
};

template <int D, int BS>
struct Cfg {
  static constexpr int kPanels = D * 2 / 128;            // 128-byte panels per row
  static constexpr int kPanelBytes = kTileKeys * 128;    // 16 KB: one panel of a tile
  static constexpr int kTileBytes = kPanels * kPanelBytes;
  static constexpr int kStageBytes = 2 * kTileBytes;     // [V tile][K tile]
  static constexpr int kStages = (kStageBytes <= 32 * 1024) ? 5 : 3;
  static constexpr int kQPanelBytes = kNH * 128;         // 2 KB
  static constexpr int kQBytes = kPanels * kQPanelBytes;
  static constexpr int kPBytes = kTileKeys * kNH * 2;
  static constexpr int kBlocksPerTile = kTileKeys / BS;
  static constexpr int kQKSteps = D / 16;
  static constexpr int kPVSteps = kTileKeys / 16;
  static constexpr int kPLbo = 256;                      // P^T: stride of 8-key groups
  static constexpr uint32_t kIdescQK = make_idesc(128, kNH, 1u, false, false);
  static constexpr uint32_t kIdescPV = make_idesc(128, kNH, 1u, true, true);
  static constexpr int kOffStages = 0;
  static constexpr int kOffQ = kStages * kStageBytes;
  static constexpr int kOffP = kOffQ + 2 * kQBytes;
  static constexpr int kOffItems = kOffP + 2 * kPBytes;
  static constexpr int kOffRed = kOffItems + kItemSlots * (int)sizeof(Item);
  static constexpr int kOffBars = kOffRed + 2 * 4 * kNH * 4;
  static constexpr int kNumBars = 2 * kItemSlots + 4 + 2 * kStages + 12 + 2;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Bars {
  uint64_t* item_full;   // [kItemSlots]
  uint64_t* item_empty;  // [kItemSlots]
  uint64_t* q_full;      // [2]
  uint64_t* q_empty;     // [2]
  uint64_t* kv_full;     // [kStages]
  uint64_t* kv_empty;    // [kStages]
  uint64_t* s_full;      // [2]
  uint64_t* s_empty;     // [2]
  uint64_t* p_full;      // [2]
  uint64_t* p_empty;     // [2]
  uint64_t* o_full;      // [2]
  uint64_t* o_empty;     // [2]
  uint64_t* mma_done;    // [1]
  uint64_t* wg;          // [1] softmax warpgroup barrier
};

__device__ __forceinline__ void decode_item(const Params& p, int item, int& b, int& hkv, int& t) {
  t = item % p.T;
  const int r = item / p.T;
  hkv = r % p.Hkv;
  b = r / p.Hkv;
}

// Reduce 16 per-lane values over the 32 lanes of a warp (max or sum); on return lane
// L holds the result for head (L >> 1) & 15.
template <bool kMax>
__device__ __forceinline__ float warp_reduce_scatter16(const float* v, int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float a[8], b4[4], c2[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float send = u16 ? v[j] : v[j + 8];
    const float keep = u16 ? v[j + 8] : v[j];
    a[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float send = u8 ? a[j] : a[j + 4];
    const float keep = u8 ? a[j + 4] : a[j];
    b4[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const float send = u4 ? b4[j] : b4[j + 2];
    const float keep = u4 ? b4[j + 2] : b4[j];
    c2[j] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  const float send = u2 ? c2[0] : c2[1];
  const float keep = u2 ? c2[1] : c2[0];
  float d = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  return op(d, __shfl_xor_sync(0xffffffffu, d, 1));
}

// Sequence of token t (cu_seqlens may be NULL): start row, length, position inside.
// Returns false (and flags the input error) when cu_seqlens is malformed.
__device__ __forceinline__ bool locate_token(const Params& p, int b, int t, int& cached_seq,
                                             int& seq_tok0, int& seq_len, int& t_rel) {
  seq_tok0 = b * p.T;
  seq_len = p.T;
  t_rel = t;
  if (p.cu_seqlens == nullptr) return true;
  int s = cached_seq;
  int c0 = p.cu_seqlens[s], c1 = p.cu_seqlens[s + 1];
  if (!(c0 <= t && t < c1)) {
    int lo = 0, hi = p.num_seqs;  // largest s with cu[s] <= t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.cu_seqlens[mid] <= t) lo = mid; else hi = mid;
    }
    s = lo;
    c0 = p.cu_seqlens[s];
    c1 = p.cu_seqlens[s + 1];
  }
  if (!(c0 <= t && t < c1) || p.cu_seqlens[0] != 0 || p.cu_seqlens[p.num_seqs] != p.T) {
    atomicOr(&g_err_nsa.flags, kDevErrInput);
    return false;
  }
  cached_seq = s;
  seq_tok0 = c0;
  seq_len = c1 - c0;
  t_rel = t - c0;
  return true;
}

// Filter + deduplicate the token's block list across one warp (lane i reads entry i).
// Returns the ballot of surviving lanes; `e` is this lane's block id.
__device__ __forceinline__ unsigned select_blocks(const Params& p, long long row, int count,
                                                  int seq_len, int t_rel, int bs, int lane, int& e) {
  const int nb = (seq_len + bs - 1) / bs;
  e = -1;
  if (lane < count) e = p.block_indices[row * p.S + lane];
  bool valid = lane < count && e >= 0 && e < nb && (!p.causal || e * bs <= t_rel);
  bool dup = false;
  for (int j = 0; j < kMaxSel; ++j) {
    const int ej = __shfl_sync(0xffffffffu, e, j);
    const bool vj = __shfl_sync(0xffffffffu, valid, j);
    if (j < lane && vj && ej == e) dup = true;
  }
  return __ballot_sync(0xffffffffu, valid && !dup);
}

template <int D, int BS>
__global__ void __launch_bounds__(kThreads, 1)
nsa_select_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<D, BS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Item* items = reinterpret_cast<Item*>(smem + C::kOffItems);
  float* red = reinterpret_cast<float*>(smem + C::kOffRed);  // [2][4][16]
  uint64_t* bar_base = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const Abort ab{abort_flag, &g_err_nsa, 1u};

  Bars bars;
  {
    uint64_t* b = bar_base;
    bars.item_full = b; b += kItemSlots;
    bars.item_empty = b; b += kItemSlots;
    bars.q_full = b; b += 2;
    bars.q_empty = b; b += 2;
    bars.kv_full = b; b += C::kStages;
    bars.kv_empty = b; b += C::kStages;
    bars.s_full = b; b += 2;
    bars.s_empty = b; b += 2;
    bars.p_full = b; b += 2;
    bars.p_empty = b; b += 2;
    bars.o_full = b; b += 2;
    bars.o_empty = b; b += 2;
    bars.mma_done = b; b += 1;
    bars.wg = b;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kItemSlots; ++i) { mbar_init(&bars.item_full[i], 1); mbar_init(&bars.item_empty[i], 2); }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1); mbar_init(&bars.q_empty[i], 1);
      mbar_init(&bars.s_full[i], 1); mbar_init(&bars.s_empty[i], 4);
      mbar_init(&bars.p_full[i], 4); mbar_init(&bars.p_empty[i], 1);
      mbar_init(&bars.o_full[i], 1); mbar_init(&bars.o_empty[i], 4);
    }
    for (int i = 0; i < C::kStages; ++i) { mbar_init(&bars.kv_full[i], 1); mbar_init(&bars.kv_empty[i], 1); }
    mbar_init(bars.mma_done, 1);
    mbar_init(bars.wg, 4);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 64);
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
    int qslot = 0; uint32_t qphase = 0;
    int stage = 0; uint32_t kvphase = 0;
    uint32_t last_kv_parity[8];
    bool kv_issued[8];
    bool q_issued[2] = {false, false};
    uint32_t last_q_parity[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < 8; ++i) { kv_issued[i] = false; last_kv_parity[i] = 0; }
    int cached_seq = 0;
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
      int b, hkv, t;
      decode_item(p, item, b, hkv, t);
      int seq_tok0, seq_len, t_rel;
      const bool seq_ok = locate_token(p, b, t, cached_seq, seq_tok0, seq_len, t_rel);
      const long long row = ((long long)b * p.T + t) * p.Hkv + hkv;
      int count = p.block_counts ? p.block_counts[row] : p.count_scalar;
      count = seq_ok ? min(max(count, 0), p.S) : 0;
      int e;
      const unsigned ballot = select_blocks(p, row, count, seq_len, t_rel, BS, lane, e);
      const int n_blocks = __popc(ballot);
      if (!warp_wait(&bars.item_empty[islot], iphase ^ 1, ab, kRoleProducer, kBarItemEmpty, item)) break;
      Item& it = items[islot];
      if ((ballot >> lane) & 1u) it.blocks[__popc(ballot & ((1u << lane) - 1u))] = e;
      if (lane == 0) {
        it.tok = b * p.T + t;
        it.hkv = hkv;
        it.t_rel = t_rel;
        it.seq_len = seq_len;
        it.seq_tok0 = seq_tok0;
        it.n_blocks = n_blocks;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.item_full[islot]);
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
      if (n_blocks == 0) continue;

      if (!warp_wait(&bars.q_empty[qslot], qphase ^ 1, ab, kRoleProducer, kBarQEmpty, item)) break;
      if (lane == 0) {
        uint64_t* fb = &bars.q_full[qslot];
        mbar_arrive_expect_tx(fb, C::kQBytes);
        uint8_t* dst = smem + C::kOffQ + qslot * C::kQBytes;
        const int qrow = (b * p.T + t) * p.Hq + hkv * p.G;
#pragma unroll
        for (int pn = 0; pn < C::kPanels; ++pn)
          tma_load_2d(dst + pn * C::kQPanelBytes, &tm_q, fb, pn * 64, qrow);
      }
      q_issued[qslot] = true;
      last_q_parity[qslot] = qphase;
      if (++qslot == 2) { qslot = 0; qphase ^= 1; }

      const int tiles = (n_blocks + C::kBlocksPerTile - 1) / C::kBlocksPerTile;
      for (int ti = 0; ti < tiles; ++ti) {
        if (!warp_wait(&bars.kv_empty[stage], kvphase ^ 1, ab, kRoleProducer, kBarKvEmpty, item)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint64_t* fb = &bars.kv_full[stage];
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          uint8_t* vdst = smem + C::kOffStages + stage * C::kStageBytes;
          uint8_t* kdst = vdst + C::kTileBytes;
#pragma unroll
          for (int sub = 0; sub < C::kBlocksPerTile; ++sub) {
            const int bi = ti * C::kBlocksPerTile + sub;
            // a missing block is read from beyond the last token: TMA fills zeros
            const int tok0 = bi < n_blocks ? seq_tok0 + it.blocks[bi] * BS : p.n_tok;
#pragma unroll
            for (int pn = 0; pn < C::kPanels; ++pn) {
              const int off = pn * C::kPanelBytes + sub * BS * 128;
              tma_load_3d(kdst + off, &tm_k, fb, pn * 64, hkv, tok0);
              tma_load_3d(vdst + off, &tm_v, fb, pn * 64, hkv, tok0);
            }
          }
        }
        kv_issued[stage] = true;
        last_kv_parity[stage] = kvphase;
        if (++stage == C::kStages) { stage = 0; kvphase ^= 1; }
      }
    }
    // Drain: wait (bounded) for every copy this warp issued before the CTA exits.
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s)
        if (kv_issued[s]) drain_wait(&bars.kv_full[s], last_kv_parity[s]);
      for (int s = 0; s < 2; ++s)
        if (q_issued[s]) drain_wait(&bars.q_full[s], last_q_parity[s]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int islot = 0; uint32_t iphase = 0;
      int qslot = 0; uint32_t qphase = 0;
      int stage = 0; uint32_t kvphase = 0;
      int sbuf = 0; uint32_t sphase = 0;
      int pbuf = 0; uint32_t pphase = 0;
      int obuf = 0; uint32_t ophase = 0;
      int pending_stage = -1;
      int cur_item = -1;
      bool ok = true;
      auto issue_pv = [&](int st) -> bool {
        if (!bounded_wait(&bars.p_full[pbuf], pphase, ab, kRoleMma, kBarPFull, cur_item)) return false;
        if (!bounded_wait(&bars.o_empty[obuf], ophase ^ 1, ab, kRoleMma, kBarOEmpty, cur_item)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_base + C::kOffStages + st * C::kStageBytes;
        const uint32_t p_addr = smem_base + C::kOffP + pbuf * C::kPBytes;
        const uint32_t d_tmem = tmem + 32 + obuf * 16;
#pragma unroll
        for (int k = 0; k < C::kPVSteps; ++k) {
          const uint64_t a = make_sdesc(v_addr + k * 16 * 128, C::kPanelBytes, 1024, kLayoutSW128);
          const uint64_t bd = make_sdesc(p_addr + k * 2 * C::kPLbo, C::kPLbo, 128, kLayoutNone);
          mma_f16_ss(d_tmem, a, bd, C::kIdescPV, k > 0);
        }
        mma_commit(&bars.kv_empty[st]);
        mma_commit(&bars.p_empty[pbuf]);
        mma_commit(&bars.o_full[obuf]);
        if (++pbuf == 2) { pbuf = 0; pphase ^= 1; }
        if (++obuf == 2) { obuf = 0; ophase ^= 1; }
        return true;
      };
      for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        cur_item = item;
        if (!bounded_wait(&bars.item_full[islot], iphase, ab, kRoleMma, kBarItemFull, item)) break;
        const int n_blocks = items[islot].n_blocks;
        const int tiles = (n_blocks + C::kBlocksPerTile - 1) / C::kBlocksPerTile;
        if (tiles == 0) {
          // nothing to compute: release the deferred PV now so the softmax group, which
          // waits for it before finishing the previous item, never starves
          if (pending_stage >= 0) {
            if (!issue_pv(pending_stage)) break;
            pending_stage = -1;
          }
          mbar_arrive(&bars.item_empty[islot]);
          if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
          continue;
        }
        if (!bounded_wait(&bars.q_full[qslot], qphase, ab, kRoleMma, kBarQFull, item)) break;
        const uint32_t q_addr = smem_base + C::kOffQ + qslot * C::kQBytes;
        for (int ti = 0; ti < tiles; ++ti) {
          if (!bounded_wait(&bars.kv_full[stage], kvphase, ab, kRoleMma, kBarKvFull, item) ||
              !bounded_wait(&bars.s_empty[sbuf], sphase ^ 1, ab, kRoleMma, kBarSEmpty, item)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t k_addr = smem_base + C::kOffStages + stage * C::kStageBytes + C::kTileBytes;
          const uint32_t d_tmem = tmem + sbuf * 16;
#pragma unroll
          for (int k = 0; k < C::kQKSteps; ++k) {
            const int pn = k / 4, kk = k % 4;
            const uint64_t a = make_sdesc(k_addr + pn * C::kPanelBytes + kk * 32, 16, 1024, kLayoutSW128);
            const uint64_t bd = make_sdesc(q_addr + pn * C::kQPanelBytes + kk * 32, 16, 1024, kLayoutSW128);
            mma_f16_ss(d_tmem, a, bd, C::kIdescQK, k > 0);
          }
          mma_commit(&bars.s_full[sbuf]);
          if (ti == tiles - 1) mma_commit(&bars.q_empty[qslot]);
          if (pending_stage >= 0 && !issue_pv(pending_stage)) { ok = false; break; }
          pending_stage = stage;
          if (++stage == C::kStages) { stage = 0; kvphase ^= 1; }
          if (++sbuf == 2) { sbuf = 0; sphase ^= 1; }
        }
        if (!ok) break;
        mbar_arrive(&bars.item_empty[islot]);
        if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
        if (++qslot == 2) { qslot = 0; qphase ^= 1; }
      }
      if (ok && pending_stage >= 0) issue_pv(pending_stage);
      // every tcgen05 op issued by this thread has finished once mma_done fires
      mma_commit(bars.mma_done);
      drain_wait(bars.mma_done, 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    const int q4 = warp - 4;            // TMEM lane quadrant
    const int r = q4 * 32 + lane;       // key lane (S^T) and head-dim lane (O^T)
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    int islot = 0; uint32_t iphase = 0;
    int sbuf = 0; uint32_t sphase = 0;
    int pbuf = 0; uint32_t pphase = 0;
    int obuf = 0; uint32_t ophase = 0;
    uint32_t wg_phase = 0;
    int par = 0;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
      if (!warp_wait(&bars.item_full[islot], iphase, ab, kRoleSoftmax, kBarItemFull, item)) break;
      const Item& it = items[islot];
      const int n_blocks = it.n_blocks;
      const int tiles = (n_blocks + C::kBlocksPerTile - 1) / C::kBlocksPerTile;
      const int tok = it.tok, hkv = it.hkv, t_rel = it.t_rel, seq_len = it.seq_len;
      const long long out_row0 = (long long)tok * p.Hq + (long long)hkv * p.G;
      float m[kNH], l[kNH], o[kNH], m_acc[kNH], m_pend[kNH];
#pragma unroll
      for (int h = 0; h < kNH; ++h) { m[h] = -INFINITY; l[h] = 0.f; o[h] = 0.f; m_acc[h] = -INFINITY; m_pend[h] = -INFINITY; }
      bool ok = true;
      auto accumulate_o = [&]() -> bool {
        if (!warp_wait(&bars.o_full[obuf], ophase, ab, kRoleSoftmax, kBarOFull, item)) return false;
        tc_fence_after();
        float ov[kNH];
        tmem_ld_32x32b_x16(tmem + lane_off + 32 + obuf * 16, ov);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.o_empty[obuf]);
        if (++obuf == 2) { obuf = 0; ophase ^= 1; }
#pragma unroll
        for (int h = 0; h < kNH; ++h) {
          const float f = m_acc[h] == -INFINITY ? 0.f : ex2(m_acc[h] - m_pend[h]);
          o[h] = o[h] * f + ov[h];
          m_acc[h] = m_pend[h];
        }
        return true;
      };
      for (int ti = 0; ti < tiles; ++ti) {
        if (!warp_wait(&bars.s_full[sbuf], sphase, ab, kRoleSoftmax, kBarSFull, item)) { ok = false; break; }
        tc_fence_after();
        float x[kNH];
        tmem_ld_32x32b_x16(tmem + lane_off + sbuf * 16, x);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.s_empty[sbuf]);
        if (++sbuf == 2) { sbuf = 0; sphase ^= 1; }
        // key of this lane
        const int bi = ti * C::kBlocksPerTile + r / BS;
        const int blk = bi < n_blocks ? it.blocks[bi] : -1;
        const int key = blk * BS + (r % BS);
        const bool valid = blk >= 0 && key < seq_len && (!p.causal || key <= t_rel);
#pragma unroll
        for (int h = 0; h < kNH; ++h) x[h] = valid ? x[h] * p.scale_log2 : -INFINITY;
        // per-head tile maxima over the 128 key lanes
        const float wmax = warp_reduce_scatter16<true>(x, lane);
        if ((lane & 1) == 0) red[(par * 4 + q4) * kNH + (lane >> 1)] = wmax;
        if (!warps_barrier(bars.wg, wg_phase, ab, kRoleSoftmax, kBarWg, item)) { ok = false; break; }
        float tmax[kNH];
#pragma unroll
        for (int h = 0; h < kNH; h += 4) {
          float4 a0 = *reinterpret_cast<const float4*>(&red[(par * 4 + 0) * kNH + h]);
          float4 a1 = *reinterpret_cast<const float4*>(&red[(par * 4 + 1) * kNH + h]);
          float4 a2 = *reinterpret_cast<const float4*>(&red[(par * 4 + 2) * kNH + h]);
          float4 a3 = *reinterpret_cast<const float4*>(&red[(par * 4 + 3) * kNH + h]);
          tmax[h + 0] = fmaxf(fmaxf(a0.x, a1.x), fmaxf(a2.x, a3.x));
          tmax[h + 1] = fmaxf(fmaxf(a0.y, a1.y), fmaxf(a2.y, a3.y));
          tmax[h + 2] = fmaxf(fmaxf(a0.z, a1.z), fmaxf(a2.z, a3.z));
          tmax[h + 3] = fmaxf(fmaxf(a0.w, a1.w), fmaxf(a2.w, a3.w));
        }
        par ^= 1;
        float pv[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h) {
          const float mn = fmaxf(m[h], tmax[h]);
          const float alpha = m[h] == -INFINITY ? 0.f : ex2(m[h] - mn);
          pv[h] = mn == -INFINITY ? 0.f : ex2(x[h] - mn);
          l[h] = l[h] * alpha + pv[h];
          m[h] = mn;
        }
        // P^T row of this key lane -> shared memory (MN-major, 16-byte core rows)
        if (!warp_wait(&bars.p_empty[pbuf], pphase ^ 1, ab, kRoleSoftmax, kBarPEmpty, item)) { ok = false; break; }
        const uint32_t prow = smem_base + C::kOffP + pbuf * C::kPBytes + (r >> 3) * C::kPLbo + (r & 7) * 16;
#pragma unroll
        for (int hg = 0; hg < 2; ++hg) {
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(pv[8 * hg + 2 * j], pv[8 * hg + 2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t*>(&h2);
          }
          st_shared_v4(prow + hg * 128, w[0], w[1], w[2], w[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.p_full[pbuf]);
        if (++pbuf == 2) { pbuf = 0; pphase ^= 1; }
        if (ti > 0 && !accumulate_o()) { ok = false; break; }
#pragma unroll
        for (int h = 0; h < kNH; ++h) m_pend[h] = m[h];
      }
      if (!ok) break;
      if (tiles > 0) {
        if (!accumulate_o()) break;
        // l: sum of the per-lane partial sums over the 128 key lanes
        const float wsum = warp_reduce_scatter16<false>(l, lane);
        if ((lane & 1) == 0) red[(par * 4 + q4) * kNH + (lane >> 1)] = wsum;
        if (!warps_barrier(bars.wg, wg_phase, ab, kRoleSoftmax, kBarWg, item)) break;
        float lt[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h)
          lt[h] = red[(par * 4 + 0) * kNH + h] + red[(par * 4 + 1) * kNH + h] +
                  red[(par * 4 + 2) * kNH + h] + red[(par * 4 + 3) * kNH + h];
        par ^= 1;
        if (r < D) {
#pragma unroll
          for (int h = 0; h < kNH; ++h)
            if (h < p.G) out[(out_row0 + h) * D + r] = __float2bfloat16_rn(o[h] / lt[h]);
        }
        if (p.lse != nullptr && r < p.G) {
          float mr = m[0], lr = lt[0];
#pragma unroll
          for (int h = 1; h < kNH; ++h) if (h == r) { mr = m[h]; lr = lt[h]; }
          p.lse[out_row0 + r] = (mr + log2f(lr)) * kLn2;
        }
      } else {
        if (r < D)
          for (int h = 0; h < p.G; ++h) out[(out_row0 + h) * D + r] = __float2bfloat16_rn(0.f);
        if (p.lse != nullptr && r < p.G) p.lse[out_row0 + r] = -INFINITY;
      }
      // all four warps are done with the item descriptor before it is released
      if (!warps_barrier(bars.wg, wg_phase, ab, kRoleSoftmax, kBarWg, item)) break;
      if (r == 0) mbar_arrive(&bars.item_empty[islot]);
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// ---------------------------------------------------------------------------- fp32
constexpr int kF32Threads = 128;

template <int D>
__global__ void __launch_bounds__(kF32Threads)
nsa_select_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                      const float* __restrict__ v, const Params p) {
  __shared__ float q_s[kNH][D];
  __shared__ float s_s[kNH][kTileKeys + 1];
  __shared__ float m_s[kNH], a_s[kNH];
  __shared__ int blocks_s[kMaxSel];
  __shared__ int meta_s[4];
  const int tid = threadIdx.x, lane = tid & 31;
  float* out = static_cast<float*>(p.out);
  int cached_seq = 0;
  for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
    int b, hkv, t;
    decode_item(p, item, b, hkv, t);
    const long long out_row0 = ((long long)b * p.T + t) * p.Hq + (long long)hkv * p.G;
    __syncthreads();
    if (tid < 32) {
      int seq_tok0, seq_len, t_rel;
      const bool seq_ok = locate_token(p, b, t, cached_seq, seq_tok0, seq_len, t_rel);
      const long long row = ((long long)b * p.T + t) * p.Hkv + hkv;
      int count = p.block_counts ? p.block_counts[row] : p.count_scalar;
      count = seq_ok ? min(max(count, 0), p.S) : 0;
      int e;
      const unsigned ballot = select_blocks(p, row, count, seq_len, t_rel, p.bs, lane, e);
      if ((ballot >> lane) & 1u) blocks_s[__popc(ballot & ((1u << lane) - 1u))] = e;
      if (lane == 0) {
        meta_s[0] = __popc(ballot);
        meta_s[1] = seq_tok0;
        meta_s[2] = t_rel;
        meta_s[3] = seq_len;
      }
    }
    for (int i = tid; i < kNH * D; i += kF32Threads) {
      const int h = i / D, d = i % D;
      q_s[h][d] = h < p.G ? q[(out_row0 + h) * D + d] : 0.f;
    }
    __syncthreads();
    const int n_blocks = meta_s[0], seq_tok0 = meta_s[1], t_rel = meta_s[2], seq_len = meta_s[3];
    const int bsz = p.bs;
    float m_run = -INFINITY, l_run = 0.f;  // valid in threads h < G
    float o[kNH];
#pragma unroll
    for (int h = 0; h < kNH; ++h) o[h] = 0.f;
    for (int bi = 0; bi < n_blocks; ++bi) {
      const int blk = blocks_s[bi];
      // scores: thread j handles key blk * bsz + j
      if (tid < bsz) {
        const int key = blk * bsz + tid;
        const bool valid = key < seq_len && (!p.causal || key <= t_rel);
        float acc[kNH];
#pragma unroll
        for (int h = 0; h < kNH; ++h) acc[h] = 0.f;
        if (valid) {
          const float* kr = k + ((long long)(seq_tok0 + key) * p.Hkv + hkv) * D;
          for (int d = 0; d < D; ++d) {
            const float kd = kr[d];
#pragma unroll
            for (int h = 0; h < kNH; ++h) acc[h] = fmaf(q_s[h][d], kd, acc[h]);
          }
        }
#pragma unroll
        for (int h = 0; h < kNH; ++h) s_s[h][tid] = valid ? acc[h] * p.scale : -INFINITY;
      }
      __syncthreads();
      if (tid >= p.G && tid < kNH) a_s[tid] = 0.f;
      if (tid < p.G) {
        float mx = -INFINITY;
        for (int j = 0; j < bsz; ++j) mx = fmaxf(mx, s_s[tid][j]);
        const float mn = fmaxf(m_run, mx);
        a_s[tid] = m_run == -INFINITY ? 0.f : expf(m_run - mn);
        m_s[tid] = mn;
        m_run = mn;
      }
      __syncthreads();
      for (int i = tid; i < kNH * bsz; i += kF32Threads) {
        const int h = i / bsz, j = i % bsz;
        if (h < p.G) s_s[h][j] = m_s[h] == -INFINITY ? 0.f : expf(s_s[h][j] - m_s[h]);
      }
      __syncthreads();
      if (tid < p.G) {
        float sum = 0.f;
        for (int j = 0; j < bsz; ++j) sum += s_s[tid][j];
        l_run = l_run * a_s[tid] + sum;
      }
      if (tid < D) {
#pragma unroll
        for (int h = 0; h < kNH; ++h) o[h] *= a_s[h];
        for (int j = 0; j < bsz; ++j) {
          const int key = blk * bsz + j;
          if (key >= seq_len || (p.causal && key > t_rel)) break;
          const float vd = v[((long long)(seq_tok0 + key) * p.Hkv + hkv) * D + tid];
#pragma unroll
          for (int h = 0; h < kNH; ++h) o[h] = fmaf(s_s[h][j], vd, o[h]);
        }
      }
      __syncthreads();
    }
    if (tid < p.G) {
      a_s[tid] = l_run;
      m_s[tid] = m_run;
    }
    __syncthreads();
    if (tid < D) {
#pragma unroll
      for (int h = 0; h < kNH; ++h)
        if (h < p.G) out[(out_row0 + h) * D + tid] = a_s[h] > 0.f ? o[h] / a_s[h] : 0.f;
    }
    if (p.lse != nullptr && tid < p.G)
      p.lse[out_row0 + tid] = a_s[tid] > 0.f ? m_s[tid] + logf(a_s[tid]) : -INFINITY;
  }
}

template <int D, int BS>
int launch_bf16(const void* q, const void* k, const void* v, const Params& p, cudaStream_t stream) {
  using C = Cfg<D, BS>;
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tq, tk, tv;
  {
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.B * p.T * p.Hq};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kNH};
    if (encode_tensor_map(&tq, dt, 2, const_cast<void*>(q), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "nsa_select: tensor map (q) failed");
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hkv, (cuuint64_t)p.B * p.T};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hkv * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)BS};
    if (encode_tensor_map(&tk, dt, 3, const_cast<void*>(k), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&tv, dt, 3, const_cast<void*>(v), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "nsa_select: tensor map (k/v) failed");
  }
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(nsa_select_kernel<D, BS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return cuda_error(e, "nsa_select: set smem attribute");
    attr_done = true;
  }
  const int grid = std::min(p.n_items, num_sms());
  nsa_select_kernel<D, BS><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "nsa_select launch");
  return SBA_OK;
}

template <int D>
int dispatch_bs(int bs, const void* q, const void* k, const void* v, const Params& p, cudaStream_t s) {
  switch (bs) {
    case 32: return launch_bf16<D, 32>(q, k, v, p, s);
    case 64: return launch_bf16<D, 64>(q, k, v, p, s);
    case 128: return launch_bf16<D, 128>(q, k, v, p, s);
  }
  return set_error(SBA_ERR_UNSUPPORTED, "nsa_select: block_size");
}

}  // namespace

unsigned read_and_clear_error_nsa(cudaStream_t, std::string* where) {
  DevError w{0u, 0u, 0}, zero{0u, 0u, 0};
  cudaMemcpyFromSymbol(&w, g_err_nsa, sizeof(w));
  if (w.flags) {
    cudaMemcpyToSymbol(g_err_nsa, &zero, sizeof(zero));
    if (where && w.where) {
      char buf[96];
      snprintf(buf, sizeof(buf), " [nsa_select role %u barrier %u item %d]", (w.where >> 16) & 0xFFu,
               w.where & 0xFFFFu, w.item);
      *where += buf;
    }
  }
  return w.flags;
}

int launch_nsa_select(const void* q, const void* k, const void* v, const int32_t* block_indices,
                      const int32_t* block_counts, int block_count_scalar, int S,
                      const int32_t* cu_seqlens, int num_seqs, int B, int T, int Hq, int Hkv,
                      int D, int block_size, int causal, float scale, int dtype, void* out,
                      float* lse, cudaStream_t stream) {
  Params p;
  p.block_indices = block_indices;
  p.block_counts = block_counts;
  p.cu_seqlens = cu_seqlens;
  p.out = out;
  p.lse = lse;
  p.count_scalar = block_count_scalar;
  p.S = S;
  p.num_seqs = num_seqs;
  p.B = B; p.T = T; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv;
  p.causal = causal;
  p.bs = block_size;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  if ((long long)B * T * Hkv >= (1LL << 31)) return set_error(SBA_ERR_UNSUPPORTED, "nsa_select: too many items");
  p.n_items = B * T * Hkv;
  p.n_tok = B * T;
  if (dtype == SBA_BF16) {
    if (D == 128) return dispatch_bs<128>(block_size, q, k, v, p, stream);
    return dispatch_bs<64>(block_size, q, k, v, p, stream);
  }
  const int grid = std::min(p.n_items, 1 << 20);
  if (D == 128)
    nsa_select_f32_kernel<128><<<grid, kF32Threads, 0, stream>>>(
        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v), p);
  else
    nsa_select_f32_kernel<64><<<grid, kF32Threads, 0, stream>>>(
        static_cast<const float*>(q), static_cast<const float*>(k), static_cast<const float*>(v), p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "nsa_select (fp32) launch");
  return SBA_OK;
}

}  // namespace sba
