// Attention over SparseMask block bounds, for sm_103a.
//
// Follows "ejkernel.kernels._triton.blocksparse_attention._mask" (module source page),
// module docstring and SparseMask docstring: for each query block only the key blocks
// in [lower, upper) are computed, and blocks in [lower_full, upper_full) need no
// per-token mask.  The token mask used elsewhere (same segment, neither padding,
// causal and inclusive window on positions) is applied to every other block.
//
// Work item = (batch row, query block of 128 tokens, KV head, pair of its query heads):
// two 128-row problems that read the same keys / values and share the token mask.  Keys
// are walked in tiles of 64 (a key block of 128 is two tiles).  A persistent CTA per SM
// runs a warp-specialised pipeline:
//   warp 0      loader: publishes the item (its tile range and full-tile range), then TMA
//               loads Q of each head into its own buffer and, per key tile, K into a K
//               ring and V plus the tile's key positions / segment ids into a V ring;
//   warps 1, 2  one MMA-issuing warp per head slot w (converged; an elected lane
//               issues): S_w = Q_w K^T (both operands in shared memory, N = 64 keys) into
//               one of two S buffers of the head, and O_w += P_w V (P_w read from tensor
//               memory over the S buffer it replaced), in the order S(0) S(1) | PV(t)
//               S(t + 2) | ...; so the scores of tile t + 1 are ready while the softmax
//               still works on tile t, and each warp's barrier waits overlap the other
//               head's MMAs;
//   warps 4..7  softmax of head slot 0, warps 8..11 of head slot 1: one thread per query
//               row; the row's 64 scores of a tile come out of tensor memory in one pass
//               into registers, are masked outside the full tile range (an exact per-row
//               key interval when the tile's keys are consecutive positions of at most
//               two segments, else a test per key), and P (bf16) is
//               written in place over the tile's S buffer; lazy online softmax (O_w
//               rescaled only when the row maximum grows by > 2^8, after the previous
//               tile's PV has landed); epilogue: O_w leaves tensor memory at once (the
//               next item's PV may start), O / l in bf16 is staged in shared memory and
//               written by TMA stores.
// Tensor memory: S_w,0 S_w,1 (64 fp32 columns each, P aliased in place) for w = 0, 1,
// then O_0, O_1 (D columns each): 512 columns at D = 128.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace sba {

static __device__ DevError g_err_bsa = {0u, 0u, 0};
// Item counters of the launches: [next item, CTAs done] per slot; launches take the slots
// in turn, so up to kSchedSlots launches (on any streams) may run at once.  Each launch
// finds its slot zero and leaves it zero.
constexpr int kSchedSlots = 64;
static __device__ int g_bsa_sched[2 * kSchedSlots];

namespace {

using namespace ptx;

// Warp 0 loader, warps 1 and 2 MMA issuers (warp 3 idle), warps 4-11 two softmax
// warpgroups.  No register split: a row of 64 scores fits the 168 registers a thread
// of a 384-thread CTA gets.
constexpr int kThreads = 384;
constexpr int kM = 128;         // query rows per head slot
constexpr int kKT = 64;         // keys per tile (N of S = Q K^T, K of O += P V)
constexpr int kItemSlots = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Item {
  int qpos[kM];              // positions / segment ids of the query block's rows (copied in
  int qseg[kM];              // by the loader with the item; SparseMask mode)
  int b, hkv, qblk, h0, nh;  // heads h0 .. h0 + nh - 1 (nh = 1 or 2)
  int tlo, tup, tlof, tupf;  // key tiles [tlo, tup); [tlof, tupf) need no token mask
  int n_tiles;               // = tup - tlo; -1: no more items (the loader's last publication)
  int start, end;            // ragged mode: the row's key range
  int idx;                   // item index (for error reports)
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
  const int* seq_start;  // ragged mode: per batch row [start, end) of the key range
  const int* seq_end;
  __nv_bfloat16* out;
  float* lse;
  int B, T, Hq, Hkv, G, nbq, causal, window_left, window_right, pad_id;
  int q_rows, kv_rows;   // query / key rows per batch row (T and T; ragged: Q and S)
  int kv_block;          // key block of the bounds (64 or 128; ragged: 128)
  float scale_log2;
  int n_pairs, n_items;
  long long wait_limit;  // cycles a bounded wait may take
  int* sched;            // [next item, CTAs done] of this launch (zero at launch, left zero)
};

enum Role : unsigned { kRoleLoader = 1, kRoleMma = 2, kRoleSoftmax = 3 };
enum BarId : unsigned {
  kBarItemFull = 1, kBarItemEmpty, kBarQFull, kBarQEmpty, kBarKFull, kBarKEmpty, kBarVFull,
  kBarVEmpty, kBarSFull, kBarPFull, kBarPvTile, kBarPvLast, kBarOEmpty
};

template <int D>
struct Cfg {
  static constexpr int kPanels = D / 64;                   // 64-element (128-byte) panels
  static constexpr int kQPanelBytes = kM * 128;
  static constexpr int kQBytes = kPanels * kQPanelBytes;   // Q of one head slot
  static constexpr int kTPanelBytes = kKT * 128;
  static constexpr int kTBytes = kPanels * kTPanelBytes;   // K (or V) of one key tile
  static constexpr int kPosSegBytes = 2 * kKT * 4;
  static constexpr int kVStageBytes = (kTBytes + kPosSegBytes + 1023) & ~1023;
  static constexpr int kItemBytes = (static_cast<int>(sizeof(Item)) + 15) & ~15;
  static constexpr int kStages = 3;                        // V ring (V + key positions / segments)
  static constexpr int kStagesK = 2;                       // K ring (a K stage is free once both S MMAs read it)
  // output staging: per softmax warp two halves of 16 rows x D bf16 (one 128-byte
  // swizzled panel per 64 columns each), stored to global memory by TMA; the second half
  // does not wait for the first half's store to leave shared memory
  static constexpr int kStgPanelBytes = 16 * 128;
  static constexpr int kStgHalfBytes = kPanels * kStgPanelBytes;
  static constexpr int kStgWarpBytes = 2 * kStgHalfBytes;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kQBytes;
  static constexpr int kOffV = kOffK + kStagesK * kTBytes;
  static constexpr int kOffStage = kOffV + kStages * kVStageBytes;
  static constexpr int kOffItems = kOffStage + 8 * kStgWarpBytes;
  static constexpr int kOffBars = (kOffItems + kItemSlots * kItemBytes + 7) & ~7;
  static constexpr int kNumBars = 2 * kItemSlots + 4 + 2 * kStagesK + 2 * kStages + 4 + 4 + 2 + 2 + 2 + 2;
  static constexpr int kOffMisc = ((kOffBars + kNumBars * 8) + 15) & ~15;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  // tensor memory columns: S_w,buf at (2 w + buf) * kKT (P aliased), O_w at kOCol + w * D
  static constexpr int kOCol = 4 * kKT;
  static constexpr int kTmemNeed = 4 * kKT + 2 * D;
  static constexpr int kTmemCols = kTmemNeed <= 256 ? 256 : 512;
  static constexpr uint32_t kIdescQK = make_idesc(128, kKT, 1u, false, false);
  static constexpr uint32_t kIdescPV = make_idesc(128, D, 1u, false, true);
  static_assert(kOffStage % 1024 == 0, "staging panels must start on 1024-byte swizzle atoms");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kTmemNeed <= 512, "tensor memory budget");
};

// item = ((b * Hkv + hkv) * nbq + qblk) * n_pairs + pair: consecutive items share K/V
__device__ __forceinline__ void decode_item(const Params& p, int item, int& b, int& hkv, int& qblk,
                                            int& h0, int& nh) {
  const int pair = item % p.n_pairs;
  int r = item / p.n_pairs;
  qblk = r % p.nbq;
  r /= p.nbq;
  hkv = r % p.Hkv;
  b = r / p.Hkv;
  h0 = hkv * p.G + 2 * pair;
  nh = min(2, p.G - 2 * pair);
}

// Scores of a tile outside the column interval [jlo, jhi] set to -inf, the interval held
// as keep bits in two 32-bit words: per score one bit test against a constant and one
// select (a compare of the column against both ends per score costs several times more).
__device__ __forceinline__ void mask_interval(float (&x)[kKT], int jlo, int jhi) {
  static_assert(kKT == 64, "two 32-bit keep words");
  const uint32_t w0 = (jlo <= 31 && jhi >= 0)
      ? ((jhi >= 31 ? 0xffffffffu : ((2u << jhi) - 1u)) & (0xffffffffu << min(max(jlo, 0), 31))) : 0u;
  const uint32_t w1 = (jhi >= 32 && jlo <= 63)
      ? ((jhi >= 63 ? 0xffffffffu : ((2u << (jhi - 32)) - 1u)) & (0xffffffffu << max(jlo - 32, 0))) : 0u;
#pragma unroll
  for (int j = 0; j < 32; ++j) x[j] = (w0 & (1u << j)) ? x[j] : -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) x[32 + j] = (w1 & (1u << j)) ? x[32 + j] : -INFINITY;
}

// Ragged form: key tiles [tlo, tup) of query block qblk of row b and the full ones
// [tlof, tupf): rows i0 .. i1 of the block sit at end - Q + i; their windows' union is
// [kmin(i0), kmax(i1)] and the keys every row sees are [kmin(i1), kmax(i0)].
__device__ __forceinline__ void ragged_tiles(const Params& p, int b, int qblk, int& start, int& end,
                                             int& tlo, int& tup, int& tlof, int& tupf) {
  start = min(max(p.seq_start[b], 0), p.kv_rows);
  end = min(max(p.seq_end[b], 0), p.kv_rows);
  tlo = tup = tlof = tupf = 0;
  const int i0 = qblk * kM, i1 = min(i0 + kM, p.q_rows) - 1;
  auto kmin = [&](int i) -> long long {
    const long long pos = (long long)end - p.q_rows + i;
    return p.window_left >= 0 ? max((long long)start, pos - p.window_left) : (long long)start;
  };
  auto kmax = [&](int i) -> long long {
    const long long pos = (long long)end - p.q_rows + i;
    return p.window_right >= 0 ? min((long long)end - 1, pos + p.window_right) : (long long)end - 1;
  };
  const long long klo = kmin(i0), khi = kmax(i1);
  if (end > start && khi >= klo) {
    tlo = static_cast<int>(klo / kKT);
    tup = static_cast<int>(khi / kKT) + 1;
    const long long flo = kmin(i1), fhi = kmax(i0);
    tlof = static_cast<int>((flo + kKT - 1) / kKT);
    tupf = fhi >= flo ? static_cast<int>((fhi + 1) / kKT) : tlof;
  }
}

// kRagged: the ragged multi-query form of the same computation (queries are the last Q
// tokens of [start, end) of a KV cache, each with its own inclusive window); the key
// range and the full tiles of a query block follow from start, end and the window, and
// the per-row key range replaces the position / segment test.
template <int D, bool kRagged>
__global__ void __launch_bounds__(kThreads, 1)
blocksparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const Params p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bb = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* item_full = bb;   bb += kItemSlots;
  uint64_t* item_empty = bb;  bb += kItemSlots;
  uint64_t* q_full = bb;      bb += 2;   // per head slot
  uint64_t* q_empty = bb;     bb += 2;
  uint64_t* k_full = bb;      bb += C::kStagesK;
  uint64_t* k_empty = bb;     bb += C::kStagesK;
  uint64_t* v_full = bb;      bb += C::kStages;
  uint64_t* v_empty = bb;     bb += C::kStages;
  uint64_t* s_full = bb;      bb += 4;   // [2 w + buf]: S_w of the buffer written
  uint64_t* p_full = bb;      bb += 4;   // [2 w + buf]: P_w stored, O_w rescaled
  uint64_t* pv_tile = bb;     bb += 2;   // each PV_w done
  uint64_t* pv_last = bb;     bb += 2;   // last PV_w of an item done
  uint64_t* o_empty = bb;     bb += 2;   // epilogue has read O_w
  uint64_t* mma_done = bb;    bb += 2;   // teardown: every MMA of issuer w finished
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const Abort ab{abort_flag, &g_err_bsa, 2u, p.wait_limit};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto item_at = [&](int slot) -> Item& {
    return *reinterpret_cast<Item*>(smem + C::kOffItems + slot * C::kItemBytes);
  };

  if (threadIdx.x == 0) {
    // an item slot is read by the two MMA threads and the eight softmax warps; a K / V
    // stage is released by both MMA threads
    for (int i = 0; i < kItemSlots; ++i) { mbar_init(&item_full[i], 1); mbar_init(&item_empty[i], 10); }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&q_full[w], 1); mbar_init(&q_empty[w], 1);
      mbar_init(&pv_tile[w], 1); mbar_init(&pv_last[w], 1);
      mbar_init(&o_empty[w], 4); mbar_init(&mma_done[w], 1);
    }
    for (int i = 0; i < 4; ++i) { mbar_init(&s_full[i], 1); mbar_init(&p_full[i], 4); }
    for (int i = 0; i < C::kStagesK; ++i) { mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 2); }
    for (int i = 0; i < C::kStages; ++i) { mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 2); }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
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
  const int nbkv = (p.kv_rows + p.kv_block - 1) / p.kv_block;

  if (warp == 0) {
    // ------------------------------------------------------------------ loader
    int islot = 0; uint32_t iphase = 0;
    // Per-slot / per-stage flags and phases are bit sets (bit i: slot or stage i): indexed
    // at run time, small arrays would live in local memory.
    uint32_t qphase = 0u, q_issued = 0u, q_last = 0u;
    int ks = 0; uint32_t kphase = 0;
    int vs = 0; uint32_t vphase = 0;
    uint32_t k_issued = 0u, k_last = 0u, v_issued = 0u, v_last = 0u;
    bool ok = true;
    // Items are handed out one at a time from the launch's counter, so a CTA that drew
    // short items takes more: the kernel ends near the average CTA load instead of the
    // heaviest fixed share.  The ragged form hands the largest items out first: with at
    // most 32 (row, query block) groups each lane ranks one group by its tile count (ties
    // by index) and the groups go out in rank order (all KV heads and head pairs of a
    // group together); with at most 32 rows, the rows by clamped length; otherwise items
    // go in index order.  Each CTA's loader ranks once, at the start.
    const int ng = p.B * p.nbq;
    const int by_group = kRagged && ng <= 32 ? 1 : (kRagged && p.B <= 32 ? 2 : 0);
    int of_rank = lane;  // lane r: the group (1) or row (2) of rank r
    if (by_group != 0) {
      const int n = by_group == 1 ? ng : p.B;
      int size = -1;
      if (lane < n) {
        if (by_group == 1) {
          int st, en, t0, t1, f0, f1;
          ragged_tiles(p, lane / p.nbq, lane % p.nbq, st, en, t0, t1, f0, f1);
          size = t1 - t0;
        } else {
          size = max(min(max(p.seq_end[lane], 0), p.kv_rows) - min(max(p.seq_start[lane], 0), p.kv_rows), 0);
        }
      }
      int rank = 0;
      for (int j = 0; j < n; ++j) {
        const int sj = __shfl_sync(0xffffffffu, size, j);
        rank += (sj > size || (sj == size && j < lane)) ? 1 : 0;
      }
      for (int j = 0; j < n; ++j)
        if (__shfl_sync(0xffffffffu, rank, j) == lane) of_rank = j;
    }
    const int per_row = p.Hkv * p.nbq * p.n_pairs, per_group = p.Hkv * p.n_pairs;
    while (ok) {
      int k = 0;
      if (lane == 0) k = atomicAdd(&p.sched[0], 1);
      k = __shfl_sync(0xffffffffu, k, 0);
      int item = k;
      if (by_group == 1 && k < p.n_items) {
        // group (b, qblk) of rank k / per_group; its (hkv, pair) from the remainder
        const int g = __shfl_sync(0xffffffffu, of_rank, k / per_group), rem = k % per_group;
        const int gb = g / p.nbq, gq = g % p.nbq, hkv = rem / p.n_pairs, pair = rem % p.n_pairs;
        item = ((gb * p.Hkv + hkv) * p.nbq + gq) * p.n_pairs + pair;
      } else if (by_group == 2 && k < p.n_items) {
        item = __shfl_sync(0xffffffffu, of_rank, k / per_row) * per_row + k % per_row;
      }
      if (k >= p.n_items) {
        // no more items: publish the end marker
        if (!warp_wait(&item_empty[islot], iphase ^ 1, ab, kRoleLoader, kBarItemEmpty, item)) break;
        if (lane == 0) {
          item_at(islot).n_tiles = -1;
          mbar_arrive(&item_full[islot]);
        }
        __syncwarp();
        break;
      }
      int b, hkv, qblk, h0, nh;
      decode_item(p, item, b, hkv, qblk, h0, nh);
      int tlo = 0, tup = 0, tlof = 0, tupf = 0, start = 0, end = 0;
      if constexpr (kRagged) {
        ragged_tiles(p, b, qblk, start, end, tlo, tup, tlof, tupf);
      } else {
        // block bounds in tiles: a key block of kv_block keys is kv_block / kKT tiles
        const int tpb = p.kv_block / kKT;
        const long long brow = (long long)b * p.nbq + qblk;
        const int lo = max(p.lower[brow], 0), up = min(p.upper[brow], nbkv);
        if (up > lo) {
          tlo = lo * tpb;
          tup = up * tpb;
          tlof = p.lower_full[brow] * tpb;
          tupf = p.upper_full[brow] * tpb;
        }
      }
      const int nt = tup > tlo ? tup - tlo : 0;
      if (!warp_wait(&item_empty[islot], iphase ^ 1, ab, kRoleLoader, kBarItemEmpty, item)) break;
      if (lane == 0) {
        Item& it = item_at(islot);
        it.b = b; it.hkv = hkv; it.qblk = qblk; it.h0 = h0; it.nh = nh;
        it.tlo = tlo; it.tup = tup; it.tlof = tlof; it.tupf = tupf;
        it.n_tiles = nt;
        it.start = start; it.end = end;
        it.idx = item;
        if (!kRagged && nt > 0) {
          // the rows' positions and segment ids ride on the item barrier
          const long long row0 = (long long)b * p.q_rows + qblk * kM;
          bulk_load(it.qpos, p.q_pos + row0, kM * 4, &item_full[islot]);
          bulk_load(it.qseg, p.q_seg + row0, kM * 4, &item_full[islot]);
          mbar_arrive_expect_tx(&item_full[islot], 2 * kM * 4);
        } else {
          mbar_arrive(&item_full[islot]);
        }
      }
      __syncwarp();
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
      if (nt == 0) continue;
      for (int w = 0; w < nh; ++w) {
        if (!warp_wait(&q_empty[w], ((qphase >> w) & 1u) ^ 1u, ab, kRoleLoader, kBarQEmpty, item)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&q_full[w], C::kQBytes);
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smem + C::kOffQ + w * C::kQBytes + pn * C::kQPanelBytes, &tm_q, &q_full[w],
                        pn * 64, h0 + w, b * p.q_rows + qblk * kM);
        }
        q_issued |= 1u << w;
        q_last = (q_last & ~(1u << w)) | (qphase & (1u << w));
        qphase ^= 1u << w;
      }
      if (!ok) break;
      for (int t = 0; t < nt; ++t) {
        const int tok0 = b * p.kv_rows + (tlo + t) * kKT;
        if (!warp_wait(&k_empty[ks], kphase ^ 1, ab, kRoleLoader, kBarKEmpty, item)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&k_full[ks], C::kTBytes);
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smem + C::kOffK + ks * C::kTBytes + pn * C::kTPanelBytes, &tm_k, &k_full[ks],
                        pn * 64, hkv, tok0);
        }
        k_issued |= 1u << ks;
        k_last = (k_last & ~(1u << ks)) | (kphase << ks);
        if (++ks == C::kStagesK) { ks = 0; kphase ^= 1; }
        if (!warp_wait(&v_empty[vs], vphase ^ 1, ab, kRoleLoader, kBarVEmpty, item)) { ok = false; break; }
        if (lane == 0) {
          uint8_t* vdst = smem + C::kOffV + vs * C::kVStageBytes;
          mbar_arrive_expect_tx(&v_full[vs], C::kTBytes + (kRagged ? 0 : C::kPosSegBytes));
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(vdst + pn * C::kTPanelBytes, &tm_v, &v_full[vs], pn * 64, hkv, tok0);
          if (!kRagged) {
            bulk_load(vdst + C::kTBytes, p.kv_pos + tok0, kKT * 4, &v_full[vs]);
            bulk_load(vdst + C::kTBytes + kKT * 4, p.kv_seg + tok0, kKT * 4, &v_full[vs]);
          }
        }
        v_issued |= 1u << vs;
        v_last = (v_last & ~(1u << vs)) | (vphase << vs);
        if (++vs == C::kStages) { vs = 0; vphase ^= 1; }
      }
    }
    // Drain: wait (bounded) for every copy this warp issued before the CTA exits.
    if (lane == 0) {
      for (int s = 0; s < C::kStagesK; ++s)
        if ((k_issued >> s) & 1u) drain_wait(&k_full[s], (k_last >> s) & 1u);
      for (int s = 0; s < C::kStages; ++s)
        if ((v_issued >> s) & 1u) drain_wait(&v_full[s], (v_last >> s) & 1u);
      for (int w = 0; w < 2; ++w)
        if ((q_issued >> w) & 1u) drain_wait(&q_full[w], (q_last >> w) & 1u);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------------ MMA issuer of head slot w
    // The whole warp runs the loop (converged); one elected lane issues the MMAs and
    // commits, lane 0 the plain arrivals.
    {
      const int w = warp - 1;
      const uint32_t leader = elect_one();
      int islot = 0; uint32_t iphase = 0;
      uint32_t qph = 0u, oph = 0u, pph = 0u;  // pph: P-full phase of S buffer i in bit i
      int ks = 0; uint32_t kphase = 0;   // next K tile to consume (for an S)
      int vs = 0; uint32_t vphase = 0;   // next V tile to consume (for a PV)
      bool ok = true;
      // descriptors of the shared-memory operands; a byte offset x adds x >> 4
      const uint64_t q_desc = make_sdesc(smem_base + C::kOffQ + w * C::kQBytes, 16, 1024, kLayoutSW128);
      const uint64_t k_desc0 = make_sdesc(smem_base + C::kOffK, 16, 1024, kLayoutSW128);
      const uint64_t v_desc0 = make_sdesc(smem_base + C::kOffV, C::kTPanelBytes, 1024, kLayoutSW128);
      const uint32_t o_tmem = tmem + C::kOCol + w * D;
      auto s_tmem = [&](int buf) { return tmem + (2 * w + buf) * kKT; };
      auto kstep = [](int kk, int panel_bytes) -> uint64_t {
        return static_cast<uint64_t>(((kk / 4) * panel_bytes + (kk % 4) * 32) >> 4);
      };
      auto next_k = [&]() { if (++ks == C::kStagesK) { ks = 0; kphase ^= 1; } };
      auto next_v = [&]() { if (++vs == C::kStages) { vs = 0; vphase ^= 1; } };
      // S_w,buf = Q_w K^T of the next K tile, then release the K stage
      auto issue_s = [&](int buf, int item) -> bool {
        if (!warp_wait(&k_full[ks], kphase, ab, kRoleMma, kBarKFull, item)) return false;
        tc_fence_after();
        const uint64_t kd = k_desc0 + static_cast<uint64_t>((ks * C::kTBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16_ss_by(leader, s_tmem(buf), q_desc + kstep(kk, C::kQPanelBytes), kd + kstep(kk, C::kTPanelBytes),
                     C::kIdescQK, kk > 0 ? 1u : 0u);
        mma_commit_by(leader, &s_full[2 * w + buf]);
        mma_commit_by(leader, &k_empty[ks]);
        next_k();
        return true;
      };
      while (ok) {
        if (!warp_wait(&item_full[islot], iphase, ab, kRoleMma, kBarItemFull, -1)) break;
        const int nt = item_at(islot).n_tiles, nh = item_at(islot).nh, item = item_at(islot).idx;
        if (nt < 0) break;  // no more items
        if (lane == 0) mbar_arrive(&item_empty[islot]);
        if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
        if (nt == 0) continue;
        if (w >= nh) {
          // no head in this slot: release each K / V stage once it has been loaded, so
          // the rings stay in step with the loader and the other MMA thread
          for (int t = 0; t < nt && ok; ++t) {
            if (!warp_wait(&k_full[ks], kphase, ab, kRoleMma, kBarKFull, item)) { ok = false; break; }
            if (lane == 0) mbar_arrive(&k_empty[ks]);
            next_k();
            if (!warp_wait(&v_full[vs], vphase, ab, kRoleMma, kBarVFull, item)) { ok = false; break; }
            if (lane == 0) mbar_arrive(&v_empty[vs]);
            next_v();
          }
          continue;
        }
        if (!warp_wait(&q_full[w], qph, ab, kRoleMma, kBarQFull, item)) break;
        qph ^= 1;
        // S of tiles 0 and 1 into the two buffers
        for (int t = 0; t < 2 && t < nt && ok; ++t) {
          if (!issue_s(t, item)) { ok = false; break; }
          if (t == nt - 1) mma_commit_by(leader, &q_empty[w]);
        }
        for (int t = 0; t < nt && ok; ++t) {
          const int buf = t & 1;
          if (!warp_wait(&v_full[vs], vphase, ab, kRoleMma, kBarVFull, item)) { ok = false; break; }
          if (t == 0) {
            if (!warp_wait(&o_empty[w], oph ^ 1, ab, kRoleMma, kBarOEmpty, item)) { ok = false; break; }
            oph ^= 1;
          }
          if (!warp_wait(&p_full[2 * w + buf], (pph >> buf) & 1u, ab, kRoleMma, kBarPFull, item)) { ok = false; break; }
          pph ^= 1u << buf;
          tc_fence_after();
          // O_w (+)= P_w V of this tile (P_w: bf16 pairs over the S_w,buf columns)
          const uint64_t vd = v_desc0 + static_cast<uint64_t>((vs * C::kVStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < kKT / 16; ++kk)
            mma_f16_ts_by(leader, o_tmem, s_tmem(buf) + kk * 8, vd + static_cast<uint64_t>((kk * 16 * 128) >> 4),
                       C::kIdescPV, (t == 0 && kk == 0) ? 0u : 1u);
          mma_commit_by(leader, &pv_tile[w]);
          if (t == nt - 1) mma_commit_by(leader, &pv_last[w]);
          mma_commit_by(leader, &v_empty[vs]);
          next_v();
          // S of tile t + 2 into the buffer PV(t) has just read (issued after it, so it
          // overwrites P only once the PV has consumed it)
          if (t + 2 < nt) {
            if (!issue_s(buf, item)) { ok = false; break; }
            if (t + 2 == nt - 1) mma_commit_by(leader, &q_empty[w]);
          }
        }
      }
      // every tcgen05 op issued by this thread has finished once mma_done fires
      mma_commit_by(leader, &mma_done[w]);
      drain_wait(&mma_done[w], 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    const int w = (warp - 4) >> 2;   // head slot of this warpgroup
    const int q4 = warp & 3;         // TMEM lane quadrant of this warp
    const int r = q4 * 32 + lane;    // query row of the item = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t o_col = tmem + lane_off + C::kOCol + w * D;
    int islot = 0; uint32_t iphase = 0;
    int vs = 0; uint32_t vphase = 0;
    uint32_t sph = 0u;  // S-full phase of buffer i in bit i (a bit set: no local memory)
    uint32_t pvt_ph = 0u;  // parity of the next pv_tile completion not yet passed
    uint32_t pvl_ph = 0u;
    while (true) {
      if (!warp_wait(&item_full[islot], iphase, ab, kRoleSoftmax, kBarItemFull, -1)) break;
      const Item& it = item_at(islot);  // valid until this warp releases the slot
      const int nt = it.n_tiles, item = it.idx;
      if (nt < 0) break;  // no more items
      const bool mine = w < it.nh;
      const long long tok = (long long)it.b * p.q_rows + it.qblk * kM + r;
      const int hq = it.h0 + w;
      const bool row_ok = !kRagged || it.qblk * kM + r < p.q_rows;  // ragged: last block partial
      bool ok = true;
      if (!mine || nt == 0) {
        if (mine && row_ok) {  // nothing attended: zeros and -inf
          __nv_bfloat16* orow = p.out + (tok * p.Hq + hq) * D;
#pragma unroll
          for (int j = 0; j < D; j += 8) *reinterpret_cast<uint4*>(orow + j) = make_uint4(0u, 0u, 0u, 0u);
          if (p.lse != nullptr) p.lse[tok * p.Hq + hq] = -INFINITY;
        }
        // keep the V ring position in step with the loader
        for (int t = 0; t < nt; ++t)
          if (++vs == C::kStages) { vs = 0; vphase ^= 1; }
        __syncwarp();
        if (lane == 0) mbar_arrive(&item_empty[islot]);
        if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
        continue;
      }
      int qs = 0;
      long long klo = INT_MIN, khi = INT_MAX;
      if constexpr (kRagged) {
        // keys of this row: [start, end) inside the inclusive window of its position
        const long long qpos = (long long)it.end - p.q_rows + it.qblk * kM + r;
        klo = it.start;
        khi = (long long)it.end - 1;
        if (p.window_left >= 0) klo = max(klo, qpos - p.window_left);
        if (p.window_right >= 0) khi = min(khi, qpos + p.window_right);
        if (!row_ok) { klo = 1; khi = 0; }
      } else {
        const int qp = it.qpos[r];
        qs = it.qseg[r];
        // key positions this row may attend (causal and inclusive window, exact in 64
        // bits, then clamped to the int32 range of the positions); padding sees none
        if (p.causal) khi = min(khi, (long long)qp);
        if (p.window_left >= 0) klo = max(klo, (long long)qp - p.window_left);
        if (p.window_right >= 0) khi = min(khi, (long long)qp + p.window_right);
        if (qs == p.pad_id) { klo = 1; khi = 0; }
      }
      const int kmin = static_cast<int>(max(klo, (long long)INT_MIN));
      const int kmax = static_cast<int>(min(khi, (long long)INT_MAX));
      const bool none = klo > khi;
      float m = -INFINITY, l = 0.f;  // log2 units, lazily moved reference max
      for (int t = 0; t < nt; ++t) {
        const int buf = t & 1;
        const int ti = it.tlo + t;
        const bool full = ti >= it.tlof && ti < it.tupf;
        const uint32_t s_col = tmem + lane_off + (2 * w + buf) * kKT;
        if (!warp_wait(&s_full[2 * w + buf], (sph >> buf) & 1u, ab, kRoleSoftmax, kBarSFull, item)) { ok = false; break; }
        sph ^= 1u << buf;
        const int* ps = nullptr;
        if (!full && !kRagged) {
          // the tile's key positions / segment ids arrived with its V
          if (!warp_wait(&v_full[vs], vphase, ab, kRoleSoftmax, kBarVFull, item)) { ok = false; break; }
          ps = reinterpret_cast<const int*>(smem + C::kOffV + vs * C::kVStageBytes + C::kTBytes);
        }
        if (++vs == C::kStages) { vs = 0; vphase ^= 1; }
        // the row's 64 raw scores: two loads in flight, one wait
        float x[kKT];
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kKT / 32; ++c) tmem_ld_32x32b_x32_nw(s_col + c * 32, x + c * 32);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < kKT; ++j) tmem_ld_ready(x[j]);
        if (!full && kRagged) {
          // the row's keys [kmin, kmax] as columns of this tile (key index of column 0:
          // ti * 64)
          const long long key0 = (long long)ti * kKT;
          int jlo = 0, jhi = -1;
          if (!none) {
            jlo = static_cast<int>(min(max((long long)kmin - key0, 0LL), (long long)kKT));
            jhi = static_cast<int>(max(min((long long)kmax - key0, (long long)kKT - 1), -1LL));
          }
          mask_interval(x, jlo, jhi);
        } else if (!full) {
          // A tile whose keys have consecutive positions p0, p0 + 1, ... and one segment
          // s0 (the causal diagonal, a window edge inside a document) admits for this row
          // exactly the key indices j in [kmin - p0, kmax - p0] when s0 is the row's
          // segment: an interval test per key, no per-key loads.  Other tiles test every
          // key's position and segment.
          // Consecutive positions split into two runs of one segment each (a document
          // boundary or the start of padding inside the tile: keys [0, j0) of segment s0,
          // [j0, 64) of s1) still give every row one interval, inside its own segment's run.
          const int p0 = ps[0], s0 = ps[kKT], s1 = ps[kKT + kKT - 1];
          const int sg0 = ps[kKT + lane], sg1 = ps[kKT + 32 + lane];
          const bool consec = (long long)ps[lane] == (long long)p0 + lane &&
                              (long long)ps[32 + lane] == (long long)p0 + 32 + lane;
          const unsigned b0 = __ballot_sync(0xffffffffu, sg0 == s0);
          const unsigned b1 = __ballot_sync(0xffffffffu, sg1 == s0);
          const int j0 = __popc(b0) + __popc(b1);  // keys of segment s0, a prefix if contiguous
          const bool runs = (sg0 == s0 || sg0 == s1) && (sg1 == s0 || sg1 == s1) &&
                            b0 == (j0 >= 32 ? 0xffffffffu : (1u << j0) - 1u) &&
                            b1 == (j0 <= 32 ? 0u : (j0 >= 64 ? 0xffffffffu : (1u << (j0 - 32)) - 1u));
          if (__all_sync(0xffffffffu, consec && runs)) {
            int jlo = 0, jhi = -1;  // empty unless the row attends some of the tile
            if (!none && (s0 == qs || s1 == qs)) {
              const bool first = s0 == qs;  // the row's run: [0, j0) or [j0, 64)
              const long long rlo = first ? 0 : j0, rhi = first ? j0 - 1 : kKT - 1;
              jlo = static_cast<int>(min(max((long long)kmin - p0, rlo), (long long)kKT));
              jhi = static_cast<int>(max(min((long long)kmax - p0, rhi), -1LL));
            }
            mask_interval(x, jlo, jhi);
          } else {
#pragma unroll
            for (int j = 0; j < kKT; ++j) {
              const int kp = ps[j], ksg = ps[kKT + j];
              const bool ok_k = !none && ksg == qs && kp >= kmin && kp <= kmax;
              if (!ok_k) x[j] = -INFINITY;
            }
          }
        }
        // row maximum: eight chains of three-input max; chain u takes the scores u,
        // u + 8, u + 16, ... of the tile
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = fmaxf(x[u], x[u + 8]);
#pragma unroll
        for (int j = 16; j < kKT; j += 16) {
#pragma unroll
          for (int u = 0; u < 8; ++u) mx[u] = fmax3f(mx[u], x[j + u], x[j + 8 + u]);
        }
        const float tmax = fmax3f(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], mx[5]),
                                  fmaxf(mx[6], mx[7])) * p.scale_log2;
        // lazy online softmax: move the reference max only when it grows by > 2^8
        float m_new = m;
        if (tmax > m + kRescaleThreshold || (m == -INFINITY && tmax != -INFINITY)) m_new = tmax;
        const float alpha = (m == -INFINITY || m_new == m) ? (m_new == m ? 1.f : 0.f) : ex2(m - m_new);
        // exponentials; P (bf16 pairs) over the S_w,buf columns, 32 keys at a time.  The
        // argument x * scale - m and the row sum run two lanes per instruction.
        float psum = 0.f;
        {
          uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};
          const uint64_t scale2 = pack_f32x2(p.scale_log2, p.scale_log2);
          const uint64_t negm2 = pack_f32x2(-m_new, -m_new);
#pragma unroll
          for (int c = 0; c < kKT / 32; ++c) {
            uint32_t pk[16];
            if (m_new == -INFINITY) {
#pragma unroll
              for (int j = 0; j < 16; ++j) pk[j] = 0u;
            } else {
#pragma unroll
              for (int j = 0; j < 32; j += 2) {
                const uint64_t a2 = fma_f32x2(pack_f32x2(x[c * 32 + j], x[c * 32 + j + 1]), scale2, negm2);
                float a0, a1;
                unpack_f32x2(a2, a0, a1);
                const float e0 = ex2(a0), e1 = ex2(a1);
                ps2[(j >> 1) & 3] = add_f32x2(ps2[(j >> 1) & 3], pack_f32x2(e0, e1));
                __nv_bfloat162 h2 = __floats2bfloat162_rn(e0, e1);
                pk[j >> 1] = *reinterpret_cast<uint32_t*>(&h2);
              }
            }
            tmem_st_32x32b_x16_u_nw(s_col + c * 16, pk);
          }
          tmem_wait_st();
          const uint64_t s01 = add_f32x2(ps2[0], ps2[1]), s23 = add_f32x2(ps2[2], ps2[3]);
          float lo, hi;
          unpack_f32x2(add_f32x2(s01, s23), lo, hi);
          psum = lo + hi;
        }
        if (t > 0) {
          // O_w holds PV(0 .. t - 2) for sure (S(t) was issued after PV(t - 2)); a rescale
          // also waits for PV(t - 1).  TMEM loads/stores are warp-collective, so the whole
          // warp rescales when any of its rows moved.
          const bool my_rescale = m_new != m && m != -INFINITY;
          if (__any_sync(0xffffffffu, my_rescale)) {
            if (!warp_wait(&pv_tile[w], pvt_ph, ab, kRoleSoftmax, kBarPvTile, item)) { ok = false; break; }
            tc_fence_after();
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
          pvt_ph ^= 1u;  // PV(t - 1) passed
        }
        l = l * alpha + psum;
        m = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[2 * w + buf]);
      }
      if (!ok) break;
      if (!warp_wait(&pv_last[w], pvl_ph, ab, kRoleSoftmax, kBarPvLast, item)) break;
      pvl_ph ^= 1u;
      pvt_ph ^= 1u;  // PV(nt - 1) passed
      tc_fence_after();
      // rows of this warp in two halves of 16, each in its own buffer (lanes 0-15 the
      // first, 16-31 the second, written at once): staged in the 128-byte swizzle the
      // tensor map expects (16-byte chunk c of row i at c ^ (i % 8)), then one TMA store per
      // half and 64-column panel; rows past the query range are clipped by the map
      uint8_t* stg = smem + C::kOffStage + (warp - 4) * C::kStgWarpBytes;
      // the staging rows are free once the previous item's stores have read them
      if (lane == 0) bulk_wait_group_read<0>();
      __syncwarp();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const uint64_t inv2 = pack_f32x2(inv, inv);
      const int half = lane >> 4, rr = lane & 15;
      // O_w leaves tensor memory one 64-column panel at a time (fewer live registers); the
      // next item's first PV may overwrite it once the last panel is in registers
#pragma unroll
      for (int pn = 0; pn < C::kPanels; ++pn) {
        float ov[64];
        tmem_ld_32x32b_x32_nw(o_col + pn * 64, ov);
        tmem_ld_32x32b_x32_nw(o_col + pn * 64 + 32, ov + 32);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 64; ++j) tmem_ld_ready(ov[j]);
        if (pn == C::kPanels - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&o_empty[w]);
        }
        uint32_t wv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          float a, c;
          unpack_f32x2(mul_f32x2(pack_f32x2(ov[2 * j], ov[2 * j + 1]), inv2), a, c);
          __nv_bfloat162 h2 = __floats2bfloat162_rn(a, c);
          wv[j] = *reinterpret_cast<uint32_t*>(&h2);
        }
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8)
          *reinterpret_cast<uint4*>(stg + half * C::kStgHalfBytes + pn * C::kStgPanelBytes + rr * 128 +
                                    ((c8 ^ (rr & 7)) * 16)) =
              make_uint4(wv[c8 * 4], wv[c8 * 4 + 1], wv[c8 * 4 + 2], wv[c8 * 4 + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_store_4d(&tm_o, stg + hh * C::kStgHalfBytes + pn * C::kStgPanelBytes, pn * 64, hq,
                         it.qblk * kM + q4 * 32 + hh * 16, it.b);
        }
        bulk_commit_group();
      }
      if (p.lse != nullptr && row_ok) p.lse[tok * p.Hq + hq] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[islot]);
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
    }
    if (lane == 0) bulk_wait_group<0>();  // this warp's output stores have completed
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  // every loader of the launch has stopped drawing items once all CTAs counted
  // themselves here: the last one leaves the counter zero for the next launch
  if (threadIdx.x == 0 && atomicAdd(&p.sched[1], 1) == static_cast<int>(gridDim.x) - 1) {
    p.sched[0] = 0;
    p.sched[1] = 0;
    __threadfence();
  }
}

// Device address of this launch's item counters (the slot after the previous launch's).
int sched_slot(int** out) {
  static std::mutex mu;
  static int* base[64] = {};
  static unsigned next = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "blocksparse_attn: cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(SBA_ERR_UNSUPPORTED, "blocksparse_attn: device ordinal >= 64");
  std::lock_guard<std::mutex> lock(mu);
  if (base[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_bsa_sched);
    if (e != cudaSuccess || ptr == nullptr) return cuda_error(e, "blocksparse_attn: item counters");
    base[dev] = static_cast<int*>(ptr);
  }
  *out = base[dev] + 2 * (next++ % kSchedSlots);
  return SBA_OK;
}

template <int D, bool kRagged>
int launch_impl(const void* q, const void* k, const void* v, const Params& p_in, cudaStream_t stream) {
  Params p = p_in;
  if (int rc = sched_slot(&p.sched)) return rc;
  using C = Cfg<D>;
  CUtensorMap tq, tk, tv;
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.B * p.q_rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hq * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kM};
    if (encode_tensor_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "blocksparse_attn: tensor map (q) failed");
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hkv, (cuuint64_t)p.B * p.kv_rows};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hkv * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)kKT};
    if (encode_tensor_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "blocksparse_attn: tensor map (k/v) failed");
  }
  CUtensorMap to;
  {
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.q_rows, (cuuint64_t)p.B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hq * D * 2, (cuuint64_t)p.q_rows * p.Hq * D * 2};
    cuuint32_t box[4] = {64, 1, 16, 1};
    if (encode_tensor_map(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.out, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "blocksparse_attn: tensor map (out) failed");
  }
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(blocksparse_attn_kernel<D, kRagged>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return cuda_error(e, "blocksparse_attn: set smem attribute");
    attr_done = true;
  }
  const int grid = std::min(p.n_items, num_sms());
  blocksparse_attn_kernel<D, kRagged><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, to, p);
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
  p.q_rows = T;
  p.kv_rows = T;
  p.kv_block = kv_block;
  p.seq_start = nullptr;
  p.seq_end = nullptr;
  p.nbq = T / kM;
  p.causal = causal;
  p.window_left = window_left;
  p.window_right = window_right;
  p.pad_id = pad_id;
  p.scale_log2 = scale * kLog2e;
  p.n_pairs = (p.G + 1) / 2;
  p.wait_limit = wait_timeout_cycles();
  const long long n_items = (long long)B * Hkv * p.nbq * p.n_pairs;
  if (n_items >= (1LL << 31)) return set_error(SBA_ERR_UNSUPPORTED, "blocksparse_attn: too many items");
  p.n_items = static_cast<int>(n_items);
  if (D == 128) return launch_impl<128, false>(q, k, v, p, stream);
  return launch_impl<64, false>(q, k, v, p, stream);
}

// Ragged multi-query attention on the block pipeline (no soft cap, no sinks): queries
// q [B, Q, Hq, 128] at positions end - Q + i, keys / values [B, S, Hkv, 128].
int launch_ragged_chunk(const void* q, const void* k, const void* v, const int32_t* seq_start,
                        const int32_t* seq_end, int B, int Qn, int Hq, int Hkv, int S,
                        float scale, int window_left, int window_right, void* out, float* lse,
                        cudaStream_t stream) {
  Params p{};
  p.seq_start = seq_start;
  p.seq_end = seq_end;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.lse = lse;
  p.B = B; p.T = 0; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv;
  p.q_rows = Qn;
  p.kv_rows = S;
  p.kv_block = 128;
  p.nbq = (Qn + kM - 1) / kM;
  p.causal = 0;  // causality comes from window_right = 0
  p.window_left = window_left;
  p.window_right = window_right;
  p.pad_id = 0;
  p.scale_log2 = scale * kLog2e;
  p.n_pairs = (p.G + 1) / 2;
  p.wait_limit = wait_timeout_cycles();
  const long long n_items = (long long)B * Hkv * p.nbq * p.n_pairs;
  if (n_items >= (1LL << 31) || (long long)B * S >= (1LL << 31) || (long long)B * Qn >= (1LL << 31))
    return set_error(SBA_ERR_UNSUPPORTED, "ragged attention: too many rows");
  p.n_items = static_cast<int>(n_items);
  return launch_impl<128, true>(q, k, v, p, stream);
}

}  // namespace sba
