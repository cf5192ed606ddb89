// Attention over SparseMask block bounds, for sm_103a.
//
// Follows "ejkernel.kernels._triton.blocksparse_attention._mask" (module source page),
// module docstring and SparseMask docstring: for each query block only the key blocks
// in [lower, upper) are computed, and blocks in [lower_full, upper_full) need no
// per-token mask.  The token mask used elsewhere (same segment, neither padding,
// causal and inclusive window on positions) is applied to every other block.
//
// Work item = (batch row, query block of 128 tokens, KV head, pair of its query heads):
// two 128-row problems that read the same key/value blocks and share the token mask.
// A persistent CTA per SM runs a warp-specialised pipeline:
//   warp 0      loader: publishes the item (bounds of its query block), then TMA loads
//               Q of each head into its own buffer and, per key block, K into a K ring
//               and V plus the block's key positions / segment ids into a V ring;
//   warp 1      MMA issuer (one thread): S_w = Q_w K^T (both operands in shared
//               memory, N = one key block) and O_w += P_w V (P_w read from tensor
//               memory), in the order S0(j) S1(j) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ...
//               so that the tensor core runs one head's MMAs while the other head's
//               softmax works;
//   warps 4..7  softmax of head slot 0, warps 8..11 of head slot 1: one thread per query
//               row; the row's scores of S_w come out of tensor memory in one pass (four
//               loads under one wait) into registers, are masked outside the full block
//               range, and P_w (bf16) is written in place over the S_w columns; lazy
//               online softmax (O_w rescaled only when the row maximum grows by > 2^8);
//               epilogue O_w / l.
// Tensor memory: S0, S1 (one key block of fp32 columns each, P aliased in place), O0,
// O1 (D columns each).  A commit after S_w(j + 1) also covers PV_w(j), so a softmax
// warpgroup that sees S_w(j + 1) may rescale O_w without a further wait.
#include <cuda_bf16.h>

#include <climits>
#include <cmath>

#include "common.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace sba {

static __device__ DevError g_err_bsa = {0u, 0u, 0};

namespace {

using namespace ptx;

// Warpgroup 0: warp 0 loader, warp 1 MMA issuer (warps 2, 3 idle), 72 registers each;
// warpgroups 1 and 2: softmax, 192 registers each (a row's 128 scores stay in
// registers).  The pool at launch is 384 threads x 168 registers = 64512 >=
// 128 x 72 + 256 x 192 = 58368.
constexpr int kThreads = 384;
constexpr int kRegsLow = 72;
constexpr int kRegsHigh = 192;
static_assert(128 * kRegsLow + 256 * kRegsHigh <= 384 * 168, "register split exceeds the pool");
constexpr int kM = 128;         // query rows per head slot
constexpr int kItemSlots = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct Item {
  int b, hkv, qblk, h0, nh;  // heads h0 .. h0 + nh - 1 (nh = 1 or 2)
  int lo, up, lof, upf;      // kv blocks [lo, up); [lof, upf) need no token mask
  int n_tiles;               // = up - lo (one key block per tile)
  int start, end;            // ragged mode: the row's key range
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
  float scale_log2;
  int n_pairs, n_items;
  long long wait_limit;  // cycles a bounded wait may take
};

enum Role : unsigned { kRoleLoader = 1, kRoleMma = 2, kRoleSoftmax = 3 };
enum BarId : unsigned {
  kBarItemFull = 1, kBarItemEmpty, kBarQFull, kBarQEmpty, kBarKFull, kBarKEmpty, kBarVFull,
  kBarVEmpty, kBarSFull, kBarPFull, kBarPvDone, kBarOEmpty
};

template <int D, int KB>
struct Cfg {
  static constexpr int kPanels = D / 64;                   // 64-element (128-byte) panels
  static constexpr int kQPanelBytes = kM * 128;
  static constexpr int kQBytes = kPanels * kQPanelBytes;   // Q of one head slot
  static constexpr int kKPanelBytes = KB * 128;
  static constexpr int kKBytes = kPanels * kKPanelBytes;   // K (or V) of one key block
  static constexpr int kPosSegBytes = 2 * KB * 4;
  static constexpr int kVStageBytes = (kKBytes + kPosSegBytes + 1023) & ~1023;
  static constexpr int kItemBytes = (static_cast<int>(sizeof(Item)) + 15) & ~15;
  static constexpr int kFixed = 2 * kQBytes + kItemSlots * kItemBytes + 1024 + 1024;
  static constexpr int kRingFit = (232448 - kFixed) / (kKBytes + kVStageBytes);
  static constexpr int kStages = kRingFit > 4 ? 4 : kRingFit;   // K and V rings
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKBytes;
  static constexpr int kOffItems = kOffV + kStages * kVStageBytes;
  static constexpr int kOffBars = (kOffItems + kItemSlots * kItemBytes + 7) & ~7;
  static constexpr int kNumBars = 2 * kItemSlots + 4 + 4 * kStages + 8;
  static constexpr int kOffMisc = ((kOffBars + kNumBars * 8) + 15) & ~15;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  // tensor memory columns: S_w (P_w aliased) and O_w per head slot
  static constexpr int kSCol = 0;                          // S_w at w * KB
  static constexpr int kOCol = 2 * KB;                     // O_w at kOCol + w * D
  static constexpr int kTmemNeed = 2 * KB + 2 * D;
  static constexpr int kTmemCols = kTmemNeed <= 256 ? 256 : 512;
  static constexpr uint32_t kIdescQK = make_idesc(128, KB, 1u, false, false);
  static constexpr uint32_t kIdescPV = make_idesc(128, D, 1u, false, true);
  static_assert(kStages >= 2, "pipeline depth");
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

// kRagged: the ragged multi-query form of the same computation (queries are the last Q
// tokens of [start, end) of a KV cache, each with its own inclusive window); the key
// range and the full blocks of a query block follow from start, end and the window, and
// the per-row key range replaces the position / segment test.
template <int D, int KB, bool kRagged>
__global__ void __launch_bounds__(kThreads, 1)
blocksparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<D, KB>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bb = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* item_full = bb;   bb += kItemSlots;
  uint64_t* item_empty = bb;  bb += kItemSlots;
  uint64_t* q_full = bb;      bb += 2;   // per head slot
  uint64_t* q_empty = bb;     bb += 2;
  uint64_t* k_full = bb;      bb += C::kStages;
  uint64_t* k_empty = bb;     bb += C::kStages;
  uint64_t* v_full = bb;      bb += C::kStages;
  uint64_t* v_empty = bb;     bb += C::kStages;
  uint64_t* s_full = bb;      bb += 2;   // S_w(j) written (and PV_w(j - 1) done)
  uint64_t* p_full = bb;      bb += 2;   // P_w(j) stored, O_w rescaled
  uint64_t* pv_done = bb;     bb += 2;   // last PV_w of an item done
  uint64_t* o_empty = bb;     bb += 2;   // epilogue has read O_w
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  uint64_t* mma_done = reinterpret_cast<uint64_t*>(smem + C::kOffMisc + 8);
  const Abort ab{abort_flag, &g_err_bsa, 2u, p.wait_limit};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto item_at = [&](int slot) -> Item& {
    return *reinterpret_cast<Item*>(smem + C::kOffItems + slot * C::kItemBytes);
  };

  if (threadIdx.x == 0) {
    // an item slot is read by the MMA thread and the eight softmax warps
    for (int i = 0; i < kItemSlots; ++i) { mbar_init(&item_full[i], 1); mbar_init(&item_empty[i], 9); }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&q_full[w], 1); mbar_init(&q_empty[w], 1);
      mbar_init(&s_full[w], 1); mbar_init(&p_full[w], 4);
      mbar_init(&pv_done[w], 1); mbar_init(&o_empty[w], 4);
    }
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&k_full[i], 1); mbar_init(&k_empty[i], 1);
      mbar_init(&v_full[i], 1); mbar_init(&v_empty[i], 1);
    }
    mbar_init(mma_done, 1);
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
  const int nbkv = (p.kv_rows + KB - 1) / KB;

  if (warp < 4) {
    setmaxnreg_dec<kRegsLow>();
  if (warp == 0) {
    // ------------------------------------------------------------------ loader
    int islot = 0; uint32_t iphase = 0;
    uint32_t qphase[2] = {0u, 0u};
    bool q_issued[2] = {false, false};
    uint32_t q_last[2] = {0u, 0u};
    int ks = 0; uint32_t kphase = 0;
    int vs = 0; uint32_t vphase = 0;
    bool k_issued[C::kStages], v_issued[C::kStages];
    uint32_t k_last[C::kStages], v_last[C::kStages];
#pragma unroll
    for (int i = 0; i < C::kStages; ++i) { k_issued[i] = v_issued[i] = false; k_last[i] = v_last[i] = 0; }
    bool ok = true;
    for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
      int b, hkv, qblk, h0, nh;
      decode_item(p, item, b, hkv, qblk, h0, nh);
      int lo = 0, up = 0, lof = 0, upf = 0, start = 0, end = 0;
      if constexpr (kRagged) {
        // rows i0 .. i1 of this query block sit at end - Q + i; their windows' union is
        // [kmin(i0), kmax(i1)] and the keys every row sees are [kmin(i1), kmax(i0)]
        start = min(max(p.seq_start[b], 0), p.kv_rows);
        end = min(max(p.seq_end[b], 0), p.kv_rows);
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
          lo = static_cast<int>(klo / KB);
          up = static_cast<int>(khi / KB) + 1;
          const long long flo = kmin(i1), fhi = kmax(i0);
          lof = static_cast<int>((flo + KB - 1) / KB);
          upf = fhi >= flo ? static_cast<int>((fhi + 1) / KB) : lof;
        }
      } else {
        const long long brow = (long long)b * p.nbq + qblk;
        lo = max(p.lower[brow], 0);
        up = min(p.upper[brow], nbkv);
        lof = p.lower_full[brow];
        upf = p.upper_full[brow];
      }
      const int nt = up > lo ? up - lo : 0;
      if (!warp_wait(&item_empty[islot], iphase ^ 1, ab, kRoleLoader, kBarItemEmpty, item)) break;
      if (lane == 0) {
        Item& it = item_at(islot);
        it.b = b; it.hkv = hkv; it.qblk = qblk; it.h0 = h0; it.nh = nh;
        it.lo = lo; it.up = up; it.lof = lof; it.upf = upf;
        it.n_tiles = nt;
        it.start = start; it.end = end;
        mbar_arrive(&item_full[islot]);
      }
      __syncwarp();
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
      if (nt == 0) continue;
      for (int w = 0; w < nh; ++w) {
        if (!warp_wait(&q_empty[w], qphase[w] ^ 1, ab, kRoleLoader, kBarQEmpty, item)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&q_full[w], C::kQBytes);
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smem + C::kOffQ + w * C::kQBytes + pn * C::kQPanelBytes, &tm_q, &q_full[w],
                        pn * 64, h0 + w, b * p.q_rows + qblk * kM);
        }
        q_issued[w] = true;
        q_last[w] = qphase[w];
        qphase[w] ^= 1;
      }
      if (!ok) break;
      for (int t = 0; t < nt; ++t) {
        const int tok0 = b * p.kv_rows + (lo + t) * KB;
        if (!warp_wait(&k_empty[ks], kphase ^ 1, ab, kRoleLoader, kBarKEmpty, item)) { ok = false; break; }
        if (lane == 0) {
          mbar_arrive_expect_tx(&k_full[ks], C::kKBytes);
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(smem + C::kOffK + ks * C::kKBytes + pn * C::kKPanelBytes, &tm_k, &k_full[ks],
                        pn * 64, hkv, tok0);
        }
        k_issued[ks] = true;
        k_last[ks] = kphase;
        if (++ks == C::kStages) { ks = 0; kphase ^= 1; }
        if (!warp_wait(&v_empty[vs], vphase ^ 1, ab, kRoleLoader, kBarVEmpty, item)) { ok = false; break; }
        if (lane == 0) {
          uint8_t* vdst = smem + C::kOffV + vs * C::kVStageBytes;
          mbar_arrive_expect_tx(&v_full[vs], C::kKBytes + (kRagged ? 0 : C::kPosSegBytes));
#pragma unroll
          for (int pn = 0; pn < C::kPanels; ++pn)
            tma_load_3d(vdst + pn * C::kKPanelBytes, &tm_v, &v_full[vs], pn * 64, hkv, tok0);
          if (!kRagged) {
            bulk_load(vdst + C::kKBytes, p.kv_pos + tok0, KB * 4, &v_full[vs]);
            bulk_load(vdst + C::kKBytes + KB * 4, p.kv_seg + tok0, KB * 4, &v_full[vs]);
          }
        }
        v_issued[vs] = true;
        v_last[vs] = vphase;
        if (++vs == C::kStages) { vs = 0; vphase ^= 1; }
      }
    }
    // Drain: wait (bounded) for every copy this warp issued before the CTA exits.
    if (lane == 0) {
      for (int s = 0; s < C::kStages; ++s) {
        if (k_issued[s]) drain_wait(&k_full[s], k_last[s]);
        if (v_issued[s]) drain_wait(&v_full[s], v_last[s]);
      }
      for (int w = 0; w < 2; ++w)
        if (q_issued[w]) drain_wait(&q_full[w], q_last[w]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int islot = 0; uint32_t iphase = 0;
      uint32_t qph[2] = {0u, 0u}, pph[2] = {0u, 0u}, oph[2] = {0u, 0u};
      int ks = 0; uint32_t kphase = 0;
      int vs = 0; uint32_t vphase = 0;
      bool ok = true;
      // descriptors of the shared-memory operands; a byte offset x adds x >> 4
      const uint64_t q_desc0 = make_sdesc(smem_base + C::kOffQ, 16, 1024, kLayoutSW128);
      const uint64_t k_desc0 = make_sdesc(smem_base + C::kOffK, 16, 1024, kLayoutSW128);
      const uint64_t v_desc0 = make_sdesc(smem_base + C::kOffV, C::kKPanelBytes, 1024, kLayoutSW128);
      auto kstep = [](int kk, int panel_bytes) -> uint64_t {
        return static_cast<uint64_t>(((kk / 4) * panel_bytes + (kk % 4) * 32) >> 4);
      };
      // S_w = Q_w K^T of the K stage `stage`
      auto issue_s = [&](int w, int stage) {
        const uint64_t qd = q_desc0 + static_cast<uint64_t>((w * C::kQBytes) >> 4);
        const uint64_t kd = k_desc0 + static_cast<uint64_t>((stage * C::kKBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16_ss(tmem + C::kSCol + w * KB, qd + kstep(kk, C::kQPanelBytes),
                     kd + kstep(kk, C::kKPanelBytes), C::kIdescQK, kk > 0 ? 1u : 0u);
        mma_commit(&s_full[w]);
      };
      // O_w (+)= P_w V of the V stage `stage` (P_w: bf16 pairs over the S_w columns)
      auto issue_pv = [&](int w, int stage, bool first) {
        const uint64_t vd = v_desc0 + static_cast<uint64_t>((stage * C::kVStageBytes) >> 4);
#pragma unroll
        for (int kk = 0; kk < KB / 16; ++kk)
          mma_f16_ts(tmem + C::kOCol + w * D, tmem + C::kSCol + w * KB + kk * 8,
                     vd + static_cast<uint64_t>((kk * 16 * 128) >> 4), C::kIdescPV,
                     (first && kk == 0) ? 0u : 1u);
      };
      for (int item = blockIdx.x; item < p.n_items && ok; item += gridDim.x) {
        if (!bounded_wait(&item_full[islot], iphase, ab, kRoleMma, kBarItemFull, item)) break;
        const int nt = item_at(islot).n_tiles, nh = item_at(islot).nh;
        mbar_arrive(&item_empty[islot]);
        if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
        if (nt == 0) continue;
        for (int w = 0; w < nh && ok; ++w) {
          if (!bounded_wait(&q_full[w], qph[w], ab, kRoleMma, kBarQFull, item)) ok = false;
          qph[w] ^= 1;
        }
        if (!ok) break;
        // S of tile 0 for every head slot
        if (!bounded_wait(&k_full[ks], kphase, ab, kRoleMma, kBarKFull, item)) break;
        tc_fence_after();
        for (int w = 0; w < nh; ++w) {
          issue_s(w, ks);
          if (nt == 1) mma_commit(&q_empty[w]);
        }
        mma_commit(&k_empty[ks]);
        int ks_next = ks + 1 == C::kStages ? 0 : ks + 1;
        uint32_t kphase_next = ks + 1 == C::kStages ? kphase ^ 1 : kphase;
        for (int t = 0; t < nt && ok; ++t) {
          const bool more = t + 1 < nt;
          if (!bounded_wait(&v_full[vs], vphase, ab, kRoleMma, kBarVFull, item)) { ok = false; break; }
          for (int w = 0; w < nh; ++w) {
            if (t == 0) {
              if (!bounded_wait(&o_empty[w], oph[w] ^ 1, ab, kRoleMma, kBarOEmpty, item)) { ok = false; break; }
              oph[w] ^= 1;
            }
            if (!bounded_wait(&p_full[w], pph[w], ab, kRoleMma, kBarPFull, item)) { ok = false; break; }
            pph[w] ^= 1;
            tc_fence_after();
            issue_pv(w, vs, t == 0);
            if (!more) mma_commit(&pv_done[w]);
            if (w == nh - 1) mma_commit(&v_empty[vs]);
            if (more) {
              if (w == 0) {
                if (!bounded_wait(&k_full[ks_next], kphase_next, ab, kRoleMma, kBarKFull, item)) { ok = false; break; }
                tc_fence_after();
              }
              issue_s(w, ks_next);   // also covers PV_w(t) for the softmax warpgroup
              if (t + 1 == nt - 1) mma_commit(&q_empty[w]);
              if (w == nh - 1) mma_commit(&k_empty[ks_next]);
            }
          }
          if (!ok) break;
          if (++vs == C::kStages) { vs = 0; vphase ^= 1; }
          if (more) {
            ks = ks_next; kphase = kphase_next;
            ks_next = ks + 1 == C::kStages ? 0 : ks + 1;
            kphase_next = ks + 1 == C::kStages ? kphase ^ 1 : kphase;
          }
        }
        if (!ok) break;
        // the last K stage of this item was consumed; move past it
        ks = ks_next; kphase = kphase_next;
      }
      // every tcgen05 op issued by this thread has finished once mma_done fires
      mma_commit(mma_done);
      drain_wait(mma_done, 0);
    }
    __syncwarp();
  }
  } else {
    setmaxnreg_inc<kRegsHigh>();
    // ------------------------------------------------------------------ softmax / epilogue
    const int w = (warp - 4) >> 2;   // head slot of this warpgroup
    const int q4 = warp & 3;         // TMEM lane quadrant of this warp
    const int r = q4 * 32 + lane;    // query row of the item = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t s_col = tmem + lane_off + C::kSCol + w * KB;
    const uint32_t o_col = tmem + lane_off + C::kOCol + w * D;
    int islot = 0; uint32_t iphase = 0;
    int vs = 0; uint32_t vphase = 0;
    uint32_t sph = 0, pvph = 0;
    for (int item = blockIdx.x; item < p.n_items; item += gridDim.x) {
      if (!warp_wait(&item_full[islot], iphase, ab, kRoleSoftmax, kBarItemFull, item)) break;
      const Item it = item_at(islot);
      const int nt = it.n_tiles;
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
        // keep the V ring position in step with the loader and the MMA thread
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
        const int qp = p.q_pos[tok];
        qs = p.q_seg[tok];
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
        const int blk = it.lo + t;
        const bool full = blk >= it.lof && blk < it.upf;
        if (!warp_wait(&s_full[w], sph, ab, kRoleSoftmax, kBarSFull, item)) { ok = false; break; }
        sph ^= 1;
        const int* ps = nullptr;
        if (!full && !kRagged) {
          // the block's key positions / segment ids arrived with its V
          if (!warp_wait(&v_full[vs], vphase, ab, kRoleSoftmax, kBarVFull, item)) { ok = false; break; }
          ps = reinterpret_cast<const int*>(smem + C::kOffV + vs * C::kVStageBytes + C::kKBytes);
        }
        if (++vs == C::kStages) { vs = 0; vphase ^= 1; }
        // the row's KB raw scores: four loads in flight, one wait
        float x[KB];
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < KB / 32; ++c) tmem_ld_32x32b_x32_nw(s_col + c * 32, x + c * 32);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < KB; ++j) tmem_ld_ready(x[j]);
        if (!full && kRagged) {
          const int key0 = blk * KB;  // key index of column 0
#pragma unroll
          for (int j = 0; j < KB; ++j)
            if (!(!none && key0 + j >= kmin && key0 + j <= kmax)) x[j] = -INFINITY;
        } else if (!full) {
#pragma unroll
          for (int j = 0; j < KB; j += 4) {
            const int4 kp4 = *reinterpret_cast<const int4*>(ps + j);
            const int4 ks4 = *reinterpret_cast<const int4*>(ps + KB + j);
            const int kp[4] = {kp4.x, kp4.y, kp4.z, kp4.w};
            const int ksg[4] = {ks4.x, ks4.y, ks4.z, ks4.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const bool ok_k = !none && ksg[u] == qs && kp[u] >= kmin && kp[u] <= kmax;
              if (!ok_k) x[j + u] = -INFINITY;
            }
          }
        }
        // row maximum: eight chains of three-input max (two new scores per instruction);
        // chain u takes the scores u, u + 8, u + 16, ... of the row
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = fmaxf(x[u], x[u + 8]);
#pragma unroll
        for (int j = 16; j < KB; j += 16) {
#pragma unroll
          for (int u = 0; u < 8; ++u) mx[u] = fmax3f(mx[u], x[j + u], x[j + 8 + u]);
        }
        const float tmax = fmax3f(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], mx[5]),
                                  fmaxf(mx[6], mx[7])) * p.scale_log2;
        // lazy online softmax: move the reference max only when it grows by > 2^8
        float m_new = m;
        if (tmax > m + kRescaleThreshold || (m == -INFINITY && tmax != -INFINITY)) m_new = tmax;
        const float alpha = (m == -INFINITY || m_new == m) ? (m_new == m ? 1.f : 0.f) : ex2(m - m_new);
        // exponentials; P (bf16 pairs) over the S_w columns, 32 keys at a time.  The
        // argument x * scale - m and the row sum run two lanes per instruction.
        float psum = 0.f;
        {
          uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};
          const uint64_t scale2 = pack_f32x2(p.scale_log2, p.scale_log2);
          const uint64_t negm2 = pack_f32x2(-m_new, -m_new);
#pragma unroll
          for (int c = 0; c < KB / 32; ++c) {
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
                x[c * 32 + j] = e0;
                x[c * 32 + j + 1] = e1;
                ps2[(j >> 1) & 3] = add_f32x2(ps2[(j >> 1) & 3], pack_f32x2(e0, e1));
              }
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                __nv_bfloat162 h2 = __floats2bfloat162_rn(x[c * 32 + 2 * j], x[c * 32 + 2 * j + 1]);
                pk[j] = *reinterpret_cast<uint32_t*>(&h2);
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
          // S_w(t) implies PV_w(t - 1) is done: O_w may be rescaled.  TMEM loads/stores
          // are warp-collective, so the whole warp rescales when any of its rows moved.
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
        l = l * alpha + psum;
        m = m_new;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[w]);
      }
      if (!ok) break;
      if (!warp_wait(&pv_done[w], pvph, ab, kRoleSoftmax, kBarPvDone, item)) break;
      pvph ^= 1;
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.out + (tok * p.Hq + hq) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float ov[32];
        tmem_ld_32x32b_x32(o_col + c * 32, ov);
        if (!row_ok) continue;  // warp-collective load above, no store for a padded row
#pragma unroll
        for (int j = 0; j < 32; j += 8) {
          uint32_t wv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(ov[j + 2 * u] * inv, ov[j + 2 * u + 1] * inv);
            wv[u] = *reinterpret_cast<uint32_t*>(&h2);
          }
          *reinterpret_cast<uint4*>(orow + c * 32 + j) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
      if (p.lse != nullptr && row_ok) p.lse[tok * p.Hq + hq] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&o_empty[w]);
        mbar_arrive(&item_empty[islot]);
      }
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

template <int D, int KB, bool kRagged>
int launch_impl(const void* q, const void* k, const void* v, const Params& p, cudaStream_t stream) {
  using C = Cfg<D, KB>;
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
    cuuint32_t box[3] = {64, 1, (cuuint32_t)KB};
    if (encode_tensor_map(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(k), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v), dims,
                          strides, box, CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "blocksparse_attn: tensor map (k/v) failed");
  }
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(blocksparse_attn_kernel<D, KB, kRagged>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return cuda_error(e, "blocksparse_attn: set smem attribute");
    attr_done = true;
  }
  const int grid = std::min(p.n_items, num_sms());
  blocksparse_attn_kernel<D, KB, kRagged><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
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
  if (D == 128 && kv_block == 128) return launch_impl<128, 128, false>(q, k, v, p, stream);
  if (D == 128 && kv_block == 64) return launch_impl<128, 64, false>(q, k, v, p, stream);
  if (D == 64 && kv_block == 128) return launch_impl<64, 128, false>(q, k, v, p, stream);
  return launch_impl<64, 64, false>(q, k, v, p, stream);
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
  return launch_impl<128, 128, true>(q, k, v, p, stream);
}

}  // namespace sba
