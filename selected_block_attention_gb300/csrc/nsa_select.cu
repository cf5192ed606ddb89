// Native-sparse-attention forward, selection branch, for sm_103a.
//
// Follows "ejkernel.modules.operations.native_sparse_attention" (operation API page),
// NativeSparseAttention.run / native_sparse_attention: each query token attends, per
// KV head, only to the key blocks named by block_indices[b, t, h_kv, :count]; the G
// query heads of a KV head share its keys (GQA); cu_seqlens packs sequences.
//
// bf16 path (tensor cores): "union walk".  A work item is a group of NT consecutive
// tokens and one KV head; its NT * G query rows (token-major, head-minor; NT = 8 when
// G = 16) fill the M = 128 rows of one tcgen05 MMA.  The item's key set is the union
// of the blocks its tokens selected (deduplicated, sorted by first key row), walked in
// tiles of 64 keys, two tiles per QK; every row keeps only the keys of blocks its own
// token selected (plus the causal / sequence-end limit), so a union block is gathered
// once per item and shared by all tokens that picked it.  A persistent CTA per SM runs:
//   warp 2      item builder: reads the NT tokens' index lists (cu_seqlens binary
//               search for packed sequences), filters them, and forms the union with a
//               warp bitonic sort plus a run merge into (first key row, token bitmask);
//   warp 0      loader: TMA loads into a shared-memory ring: the item's Q rows (one 3D
//               box per 64-wide panel), then K and V of each pair of tiles;
//   warp 1      QK issuer (one thread): copies Q into tensor memory (tcgen05.cp, in
//               order with its MMAs), then S = Q K^T for a pair (M = 128 rows, N = 128
//               keys, A from TMEM, fp32 in TMEM);
//   warp 3      PV issuer (one thread): O_w += P_w V_w (N = head dim, A = P_w from
//               TMEM) for each warpgroup's half of the pair.  With both A operands in
//               TMEM the MMAs read only K and V from shared memory, and with two
//               issuing threads one's barrier waits overlap the other's MMAs;
//   warps 4..11 two softmax warpgroups, one thread per row each; warpgroup w takes
//               tile w of every pair (S columns 64 w .. 64 w + 63) with its own P
//               columns, O accumulator and running (m, l).  Per tile: selection /
//               causal mask, lazy online softmax (O rescaled only when the running max
//               grows by > 2^8), P (bf16) stored to TMEM.  The epilogue merges the two
//               partial results ((m, l) exchanged through shared memory; each
//               warpgroup writes half of the head-dim columns) and writes O / l, LSE.
//
// fp32 path (CUDA cores, exact fp32 products and sums): one CTA per token group.
// Tensor cores would round fp32 inputs to tf32, which is not accurate enough for the
// float32 contract, and the fp32 workloads are small.
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "sync.cuh"

namespace sba {

static __device__ DevError g_err_nsa = {0u, 0u, 0};
// Item counters of the union kernel's launches: [next item, CTAs done] per slot; launches
// take the slots in turn, so up to kSchedSlots launches (on any streams) may run at once.
// Each launch finds its slot zero and leaves it zero.
constexpr int kSchedSlots = 64;
static __device__ int g_nsa_sched[2 * kSchedSlots];

namespace {

using namespace ptx;

constexpr int kThreads = 384;   // warps 0-3: loader, MMA, builder, spare; 4-11: two softmax warpgroups
constexpr int kRows = 128;      // MMA M: NT tokens x G query heads
constexpr int kTileKeys = 64;   // keys per pipeline tile (MMA N of S = Q K^T)
constexpr int kNH = 16;         // largest supported G
constexpr int kMaxNT = 16;      // tokens per item
constexpr int kMaxSel = 32;     // largest supported S
constexpr int kMaxUnion = kMaxNT * kMaxSel;
constexpr int kItemSlots = 3;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum Role : unsigned { kRoleLoader = 1, kRoleMma = 2, kRoleSoftmax = 3, kRoleBuilder = 4 };
enum BarId : unsigned {
  kBarItemFull = 1, kBarItemEmpty, kBarQFull, kBarQEmpty, kBarKvFull, kBarKvEmpty, kBarSFull,
  kBarSEmpty, kBarPFull, kBarPvDone, kBarOEmpty, kBarXch
};

struct Params {
  const void* g_slc;  // [B, T, Hq] gate of the output rows (query dtype), or NULL
  const int* block_indices;
  const int* block_counts;
  const int* cu_seqlens;
  void* out;
  float* lse;
  int count_scalar, S, num_seqs;
  int B, T, Hq, Hkv, G, causal, bs;
  int NT, rows;  // tokens per item, rows used (NT * G <= 128)
  int ranked;    // items are formed from count-ranked windows (see build_item)
  float scale, scale_log2;
  int n_items, n_tok;
  int item0;             // work items [item0, n_items) of this launch
  long long wait_limit;  // cycles a bounded wait may take
  int* sched;            // union kernel: [next item, CTAs done] of this launch (zero at launch, left zero)
};

// One union-walk item as the builder hands it to the other roles.
struct Item {
  int g, hkv, n_union, n_tiles;    // n_tiles = -1: no more items (the builder's last publication)
  unsigned tok_valid;              // bit i: token slot i holds a token
  int tok[kMaxNT];                 // token of slot i (-1: none)
  int limit[kMaxNT];               // last key row (absolute) token i may see; -1 if none
  int ux[kMaxUnion];               // first key row (absolute) of each union block
  unsigned short ubits[kMaxUnion]; // tokens of the group that selected it
};

template <int D, int BS>
struct Cfg {
  static constexpr int kPanels = D / 64;                   // 64-element (128-byte) panels
  static constexpr int kSegLen = BS < kTileKeys ? BS : kTileKeys;
  static constexpr int kSegs = kTileKeys / kSegLen;        // union blocks per tile (BS <= 64)
  static constexpr int kPairKeys = 2 * kTileKeys;          // one QK covers two tiles
  static constexpr int kPanelBytes = kPairKeys * 128;      // 16 KB: 128 keys x 64 elements
  static constexpr int kKBytes = kPanels * kPanelBytes;    // K (or V) of a pair; also Q staging
  static constexpr int kStageBytes = 2 * kKBytes;          // [K][V] of a pair, or an item's Q
  static constexpr int kQPanelBytes = kRows * 128;
  static constexpr int kItemBytes = (static_cast<int>(sizeof(Item)) + 127) & ~127;
  static constexpr int kMlBytes = 2 * 2 * kRows * 8;       // (m, l) per row: [item parity][wg]
  static constexpr int kFixed = kItemSlots * kItemBytes + kMaxUnion * 8 + kMlBytes + 1024 + 1024;
  static constexpr int kStagesFit = (232448 - kFixed) / kStageBytes;
  static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
  static constexpr int kOffStages = 0;
  static constexpr int kOffItems = kOffStages + kStages * kStageBytes;
  static constexpr int kOffSort = kOffItems + kItemSlots * kItemBytes;
  static constexpr int kOffMl = kOffSort + kMaxUnion * 8;
  static constexpr int kOffBars = kOffMl + kMlBytes;
  static constexpr int kNumBars = 2 * kItemSlots + 2 * kStages + 1 + 2 + 4 + 1 + 2 + 1;
  static constexpr int kOffMisc = ((kOffBars + kNumBars * 8) + 15) & ~15;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  // tensor memory columns (512 at D = 128): S of a pair, O and P per warpgroup, Q
  static constexpr int kSCol = 0;                          // S: 128 fp32, warpgroup w reads 64 at w * 64
  static constexpr int kOCol = kPairKeys;                  // O of wg w: D fp32 at kOCol + w * D
  static constexpr int kPCol = kOCol + 2 * D;              // P of wg w: 64 bf16 (32 cols) at kPCol + w * 32
  static constexpr int kQCol = kPCol + kTileKeys;          // Q: D bf16 (D / 2 cols)
  static constexpr int kTmemCols = 512;
  static constexpr uint32_t kIdescQK = make_idesc(128, kPairKeys, 1u, false, false);
  static constexpr uint32_t kIdescPV = make_idesc(128, D, 1u, false, true);
  static_assert(kStages >= 3, "pipeline depth");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kQCol + D / 2 <= kTmemCols, "tensor memory budget");
};

__device__ __forceinline__ void decode_item(const Params& p, int item, int& b, int& hkv, int& t) {
  t = item % p.T;
  const int r = item / p.T;
  hkv = r % p.Hkv;
  b = r / p.Hkv;
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

// ------------------------------------------------------------------ item builder
// Forms the union of the selected blocks of the item's NT tokens for KV head hkv.
// Keys (first key row << 16 | token bit) are sorted by one warp (bitonic network in
// shared memory); equal rows are merged by OR-ing their token bits.
//
// Tokens of an item: without ranking g*NT .. g*NT+NT-1.  With ranking the tokens of a
// window of 8*NT consecutive tokens are ranked by their selection count (ties by
// position) and item g takes ranks (g % 8)*NT .. (g % 8)*NT+NT-1 of window g / 8: tokens
// that select few blocks share items with each other, so the unions (and the tiles every
// row of an item walks) are smaller than for consecutive tokens.
template <int BS>
__device__ __forceinline__ void build_item(const Params& p, int g, int hkv, int lane,
                                           int& cached_seq, Item& it, uint64_t* keys) {
  const unsigned kFull = 0xffffffffu;
  const unsigned lt_mask = (1u << lane) - 1u;
  if (p.ranked) {
    const int wn = 8 * p.NT;            // window of 8 items (64 or 128 tokens)
    const int base = (g >> 3) * wn, r = g & 7;
    constexpr int kPer = 128 / 32;      // tokens per lane for the largest window
    int key[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int li = j * 32 + lane, t = base + li;
      int cnt = 0xFFFF;                 // past the window / the tokens: ranked last
      if (li < wn && t < p.n_tok) {
        cnt = p.block_counts ? p.block_counts[(long long)t * p.Hkv + hkv] : p.count_scalar;
        cnt = min(max(cnt, 0), p.S);
      }
      key[j] = (cnt << 8) | li;
    }
    int rank[kPer] = {0, 0, 0, 0};
    const int npl = (wn + 31) / 32;     // tokens per lane of this window (2 to 4)
    for (int src = 0; src < 32; ++src) {
#pragma unroll
      for (int jj = 0; jj < kPer; ++jj) {
        if (jj >= npl) break;           // warp-uniform
        const int other = __shfl_sync(kFull, key[jj], src);
#pragma unroll
        for (int j = 0; j < kPer; ++j)
          if (j < npl) rank[j] += other < key[j];
      }
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int li = j * 32 + lane, t = base + li;
      const int slot = rank[j] - r * p.NT;
      if (li < wn && slot >= 0 && slot < p.NT) it.tok[slot] = t < p.n_tok ? t : -1;
    }
    if (lane >= p.NT && lane < kMaxNT) it.tok[lane] = -1;
  } else {
    if (lane < kMaxNT) it.tok[lane] = (lane < p.NT && g * p.NT + lane < p.n_tok) ? g * p.NT + lane : -1;
  }
  __syncwarp();
  const int tok = lane < kMaxNT ? it.tok[lane] : -1;
  const bool tv = lane < p.NT && tok >= 0;
  int seq0 = 0, slen = 0, trel = 0, cnt = 0, limit = -1;
  if (tv) {
    const int b = p.cu_seqlens ? 0 : tok / p.T;
    const int t = p.cu_seqlens ? tok : tok - b * p.T;
    if (locate_token(p, b, t, cached_seq, seq0, slen, trel)) {
      cnt = p.block_counts ? p.block_counts[(long long)tok * p.Hkv + hkv] : p.count_scalar;
      cnt = min(max(cnt, 0), p.S);
      limit = p.causal ? tok : seq0 + slen - 1;
    }
  }
  // all index loads first (independent of the counts), then filter
  const int total = p.NT * p.S;
  constexpr int kChunks = kMaxUnion / 32;
  int ev[kChunks];
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    const int idx = c * 32 + lane;
    ev[c] = -1;
    if (c * 32 >= total) continue;  // warp-uniform
    const int i = idx < total ? idx / p.S : 0, j = idx - i * p.S;
    const int trow = __shfl_sync(kFull, tok, i);
    if (idx < total && trow >= 0) ev[c] = p.block_indices[((long long)trow * p.Hkv + hkv) * p.S + j];
  }
  // When every token of the item lies in one sequence and that sequence's blocks fit the
  // sort buffer as one 32-bit token mask per block, the union is read off a per-block
  // mask (blocks come out in row order); otherwise the (row, token bit) keys are sorted.
  const unsigned tv_bal = __ballot_sync(kFull, tv);
  bool use_map = false;
  int map_seq0 = 0, map_nb = 0;
  if (tv_bal != 0u) {
    const int src = __ffs(tv_bal) - 1;
    map_seq0 = __shfl_sync(kFull, seq0, src);
    map_nb = (__shfl_sync(kFull, slen, src) + BS - 1) / BS;
    use_map = __all_sync(kFull, !tv || seq0 == map_seq0) && map_nb <= 2 * kMaxUnion;
  }
  uint32_t* bmap = reinterpret_cast<uint32_t*>(keys);
  if (use_map) {
    for (int idx = lane; idx < map_nb; idx += 32) bmap[idx] = 0u;
    __syncwarp();
  }
  int n = 0, emax = -1;
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
    if (c * 32 >= total) break;
    const int idx = c * 32 + lane;
    const int i = idx < total ? idx / p.S : 0;
    const int j = idx - i * p.S;
    const int cnt_i = __shfl_sync(kFull, cnt, i);
    const int seq0_i = __shfl_sync(kFull, seq0, i);
    const int slen_i = __shfl_sync(kFull, slen, i);
    const int trel_i = __shfl_sync(kFull, trel, i);
    const int e = ev[c];
    const int nb = (slen_i + BS - 1) / BS;
    const bool valid = idx < total && j < cnt_i && e >= 0 && e < nb && (!p.causal || e * BS <= trel_i);
    if (use_map) {
      if (valid) {
        atomicOr(&bmap[e], 1u << i);
        emax = max(emax, e);
      }
    } else {
      const unsigned bal = __ballot_sync(kFull, valid);
      if (valid)
        keys[n + __popc(bal & lt_mask)] =
            (static_cast<uint64_t>(static_cast<uint32_t>(seq0_i + e * BS)) << 16) | (1u << i);
      n += __popc(bal);
    }
  }
  int nu = 0;
  if (use_map) {
    __syncwarp();
    const int nscan = __reduce_max_sync(kFull, emax) + 1;
    for (int base = 0; base < nscan; base += 32) {
      const int idx = base + lane;
      const uint32_t bits = idx < nscan ? bmap[idx] : 0u;
      const unsigned bal = __ballot_sync(kFull, bits != 0u);
      if (bits != 0u) {
        const int pos = nu + __popc(bal & lt_mask);
        it.ux[pos] = map_seq0 + idx * BS;
        it.ubits[pos] = static_cast<unsigned short>(bits);
      }
      nu += __popc(bal);
    }
  } else {
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
  }
  if (lane < kMaxNT) it.limit[lane] = limit;
  const unsigned tv_bits = __ballot_sync(kFull, tv);
  if (lane == 0) {
    it.g = g;
    it.hkv = hkv;
    it.n_union = nu;
    it.n_tiles = BS <= kTileKeys ? (nu * BS + kTileKeys - 1) / kTileKeys : nu * (BS / kTileKeys);
    it.tok_valid = tv_bits;
  }
  __syncwarp();
}

template <int D, int BS>
__global__ void __launch_bounds__(kThreads, 1)
nsa_union_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const Params p) {
  using C = Cfg<D, BS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem + C::kOffSort);
  float2* ml = reinterpret_cast<float2*>(smem + C::kOffMl);
  uint64_t* bb = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  uint64_t* item_full = bb;   bb += kItemSlots;
  uint64_t* item_empty = bb;  bb += kItemSlots;
  uint64_t* st_full = bb;     bb += C::kStages;  // ring: an item's Q, then one stage per pair
  uint64_t* st_empty = bb;    bb += C::kStages;
  uint64_t* q_used = bb;      bb += 1;   // last QK of an item done: TMEM Q may be replaced
  uint64_t* s_full = bb;      bb += 1;   // S of the current pair written
  uint64_t* s_empty = bb;     bb += 1;   // both warpgroups have read it
  uint64_t* p_full = bb;      bb += 2;   // per warpgroup
  uint64_t* pv_done = bb;     bb += 2;
  uint64_t* o_empty = bb;     bb += 1;
  uint64_t* mma_done = bb;    bb += 2;   // per issuing thread
  uint64_t* xch = bb;                    // (m, l) exchange between the two warpgroups
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  const Abort ab{abort_flag, &g_err_nsa, 1u, p.wait_limit};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto item_at = [&](int slot) -> Item& {
    return *reinterpret_cast<Item*>(smem + C::kOffItems + slot * C::kItemBytes);
  };

  if (threadIdx.x == 0) {
    // item slots are released by the loader, the two MMA threads and the 8 softmax warps
    for (int i = 0; i < kItemSlots; ++i) { mbar_init(&item_full[i], 1); mbar_init(&item_empty[i], 11); }
    for (int i = 0; i < C::kStages; ++i) { mbar_init(&st_full[i], 1); mbar_init(&st_empty[i], 1); }
    mbar_init(q_used, 1);
    mbar_init(s_full, 1); mbar_init(s_empty, 8);
    for (int i = 0; i < 2; ++i) { mbar_init(&p_full[i], 4); mbar_init(&pv_done[i], 1); }
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

  if (warp == 2) {
    // ------------------------------------------------------------------ item builder
    int islot = 0; uint32_t iphase = 0;
    int cached_seq = 0;
    // Items are handed out one at a time from the launch's counter once a slot is free,
    // so a CTA that drew small unions takes more: the kernel ends near the average CTA
    // load instead of the heaviest fixed share.  They go out from the last token group to
    // the first: under causal masking later tokens see more blocks, so the large unions
    // are taken first and the small ones fill the end.
    while (true) {
      if (!warp_wait(&item_empty[islot], iphase ^ 1, ab, kRoleBuilder, kBarItemEmpty, -1)) break;
      int item = 0;
      if (lane == 0) item = p.n_items - 1 - atomicAdd(&p.sched[0], 1);
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item < p.item0) {
        // no more items: publish the end marker
        if (lane == 0) {
          item_at(islot).n_tiles = -1;
          mbar_arrive(&item_full[islot]);
        }
        __syncwarp();
        break;
      }
      const int g = item / p.Hkv, hkv = item - g * p.Hkv;
      build_item<BS>(p, g, hkv, lane, cached_seq, item_at(islot), keys);
      if (lane == 0) mbar_arrive(&item_full[islot]);
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------------ loader
    int islot = 0; uint32_t iphase = 0;
    int stage = 0; uint32_t phase = 0;
    // stage i issued / parity of its last load in bit i (bit sets: indexed at run time, an
    // array would live in local memory)
    uint32_t issued = 0u, last_parity = 0u;
    const uint32_t q_box_bytes = static_cast<uint32_t>(C::kPanels * 128 * p.G * p.NT);
    bool ok = true;
    while (ok) {
      if (!warp_wait(&item_full[islot], iphase, ab, kRoleLoader, kBarItemFull, -1)) break;
      const Item& it = item_at(islot);
      const int nt = it.n_tiles, nu = it.n_union, hkv = it.hkv;
      if (nt < 0) break;  // no more items
      const int item = it.g * p.Hkv + hkv;
      const int np = (nt + 1) / 2;
      for (int pp = np > 0 ? -1 : 0; pp < np; ++pp) {  // pp = -1: the item's Q
        if (!warp_wait(&st_empty[stage], phase ^ 1, ab, kRoleLoader, kBarKvEmpty, item)) { ok = false; break; }
        if (lane == 0) {
          uint64_t* fb = &st_full[stage];
          uint8_t* kdst = smem + C::kOffStages + stage * C::kStageBytes;
          uint8_t* vdst = kdst + C::kKBytes;
          if (pp < 0) {
            mbar_arrive_expect_tx(fb, q_box_bytes);
            if (p.ranked) {
              // one box (G heads) per token slot; an empty slot reads zeros past the end
              for (int i = 0; i < p.NT; ++i) {
                const int tk = it.tok[i] >= 0 ? it.tok[i] : p.n_tok;
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                  tma_load_3d(kdst + pn * C::kQPanelBytes + i * p.G * 128, &tm_q, fb, pn * 64,
                              hkv * p.G, tk);
              }
            } else {
#pragma unroll
              for (int pn = 0; pn < C::kPanels; ++pn)
                tma_load_3d(kdst + pn * C::kQPanelBytes, &tm_q, fb, pn * 64, hkv * p.G, it.g * p.NT);
            }
          } else {
            mbar_arrive_expect_tx(fb, C::kStageBytes);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const int t = 2 * pp + hh;
#pragma unroll
              for (int e = 0; e < C::kSegs; ++e) {
                int row0;
                if constexpr (BS <= kTileKeys) {
                  const int ui = t * C::kSegs + e;
                  // a missing block is read from beyond the last token: TMA fills zeros
                  row0 = ui < nu ? it.ux[ui] : p.n_tok;
                } else {
                  const int ui = t / (BS / kTileKeys);
                  row0 = ui < nu ? it.ux[ui] + (t % (BS / kTileKeys)) * kTileKeys : p.n_tok;
                }
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn) {
                  const int off = pn * C::kPanelBytes + (hh * kTileKeys + e * C::kSegLen) * 128;
                  tma_load_3d(kdst + off, &tm_k, fb, pn * 64, hkv, row0);
                  tma_load_3d(vdst + off, &tm_v, fb, pn * 64, hkv, row0);
                }
              }
            }
          }
        }
        issued |= 1u << stage;
        last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[islot]);
      if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
    }
    // Drain: wait (bounded) for every copy this warp issued before the CTA exits.
    if (lane == 0)
      for (int s = 0; s < C::kStages; ++s)
        if ((issued >> s) & 1u) drain_wait(&st_full[s], (last_parity >> s) & 1u);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ QK issuer
    // Two warps issue the MMAs (QK here, PV in warp 3): a warp's wait on a barrier stalls
    // only its own stream while the tensor core runs the other's MMAs.  Each runs its
    // loop converged; one elected lane issues the tcgen05 operations, lane 0 the plain
    // arrivals.
    {
      const uint32_t leader = elect_one();
      int islot = 0; uint32_t iphase = 0;
      uint32_t quphase = 0, sphase = 0;
      bool q_in_use = false;  // a QK of an earlier item may still read the TMEM copy of Q
      int stage = 0; uint32_t phase = 0;
      bool ok = true;
      // descriptors of the shared-memory operands; a byte offset x adds x >> 4
      const uint64_t st_desc0 = make_sdesc(smem_base + C::kOffStages, 16, 1024, kLayoutSW128);
      while (ok) {
        if (!warp_wait(&item_full[islot], iphase, ab, kRoleMma, kBarItemFull, -1)) break;
        const int nt = item_at(islot).n_tiles;
        if (nt < 0) break;  // no more items
        const int item = item_at(islot).g * p.Hkv + item_at(islot).hkv;
        if (lane == 0) mbar_arrive(&item_empty[islot]);
        if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
        const int np = (nt + 1) / 2;
        if (np == 0) continue;
        // Q of this item (its first ring stage) -> TMEM, once the previous item's QKs are done
        if (!warp_wait(&st_full[stage], phase, ab, kRoleMma, kBarQFull, item)) break;
        if (q_in_use) {
          if (!warp_wait(q_used, quphase, ab, kRoleMma, kBarQEmpty, item)) break;
          quphase ^= 1;
        }
        tc_fence_after();
        {
          const uint64_t qd = st_desc0 + static_cast<uint64_t>((stage * C::kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tmem_cp_128x256b_by(leader, tmem + C::kQCol + kk * 8,
                             qd + static_cast<uint64_t>(((kk / 4) * C::kQPanelBytes + (kk % 4) * 32) >> 4));
        }
        mma_commit_by(leader, &st_empty[stage]);
        if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        for (int pp = 0; pp < np; ++pp) {
          if (!warp_wait(&st_full[stage], phase, ab, kRoleMma, kBarKvFull, item) ||
              !warp_wait(s_empty, sphase ^ 1, ab, kRoleMma, kBarSEmpty, item)) { ok = false; break; }
          sphase ^= 1;
          tc_fence_after();
          const uint64_t kd = st_desc0 + static_cast<uint64_t>((stage * C::kStageBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            mma_f16_ts_by(leader, tmem + C::kSCol, tmem + C::kQCol + kk * 8,
                       kd + static_cast<uint64_t>(((kk / 4) * C::kPanelBytes + (kk % 4) * 32) >> 4),
                       C::kIdescQK, kk > 0);
          mma_commit_by(leader, s_full);
          if (pp == np - 1) {
            mma_commit_by(leader, q_used);
            q_in_use = true;
          }
          if (++stage == C::kStages) { stage = 0; phase ^= 1; }
        }
      }
      // every tcgen05 op issued by this thread has finished once mma_done fires
      mma_commit_by(leader, &mma_done[0]);
      drain_wait(&mma_done[0], 0);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ------------------------------------------------------------------ PV issuer
    {
      const uint32_t leader = elect_one();
      int islot = 0; uint32_t iphase = 0;
      int stage = 0;
      uint32_t pph[2] = {0u, 0u};
      uint32_t ophase = 0;
      bool ok = true;
      const uint64_t v_desc0 =
          make_sdesc(smem_base + C::kOffStages + C::kKBytes, C::kPanelBytes, 1024, kLayoutSW128);
      while (ok) {
        if (!warp_wait(&item_full[islot], iphase, ab, kRoleMma, kBarItemFull, -1)) break;
        const int nt = item_at(islot).n_tiles;
        if (nt < 0) break;  // no more items
        const int item = item_at(islot).g * p.Hkv + item_at(islot).hkv;
        if (lane == 0) mbar_arrive(&item_empty[islot]);
        if (++islot == kItemSlots) { islot = 0; iphase ^= 1; }
        const int np = (nt + 1) / 2;
        if (np == 0) continue;
        if (++stage == C::kStages) stage = 0;  // the item's Q stage (released by the QK thread)
        // Per pair, warpgroup w's half: O_w (+)= P_w (A in TMEM, 64 keys) * V[64 w ..
        // 64 w + 63]; the first pair of an item overwrites O_w.  A PV follows its tile's
        // softmax, which follows the pair's QK, so the stage is free once both are done.
        for (int pp = 0; pp < np && ok; ++pp) {
          const uint64_t vd = v_desc0 + static_cast<uint64_t>((stage * C::kStageBytes) >> 4);
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            if (!warp_wait(&p_full[w], pph[w], ab, kRoleMma, kBarPFull, item)) { ok = false; break; }
            pph[w] ^= 1;
            if (pp == 0 && w == 0) {
              if (!warp_wait(o_empty, ophase ^ 1, ab, kRoleMma, kBarOEmpty, item)) { ok = false; break; }
              ophase ^= 1;
            }
            tc_fence_after();
#pragma unroll
            for (int k = 0; k < kTileKeys / 16; ++k)
              mma_f16_ts_by(leader, tmem + C::kOCol + w * D, tmem + C::kPCol + w * (kTileKeys / 2) + k * 8,
                         vd + static_cast<uint64_t>(((w * kTileKeys + k * 16) * 128) >> 4), C::kIdescPV,
                         (pp == 0 && k == 0) ? 0u : 1u);
            mma_commit_by(leader, &pv_done[w]);
          }
          if (!ok) break;
          mma_commit_by(leader, &st_empty[stage]);
          if (++stage == C::kStages) stage = 0;
        }
      }
      mma_commit_by(leader, &mma_done[1]);
      drain_wait(&mma_done[1], 0);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax / epilogue
    const int w = (warp - 4) >> 2;   // warpgroup: tile 2 pp + w of every pair pp
    const int q4 = warp & 3;         // TMEM lane quadrant of this warp
    const int r = q4 * 32 + lane;    // row of the tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const uint32_t s_col = tmem + lane_off + C::kSCol + w * kTileKeys;
    const uint32_t o_col = tmem + lane_off + C::kOCol + w * D;
    const uint32_t p_col = tmem + lane_off + C::kPCol + w * (kTileKeys / 2);
    const int ti = r < p.rows ? r / p.G : 0;  // token of this row within the item
    const int h = r - ti * p.G;
    int islot = 0; uint32_t iphase = 0;
    uint32_t sph = 0, pvph = 0, xph = 0;
    int par = 0;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    while (true) {
      if (!warp_wait(&item_full[islot], iphase, ab, kRoleSoftmax, kBarItemFull, -1)) break;
      const Item& it = item_at(islot);
      const int nt = it.n_tiles, nu = it.n_union;
      if (nt < 0) break;  // no more items
      const int item = it.g * p.Hkv + it.hkv;
      const int np = (nt + 1) / 2;
      const bool row_ok = r < p.rows && ((it.tok_valid >> ti) & 1u);
      const int limit = r < p.rows ? it.limit[ti] : -1;
      const unsigned tbit = 1u << ti;
      float m = -INFINITY, l = 0.f;  // log2 units, lazily moved reference max
      bool ok = true;
      for (int pp = 0; pp < np; ++pp) {
        const int t = 2 * pp + w;
        // valid keys of each segment of this warpgroup's tile for this row's token
        int nv[C::kSegs];
        int nvsum = 0;
#pragma unroll
        for (int e = 0; e < C::kSegs; ++e) {
          int ui, x0;
          if constexpr (BS <= kTileKeys) {
            ui = t * C::kSegs + e;
            x0 = ui < nu ? it.ux[ui] : 0;
          } else {
            ui = t / (BS / kTileKeys);
            x0 = ui < nu ? it.ux[ui] + (t % (BS / kTileKeys)) * kTileKeys : 0;
          }
          const bool sel = ui < nu && (it.ubits[ui] & tbit) != 0u;
          nv[e] = sel ? min(max(limit - x0 + 1, 0), C::kSegLen) : 0;
          nvsum += nv[e];
        }
        const bool any = __any_sync(0xffffffffu, nvsum > 0);
        if (!warp_wait(s_full, sph, ab, kRoleSoftmax, kBarSFull, item)) { ok = false; break; }
        sph ^= 1;
        float x[kTileKeys];
        if (any) {
          // both loads in flight, one wait
          tc_fence_after();
          tmem_ld_32x32b_x32_nw(s_col, x);
          tmem_ld_32x32b_x32_nw(s_col + 32, x + 32);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < kTileKeys; ++j) tmem_ld_ready(x[j]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty);
        float m_new = m, alpha = 1.f, psum = 0.f;
        uint32_t pk[kTileKeys / 2];
        if (any) {
          // masked raw scores (keys of a segment past its valid count), the valid keys as
          // keep bits in two 32-bit words: one bit test and one select per score
          static_assert(kTileKeys == 64 && (C::kSegLen == 32 || C::kSegLen == 64), "keep words");
          uint32_t kw[2];
          if constexpr (C::kSegLen == 64) {
            kw[0] = nv[0] >= 32 ? 0xffffffffu : (1u << nv[0]) - 1u;
            kw[1] = nv[0] >= 64 ? 0xffffffffu : (nv[0] > 32 ? (1u << (nv[0] - 32)) - 1u : 0u);
          } else {
#pragma unroll
            for (int e = 0; e < 2; ++e) kw[e] = nv[e] >= 32 ? 0xffffffffu : (1u << nv[e]) - 1u;
          }
          if (!__all_sync(0xffffffffu, (kw[0] & kw[1]) == 0xffffffffu)) {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = (kw[0] & (1u << j)) ? x[j] : -INFINITY;
#pragma unroll
            for (int j = 0; j < 32; ++j) x[32 + j] = (kw[1] & (1u << j)) ? x[32 + j] : -INFINITY;
          }
          // maximum: eight chains of three-input max; chain u takes the keys u, u + 8, ...
          float mx[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) mx[u] = fmaxf(x[u], x[u + 8]);
#pragma unroll
          for (int j = 16; j < kTileKeys; j += 16) {
#pragma unroll
            for (int u = 0; u < 8; ++u) mx[u] = fmax3f(mx[u], x[j + u], x[j + 8 + u]);
          }
          const float tmax = fmax3f(fmax3f(mx[0], mx[1], mx[2]), fmax3f(mx[3], mx[4], mx[5]),
                                    fmaxf(mx[6], mx[7])) * p.scale_log2;
          // lazy online softmax: move the reference max only when it grows by > 2^8
          if (tmax > m + kRescaleThreshold || (m == -INFINITY && tmax != -INFINITY)) m_new = tmax;
          alpha = (m == -INFINITY || m_new == m) ? (m_new == m ? 1.f : 0.f) : ex2(m - m_new);
          // exponentials, P as bf16 pairs and the row sum; the argument x * scale - m and
          // the sum run two lanes per instruction
          const uint64_t scale2 = pack_f32x2(p.scale_log2, p.scale_log2);
          const uint64_t negm2 = pack_f32x2(-m_new, -m_new);
          uint64_t ps2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int e = 0; e < C::kSegs; ++e) {
            if (nv[e] > 0) {
#pragma unroll
              for (int jj = 0; jj < C::kSegLen; jj += 2) {
                const int j = e * C::kSegLen + jj;
                const uint64_t a2 = fma_f32x2(pack_f32x2(x[j], x[j + 1]), scale2, negm2);
                float a0, a1;
                unpack_f32x2(a2, a0, a1);
                const float e0 = ex2(a0), e1 = ex2(a1);
                ps2[(j >> 1) & 3] = add_f32x2(ps2[(j >> 1) & 3], pack_f32x2(e0, e1));
                __nv_bfloat162 h2 = __floats2bfloat162_rn(e0, e1);
                pk[j >> 1] = *reinterpret_cast<uint32_t*>(&h2);
              }
            } else {
#pragma unroll
              for (int jj = 0; jj < C::kSegLen; jj += 2) pk[(e * C::kSegLen + jj) >> 1] = 0u;
            }
          }
          const uint64_t s01 = add_f32x2(ps2[0], ps2[1]), s23 = add_f32x2(ps2[2], ps2[3]);
          float lo, hi;
          unpack_f32x2(add_f32x2(s01, s23), lo, hi);
          psum = lo + hi;
        } else {
#pragma unroll
          for (int j = 0; j < kTileKeys / 2; ++j) pk[j] = 0u;
        }
        l = l * alpha + psum;
        // this warpgroup's previous PV must be done before its P is replaced and its O
        // rescaled
        if (pp > 0) {
          if (!warp_wait(&pv_done[w], pvph, ab, kRoleSoftmax, kBarPvDone, item)) { ok = false; break; }
          pvph ^= 1;
          tc_fence_after();
        }
        // P row (bf16 pairs, key order) into this warpgroup's TMEM P columns
        tmem_st_32x32b_x32_u(p_col, pk);
        if (pp > 0) {
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
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[w]);
      }
      if (!ok) break;
      if (np > 0) {
        if (!warp_wait(&pv_done[w], pvph, ab, kRoleSoftmax, kBarPvDone, item)) break;
        pvph ^= 1;
      }
      // merge the two warpgroups' partial results row by row
      ml[(par * 2 + w) * kRows + r] = make_float2(m, l);
      __syncwarp();
      if (lane == 0) mbar_arrive(xch);
      if (!warp_wait(xch, xph, ab, kRoleSoftmax, kBarXch, item)) break;
      xph ^= 1;
      const float2 oth = ml[(par * 2 + (w ^ 1)) * kRows + r];
      const float mx = fmaxf(m, oth.x);
      const float a_me = l > 0.f ? ex2(m - mx) : 0.f;
      const float a_ot = oth.y > 0.f ? ex2(oth.x - mx) : 0.f;
      const float L = l * a_me + oth.y * a_ot;
      const float a0 = w == 0 ? a_me : a_ot, a1 = w == 0 ? a_ot : a_me;
      constexpr int kOutHalf = D / 2;
      const long long orow = (long long)(row_ok ? it.tok[ti] : 0) * p.Hq + (long long)it.hkv * p.G + h;
      const float gate =
          (p.g_slc != nullptr && row_ok) ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.g_slc)[orow]) : 1.f;
      const float inv = L > 0.f ? gate / L : 0.f;
      if (np > 0) {
        tc_fence_after();
        // O = (O_0 a0 + O_1 a1) * gate / L, with the factor folded into both weights: two
        // columns per packed multiply and multiply-add
        const uint64_t a0i = pack_f32x2(a0 * inv, a0 * inv), a1i = pack_f32x2(a1 * inv, a1 * inv);
#pragma unroll
        for (int c = 0; c < kOutHalf / 32; ++c) {
          const int col = w * kOutHalf + c * 32;
          float o0[32], o1[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::kOCol + col, o0);
          tmem_ld_32x32b_x32(tmem + lane_off + C::kOCol + D + col, o1);
          if (c == kOutHalf / 32 - 1) {
            // O_0 and O_1 are read: the next item's first PV may overwrite them
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(o_empty);
          }
          if (row_ok) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              uint32_t wv[4];
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int j0 = j + 2 * u;
                float v0, v1;
                unpack_f32x2(fma_f32x2(pack_f32x2(o1[j0], o1[j0 + 1]), a1i,
                                       mul_f32x2(pack_f32x2(o0[j0], o0[j0 + 1]), a0i)),
                             v0, v1);
                __nv_bfloat162 h2 = __floats2bfloat162_rn(v0, v1);
                wv[u] = *reinterpret_cast<uint32_t*>(&h2);
              }
              *reinterpret_cast<uint4*>(out + orow * D + col + j) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
          }
        }
      } else if (row_ok) {
#pragma unroll
        for (int j = 0; j < kOutHalf; j += 8)
          *reinterpret_cast<uint4*>(out + orow * D + w * kOutHalf + j) = make_uint4(0u, 0u, 0u, 0u);
      }
      if (w == 0 && row_ok && p.lse != nullptr) p.lse[orow] = L > 0.f ? (mx + log2f(L)) * kLn2 : -INFINITY;
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
  // every builder of the launch has stopped drawing items once all CTAs counted
  // themselves here: the last one leaves the counter zero for the next launch
  if (threadIdx.x == 0 && atomicAdd(&p.sched[1], 1) == static_cast<int>(gridDim.x) - 1) {
    p.sched[0] = 0;
    p.sched[1] = 0;
    __threadfence();
  }
}


// ---------------------------------------------------------------------------- fp32
constexpr int kF32Threads = 128;
constexpr int kF32MaxBlock = 128;  // largest block size

template <int D>
__global__ void __launch_bounds__(kF32Threads)
nsa_select_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                      const float* __restrict__ v, const Params p) {
  __shared__ float q_s[kNH][D];
  __shared__ float s_s[kNH][kF32MaxBlock + 1];
  __shared__ float m_s[kNH], a_s[kNH];
  __shared__ int blocks_s[kMaxSel];
  __shared__ int meta_s[4];
  const int tid = threadIdx.x, lane = tid & 31;
  float* out = static_cast<float*>(p.out);
  int cached_seq = 0;
  for (int item = p.item0 + blockIdx.x; item < p.n_items; item += gridDim.x) {
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
    const float* gates = static_cast<const float*>(p.g_slc);
    if (tid < D) {
#pragma unroll
      for (int h = 0; h < kNH; ++h)
        if (h < p.G) {
          const float g = gates != nullptr ? gates[out_row0 + h] : 1.f;
          out[(out_row0 + h) * D + tid] = a_s[h] > 0.f ? g * (o[h] / a_s[h]) : 0.f;
        }
    }
    if (p.lse != nullptr && tid < p.G)
      p.lse[out_row0 + tid] = a_s[tid] > 0.f ? m_s[tid] + logf(a_s[tid]) : -INFINITY;
  }
}

// Device address of this launch's item counters (the slot after the previous launch's).
int sched_slot(int** out) {
  static std::mutex mu;
  static int* base[64] = {};
  static unsigned next = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "nsa_select: cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(SBA_ERR_UNSUPPORTED, "nsa_select: device ordinal >= 64");
  std::lock_guard<std::mutex> lock(mu);
  if (base[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_nsa_sched);
    if (e != cudaSuccess || ptr == nullptr) return cuda_error(e, "nsa_select: item counters");
    base[dev] = static_cast<int*>(ptr);
  }
  *out = base[dev] + 2 * (next++ % kSchedSlots);
  return SBA_OK;
}

template <int D, int BS>
int launch_bf16(const void* q, const void* k, const void* v, const Params& p_in, cudaStream_t stream) {
  using C = Cfg<D, BS>;
  Params p = p_in;
  if (int rc = sched_slot(&p.sched)) return rc;
  const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tq, tk, tv;
  {
    // Q as (D, Hq, tokens): one box = 64 head-dim elements x G heads x NT tokens, i.e.
    // rows (token-major, head-minor) of one item
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hq, (cuuint64_t)p.n_tok};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hq * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)p.G, (cuuint32_t)(p.ranked ? 1 : p.NT)};
    if (encode_tensor_map(&tq, dt, 3, const_cast<void*>(q), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "nsa_select: tensor map (q) failed");
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)p.Hkv, (cuuint64_t)p.n_tok};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)p.Hkv * D * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)C::kSegLen};
    if (encode_tensor_map(&tk, dt, 3, const_cast<void*>(k), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS ||
        encode_tensor_map(&tv, dt, 3, const_cast<void*>(v), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) != CUDA_SUCCESS)
      return set_error(SBA_ERR_CUDA, "nsa_select: tensor map (k/v) failed");
  }
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(nsa_union_kernel<D, BS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return cuda_error(e, "nsa_select: set smem attribute");
    attr_done = true;
  }
  const int grid = std::min(p.n_items - p.item0, num_sms());
  nsa_union_kernel<D, BS><<<grid, kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, p);
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

int launch_nsa_select(const void* q, const void* k, const void* v, const void* g_slc,
                      const int32_t* block_indices,
                      const int32_t* block_counts, int block_count_scalar, int S,
                      const int32_t* cu_seqlens, int num_seqs, int B, int T, int Hq, int Hkv,
                      int D, int block_size, int causal, float scale, int dtype, void* out,
                      float* lse, cudaStream_t stream, long long tok_begin, long long tok_end) {
  Params p;
  p.g_slc = g_slc;
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
  p.NT = std::min(kMaxNT, kRows / p.G);
  p.rows = p.NT * p.G;
  p.ranked = 0;
  p.item0 = 0;
  p.wait_limit = wait_timeout_cycles();
  if ((long long)B * T * Hkv >= (1LL << 31)) return set_error(SBA_ERR_UNSUPPORTED, "nsa_select: too many items");
  p.n_tok = B * T;
  if (dtype == SBA_BF16) {
    // Count-ranked items need a token's Q rows to start a 1024-byte swizzle atom in the
    // item's Q stage (G >= 8); smaller groups take consecutive tokens.
    p.ranked = p.G >= 8 ? 1 : 0;
    const long long groups = p.ranked ? (p.n_tok + 8 * p.NT - 1) / (8 * p.NT) * 8
                                      : (p.n_tok + p.NT - 1) / p.NT;
    p.n_items = static_cast<int>(groups * Hkv);
    if (tok_begin > 0 || (tok_end >= 0 && tok_end < p.n_tok)) {
      // tokens [tok_begin, tok_end) only: the host keeps both ends multiples of 128 tokens
      // (whole count-ranked windows and groups), so they map to a contiguous item range
      const long long t1 = tok_end < 0 ? p.n_tok : tok_end;
      if (tok_begin % 128 != 0 || (t1 % 128 != 0 && t1 != p.n_tok) || tok_begin >= t1)
        return set_error(SBA_ERR_INVALID_ARG, "nsa_select: token range must be 128-aligned");
      p.item0 = static_cast<int>(tok_begin / p.NT * Hkv);
      p.n_items = static_cast<int>(std::min<long long>((t1 + p.NT - 1) / p.NT * Hkv, p.n_items));
    }
    if (D == 128) return dispatch_bs<128>(block_size, q, k, v, p, stream);
    return dispatch_bs<64>(block_size, q, k, v, p, stream);
  }
  p.n_items = B * T * Hkv;
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
