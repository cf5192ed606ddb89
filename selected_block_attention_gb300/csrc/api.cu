// C ABI of libsba: argument validation, error reporting, and dispatch to the kernel
// launchers.  Nothing here computes attention; every step of the path runs in the
// kernels of the other translation units.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <string>

#include "common.cuh"

namespace sba {

static thread_local std::string g_last_error;

int set_error(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_error(cudaError_t e, const char* what) {
  return set_error(SBA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
static std::once_flag g_encode_once;

CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank,
                           void* gaddr, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                           const cuuint32_t* box, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return CUDA_ERROR_NOT_FOUND;
  cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  return g_encode(map, dtype, rank, gaddr, dims, strides_bytes, box, elem_strides,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

static std::atomic<long long> g_wait_limit{kWaitTimeoutCycles};

long long wait_timeout_cycles() { return g_wait_limit.load(std::memory_order_relaxed); }

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n = 1;
  }
  return n;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr int kHostChunks = 8;  // chunks of the host-buffer entry point (16 measured no faster)

// Two non-blocking streams per device for the host-buffer entry point: one carries the
// host-to-device copies, the other the device-to-host copies.  Created on first use and
// kept for the life of the process; calls that share a device share them.
constexpr int kCopyStreams = 1;  // per direction (two measured slower: the copies share the link)
struct CopyStreams {
  cudaStream_t in[kCopyStreams] = {}, out[kCopyStreams] = {};
};
static std::mutex g_copy_mutex;
static CopyStreams g_copy_streams[64];

static int copy_streams(CopyStreams** cs) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return set_error(SBA_ERR_UNSUPPORTED, "device ordinal must be < 64");
  std::lock_guard<std::mutex> lock(g_copy_mutex);
  CopyStreams& c = g_copy_streams[dev];
  if (c.in[0] == nullptr) {
    CopyStreams fresh;
    for (int i = 0; i < kCopyStreams && e == cudaSuccess; ++i) {
      e = cudaStreamCreateWithFlags(&fresh.in[i], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&fresh.out[i], cudaStreamNonBlocking);
    }
    if (e != cudaSuccess) {
      for (int i = 0; i < kCopyStreams; ++i) {
        if (fresh.in[i]) cudaStreamDestroy(fresh.in[i]);
        if (fresh.out[i]) cudaStreamDestroy(fresh.out[i]);
      }
      return cuda_error(e, "copy stream");
    }
    c = fresh;
  }
  *cs = &c;
  return SBA_OK;
}

// Device staging layout of the host-buffer NSA entry: every array whole (all B rows),
// each starting on a 256-byte boundary.
struct NsaHostLayout {
  size_t q, k, v, idx, cnt, g, out, lse, total;
  size_t q_row, kv_row, idx_row, cnt_row, g_row, lse_row;  // bytes per batch row
};
static size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
static NsaHostLayout nsa_host_layout(int B, int T, int Hq, int Hkv, int D, int S, int dtype,
                                     bool has_counts, bool has_gate, bool has_lse) {
  NsaHostLayout L{};
  const size_t esz = dtype == SBA_F32 ? 4 : 2;
  L.q_row = static_cast<size_t>(T) * Hq * D * esz;
  L.kv_row = static_cast<size_t>(T) * Hkv * D * esz;
  L.idx_row = static_cast<size_t>(T) * Hkv * S * 4;
  L.cnt_row = has_counts ? static_cast<size_t>(T) * Hkv * 4 : 0;
  L.g_row = has_gate ? static_cast<size_t>(T) * Hq * esz : 0;
  L.lse_row = has_lse ? static_cast<size_t>(T) * Hq * 4 : 0;
  size_t off = 0;
  L.q = off;   off += round256(L.q_row * B);
  L.k = off;   off += round256(L.kv_row * B);
  L.v = off;   off += round256(L.kv_row * B);
  L.idx = off; off += round256(L.idx_row * B);
  L.cnt = off; off += round256(L.cnt_row * B);
  L.g = off;   off += round256(L.g_row * B);
  L.out = off; off += round256(L.q_row * B);
  L.lse = off; off += round256(L.lse_row * B);
  L.total = off;
  return L;
}

}  // namespace sba

using namespace sba;

#define SBA_REQUIRE(cond, msg)                                                  \
  do {                                                                          \
    if (!(cond)) return set_error(SBA_ERR_INVALID_ARG, std::string(__func__) + ": " + (msg)); \
  } while (0)
#define SBA_SUPPORT(cond, msg)                                                  \
  do {                                                                          \
    if (!(cond)) return set_error(SBA_ERR_UNSUPPORTED, std::string(__func__) + ": " + (msg)); \
  } while (0)

extern "C" {

const char* sba_version(void) { return "sba 0.1.0 sm_103a"; }

const char* sba_last_error(void) { return g_last_error.c_str(); }

int sba_set_wait_timeout_cycles(long long cycles) {
  g_last_error.clear();
  SBA_REQUIRE(cycles >= 0, "cycles must be >= 0 (0 restores the default)");
  g_wait_limit.store(cycles == 0 ? kWaitTimeoutCycles : cycles, std::memory_order_relaxed);
  return SBA_OK;
}

long long sba_get_wait_timeout_cycles(void) { return wait_timeout_cycles(); }

int sba_nsa_select_fwd(const void* q, const void* k, const void* v, const void* g_slc,
                       const int32_t* block_indices, const int32_t* block_counts,
                       int block_count_scalar, int S, const int32_t* cu_seqlens, int num_seqs,
                       int B, int T, int Hq, int Hkv, int D, int block_size, int causal,
                       float softmax_scale, int dtype, void* out, float* lse,
                       sba_stream_t stream) {
  g_last_error.clear();
  SBA_REQUIRE(q && k && v && block_indices && out, "null tensor pointer");
  SBA_REQUIRE(B >= 1 && T >= 1 && Hq >= 1 && Hkv >= 1, "sizes must be positive");
  SBA_REQUIRE(Hq % Hkv == 0, "Hq must be a multiple of Hkv");
  SBA_REQUIRE(S >= 1, "S (selected-block slots) must be >= 1");
  SBA_REQUIRE(dtype == SBA_BF16 || dtype == SBA_F32, "dtype must be SBA_BF16 or SBA_F32");
  SBA_REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out),
              "q, k, v and out must be 16-byte aligned");
  SBA_REQUIRE(cu_seqlens == nullptr || (num_seqs >= 1 && B == 1),
              "cu_seqlens needs num_seqs >= 1 and B == 1");
  SBA_REQUIRE(block_counts != nullptr || block_count_scalar >= 0,
              "block_count_scalar must be >= 0");
  SBA_REQUIRE(std::isfinite(softmax_scale), "softmax_scale must be finite");
  SBA_SUPPORT(D == 64 || D == 128, "D must be 64 or 128");
  SBA_SUPPORT(block_size == 32 || block_size == 64 || block_size == 128,
              "block_size must be 32, 64 or 128");
  SBA_SUPPORT(Hq / Hkv <= 16, "Hq / Hkv must be <= 16");
  SBA_SUPPORT(S <= 32, "S must be <= 32");
  SBA_SUPPORT((long long)B * T * Hq < (1LL << 31), "B * T * Hq must be < 2^31");
  float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  return launch_nsa_select(q, k, v, g_slc, block_indices, block_counts, block_count_scalar, S,
                           cu_seqlens, cu_seqlens ? num_seqs : 0, B, T, Hq, Hkv, D, block_size,
                           causal ? 1 : 0, scale, dtype, out, lse,
                           reinterpret_cast<cudaStream_t>(stream));
}

size_t sba_nsa_select_bwd_workspace_size(int B, int T, int Hq, int Hkv, int S, int num_seqs) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || S < 1 || num_seqs < 0) return 0;
  return nsa_bwd_workspace_bytes(B, T, Hq, Hkv, S, num_seqs);
}

int sba_nsa_select_bwd(const void* q, const void* k, const void* v, const void* out,
                       const float* lse, const void* d_out, const int32_t* block_indices,
                       const int32_t* block_counts, int block_count_scalar, int S,
                       const int32_t* cu_seqlens, int num_seqs, int B, int T, int Hq, int Hkv, int D,
                       int block_size, int causal, float softmax_scale, int dtype, void* dq,
                       void* dk, void* dv, void* workspace, size_t workspace_bytes,
                       sba_stream_t stream) {
  g_last_error.clear();
  SBA_REQUIRE(q && k && v && out && lse && d_out && block_indices && dq && dk && dv,
              "null tensor pointer");
  SBA_REQUIRE(B >= 1 && T >= 1 && Hq >= 1 && Hkv >= 1, "sizes must be positive");
  SBA_REQUIRE(Hq % Hkv == 0, "Hq must be a multiple of Hkv");
  SBA_REQUIRE(S >= 1, "S (selected-block slots) must be >= 1");
  SBA_REQUIRE(dtype == SBA_BF16 || dtype == SBA_F32, "dtype must be SBA_BF16 or SBA_F32");
  SBA_REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out) && aligned16(d_out) &&
                  aligned16(dq) && aligned16(dk) && aligned16(dv) && aligned16(lse),
              "tensors must be 16-byte aligned");
  SBA_REQUIRE(cu_seqlens == nullptr || (num_seqs >= 1 && B == 1),
              "cu_seqlens needs num_seqs >= 1 and B == 1");
  SBA_REQUIRE(block_counts != nullptr || block_count_scalar >= 0,
              "block_count_scalar must be >= 0");
  SBA_REQUIRE(std::isfinite(softmax_scale), "softmax_scale must be finite");
  SBA_SUPPORT(dtype == SBA_BF16, "the backward supports bf16 only");
  SBA_SUPPORT(D == 128, "the backward supports D == 128 only");
  SBA_SUPPORT(block_size == 64, "the backward supports block_size == 64 only");
  SBA_SUPPORT(Hq / Hkv == 8 || Hq / Hkv == 16, "the backward supports Hq / Hkv in {8, 16}");
  SBA_SUPPORT(S <= 32, "S must be <= 32");
  SBA_SUPPORT((long long)B * T * Hq < (1LL << 31), "B * T * Hq must be < 2^31");
  const int ns = cu_seqlens ? num_seqs : 0;
  SBA_REQUIRE(workspace != nullptr && (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0 &&
                  workspace_bytes >= nsa_bwd_workspace_bytes(B, T, Hq, Hkv, S, ns),
              "workspace missing, not 256-byte aligned or smaller than "
              "sba_nsa_select_bwd_workspace_size()");
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  return launch_nsa_select_bwd(q, k, v, out, lse, d_out, block_indices, block_counts,
                               block_count_scalar, S, cu_seqlens, ns, B, T, Hq, Hkv, causal ? 1 : 0,
                               scale, dq, dk, dv, workspace, reinterpret_cast<cudaStream_t>(stream));
}

size_t sba_nsa_select_host_workspace_size(int B, int T, int Hq, int Hkv, int D, int S,
                                          int dtype, int has_counts, int has_gate,
                                          int has_lse) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || S < 1) return 0;
  if (dtype != SBA_BF16 && dtype != SBA_F32) return 0;
  return nsa_host_layout(B, T, Hq, Hkv, D, S, dtype, has_counts != 0, has_gate != 0,
                         has_lse != 0).total;
}

int sba_nsa_select_fwd_host(const void* q_h, const void* k_h, const void* v_h,
                            const void* g_slc_h, const int32_t* block_indices_h,
                            const int32_t* block_counts_h, int block_count_scalar, int S, int B,
                            int T, int Hq, int Hkv, int D, int block_size, int causal,
                            float softmax_scale, int dtype, void* out_h, float* lse_h,
                            void* workspace, size_t workspace_bytes, sba_stream_t stream) {
  g_last_error.clear();
  SBA_REQUIRE(q_h && k_h && v_h && block_indices_h && out_h, "null host pointer");
  SBA_REQUIRE(workspace != nullptr, "null workspace");
  SBA_REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 255u) == 0,
              "workspace must be 256-byte aligned");
  SBA_REQUIRE(B >= 1 && T >= 1 && Hq >= 1 && Hkv >= 1, "sizes must be positive");
  SBA_REQUIRE(Hq % Hkv == 0, "Hq must be a multiple of Hkv");
  SBA_REQUIRE(S >= 1, "S (selected-block slots) must be >= 1");
  SBA_REQUIRE(dtype == SBA_BF16 || dtype == SBA_F32, "dtype must be SBA_BF16 or SBA_F32");
  SBA_REQUIRE(block_counts_h != nullptr || block_count_scalar >= 0,
              "block_count_scalar must be >= 0");
  SBA_REQUIRE(std::isfinite(softmax_scale), "softmax_scale must be finite");
  SBA_SUPPORT(D == 64 || D == 128, "D must be 64 or 128");
  SBA_SUPPORT(block_size == 32 || block_size == 64 || block_size == 128,
              "block_size must be 32, 64 or 128");
  SBA_SUPPORT(Hq / Hkv <= 16, "Hq / Hkv must be <= 16");
  SBA_SUPPORT(S <= 32, "S must be <= 32");
  SBA_SUPPORT((long long)B * T * Hq < (1LL << 31), "B * T * Hq must be < 2^31");
  const NsaHostLayout L = nsa_host_layout(B, T, Hq, Hkv, D, S, dtype, block_counts_h != nullptr,
                                          g_slc_h != nullptr, lse_h != nullptr);
  SBA_REQUIRE(workspace_bytes >= L.total,
              "workspace too small (see sba_nsa_select_host_workspace_size)");
  CopyStreams* cs = nullptr;
  if (int rc = copy_streams(&cs)) return rc;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  // Chunks: for bf16 with T a multiple of 128, (batch row, token range) pieces of whole
  // 128-token spans, token-range major; a chunk's queries see keys up to its last token,
  // so under causal masking it only needs the K/V rows it adds to what earlier chunks of
  // its row copied (without causal masking the first chunk of a row copies the row's
  // K/V).  Otherwise whole batch rows.
  struct Chunk { int b0, rows; long long t0, t1, kv0, kv1; };
  Chunk chunks[kHostChunks];
  int nchunks = 0;
  if (dtype == SBA_BF16 && T % 128 == 0 && T >= 256 && B < kHostChunks) {
    const int per_row = std::max(1, std::min(kHostChunks / B, T / 128));
    const long long span = (static_cast<long long>(T) / 128 + per_row - 1) / per_row * 128;
    for (long long t0 = 0; t0 < T; t0 += span)
      for (int b = 0; b < B; ++b) {
        const long long t1 = std::min<long long>(t0 + span, T);
        const long long kv0 = causal ? t0 : (t0 == 0 ? 0 : T);
        const long long kv1 = causal ? t1 : T;
        chunks[nchunks++] = Chunk{b, 1, t0, t1, kv0, std::max(kv0, kv1)};
      }
  } else {
    const int n = B < kHostChunks ? B : kHostChunks;
    for (int c = 0; c < n; ++c) {
      const int r0 = static_cast<int>(static_cast<long long>(B) * c / n);
      const int rows = static_cast<int>(static_cast<long long>(B) * (c + 1) / n) - r0;
      chunks[nchunks++] = Chunk{r0, rows, 0, T, 0, T};
    }
  }

  // events: start, then per chunk "inputs copied" and "computed", then "outputs copied"
  // events: start, per chunk "inputs copied" and "computed", per output stream "done"
  cudaEvent_t ev[1 + 2 * kHostChunks + kCopyStreams];
  int nev = 0;
  auto cleanup = [&]() {
    for (int i = 0; i < nev; ++i) cudaEventDestroy(ev[i]);  // released once they complete
  };
  for (; nev < 1 + 2 * nchunks + kCopyStreams; ++nev) {
    cudaError_t e = cudaEventCreateWithFlags(&ev[nev], cudaEventDisableTiming);
    if (e != cudaSuccess) { cleanup(); return cuda_error(e, "event create"); }
  }
  cudaEvent_t ev_start = ev[0];
  cudaError_t e = cudaEventRecord(ev_start, st);
  for (int i = 0; i < kCopyStreams && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(cs->in[i], ev_start, 0);
  if (e != cudaSuccess) { cleanup(); return cuda_error(e, "stream ordering"); }
  cudaStream_t in_s = cs->in[0], out_s = cs->out[0];

  // rows [r0, r0 + rows) x tokens [t0, t1) of an array with `tok_bytes` per token: one
  // contiguous range when it covers one row or whole rows
  auto span_bytes = [&](size_t tok_bytes, int r0, int rows, long long t0, long long t1,
                        size_t& off, size_t& bytes) {
    off = (static_cast<size_t>(r0) * T + static_cast<size_t>(t0)) * tok_bytes;
    bytes = (rows == 1 ? static_cast<size_t>(t1 - t0) : static_cast<size_t>(rows) * T) * tok_bytes;
  };
  auto h2d = [&](size_t base, const void* src, size_t row_bytes, int r0, int rows, long long t0,
                 long long t1) {
    if (row_bytes == 0 || t1 <= t0) return cudaSuccess;
    size_t off, bytes;
    span_bytes(row_bytes / T, r0, rows, t0, t1, off, bytes);
    return cudaMemcpyAsync(ws + base + off, static_cast<const uint8_t*>(src) + off, bytes,
                           cudaMemcpyHostToDevice, in_s);
  };
  auto d2h = [&](void* dst, size_t base, size_t row_bytes, int r0, int rows, long long t0,
                 long long t1) {
    if (row_bytes == 0) return cudaSuccess;
    size_t off, bytes;
    span_bytes(row_bytes / T, r0, rows, t0, t1, off, bytes);
    return cudaMemcpyAsync(static_cast<uint8_t*>(dst) + off, ws + base + off, bytes,
                           cudaMemcpyDeviceToHost, out_s);
  };
  const bool split = nchunks > 0 && (chunks[0].t0 != 0 || chunks[0].t1 != T || nchunks > B);
  for (int c = 0; c < nchunks; ++c) {
    const Chunk& ch = chunks[c];
    cudaEvent_t ev_in = ev[1 + 2 * c], ev_k = ev[2 + 2 * c];
    // consecutive chunks alternate between the copy streams of each direction; the
    // compute stream waits for every chunk's inputs in chunk order, so a chunk's K/V
    // prefix (copied by earlier chunks on either stream) is complete when it runs
    in_s = cs->in[c % kCopyStreams];
    out_s = cs->out[c % kCopyStreams];
    e = h2d(L.q, q_h, L.q_row, ch.b0, ch.rows, ch.t0, ch.t1);
    if (e == cudaSuccess) e = h2d(L.k, k_h, L.kv_row, ch.b0, ch.rows, ch.kv0, ch.kv1);
    if (e == cudaSuccess) e = h2d(L.v, v_h, L.kv_row, ch.b0, ch.rows, ch.kv0, ch.kv1);
    if (e == cudaSuccess) e = h2d(L.idx, block_indices_h, L.idx_row, ch.b0, ch.rows, ch.t0, ch.t1);
    if (e == cudaSuccess && block_counts_h)
      e = h2d(L.cnt, block_counts_h, L.cnt_row, ch.b0, ch.rows, ch.t0, ch.t1);
    if (e == cudaSuccess && g_slc_h) e = h2d(L.g, g_slc_h, L.g_row, ch.b0, ch.rows, ch.t0, ch.t1);
    if (e == cudaSuccess) e = cudaEventRecord(ev_in, in_s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_in, 0);
    if (e != cudaSuccess) { cleanup(); return cuda_error(e, "host-to-device copy"); }
    int rc;
    if (split) {
      // the whole staged batch, restricted to this chunk's tokens
      rc = launch_nsa_select(
          ws + L.q, ws + L.k, ws + L.v, g_slc_h ? ws + L.g : nullptr,
          reinterpret_cast<const int32_t*>(ws + L.idx),
          block_counts_h ? reinterpret_cast<const int32_t*>(ws + L.cnt) : nullptr,
          block_count_scalar, S, nullptr, 0, B, T, Hq, Hkv, D, block_size, causal ? 1 : 0, scale,
          dtype, ws + L.out, lse_h ? reinterpret_cast<float*>(ws + L.lse) : nullptr, st,
          static_cast<long long>(ch.b0) * T + ch.t0, static_cast<long long>(ch.b0) * T + ch.t1);
    } else {
      const int r0 = ch.b0, rows = ch.rows;
      rc = launch_nsa_select(
          ws + L.q + L.q_row * r0, ws + L.k + L.kv_row * r0, ws + L.v + L.kv_row * r0,
          g_slc_h ? ws + L.g + L.g_row * r0 : nullptr,
          reinterpret_cast<const int32_t*>(ws + L.idx + L.idx_row * r0),
          block_counts_h ? reinterpret_cast<const int32_t*>(ws + L.cnt + L.cnt_row * r0) : nullptr,
          block_count_scalar, S, nullptr, 0, rows, T, Hq, Hkv, D, block_size, causal ? 1 : 0, scale,
          dtype, ws + L.out + L.q_row * r0,
          lse_h ? reinterpret_cast<float*>(ws + L.lse + L.lse_row * r0) : nullptr, st);
    }
    if (rc != SBA_OK) { cleanup(); return rc; }
    e = cudaEventRecord(ev_k, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(out_s, ev_k, 0);
    if (e == cudaSuccess) e = d2h(out_h, L.out, L.q_row, ch.b0, ch.rows, ch.t0, ch.t1);
    if (e == cudaSuccess && lse_h) e = d2h(lse_h, L.lse, L.lse_row, ch.b0, ch.rows, ch.t0, ch.t1);
    if (e != cudaSuccess) { cleanup(); return cuda_error(e, "device-to-host copy"); }
  }
  for (int i = 0; i < kCopyStreams && e == cudaSuccess; ++i) {
    cudaEvent_t ev_done = ev[1 + 2 * nchunks + i];
    e = cudaEventRecord(ev_done, cs->out[i]);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_done, 0);
  }
  cleanup();
  if (e != cudaSuccess) return cuda_error(e, "stream ordering");
  return SBA_OK;
}

int sba_sparse_mask_bounds(const int32_t* q_pos, const int32_t* q_seg, const int32_t* kv_pos,
                           const int32_t* kv_seg, int B, int Tq, int Tkv, int q_block,
                           int kv_block, int causal, int window_left, int window_right,
                           int padding_segment_id, int32_t* lower, int32_t* upper,
                           int32_t* lower_full, int32_t* upper_full, sba_stream_t stream) {
  g_last_error.clear();
  SBA_REQUIRE(q_pos && q_seg && kv_pos && kv_seg && lower && upper && lower_full && upper_full,
              "null pointer");
  SBA_REQUIRE(B >= 1 && Tq >= 1 && Tkv >= 1, "sizes must be positive");
  SBA_REQUIRE(q_block >= 1 && kv_block >= 1, "block sizes must be positive");
  SBA_REQUIRE(window_left >= -1 && window_right >= -1, "windows must be >= -1");
  SBA_SUPPORT(q_block <= 4096 && kv_block <= 4096, "block sizes must be <= 4096");
  SBA_SUPPORT(B <= 65535, "B must be <= 65535");
  SBA_SUPPORT((long long)B * ((Tq + q_block - 1) / q_block) < (1LL << 31), "too many blocks");
  return launch_sparse_mask_bounds(q_pos, q_seg, kv_pos, kv_seg, B, Tq, Tkv, q_block, kv_block,
                                   causal ? 1 : 0, window_left, window_right, padding_segment_id,
                                   lower, upper, lower_full, upper_full, 0,
                                   reinterpret_cast<cudaStream_t>(stream));
}

int sba_sparse_mask_dkdv_bounds(const int32_t* q_pos, const int32_t* q_seg,
                                const int32_t* kv_pos, const int32_t* kv_seg, int B, int Tq,
                                int Tkv, int q_block, int kv_block, int causal, int window_left,
                                int window_right, int padding_segment_id, int32_t* lower,
                                int32_t* upper, int32_t* lower_full, int32_t* upper_full,
                                sba_stream_t stream) {
  g_last_error.clear();
  SBA_REQUIRE(q_pos && q_seg && kv_pos && kv_seg && lower && upper && lower_full && upper_full,
              "null pointer");
  SBA_REQUIRE(B >= 1 && Tq >= 1 && Tkv >= 1, "sizes must be positive");
  SBA_REQUIRE(q_block >= 1 && kv_block >= 1, "block sizes must be positive");
  SBA_REQUIRE(window_left >= -1 && window_right >= -1, "windows must be >= -1");
  SBA_SUPPORT(q_block <= 4096 && kv_block <= 4096, "block sizes must be <= 4096");
  SBA_SUPPORT(B <= 65535, "B must be <= 65535");
  SBA_SUPPORT((long long)B * ((Tkv + kv_block - 1) / kv_block) < (1LL << 31), "too many blocks");
  return launch_sparse_mask_bounds(q_pos, q_seg, kv_pos, kv_seg, B, Tq, Tkv, q_block, kv_block,
                                   causal ? 1 : 0, window_left, window_right, padding_segment_id,
                                   lower, upper, lower_full, upper_full, 1,
                                   reinterpret_cast<cudaStream_t>(stream));
}

int sba_blocksparse_attn_fwd(const void* q, const void* k, const void* v, const int32_t* q_pos,
                             const int32_t* q_seg, const int32_t* kv_pos, const int32_t* kv_seg,
                             const int32_t* lower, const int32_t* upper,
                             const int32_t* lower_full, const int32_t* upper_full, int B, int T,
                             int Hq, int Hkv, int D, int q_block, int kv_block, int causal,
                             int window_left, int window_right, int padding_segment_id,
                             float softmax_scale, void* out, float* lse, sba_stream_t stream) {
  g_last_error.clear();
  SBA_REQUIRE(q && k && v && q_pos && q_seg && kv_pos && kv_seg && lower && upper &&
                  lower_full && upper_full && out,
              "null pointer");
  SBA_REQUIRE(B >= 1 && T >= 1 && Hq >= 1 && Hkv >= 1 && Hq % Hkv == 0, "bad head/size arguments");
  SBA_REQUIRE(window_left >= -1 && window_right >= -1, "windows must be >= -1");
  SBA_REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out) &&
                  aligned16(q_pos) && aligned16(q_seg) && aligned16(kv_pos) && aligned16(kv_seg),
              "q, k, v, out, q_pos, q_seg, kv_pos and kv_seg must be 16-byte aligned");
  SBA_REQUIRE(std::isfinite(softmax_scale), "softmax_scale must be finite");
  SBA_SUPPORT(q_block == 128, "q_block must be 128");
  SBA_SUPPORT(kv_block == 64 || kv_block == 128, "kv_block must be 64 or 128");
  SBA_SUPPORT(T % 128 == 0, "T must be a multiple of 128");
  SBA_SUPPORT(D == 64 || D == 128, "D must be 64 or 128");
  SBA_SUPPORT((long long)B * T * Hq < (1LL << 31), "B * T * Hq must be < 2^31");
  float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  return launch_blocksparse_attn(q, k, v, q_pos, q_seg, kv_pos, kv_seg, lower, upper, lower_full,
                                 upper_full, B, T, Hq, Hkv, D, q_block, kv_block, causal ? 1 : 0,
                                 window_left, window_right, padding_segment_id, scale, out, lse,
                                 reinterpret_cast<cudaStream_t>(stream));
}

size_t sba_ragged_decode_workspace_size(int B, int Hq, int S, int D, int window_left) {
  if (B < 1 || Hq < 1 || S < 1 || D < 1) return 0;
  return decode_workspace_bytes(B, Hq, S, D, window_left);
}

int sba_ragged_decode_fwd(const void* q, const void* k, const void* v, const int32_t* seq_start,
                          const int32_t* seq_end, int B, int Hq, int Hkv, int S, int D,
                          float softmax_scale, int window_left, int window_right,
                          float logits_soft_cap, const float* sink_bias, int num_sinks,
                          int sink_bias_per_head, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, sba_stream_t stream) {
  g_last_error.clear();
  SBA_REQUIRE(q && k && v && seq_start && seq_end && out, "null pointer");
  SBA_REQUIRE(B >= 1 && Hq >= 1 && Hkv >= 1 && S >= 1 && Hq % Hkv == 0, "bad sizes");
  SBA_REQUIRE(window_left >= -1 && window_right >= -1, "windows must be >= -1");
  SBA_REQUIRE(num_sinks >= 0 && (num_sinks == 0 || sink_bias != nullptr),
              "num_sinks > 0 needs sink_bias");
  SBA_REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out),
              "q, k, v and out must be 16-byte aligned");
  SBA_REQUIRE(std::isfinite(softmax_scale) && std::isfinite(logits_soft_cap),
              "scale and cap must be finite");
  SBA_SUPPORT(D == 128, "D must be 128");
  SBA_SUPPORT(Hq / Hkv <= 16, "Hq / Hkv must be <= 16");
  SBA_SUPPORT(num_sinks <= 16, "num_sinks must be <= 16");
  size_t need = decode_workspace_bytes(B, Hq, S, D, window_left);
  SBA_REQUIRE(workspace != nullptr && aligned16(workspace) && workspace_bytes >= need,
              "workspace missing, misaligned or smaller than sba_ragged_decode_workspace_size()");
  float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  return launch_ragged_decode(q, k, v, seq_start, seq_end, B, Hq, Hkv, S, D, scale, window_left,
                              window_right, logits_soft_cap, sink_bias, num_sinks,
                              sink_bias_per_head ? 1 : 0, out, lse, workspace, workspace_bytes,
                              reinterpret_cast<cudaStream_t>(stream));
}

size_t sba_ragged_flash_attention_workspace_size(int B, int Q, int Hq, int S, int D,
                                                 int window_left, int window_right) {
  if (B < 1 || Q < 1 || Hq < 1 || S < 1 || D < 1) return 0;
  return ragged_mq_workspace_bytes(B, Q, Hq, S, window_left, window_right);
}

int sba_ragged_flash_attention_fwd(const void* q, const void* k, const void* v,
                                   const int32_t* seq_start, const int32_t* seq_end, int B, int Q,
                                   int Hq, int Hkv, int S, int D, float softmax_scale,
                                   int window_left, int window_right, float logits_soft_cap,
                                   const float* sink_bias, int num_sinks, int sink_bias_per_head,
                                   void* out, float* lse, void* workspace, size_t workspace_bytes,
                                   sba_stream_t stream) {
  g_last_error.clear();
  SBA_REQUIRE(q && k && v && seq_start && seq_end && out, "null pointer");
  SBA_REQUIRE(B >= 1 && Q >= 1 && Hq >= 1 && Hkv >= 1 && S >= 1 && Hq % Hkv == 0, "bad sizes");
  SBA_REQUIRE(window_left >= -1 && window_right >= -1, "windows must be >= -1");
  SBA_REQUIRE(num_sinks >= 0 && (num_sinks == 0 || sink_bias != nullptr),
              "num_sinks > 0 needs sink_bias");
  SBA_REQUIRE(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out),
              "q, k, v and out must be 16-byte aligned");
  SBA_REQUIRE(std::isfinite(softmax_scale) && std::isfinite(logits_soft_cap),
              "scale and cap must be finite");
  SBA_SUPPORT(D == 128, "D must be 128");
  SBA_SUPPORT(num_sinks <= 16, "num_sinks must be <= 16");
  SBA_SUPPORT((long long)B * Q * Hq < (1LL << 31) && (long long)B * S * Hkv < (1LL << 31),
              "B * Q * Hq and B * S * Hkv must be < 2^31");
  const size_t need = ragged_mq_workspace_bytes(B, Q, Hq, S, window_left, window_right);
  SBA_REQUIRE(workspace != nullptr && aligned16(workspace) && workspace_bytes >= need,
              "workspace missing, misaligned or smaller than "
              "sba_ragged_flash_attention_workspace_size()");
  float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  return launch_ragged_mq(q, k, v, seq_start, seq_end, B, Q, Hq, Hkv, S, scale, window_left,
                          window_right, logits_soft_cap, sink_bias, num_sinks,
                          sink_bias_per_head ? 1 : 0, out, lse, workspace,
                          reinterpret_cast<cudaStream_t>(stream));
}

int sba_l2_read_probe(const void* buf, size_t bytes, int reps, uint32_t* sink,
                      sba_stream_t stream) {
  g_last_error.clear();
  SBA_REQUIRE(buf && sink, "null pointer");
  SBA_REQUIRE(aligned16(buf) && bytes >= 16 && bytes % 16 == 0,
              "buf must be 16-byte aligned and bytes a positive multiple of 16");
  SBA_REQUIRE(reps >= 1, "reps must be >= 1");
  return launch_l2_read_probe(buf, bytes, reps, sink, reinterpret_cast<cudaStream_t>(stream));
}

int sba_check_error(sba_stream_t stream) {
  g_last_error.clear();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_error(e, "sba_check_error: stream synchronize");
  std::string where;
  unsigned w = read_and_clear_error_nsa(s, &where) | read_and_clear_error_mask(s, &where) |
               read_and_clear_error_blocksparse(s, &where) | read_and_clear_error_decode(s, &where) |
               read_and_clear_error_nsa_bwd(s, &where);
  if (w & kDevErrTimeout)
    return set_error(SBA_ERR_TIMEOUT, "a kernel gave up on a bounded internal wait" + where);
  if (w & kDevErrInput)
    return set_error(SBA_ERR_DEVICE_INPUT, "a kernel found malformed device-side input" + where);
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "sba_check_error");
  return SBA_OK;
}

}  // extern "C"
