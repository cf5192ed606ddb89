// Shared host/device helpers of libsba: status codes, error words, bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/sba.h"

namespace sba {

// Bits of the per-translation-unit device error word.
enum : unsigned {
  kDevErrTimeout = 1u,  // a bounded wait expired; the kernel returned early
  kDevErrInput = 2u,    // malformed device-side input (e.g. cu_seqlens)
};

// Roughly two seconds at the GB300 boost clock: by default every spin-wait on an
// mbarrier gives up after this many SM cycles, flags kDevErrTimeout and unwinds.  The
// limit a launch uses is wait_timeout_cycles() (settable through the C ABI); the
// teardown drains of copies already in flight always use this default.
constexpr long long kWaitTimeoutCycles = 4000000000LL;

// Current limit for the bounded waits of the next launches (api.cu).
long long wait_timeout_cycles();

// Host-side error reporting (defined in api.cu).
int set_error(int code, const std::string& msg);
int cuda_error(cudaError_t e, const char* what);

// Per-translation-unit error word readers (each kernel file defines one).
// Each returns the kDevErr* flags and appends a short location note to *where.
unsigned read_and_clear_error_nsa(cudaStream_t s, std::string* where);
unsigned read_and_clear_error_mask(cudaStream_t s, std::string* where);
unsigned read_and_clear_error_blocksparse(cudaStream_t s, std::string* where);
unsigned read_and_clear_error_decode(cudaStream_t s, std::string* where);
unsigned read_and_clear_error_nsa_bwd(cudaStream_t s, std::string* where);

// Launch entry points implemented by the kernel files (arguments already validated).
int launch_nsa_select(const void* q, const void* k, const void* v, const void* g_slc,
                      const int32_t* block_indices,
                      const int32_t* block_counts, int block_count_scalar, int S,
                      const int32_t* cu_seqlens, int num_seqs, int B, int T, int Hq, int Hkv,
                      int D, int block_size, int causal, float scale, int dtype, void* out,
                      float* lse, cudaStream_t stream, long long tok_begin = 0,
                      long long tok_end = -1);
int launch_sparse_mask_bounds(const int32_t* q_pos, const int32_t* q_seg, const int32_t* kv_pos,
                              const int32_t* kv_seg, int B, int Tq, int Tkv, int q_block,
                              int kv_block, int causal, int window_left, int window_right,
                              int pad_id, int32_t* lower, int32_t* upper, int32_t* lower_full,
                              int32_t* upper_full, int dkdv, cudaStream_t stream);
int launch_blocksparse_attn(const void* q, const void* k, const void* v, const int32_t* q_pos,
                            const int32_t* q_seg, const int32_t* kv_pos, const int32_t* kv_seg,
                            const int32_t* lower, const int32_t* upper, const int32_t* lower_full,
                            const int32_t* upper_full, int B, int T, int Hq, int Hkv, int D,
                            int q_block, int kv_block, int causal, int window_left,
                            int window_right, int pad_id, float scale, void* out, float* lse,
                            cudaStream_t stream);
size_t decode_workspace_bytes(int B, int Hq, int S, int D, int window_left);
int launch_ragged_decode(const void* q, const void* k, const void* v, const int32_t* seq_start,
                         const int32_t* seq_end, int B, int Hq, int Hkv, int S, int D,
                         float scale, int window_left, int window_right, float cap,
                         const float* sink_bias, int num_sinks, int sink_per_head, void* out,
                         float* lse, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream);
size_t ragged_mq_workspace_bytes(int B, int Qn, int Hq, int S, int window_left,
                                 int window_right);
int launch_ragged_mq(const void* q, const void* k, const void* v, const int32_t* seq_start,
                     const int32_t* seq_end, int B, int Qn, int Hq, int Hkv, int S, float scale,
                     int window_left, int window_right, float cap, const float* sink_bias,
                     int num_sinks, int sink_per_head, void* out, float* lse, void* workspace,
                     cudaStream_t stream);

int launch_ragged_chunk(const void* q, const void* k, const void* v, const int32_t* seq_start,
                        const int32_t* seq_end, int B, int Qn, int Hq, int Hkv, int S,
                        float scale, int window_left, int window_right, void* out, float* lse,
                        cudaStream_t stream);
size_t nsa_bwd_workspace_bytes(int B, int T, int Hq, int Hkv, int S, int num_seqs);
int launch_nsa_select_bwd(const void* q, const void* k, const void* v, const void* out,
                          const float* lse, const void* d_out, const int32_t* block_indices,
                          const int32_t* block_counts, int block_count_scalar, int S,
                          const int32_t* cu_seqlens, int num_seqs, int B, int T, int Hq, int Hkv,
                          int causal, float scale, void* dq, void* dk, void* dv, void* workspace,
                          cudaStream_t stream);
int launch_l2_read_probe(const void* buf, size_t bytes, int reps, unsigned* sink,
                         cudaStream_t stream);

// Driver entry point for tensor-map encoding, resolved once through the runtime.
CUresult encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, cuuint32_t rank,
                           void* gaddr, const cuuint64_t* dims, const cuuint64_t* strides_bytes,
                           const cuuint32_t* box, CUtensorMapSwizzle swizzle);

int num_sms();

}  // namespace sba
