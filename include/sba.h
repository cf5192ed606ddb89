/*
 * sba.h -- C ABI of libsba, selected-block sparse attention for NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every function returns an int status: SBA_OK (0) or a negative SBA_ERR_* code.
 *    On error nothing is launched and sba_last_error() (thread-local) describes why.
 *    No C++ exception crosses this boundary.
 *  - Every tensor pointer is caller-owned DEVICE memory (from cudaMalloc, a caching
 *    allocator, ...), dense row-major in the layout given per argument, 16-byte aligned.
 *    The library keeps no pointer after a call returns and allocates no device memory.
 *  - Work is enqueued asynchronously on `stream` (0 = legacy default stream); nothing
 *    synchronises.  Errors a kernel detects while running (a malformed cu_seqlens, an
 *    internal wait that timed out) are recorded in a device-side error word and
 *    reported by sba_check_error().
 *  - dtype codes: SBA_BF16 = 0 (bfloat16), SBA_F32 = 1 (float32).
 *  - softmax_scale <= 0 selects 1 / sqrt(D).
 *  - Log-sum-exp outputs are natural-log, float32; a row with no admissible key gets
 *    output 0 and LSE = -inf.
 */
#ifndef SBA_H_
#define SBA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SBA_API __attribute__((visibility("default")))
#else
#define SBA_API
#endif

typedef struct CUstream_st* sba_stream_t; /* same object as cudaStream_t */

enum {
  SBA_OK = 0,
  SBA_ERR_INVALID_ARG = -1, /* a size, pointer, alignment or flag is out of range   */
  SBA_ERR_UNSUPPORTED = -2, /* valid arguments this build has no kernel for         */
  SBA_ERR_CUDA = -3,        /* a CUDA runtime/driver call failed (message attached) */
  SBA_ERR_TIMEOUT = -4,     /* a kernel gave up on an internal wait (see check)     */
  SBA_ERR_DEVICE_INPUT = -5 /* a kernel found malformed device-side input           */
};

enum { SBA_BF16 = 0, SBA_F32 = 1 };

/* Library version string, e.g. "sba 0.1.0 sm_103a". */
SBA_API const char* sba_version(void);

/* Message of the last failing call on this host thread ("" if none). */
SBA_API const char* sba_last_error(void);

/*
 * sba_set_wait_timeout_cycles -- limit, in SM clock cycles, on every internal wait of
 * the warp-specialised kernels (the NSA selection forward on tensor cores and the
 * block-sparse / ragged block attention).  No counterpart on the pages: it is the
 * library's failure detection.  A wait that runs past the limit records the kernel,
 * role, barrier and work item in the device error word, makes every other wait of its
 * CTA return at once, drains the copies already issued, frees its tensor memory and
 * returns; sba_check_error() then reports SBA_ERR_TIMEOUT with that location and the
 * outputs of that launch are undefined.  Applies to launches made after the call, from
 * any host thread (process-wide).  cycles == 0 restores the default (4e9 cycles, about
 * two seconds at the boost clock); a limit far below a kernel's normal wait times
 * makes its launches fail.  Returns SBA_ERR_INVALID_ARG for cycles < 0.
 * sba_get_wait_timeout_cycles returns the limit in force.
 */
SBA_API int sba_set_wait_timeout_cycles(long long cycles);
SBA_API long long sba_get_wait_timeout_cycles(void);

/*
 * sba_nsa_select_fwd -- native-sparse-attention forward, selection branch.
 *
 * Defined by: "ejkernel.modules.operations.native_sparse_attention" (operation API
 * page), method NativeSparseAttention.run and function native_sparse_attention.
 * Each query token attends, per KV head, only to the key blocks of `block_size`
 * tokens named by block_indices[b, t, h_kv, :count]; Hq query heads share Hkv KV
 * heads (query head hq reads KV head hq / (Hq / Hkv)); cu_seqlens packs
 * variable-length sequences into one batch row; the output has the query's shape.
 *
 *  q             [B, T, Hq, D]  dtype        (B == 1 when cu_seqlens != NULL)
 *  k, v          [B, T, Hkv, D] dtype
 *  g_slc         [B, T, Hq] dtype, or NULL: gate of the selection branch (the
 *                operation's g_slc argument); the output row of (b, t, hq) is
 *                multiplied by g_slc[b, t, hq].  The LSE is not gated.  (The
 *                compressed branch and its gate g_cmp are not part of this call.)
 *  block_indices [B, T, Hkv, S] int32: block ids relative to the start of the
 *                token's own sequence.  Entries < 0, >= ceil(L / block_size) (L = the
 *                sequence's length) or, when causal, after the token's own block are
 *                ignored.  Order does not matter; duplicates count once.
 *  block_counts  [B, T, Hkv] int32, or NULL to use block_count_scalar for every
 *                token; only the first min(count, S) entries are read.
 *  cu_seqlens    [num_seqs + 1] int32 (0 = c[0] <= c[1] <= ... <= c[num_seqs] = T),
 *                or NULL for fixed-length rows of T tokens.
 *  causal        nonzero: key k of a token at sequence position t is visible iff k <= t.
 *  out           [B, T, Hq, D] dtype (written).
 *  lse           [B, T, Hq] float32 (written), or NULL.
 * Supported: D in {64, 128}; block_size in {32, 64, 128}; 1 <= Hq/Hkv <= 16;
 * 1 <= S <= 32; dtype bf16 (tensor cores, bf16 inputs, fp32 accumulation, P rounded
 * to bf16) or f32 (CUDA cores, exact fp32 products and sums).
 */
SBA_API int sba_nsa_select_fwd(const void* q, const void* k, const void* v, const void* g_slc,
                       const int32_t* block_indices, const int32_t* block_counts,
                       int block_count_scalar, int S,
                       const int32_t* cu_seqlens, int num_seqs,
                       int B, int T, int Hq, int Hkv, int D, int block_size, int causal,
                       float softmax_scale, int dtype,
                       void* out, float* lse, sba_stream_t stream);

/*
 * sba_nsa_select_bwd_workspace_size -- bytes of device workspace sba_nsa_select_bwd
 * needs (Delta per query row, and the per-key-block token lists).  num_seqs = 0 for
 * fixed-length rows.  Returns 0 for invalid sizes.
 */
SBA_API size_t sba_nsa_select_bwd_workspace_size(int B, int T, int Hq, int Hkv, int S,
                                                 int num_seqs);

/*
 * sba_nsa_select_bwd -- gradients of sba_nsa_select_fwd with respect to q, k and v.
 *
 * Defined by: "ejkernel.modules.operations.native_sparse_attention" (operation API
 * page), NativeSparseAttention.run / native_sparse_attention, which is differentiable
 * in query, key and value.  The page gives no gradient algorithm; the result is the
 * gradient of the forward above (no gate): for each row (token, query head) with its
 * explicit key set and P = exp(scale * q.k - LSE) over that set,
 *   dV_k += P_k dO,  dS_k = P_k (dO.v_k - dO.O),  dQ = scale * sum_k dS_k k_k,
 *   dK_k += scale * dS_k q.
 * A gate g_slc applied in the forward is handled by the caller: pass dO * g_slc as
 * d_out (the gate's own gradient is rowsum(dO * O_ungated)).
 *
 *  q, k, v, block_indices, block_counts, block_count_scalar, S, cu_seqlens, num_seqs,
 *  B, T, Hq, Hkv, D, block_size, causal, softmax_scale, dtype: exactly as passed to
 *                the forward that produced `out` and `lse`
 *  out           [B, T, Hq, D] dtype: the forward's output (ungated)
 *  lse           [B, T, Hq] float32: the forward's log-sum-exp (required)
 *  d_out         [B, T, Hq, D] dtype: gradient of the loss with respect to out
 *  dq            [B, T, Hq, D] dtype (written)
 *  dk, dv        [B, T, Hkv, D] dtype (written; keys no token selected get 0)
 *  workspace     device scratch of at least sba_nsa_select_bwd_workspace_size(B, T, Hq,
 *                Hkv, S, cu_seqlens ? num_seqs : 0) bytes, 256-byte aligned, caller-owned;
 *                needs no initialisation.
 * Supported: dtype bf16 (tensor cores, fp32 accumulation; P and dS rounded to bf16
 * before their products), D == 128, block_size == 64, Hq / Hkv in {8, 16}, S <= 32;
 * other valid arguments return SBA_ERR_UNSUPPORTED.  dK / dV sum many tokens in an
 * order set by atomics, so results may differ in the last bits between runs.
 * Internally, on `stream`: a memset, three small index kernels (Delta and counts, offsets,
 * token lists), the dQ kernel and the dK/dV kernel.
 */
SBA_API int sba_nsa_select_bwd(const void* q, const void* k, const void* v, const void* out,
                               const float* lse, const void* d_out,
                               const int32_t* block_indices, const int32_t* block_counts,
                               int block_count_scalar, int S, const int32_t* cu_seqlens,
                               int num_seqs, int B, int T, int Hq, int Hkv, int D, int block_size,
                               int causal, float softmax_scale, int dtype, void* dq, void* dk,
                               void* dv, void* workspace, size_t workspace_bytes,
                               sba_stream_t stream);

/*
 * sba_nsa_select_host_workspace_size -- bytes of device staging memory that
 * sba_nsa_select_fwd_host needs for the given shapes: device copies of q, k, v,
 * block_indices, block_counts (has_counts), g_slc (has_gate), out and lse (has_lse),
 * each starting on a 256-byte boundary.  Returns 0 for sizes < 1 or an unknown dtype.
 */
SBA_API size_t sba_nsa_select_host_workspace_size(int B, int T, int Hq, int Hkv, int D, int S,
                                                  int dtype, int has_counts, int has_gate,
                                                  int has_lse);

/*
 * sba_nsa_select_fwd_host -- sba_nsa_select_fwd on HOST buffers, fixed-length rows
 * (no cu_seqlens).  Same operation, arguments, layouts and support limits as
 * sba_nsa_select_fwd; every tensor argument (q_h, k_h, v_h, g_slc_h, block_indices_h,
 * block_counts_h, out_h, lse_h) is a host pointer.  Page-locked (pinned) host memory
 * makes the copies asynchronous; pageable memory works but copies synchronously.
 *
 *  workspace        device memory of at least sba_nsa_select_host_workspace_size(B, T,
 *                   Hq, Hkv, D, S, dtype, block_counts_h != NULL, g_slc_h != NULL,
 *                   lse_h != NULL) bytes, 256-byte aligned, owned by the caller; its
 *                   contents are scratch.
 *
 * The work is split into up to eight chunks.  With bf16 inputs, T a multiple of 128 and
 * T >= 256, a chunk is a (batch row, range of 128-token spans) piece, token ranges
 * first: under causal masking a chunk copies only the K/V rows it adds to its row's
 * prefix (the earlier chunks' rows are already on the device), otherwise the row's
 * first chunk copies the row's K/V.  Else a chunk is a group of whole batch rows.  Each
 * chunk's inputs are copied to the device on a library stream, computed on `stream`,
 * and its outputs copied back on a second library stream, so that the copy of one
 * chunk overlaps the computation of its neighbours (the library keeps these two
 * non-blocking streams per device from the first call on).  Ordering: the call's work starts after the
 * work already enqueued on `stream`, and its end (the last copy to out_h / lse_h) is
 * enqueued on `stream`: synchronize `stream` before reading out_h or lse_h, and do not
 * reuse the workspace or the host buffers before that.
 * Errors: SBA_ERR_INVALID_ARG (null pointer, misaligned or short workspace, sizes),
 * SBA_ERR_UNSUPPORTED (as sba_nsa_select_fwd), SBA_ERR_CUDA (a copy, event or launch
 * failed; work enqueued before the failure may still run).
 */
SBA_API int sba_nsa_select_fwd_host(const void* q_h, const void* k_h, const void* v_h,
                                    const void* g_slc_h, const int32_t* block_indices_h,
                                    const int32_t* block_counts_h, int block_count_scalar, int S,
                                    int B, int T, int Hq, int Hkv, int D, int block_size,
                                    int causal, float softmax_scale, int dtype, void* out_h,
                                    float* lse_h, void* workspace, size_t workspace_bytes,
                                    sba_stream_t stream);

/*
 * sba_sparse_mask_bounds -- SparseMask block bounds for the forward pass.
 *
 * Defined by: "ejkernel.kernels._triton.blocksparse_attention._mask" (module source
 * page): dataclass SparseMask, kernel _compute_sparse_mask with the query as the
 * outer operand, and the padding, padding-segment remap and clip/fix-up steps of
 * define_sparse_mask_fn.  Tq and Tkv are padded to block multiples (query positions
 * with -1, key positions with INT32_MAX, segment ids with padding_segment_id), the
 * padding id is remapped to padded_Tkv + 1, each (query block, key block) pair is
 * tested for segment-range overlap, causality and the inclusive window, and the
 * half-open bounds are min/max-accumulated then clipped.  Results are bit-exact
 * integers.
 *
 *  q_pos, q_seg    [B, Tq] int32  positions / segment ids of the query tokens
 *  kv_pos, kv_seg  [B, Tkv] int32 positions / segment ids of the key tokens
 *  window_left/right  inclusive window in positions; -1 = unbounded
 *  padding_segment_id  segment id that marks padding tokens
 *  lower, upper, lower_full, upper_full  [B, 1, ceil(Tq / q_block)] int32 (written)
 * Preconditions: real segment ids < padded_Tkv + 1; |positions| + window < 2^31.
 */
SBA_API int sba_sparse_mask_bounds(const int32_t* q_pos, const int32_t* q_seg,
                           const int32_t* kv_pos, const int32_t* kv_seg,
                           int B, int Tq, int Tkv, int q_block, int kv_block, int causal,
                           int window_left, int window_right, int padding_segment_id,
                           int32_t* lower, int32_t* upper,
                           int32_t* lower_full, int32_t* upper_full,
                           sba_stream_t stream);

/*
 * sba_sparse_mask_dkdv_bounds -- SparseMask block bounds for the dK/dV backward pass.
 *
 * Defined by: "ejkernel.kernels._triton.blocksparse_attention._mask" (module source
 * page): define_sparse_mask_fn with calculate_dkdv_mask set, i.e. kernel
 * _compute_sparse_mask with the key/value blocks as the outer operand and the query
 * blocks as the inner one, then the same clip/fix-up against the number of query
 * blocks.  Padding and the padding-segment remap are those of sba_sparse_mask_bounds.
 * Position tests, as the page prints them for this operand order (o = key/value block,
 * i = query block, min/max over the block's positions; 64-bit arithmetic):
 *   causal:        attend  max_i >= min_o            full  min_i >= max_o
 *   window_left:   attend  max_i >= min_o - left     full  min_i >= min_o - left
 *   window_right:  attend  min_i <= max_o + right    full  max_i <= max_o + right
 * Results are bit-exact integers.
 *
 *  q_pos, q_seg, kv_pos, kv_seg, window_left/right, padding_segment_id: as in
 *                  sba_sparse_mask_bounds
 *  lower, upper, lower_full, upper_full  [B, 1, ceil(Tkv / kv_block)] int32 (written):
 *                  half-open ranges of query blocks per key/value block
 * All pointers are caller-owned device memory.  Returns SBA_ERR_INVALID_ARG for null
 * pointers or non-positive sizes, SBA_ERR_UNSUPPORTED for blocks > 4096 or B > 65535.
 */
SBA_API int sba_sparse_mask_dkdv_bounds(const int32_t* q_pos, const int32_t* q_seg,
                                        const int32_t* kv_pos, const int32_t* kv_seg,
                                        int B, int Tq, int Tkv, int q_block, int kv_block,
                                        int causal, int window_left, int window_right,
                                        int padding_segment_id,
                                        int32_t* lower, int32_t* upper,
                                        int32_t* lower_full, int32_t* upper_full,
                                        sba_stream_t stream);

/*
 * sba_blocksparse_attn_fwd -- attention restricted by SparseMask bounds.
 *
 * Defined by: "ejkernel.kernels._triton.blocksparse_attention._mask" (module source
 * page), module docstring and SparseMask docstring: key blocks outside
 * [lower, upper) of a query block are skipped; blocks inside
 * [lower_full, upper_full) are processed without per-token masking.  Token-level
 * mask (the page does not print one; plainest reading): same segment, neither
 * padding, causal on positions, inclusive window on positions.
 *
 *  q [B, T, Hq, D] bf16; k, v [B, T, Hkv, D] bf16 (queries and keys share T)
 *  q_pos, q_seg, kv_pos, kv_seg [B, T] int32
 *  lower, upper, lower_full, upper_full [B, 1, T / q_block] int32 (as produced by
 *  sba_sparse_mask_bounds with the same block sizes)
 *  out [B, T, Hq, D] bf16 (written); lse [B, T, Hq] float32 (written) or NULL.
 * q, k, v, out, q_pos, q_seg, kv_pos and kv_seg must be 16-byte aligned (the kernel
 * copies them with TMA / bulk copies); SBA_ERR_INVALID_ARG otherwise.
 * Supported: q_block == 128, kv_block in {64, 128}, T % 128 == 0, D in {64, 128},
 * 1 <= Hq / Hkv, bf16 only.
 */
SBA_API int sba_blocksparse_attn_fwd(const void* q, const void* k, const void* v,
                             const int32_t* q_pos, const int32_t* q_seg,
                             const int32_t* kv_pos, const int32_t* kv_seg,
                             const int32_t* lower, const int32_t* upper,
                             const int32_t* lower_full, const int32_t* upper_full,
                             int B, int T, int Hq, int Hkv, int D, int q_block, int kv_block,
                             int causal, int window_left, int window_right,
                             int padding_segment_id, float softmax_scale,
                             void* out, float* lse, sba_stream_t stream);

/*
 * sba_ragged_decode_workspace_size -- bytes of device workspace that
 * sba_ragged_decode_fwd needs for these sizes (fp32 split partials).  window_left < 0
 * means no left window.  Returns 0 for invalid sizes.
 */
SBA_API size_t sba_ragged_decode_workspace_size(int B, int Hq, int S, int D, int window_left);

/*
 * sba_ragged_decode_fwd -- ragged single-token decode attention.
 *
 * Defined by: "ejkernel.kernels._xla.ragged_decode_attention._xla_impl_fwd" (API
 * page): ragged_decode_mqa_xla / inner_decode_xla (per-row key range
 * [sequence_start, sequence_end), sliding window, logits soft cap, softmax_aux sink
 * biases), create_attention_mask (sinks are always attendable),
 * apply_logits_soft_cap and apply_attention_sinks_block.  The query sits at
 * position end - 1; key k is attendable iff start <= k < end and it lies in the
 * inclusive window or k < num_sinks.  Logit = scale * <q, k>, then
 * cap * tanh(logit / cap) when cap > 0, then + sink_bias for sink keys.
 *
 *  q          [B, Hq, D] bf16
 *  k, v       [B, S, Hkv, D] bf16 (the KV cache; rows beyond sequence_end unread)
 *  seq_start, seq_end  [B] int32
 *  sink_bias  float32 [Hq, num_sinks] (sink_bias_per_head != 0) or [num_sinks];
 *             NULL with num_sinks == 0 for none.  num_sinks <= 16.
 *  out        [B, Hq, D] bf16 (written); lse [B, Hq] float32 (written) or NULL
 *  workspace  device scratch of at least
 *             sba_ragged_decode_workspace_size(B, Hq, S, D, window_left) bytes,
 *             16-byte aligned, caller-owned; contents need no initialisation.
 * Supported: D == 128, 1 <= Hq / Hkv <= 16, num_sinks <= 16, sequence_end <= S, bf16.
 * Internally, on `stream`: a memset of the workspace's split counters and one split-KV
 * kernel whose last split of each row tile merges the partials.
 */
SBA_API int sba_ragged_decode_fwd(const void* q, const void* k, const void* v,
                          const int32_t* seq_start, const int32_t* seq_end,
                          int B, int Hq, int Hkv, int S, int D, float softmax_scale,
                          int window_left, int window_right, float logits_soft_cap,
                          const float* sink_bias, int num_sinks, int sink_bias_per_head,
                          void* out, float* lse,
                          void* workspace, size_t workspace_bytes, sba_stream_t stream);

/*
 * sba_ragged_decode_fwd_noalloc -- sba_ragged_decode_fwd without a workspace argument.
 *
 * The pages have no counterpart of this entry point; it exists for callers that cannot
 * allocate device memory when they call the library (device memory owned by another
 * allocator with a fixed budget, plugin interfaces that receive only input and output
 * buffers, loops that must not incur the device-wide synchronisation of
 * cudaMalloc/cudaFree).  The split partials live in a 16 MiB array inside the library:
 * every GPU that loads the library reserves it until the process exits.  Arguments,
 * layouts and results are those of sba_ragged_decode_fwd.
 *  - Sizes whose sba_ragged_decode_workspace_size() exceeds 16 MiB are rejected with
 *    SBA_ERR_INVALID_ARG (use sba_ragged_decode_fwd with a workspace instead).
 *  - The first call on each device looks up the array's device address (with that device
 *    current: `stream` must belong to the current device) and caches it for the life of
 *    the process; make that first call before any stream capture.  The cached address
 *    belongs to the device's context: after cudaDeviceReset() on a device, do not call
 *    this entry point on that device again in the same process.
 *  - All calls on a device share the array: calls that may overlap on the GPU (different
 *    streams, no ordering between them) race and corrupt each other's results.  Calls on
 *    one stream are ordered and safe.  The array keeps the last call's partials; every
 *    partial a call reads was written by that call, and the per-tile split counters it
 *    needs zeroed are cleared by the call itself (cudaMemsetAsync on `stream`).
 *  - Neither the call nor its first-call set-up calls cudaMalloc, cudaFree or any
 *    allocating routine.  The 16 MiB are reserved when the library's device code is
 *    loaded onto the GPU; with lazy module loading (CUDA_MODULE_LOADING=LAZY, the
 *    default) that load may happen during the first call.
 */
SBA_API int sba_ragged_decode_fwd_noalloc(const void* q, const void* k, const void* v,
                                          const int32_t* seq_start, const int32_t* seq_end,
                                          int B, int Hq, int Hkv, int S, int D,
                                          float softmax_scale, int window_left,
                                          int window_right, float logits_soft_cap,
                                          const float* sink_bias, int num_sinks,
                                          int sink_bias_per_head, void* out, float* lse,
                                          sba_stream_t stream);

/*
 * sba_ragged_flash_attention_workspace_size -- bytes of device workspace that
 * sba_ragged_flash_attention_fwd needs for these sizes (fp32 split partials).  A window
 * bound < 0 means unbounded on that side.  Returns 0 for invalid sizes.
 */
SBA_API size_t sba_ragged_flash_attention_workspace_size(int B, int Q, int Hq, int S, int D,
                                                         int window_left, int window_right);

/*
 * sba_ragged_flash_attention_fwd -- ragged multi-query attention: Q query tokens per
 * batch row against that row's slice of a KV cache.
 *
 * Defined by: "ejkernel.kernels._xla.ragged_decode_attention._xla_impl_fwd" (API
 * page): ragged_flash_attention_xla (queries [B, Q, H, D], per-row key range
 * [sequence_start, sequence_end), sliding window, logits soft cap, softmax_aux sink
 * biases) with create_attention_mask (one mask for all heads; sinks are always
 * attendable).  Readings of what the page leaves open: query i of a row sits at
 * position p_i = end - Q + i (the row's last Q tokens; Q = 1 is sba_ragged_decode_fwd);
 * there is no causal switch, so key k is attendable by query i iff start <= k < end and
 * either p_i - window_left <= k <= p_i + window_right (a bound < 0 is unbounded) or
 * k < num_sinks.  Logit = scale * <q, k>, then cap * tanh(logit / cap) when cap > 0,
 * then + sink_bias for sink keys.  A query with no attendable key gets output 0 and
 * LSE -inf.
 *
 *  q          [B, Q, Hq, D] bf16
 *  k, v       [B, S, Hkv, D] bf16 (the KV cache; Hq % Hkv == 0, query head hq reads
 *             KV head hq / (Hq / Hkv); the page's case is Hkv == Hq)
 *  seq_start, seq_end  [B] int32 (clamped to [0, S])
 *  sink_bias  float32 [Hq, num_sinks] (sink_bias_per_head != 0) or [num_sinks];
 *             NULL with num_sinks == 0 for none.  num_sinks <= 16.
 *  out        [B, Q, Hq, D] bf16 (written); lse [B, Q, Hq] float32 (written) or NULL
 *  workspace  device scratch of at least
 *             sba_ragged_flash_attention_workspace_size(B, Q, Hq, S, D, window_left,
 *             window_right) bytes, 16-byte aligned, caller-owned; needs no initialisation.
 * All pointers are caller-owned device memory.  Returns SBA_ERR_INVALID_ARG for null or
 * misaligned pointers, bad sizes or a short workspace, SBA_ERR_UNSUPPORTED outside:
 * D == 128, num_sinks <= 16, B * ceil(Q * Hq / Hkv / 16) <= 65535, Q <= 65535.
 * Internally, on `stream`: with Q >= 128, no soft cap and no sinks, one launch of the
 * tensor-memory block kernel (query blocks of 128 rows, key blocks of 128; the workspace
 * is not touched); otherwise a memset of the workspace's split counters and one split-KV
 * kernel whose last split of each row tile merges the partials.
 */
SBA_API int sba_ragged_flash_attention_fwd(const void* q, const void* k, const void* v,
                                           const int32_t* seq_start, const int32_t* seq_end,
                                           int B, int Q, int Hq, int Hkv, int S, int D,
                                           float softmax_scale, int window_left,
                                           int window_right, float logits_soft_cap,
                                           const float* sink_bias, int num_sinks,
                                           int sink_bias_per_head, void* out, float* lse,
                                           void* workspace, size_t workspace_bytes,
                                           sba_stream_t stream);

/*
 * sba_l2_read_probe -- measurement helper for the roofline's L2 term; computes nothing
 * of the attention method.
 *
 * Reads buf (bytes bytes) reps times with 16-byte loads that bypass L1, from four
 * 512-thread blocks per SM, and XORs what it read into *sink (so no load is dead).
 * With bytes at most half the L2 size, reps * bytes / elapsed time is the L2-to-SM read
 * bandwidth.  buf: caller-owned device memory, 16-byte aligned, bytes a positive
 * multiple of 16; sink: one caller-owned device word.  Returns SBA_ERR_INVALID_ARG
 * otherwise.  Asynchronous on `stream`.
 */
SBA_API int sba_l2_read_probe(const void* buf, size_t bytes, int reps, uint32_t* sink,
                              sba_stream_t stream);

/*
 * sba_check_error -- synchronise `stream`, then read and clear the device-side error
 * word of every kernel of this library.  Returns SBA_OK, SBA_ERR_TIMEOUT (a kernel
 * gave up on a bounded internal wait and returned early), SBA_ERR_DEVICE_INPUT (a
 * kernel found malformed device data such as a non-monotone cu_seqlens) or
 * SBA_ERR_CUDA (an asynchronous CUDA error).
 */
SBA_API int sba_check_error(sba_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SBA_H_ */
