/*
 * mosaic.h -- C ABI of the GB300 (sm_103a) mask-only logits library, libmosaic.so.
 *
 * The operation. "Mosaic: Unlocking Long-Context Inference for Diffusion LLMs via Global
 * Memory" (paper review), section 3, observation #2 and core component 1 "Mask-only Logits
 * Kernel": at each denoising step only the still-masked tokens are sampled, so logits are
 * computed for those tokens alone, by one gather-GEMM launch that takes the hidden states of
 * all tokens plus the mask indices, addresses the hidden rows indirectly through the indices
 * and writes no intermediate gathered buffer:
 *
 *     out[i, v] = sum_k hidden[row(i), k] * W[v, k]        0 <= i < M, 0 <= v < V
 *
 * with fp32 accumulation and bf16 (round-to-nearest-even) or fp32 output. Lazy chunking
 * ("扩散大语言模型内存优化：Mosaic系统突破与实践", section 2.3; dLLM-Serve article
 * "扩散大语言模型内存优化：从理论到系统设计", section 3.2.2): when a chunk size is given and
 * M exceeds it, consecutive row slices are computed one after another into the same output
 * buffer, and the concatenation of the slices equals the unchunked result bit for bit.
 *
 * Conventions for every call below:
 *   - All array pointers are DEVICE pointers on the handle's device unless stated otherwise;
 *     the caller allocates and owns them. The library allocates nothing per call.
 *   - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = legacy
 *     default stream). Argument errors are detected on the host and returned before anything
 *     is enqueued. Errors seen by the GPU (bad indices, a wait that ran out) are recorded in
 *     the handle's device status word and reported by mosaic_check().
 *   - Not thread-safe per handle: one host thread per handle at a time.
 */
#ifndef MOSAIC_H_
#define MOSAIC_H_

#include <stdint.h>

#if defined(__GNUC__)
#define MOSAIC_API __attribute__((visibility("default")))
#else
#define MOSAIC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOSAIC_OK = 0,
  MOSAIC_ERR_INVALID_ARG = 1, /* host-detected bad argument; nothing was enqueued          */
  MOSAIC_ERR_UNSUPPORTED = 2, /* shape/alignment/device outside what the kernel handles    */
  MOSAIC_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed                         */
  MOSAIC_ERR_INDEX = 4,       /* (mosaic_check) a mask index fell outside its sequence / H */
  MOSAIC_ERR_TIMEOUT = 5      /* (mosaic_check) a bounded on-GPU wait ran out              */
} mosaic_status;

typedef enum { MOSAIC_BF16 = 0, MOSAIC_F32 = 1 } mosaic_dtype;

typedef struct mosaic_handle mosaic_handle;

/*
 * Called on the host after chunk `chunk` has been enqueued on the stream (see
 * mosaic_masked_logits). `out` holds rows [row_begin, row_begin + rows) of the result once
 * the stream reaches this point; the consumer must enqueue its work on the same stream (or
 * otherwise order it before the next chunk) because the next chunk overwrites `out`.
 */
typedef void (*mosaic_chunk_cb)(int64_t chunk, int64_t row_begin, int64_t rows, void* out,
                                void* user);

/*
 * Create a handle bound to CUDA device `device` (made current by this call). The handle owns
 * one small device status word and the device properties used for launch sizing. Returns
 * MOSAIC_ERR_UNSUPPORTED on a device that is not sm_103, MOSAIC_ERR_CUDA if CUDA fails,
 * including when a kernel that moves registers between its warpgroups was not built with
 * exactly 128 registers per thread (checked here, before any launch).
 */
MOSAIC_API mosaic_status mosaic_create(mosaic_handle** handle, int device);

/* Free the handle (synchronises the device first). NULL is accepted. */
MOSAIC_API mosaic_status mosaic_destroy(mosaic_handle* handle);

/*
 * Mask-only logits (gather-GEMM), one persistent kernel launch per chunk.
 *
 * hidden        bf16 [L_tot, d], row-major, row stride d elements; 16-byte aligned.
 * mask_idx      int32 [M]. Flat mode (seq_offsets == mask_offsets == NULL): global rows of
 *               hidden. CSR mode: positions local to their sequence (see below). Any order,
 *               duplicates allowed; output row i always belongs to mask_idx[i].
 * seq_offsets   CSR mode: int32 [B+1], rising; sequence b owns hidden rows
 *               [seq_offsets[b], seq_offsets[b+1]), seq_offsets[B] <= L_tot.
 * mask_offsets  CSR mode: int32 [B+1], rising from 0 to M; sequence b owns
 *               mask_idx[mask_offsets[b] .. mask_offsets[b+1]), and the hidden row of such an
 *               entry is seq_offsets[b] + mask_idx[i].
 * B             number of sequences in CSR mode (>= 1), ignored in flat mode.
 * W             bf16 [V, d] LM-head weight, row-major; 16-byte aligned.
 * out           [rows_out, V] row-major in out_dtype, 16-byte aligned, where
 *               rows_out = M if chunking is off, else chunk_rows.
 * chunk_rows    <= 0 or >= M: chunking off, one launch writes out[M, V]. Otherwise rows are
 *               cut into slices [c*chunk_rows, min(M, (c+1)*chunk_rows)) of the flat index list
 *               (crossing sequence boundaries in CSR mode); each slice is written to out[0..]
 *               and then cb(c, row_begin, rows, out, user) runs on the host. cb is required
 *               when chunking is on; when chunking is off a non-NULL cb runs once (c = 0).
 * stream        cudaStream_t (as void*) to enqueue on.
 *
 * Requirements (else MOSAIC_ERR_INVALID_ARG / MOSAIC_ERR_UNSUPPORTED, nothing enqueued):
 * non-NULL pointers (except the CSR pair in flat mode, cb when unchunked), d % 8 == 0,
 * V % 8 == 0, 1 <= d, 1 <= V, 0 <= M, L_tot < 2^31, M < 2^31, both CSR arrays or neither.
 * M == 0 returns MOSAIC_OK without launching or calling cb; the array pointers are then
 * not looked at and may be NULL.
 *
 * Bad indices are not an argument error (the host cannot read them): an index outside its
 * sequence or outside hidden makes that output row all zeros and sets the status word, which
 * mosaic_check() reports as MOSAIC_ERR_INDEX. The same holds for CSR offsets that do not
 * start at 0 and end at M.
 */
MOSAIC_API mosaic_status mosaic_masked_logits(mosaic_handle* handle,
                                              const void* hidden, int64_t L_tot, int64_t d,
                                              const int32_t* mask_idx, int64_t M,
                                              const int32_t* seq_offsets,
                                              const int32_t* mask_offsets, int32_t B,
                                              const void* W, int64_t V,
                                              void* out, mosaic_dtype out_dtype,
                                              int64_t chunk_rows, mosaic_chunk_cb cb,
                                              void* user, void* stream);

/*
 * FP8 variant of mosaic_masked_logits: both operands in FP8 E4M3 ("fn": 1 sign, 4 exponent bits
 * with bias 7, 3 fraction bits, largest finite 448) with one fp32 scale per row, so that
 *
 *     out[i, v] = hidden_scale[row(i)] * w_scale[v] * sum_k hidden_q[row(i), k] * W_q[v, k]
 *
 * accumulated in fp32 on the tensor cores (kind::f8f6f4) and stored as bf16 (round to nearest
 * even) or fp32. The pages name FP8 for this step only as future work (the dLLM-Serve article
 * "扩散大语言模型内存优化：从理论到系统设计", section 5) and give no scheme: the per-row scaling
 * is this library's, and mosaic_quantize_rows_e4m3() produces operands in it.
 *
 * hidden_q      E4M3 codes [L_tot, d], one byte per element, row-major; 16-byte aligned.
 * hidden_scale  fp32 [L_tot], 4-byte aligned.
 * W_q           E4M3 codes [V, d]; 16-byte aligned.   w_scale  fp32 [V], 16-byte aligned.
 * All other arguments, the chunking, the status word and the error behaviour are those of
 * mosaic_masked_logits, except that d must be a multiple of 16 (16-byte rows of codes).
 */
MOSAIC_API mosaic_status mosaic_masked_logits_fp8(mosaic_handle* handle,
                                                  const void* hidden_q, const float* hidden_scale,
                                                  int64_t L_tot, int64_t d,
                                                  const int32_t* mask_idx, int64_t M,
                                                  const int32_t* seq_offsets,
                                                  const int32_t* mask_offsets, int32_t B,
                                                  const void* W_q, const float* w_scale,
                                                  int64_t V, void* out, mosaic_dtype out_dtype,
                                                  int64_t chunk_rows, mosaic_chunk_cb cb,
                                                  void* user, void* stream);

/*
 * Per-row E4M3 quantization for mosaic_masked_logits_fp8 (no counterpart on the pages): for each
 * row r of the bf16 matrix x [rows, d], a = max_k |x[r, k]|, scale[r] = a / 448 and
 * q[r, k] = E4M3(x[r, k] * (448 / a)) rounded to nearest even and clamped to +-448, both
 * divisions and the multiply single IEEE fp32 operations (so the result is a deterministic
 * function of x); a row of zeros gets scale 0 and zero codes. Used once for W and per step for
 * the hidden states.
 *
 * x      bf16 [rows, d] row-major, 16-byte aligned, device memory of the current device.
 * q      E4M3 codes [rows, d] (one byte each), 16-byte aligned; caller-owned.
 * scale  fp32 [rows], 4-byte aligned; caller-owned.
 * Requirements (else MOSAIC_ERR_INVALID_ARG / MOSAIC_ERR_UNSUPPORTED, nothing enqueued):
 * rows >= 0, d >= 1, d % 16 == 0, rows < 2^31. rows == 0 enqueues nothing. Enqueued on
 * `stream` (cudaStream_t as void*).
 */
MOSAIC_API mosaic_status mosaic_quantize_rows_e4m3(const void* x, int64_t rows, int64_t d,
                                                   void* q, float* scale, void* stream);

/*
 * The same quantization applied only to the hidden rows a mosaic_masked_logits_fp8 call with
 * the same (mask_idx, M, seq_offsets, mask_offsets, B) will read: for each masked position the
 * row hidden[row] is quantized into hidden_q[row] / hidden_scale[row] ([L_tot, d] / [L_tot]
 * buffers; the other rows are left as they are). Positions whose row is outside its sequence or
 * outside hidden are skipped (the logits call reports them); duplicate positions write the same
 * values. Argument rules as for mosaic_quantize_rows_e4m3 plus those of the mask arguments of
 * mosaic_masked_logits; M == 0 enqueues nothing.
 */
MOSAIC_API mosaic_status mosaic_quantize_masked_rows_e4m3(const void* hidden, int64_t L_tot,
                                                          int64_t d, const int32_t* mask_idx,
                                                          int64_t M, const int32_t* seq_offsets,
                                                          const int32_t* mask_offsets, int32_t B,
                                                          void* hidden_q, float* hidden_scale,
                                                          void* stream);

/*
 * Synchronise `stream`, read and clear the handle's device status word. Returns MOSAIC_OK,
 * MOSAIC_ERR_INDEX (a bad mask index / CSR offsets were seen), MOSAIC_ERR_TIMEOUT (a bounded
 * wait inside a kernel gave up; the kernel returned and the CUDA context stays usable) or
 * MOSAIC_ERR_CUDA.
 */
MOSAIC_API mosaic_status mosaic_check(mosaic_handle* handle, void* stream);

/*
 * Upper bound, in nanoseconds, on any single wait inside the kernel before it gives up with
 * MOSAIC_ERR_TIMEOUT (default 2e9). Tests set a tiny value to exercise the timeout path.
 */
MOSAIC_API mosaic_status mosaic_set_wait_timeout(mosaic_handle* handle, uint64_t timeout_ns);

/* Number of kernel launches enqueued through this handle since creation. */
MOSAIC_API int64_t mosaic_launch_count(const mosaic_handle* handle);

/*
 * Greedy sampling of the masked positions, fused with the mask-only logits: the step that
 * follows the logits in a denoising step (paper review, section 3, observation #2: only the
 * masked tokens are sampled). The [M, V] logits are never written; per masked position i:
 *
 *     token[i]      = argmax_v logits[i, v]          (ties: the smallest v)
 *     confidence[i] = max_v softmax(logits[i, :])_v  = 1 / sum_v exp(logits[i, v] - max)
 *
 * computed from the fp32 accumulators. Arguments as for mosaic_masked_logits, plus:
 * token       int32 [M], device; confidence fp32 [M], device (4-byte aligned).
 * workspace   device scratch of at least mosaic_masked_sample_workspace_bytes(M, V, chunk_rows)
 *             bytes, 16-byte aligned, owned by the caller (per-tile partial maxima, sums and
 *             arguments); chunk_rows (same rule as mosaic_masked_logits) only bounds its size.
 * A position whose mask index is bad gets token -1 and confidence 0 (and the status word is
 * set, see mosaic_check). Two kernel launches per chunk (the fused gather-GEMM and a per-row
 * reduction over the N tiles); results are deterministic.
 */
MOSAIC_API int64_t mosaic_masked_sample_workspace_bytes(int64_t M, int64_t V, int64_t chunk_rows);
MOSAIC_API mosaic_status mosaic_masked_sample(mosaic_handle* handle,
                                              const void* hidden, int64_t L_tot, int64_t d,
                                              const int32_t* mask_idx, int64_t M,
                                              const int32_t* seq_offsets,
                                              const int32_t* mask_offsets, int32_t B,
                                              const void* W, int64_t V,
                                              int32_t* token, float* confidence,
                                              void* workspace, int64_t workspace_bytes,
                                              int64_t chunk_rows, void* stream);

/*
 * Lazy chunking's "minimum sufficient chunk count" for the logits output
 * ("扩散大语言模型内存优化：Mosaic系统突破与实践", section 2.3: chunking stays off unless memory is
 * short, and then the smallest chunk count that fits is used; paper review section 3, core
 * component 3). Host-only arithmetic, no GPU needed.
 *
 * Given M masked rows, vocabulary V, the output dtype and a byte budget for the live output
 * buffer, writes to *chunk_rows the value to pass to mosaic_masked_logits and to *n_chunks the
 * number of launches it gives:
 *   - M * V * elt <= budget: chunking stays off, *chunk_rows = 0, *n_chunks = (M > 0);
 *   - otherwise the fewest chunks n whose rows fit (ceil(M / n) * V * elt <= budget), with the
 *     rows balanced across them: *chunk_rows = ceil(M / n) (the last chunk may be shorter).
 * MOSAIC_ERR_UNSUPPORTED if not even one row fits; MOSAIC_ERR_INVALID_ARG for M < 0, V < 1,
 * budget < 0, an unknown dtype or NULL outputs.
 */
MOSAIC_API mosaic_status mosaic_min_chunk_rows(int64_t M, int64_t V, mosaic_dtype out_dtype,
                                               int64_t budget_bytes, int64_t* chunk_rows,
                                               int64_t* n_chunks);

/*
 * VMM-backed output workspace for lazy chunking (paper review, section 3, core component 4
 * "Global Memory Manager"; "扩散大语言模型内存优化：Mosaic系统突破与实践", section 3.1: reserve
 * virtual addresses up front, bind physical pages as demand grows). A contiguous virtual range
 * of reserve_bytes is reserved on `device` without physical memory; mosaic_workspace_bind makes
 * sure the first `bytes` of it are backed (binding more pages only when the demand grows) and
 * returns its base address, which never changes, so a chunk output buffer can grow to the
 * largest chunk actually used without reallocation or fragmentation. mosaic_workspace_trim waits
 * for the device to be idle and unbinds pages beyond keep_bytes (in the units they were bound;
 * the bound size may stay above keep_bytes). Sizes round up to the allocation granularity
 * (typically 2 MiB). The bound pages are ordinary device memory of `device` and can be passed
 * as `out` to mosaic_masked_logits. Not thread-safe per workspace.
 */
typedef struct mosaic_workspace mosaic_workspace;
MOSAIC_API mosaic_status mosaic_workspace_create(mosaic_workspace** ws, int device,
                                                 int64_t reserve_bytes);
MOSAIC_API mosaic_status mosaic_workspace_bind(mosaic_workspace* ws, int64_t bytes, void** ptr);
MOSAIC_API mosaic_status mosaic_workspace_trim(mosaic_workspace* ws, int64_t keep_bytes);
MOSAIC_API int64_t mosaic_workspace_bound_bytes(const mosaic_workspace* ws);
MOSAIC_API int64_t mosaic_workspace_reserved_bytes(const mosaic_workspace* ws);
MOSAIC_API mosaic_status mosaic_workspace_destroy(mosaic_workspace* ws);

/* Text of the last error produced on the calling thread ("" if none). */
MOSAIC_API const char* mosaic_last_error_string(void);

/*
 * Allocation-free variant of mosaic_masked_logits (no counterpart in the Mosaic pages; it
 * exists for callers that cannot allocate device memory).
 *
 * Who needs it: code whose device memory is owned entirely by someone else -- a global
 * memory planner or arena that reserves and binds the whole workspace up front, a serving
 * loop where a cudaMalloc would synchronise the device, or a host that only hands this
 * library its input and output buffers. mosaic_create() allocates a status word, so such a
 * caller cannot hold a handle; this entry point needs none and allocates nothing (no
 * cudaMalloc, cudaFree or allocating library routine).
 *
 * Arguments, layouts and semantics are those of mosaic_masked_logits (same kernel, same
 * results bit for bit), on the CURRENT CUDA device. Instead of the handle's status word it
 * uses a status word per chunk held in a fixed device array inside the library, of
 * MOSAIC_NOALLOC_MAX_CHUNKS words; a call that needs more chunks than that (ceil(M /
 * chunk_rows), 1 when chunking is off) is rejected with MOSAIC_ERR_UNSUPPORTED before
 * anything is enqueued. Every GPU that loads the library holds that array until exit.
 *
 * chunk_status   optional HOST array of at least that many uint32 words. NULL: the call is
 *                asynchronous and reports only argument errors; a bad mask index then yields a
 *                zero-filled output row that nothing reports, so pass the array at least while
 *                debugging. Non-NULL: the call waits for `stream`, copies each chunk's status
 *                word there (bit 1: a bad mask index or CSR offsets, bit 2: a bounded wait ran
 *                out) and returns MOSAIC_ERR_INDEX / MOSAIC_ERR_TIMEOUT / MOSAIC_OK accordingly.
 *
 * Every wait inside the kernel gives up after a fixed 2 seconds (there is no handle, so
 * mosaic_set_wait_timeout does not apply here).
 *
 * The first call on a device sets that device up (kernel attributes, occupancy, the array's
 * device address, kept until the process exits); make it before any CUDA stream capture, and do
 * not call this entry point on a device after cudaDeviceReset() of that device (the library's
 * device code is loaded again and the kept address would be stale). All calls share the one array,
 * which keeps the last call's words: each call clears the words it uses on `stream` before
 * its kernels run, so calls that overlap on the GPU (different streams, no ordering) race
 * on the status words and their reported status is unreliable; the logits are unaffected.
 */
#define MOSAIC_NOALLOC_MAX_CHUNKS 4096
MOSAIC_API mosaic_status mosaic_masked_logits_noalloc(const void* hidden, int64_t L_tot,
                                                      int64_t d, const int32_t* mask_idx,
                                                      int64_t M, const int32_t* seq_offsets,
                                                      const int32_t* mask_offsets, int32_t B,
                                                      const void* W, int64_t V, void* out,
                                                      mosaic_dtype out_dtype,
                                                      int64_t chunk_rows, mosaic_chunk_cb cb,
                                                      void* user, uint32_t* chunk_status,
                                                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOSAIC_H_ */
