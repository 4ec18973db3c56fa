// C ABI of libmosaic.so: argument validation, TMA descriptor set-up and the lazy-chunk driver
// around the gather-GEMM kernel. The declarations and their contracts are in include/mosaic.h.
//
// Lazy chunking follows "扩散大语言模型内存优化：Mosaic系统突破与实践" (section 2.3: chunking is
// off by default and used only when asked for) and the dLLM-Serve article
// "扩散大语言模型内存优化：从理论到系统设计" (section 3.2.2: rows beyond the cap are cut into
// consecutive slices, each run through the LM head). Here every slice reuses one output buffer
// and the kernel's per-element arithmetic does not depend on where a row falls in a slice, so
// the concatenated slices equal the unchunked result bit for bit.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include "../../include/mosaic.h"
#include "gather_gemm.h"
#include "status.h"

struct mosaic_handle {
  int device = 0;
  int num_sms = 0;
  int max_clusters[2][2] = {};  // [out_f32][pair]: clusters resident at once
  int max_clusters_sample[2] = {};  // [pair], sampling epilogue
  int max_clusters_fp8[2][2] = {};  // [out_f32][pair], FP8 operands
  uint32_t* d_status = nullptr;
  uint64_t timeout_ns = 2000000000ull;
  int64_t launches = 0;
};

namespace {

thread_local std::string g_last_error;

}  // namespace

void mosaic::set_last_error(const char* msg) { g_last_error = msg; }

namespace {

mosaic_status fail(mosaic_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

mosaic_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOSAIC_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Device memory the handle's GPU can address (device or managed allocation).
bool is_device_ptr(const void* p, int device) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeDevice) return a.device == device;
  return a.type == cudaMemoryTypeManaged;
}

// 2-D row-major tensor [rows, cols] of `elt`-byte elements, box {box_cols, box_rows}, swizzled
// at the width of a box row (box_cols * elt: 64 or 128 bytes), zero fill outside the tensor.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t elt, const void* base,
               uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * elt};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  box_cols * elt == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// L2 bytes a raster group's gathered rows may take (compile-time, for tuning runs).
#ifndef MOSAIC_L2_GROUP_BYTES
#define MOSAIC_L2_GROUP_BYTES (64ll << 20)
#endif

// M units per raster group: as many as keep the group's gathered rows (cluster_m x BM rows of
// row_bytes per unit) within MOSAIC_L2_GROUP_BYTES of L2, so that W panels are streamed once per
// group.
int pick_group_u(int m_units, int cm, int64_t row_bytes) {
  const int64_t per_unit = static_cast<int64_t>(cm) * mosaic::gather_gemm_block_m() * row_bytes;
  int64_t g = static_cast<int64_t>(MOSAIC_L2_GROUP_BYTES) / per_unit;
  if (g < 1) g = 1;
  if (g > m_units) g = m_units;
  return static_cast<int>(g);
}

}  // namespace

extern "C" {

const char* mosaic_last_error_string(void) { return g_last_error.c_str(); }

mosaic_status mosaic_min_chunk_rows(int64_t M, int64_t V, mosaic_dtype out_dtype,
                                    int64_t budget_bytes, int64_t* chunk_rows,
                                    int64_t* n_chunks) {
  if (!chunk_rows || !n_chunks) return fail(MOSAIC_ERR_INVALID_ARG, "NULL output pointer");
  if (M < 0 || V < 1 || budget_bytes < 0)
    return fail(MOSAIC_ERR_INVALID_ARG, "need M >= 0, V >= 1, budget_bytes >= 0");
  if (out_dtype != MOSAIC_BF16 && out_dtype != MOSAIC_F32)
    return fail(MOSAIC_ERR_INVALID_ARG, "unknown out_dtype %d", static_cast<int>(out_dtype));
  const int64_t row_bytes = V * (out_dtype == MOSAIC_F32 ? 4 : 2);
  const int64_t fit = budget_bytes / row_bytes;  // most rows the budget holds
  if (M <= fit) {  // everything fits: chunking stays off
    *chunk_rows = 0;
    *n_chunks = M > 0 ? 1 : 0;
    return MOSAIC_OK;
  }
  if (fit < 1)
    return fail(MOSAIC_ERR_UNSUPPORTED, "a budget of %lld bytes holds no output row of %lld bytes",
                static_cast<long long>(budget_bytes), static_cast<long long>(row_bytes));
  const int64_t n = (M + fit - 1) / fit;      // fewest chunks whose rows fit
  const int64_t rows = (M + n - 1) / n;       // balanced: rows <= fit
  *chunk_rows = rows;
  *n_chunks = (M + rows - 1) / rows;
  return MOSAIC_OK;
}

mosaic_status mosaic_create(mosaic_handle** handle, int device) {
  if (!handle) return fail(MOSAIC_ERR_INVALID_ARG, "handle out-pointer is NULL");
  *handle = nullptr;
  cudaError_t e = cudaSetDevice(device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
  if (prop.major != 10 || prop.minor != 3)
    return fail(MOSAIC_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                device, prop.major, prop.minor);
  if (!encode_fn()) return fail(MOSAIC_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
  auto* h = new mosaic_handle();
  h->device = device;
  h->num_sms = prop.multiProcessorCount;
  for (int f32 = 0; f32 < 2; ++f32) {
    for (int pair = 0; pair < 2 && e == cudaSuccess; ++pair) {
      e = mosaic::gather_gemm_prepare(f32 != 0, pair != 0, &h->max_clusters[f32][pair]);
      if (e == cudaSuccess && h->max_clusters[f32][pair] < 1) e = cudaErrorInvalidConfiguration;
    }
    if (e != cudaSuccess) {
      delete h;
      return cuda_fail(e, "kernel attributes (registers per thread) / cluster occupancy");
    }
  }
  for (int pair = 0; pair < 2 && e == cudaSuccess; ++pair) {
    e = mosaic::gather_gemm_prepare_sample(pair != 0, &h->max_clusters_sample[pair]);
    if (e == cudaSuccess && h->max_clusters_sample[pair] < 1) e = cudaErrorInvalidConfiguration;
  }
  for (int f32 = 0; f32 < 2 && e == cudaSuccess; ++f32)
    for (int pair = 0; pair < 2 && e == cudaSuccess; ++pair) {
      e = mosaic::gather_gemm_prepare_fp8(f32 != 0, pair != 0, &h->max_clusters_fp8[f32][pair]);
      if (e == cudaSuccess && h->max_clusters_fp8[f32][pair] < 1) e = cudaErrorInvalidConfiguration;
    }
  if (e != cudaSuccess) {
    delete h;
    return cuda_fail(e, "sampling / FP8 kernel attributes (registers per thread), cluster occupancy");
  }
  e = cudaMalloc(&h->d_status, 256);
  if (e == cudaSuccess) e = cudaMemset(h->d_status, 0, 256);
  if (e != cudaSuccess) {
    if (h->d_status) cudaFree(h->d_status);
    delete h;
    return cuda_fail(e, "status word allocation");
  }
  *handle = h;
  g_last_error.clear();
  return MOSAIC_OK;
}

mosaic_status mosaic_destroy(mosaic_handle* h) {
  if (!h) return MOSAIC_OK;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  cudaFree(h->d_status);
  delete h;
  return MOSAIC_OK;
}

mosaic_status mosaic_set_wait_timeout(mosaic_handle* h, uint64_t timeout_ns) {
  if (!h) return fail(MOSAIC_ERR_INVALID_ARG, "NULL handle");
  h->timeout_ns = timeout_ns;
  return MOSAIC_OK;
}

int64_t mosaic_launch_count(const mosaic_handle* h) { return h ? h->launches : -1; }

mosaic_status mosaic_check(mosaic_handle* h, void* stream) {
  if (!h) return fail(MOSAIC_ERR_INVALID_ARG, "NULL handle");
  cudaSetDevice(h->device);
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t word = 0;
  e = cudaMemcpy(&word, h->d_status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
  e = cudaMemset(h->d_status, 0, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
  if (word & mosaic::MOSAIC_STATUS_TIMEOUT)
    return fail(MOSAIC_ERR_TIMEOUT, "a bounded wait inside the kernel ran out");
  if (word & mosaic::MOSAIC_STATUS_INDEX)
    return fail(MOSAIC_ERR_INDEX, "a mask index (or CSR offset) was outside its sequence");
  return MOSAIC_OK;
}

}  // extern "C"

namespace {

// The lazy-chunk driver of mosaic_masked_logits and mosaic_masked_logits_fp8. fp8: hidden and W
// hold E4M3 codes (one byte per element) with per-row scales h_scale [L_tot] and w_scale [V].
mosaic_status logits_impl(mosaic_handle* h, const void* hidden, const float* h_scale,
                          int64_t L_tot, int64_t d, const int32_t* mask_idx, int64_t M,
                          const int32_t* seq_offsets, const int32_t* mask_offsets, int32_t B,
                          const void* W, const float* w_scale, int64_t V, void* out,
                          mosaic_dtype out_dtype, int64_t chunk_rows, mosaic_chunk_cb cb,
                          void* user, void* stream_ptr, bool fp8) {
  if (!h) return fail(MOSAIC_ERR_INVALID_ARG, "NULL handle");
  if (M < 0) return fail(MOSAIC_ERR_INVALID_ARG, "M < 0");
  if (M >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "M >= 2^31");
  if (out_dtype != MOSAIC_BF16 && out_dtype != MOSAIC_F32)
    return fail(MOSAIC_ERR_INVALID_ARG, "unknown out_dtype %d", static_cast<int>(out_dtype));
  if ((seq_offsets == nullptr) != (mask_offsets == nullptr))
    return fail(MOSAIC_ERR_INVALID_ARG, "CSR mode needs both seq_offsets and mask_offsets");
  const bool csr = seq_offsets != nullptr;
  if (csr && B < 1) return fail(MOSAIC_ERR_INVALID_ARG, "CSR mode needs B >= 1");
  const bool chunked = chunk_rows > 0 && chunk_rows < M;
  if (chunked && !cb) return fail(MOSAIC_ERR_INVALID_ARG, "chunking on (chunk_rows < M) needs a callback");
  if (M == 0) return MOSAIC_OK;  // nothing to read or write: no launch, no callback
  if (!hidden || !W || !out || !mask_idx)
    return fail(MOSAIC_ERR_INVALID_ARG, "NULL hidden, W, out or mask_idx");
  if (d < 1 || V < 1 || L_tot < 1) return fail(MOSAIC_ERR_INVALID_ARG, "d, V and L_tot must be >= 1");
  if (d % 8 != 0) return fail(MOSAIC_ERR_UNSUPPORTED, "d must be a multiple of 8 (16-byte rows)");
  if (V % 8 != 0) return fail(MOSAIC_ERR_UNSUPPORTED, "V must be a multiple of 8 (16-byte rows)");
  if (L_tot >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "L_tot >= 2^31");
  if (V >= (1ll << 31) || d >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "V or d too large");
  if (!aligned16(hidden) || !aligned16(W) || !aligned16(out))
    return fail(MOSAIC_ERR_INVALID_ARG, "hidden, W and out must be 16-byte aligned");
  if (fp8) {
    if (d % 16 != 0) return fail(MOSAIC_ERR_UNSUPPORTED, "d must be a multiple of 16 (16-byte E4M3 rows)");
    if (!h_scale || !w_scale) return fail(MOSAIC_ERR_INVALID_ARG, "NULL hidden_scale or w_scale");
    if (!aligned16(w_scale) || reinterpret_cast<uintptr_t>(h_scale) % 4 != 0)
      return fail(MOSAIC_ERR_INVALID_ARG, "w_scale must be 16-byte aligned, hidden_scale 4-byte aligned");
  }

  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  if (!is_device_ptr(hidden, h->device) || !is_device_ptr(W, h->device) ||
      !is_device_ptr(out, h->device) || !is_device_ptr(mask_idx, h->device) ||
      (csr && (!is_device_ptr(seq_offsets, h->device) || !is_device_ptr(mask_offsets, h->device))) ||
      (fp8 && (!is_device_ptr(h_scale, h->device) || !is_device_ptr(w_scale, h->device))))
    return fail(MOSAIC_ERR_INVALID_ARG, "every array must be device memory of device %d", h->device);

  const bool f32 = out_dtype == MOSAIC_F32;
  const int BM = mosaic::gather_gemm_block_m(), BN = mosaic::gather_gemm_block_n(),
            BK = fp8 ? mosaic::gather_gemm_block_k_fp8() : mosaic::gather_gemm_block_k();
  const int elt = fp8 ? 1 : 2;
  const int64_t cr = chunked ? chunk_rows : M;
  const int64_t n_tiles = (V + BN - 1) / BN;
  const int64_t m_tiles_max = (cr + BM - 1) / BM;
  if (m_tiles_max * n_tiles >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "too many tiles");

  // A CTA pair (256-row tiles) whenever there is more than one M tile; the choice is fixed for
  // the whole call (from the largest chunk) so every chunk runs the same kernel.
  const bool pair = m_tiles_max >= 2;
  const int cm = pair ? 2 : 1;
  CUtensorMap tm_w, tm_out;
  if (!encode_2d(&tm_w, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                 elt, W, V, d, mosaic::gather_gemm_w_box_rows(pair), BK))
    return fail(MOSAIC_ERR_UNSUPPORTED, "tensor map for W rejected");

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int64_t n_chunks = (M + cr - 1) / cr;
  for (int64_t c = 0; c < n_chunks; ++c) {
    const int64_t rb = c * cr;
    const int64_t rows = (M - rb < cr) ? (M - rb) : cr;
    const CUtensorMapDataType odt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!encode_2d(&tm_out, odt, f32 ? 4 : 2, out, rows, V, BM, mosaic::gather_gemm_epi_cols(f32)))
      return fail(MOSAIC_ERR_UNSUPPORTED, "tensor map for out rejected");
    mosaic::GatherGemmParams p = {};  // fields a variant does not use stay null
    p.hidden = hidden;
    p.idx = mask_idx;
    p.seq_offsets = csr ? seq_offsets : nullptr;
    p.mask_offsets = csr ? mask_offsets : nullptr;
    p.L_tot = L_tot;
    p.B = csr ? B : 0;
    p.M_total = static_cast<int32_t>(M);
    p.row_begin = static_cast<int32_t>(rb);
    p.rows = static_cast<int32_t>(rows);
    p.chunk_index = static_cast<int32_t>(c);
    p.V = static_cast<int32_t>(V);
    p.d = static_cast<int32_t>(d);
    p.k_blocks = static_cast<int32_t>((d + BK - 1) / BK);
    p.m_tiles = static_cast<int32_t>((rows + BM - 1) / BM);
    p.n_tiles = static_cast<int32_t>(n_tiles);
    p.cluster_m = cm;
    p.m_units = (p.m_tiles + cm - 1) / cm;
    p.group_u = pick_group_u(p.m_units, cm, d * elt);
    p.status = h->d_status;
    p.timeout_ns = h->timeout_ns;
    p.a_scale = h_scale;
    p.b_scale = w_scale;
    if (fp8) {
      const int grid =
          mosaic::gather_gemm_schedule(p, h->max_clusters_fp8[f32 ? 1 : 0][pair ? 1 : 0]);
      e = mosaic::gather_gemm_launch_fp8(tm_w, tm_out, p, f32, grid, stream);
    } else {
      const int grid = mosaic::gather_gemm_schedule(p, h->max_clusters[f32 ? 1 : 0][pair ? 1 : 0]);
      e = mosaic::gather_gemm_launch(tm_w, tm_out, p, f32, grid, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "gather-GEMM launch");
    ++h->launches;
    if (cb) cb(c, rb, rows, out, user);
  }
  return MOSAIC_OK;
}

}  // namespace

extern "C" {

mosaic_status mosaic_masked_logits(mosaic_handle* h, const void* hidden, int64_t L_tot,
                                   int64_t d, const int32_t* mask_idx, int64_t M,
                                   const int32_t* seq_offsets, const int32_t* mask_offsets,
                                   int32_t B, const void* W, int64_t V, void* out,
                                   mosaic_dtype out_dtype, int64_t chunk_rows,
                                   mosaic_chunk_cb cb, void* user, void* stream_ptr) {
  return logits_impl(h, hidden, nullptr, L_tot, d, mask_idx, M, seq_offsets, mask_offsets, B, W,
                     nullptr, V, out, out_dtype, chunk_rows, cb, user, stream_ptr, false);
}

mosaic_status mosaic_masked_logits_fp8(mosaic_handle* h, const void* hidden_q,
                                       const float* hidden_scale, int64_t L_tot, int64_t d,
                                       const int32_t* mask_idx, int64_t M,
                                       const int32_t* seq_offsets, const int32_t* mask_offsets,
                                       int32_t B, const void* W_q, const float* w_scale,
                                       int64_t V, void* out, mosaic_dtype out_dtype,
                                       int64_t chunk_rows, mosaic_chunk_cb cb, void* user,
                                       void* stream_ptr) {
  return logits_impl(h, hidden_q, hidden_scale, L_tot, d, mask_idx, M, seq_offsets, mask_offsets,
                     B, W_q, w_scale, V, out, out_dtype, chunk_rows, cb, user, stream_ptr, true);
}

mosaic_status mosaic_quantize_masked_rows_e4m3(const void* hidden, int64_t L_tot, int64_t d,
                                               const int32_t* mask_idx, int64_t M,
                                               const int32_t* seq_offsets,
                                               const int32_t* mask_offsets, int32_t B,
                                               void* hidden_q, float* hidden_scale,
                                               void* stream_ptr) {
  if (M < 0 || L_tot < 1 || d < 1) return fail(MOSAIC_ERR_INVALID_ARG, "M < 0, L_tot < 1 or d < 1");
  if (d % 16 != 0) return fail(MOSAIC_ERR_UNSUPPORTED, "d must be a multiple of 16");
  if (M >= (1ll << 31) || L_tot >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "M or L_tot >= 2^31");
  if ((seq_offsets == nullptr) != (mask_offsets == nullptr))
    return fail(MOSAIC_ERR_INVALID_ARG, "CSR mode needs both seq_offsets and mask_offsets");
  const bool csr = seq_offsets != nullptr;
  if (csr && B < 1) return fail(MOSAIC_ERR_INVALID_ARG, "CSR mode needs B >= 1");
  if (M == 0) return MOSAIC_OK;
  if (!hidden || !mask_idx || !hidden_q || !hidden_scale)
    return fail(MOSAIC_ERR_INVALID_ARG, "NULL hidden, mask_idx, hidden_q or hidden_scale");
  if (!aligned16(hidden) || !aligned16(hidden_q) || reinterpret_cast<uintptr_t>(hidden_scale) % 4 != 0)
    return fail(MOSAIC_ERR_INVALID_ARG, "hidden and hidden_q must be 16-byte aligned, hidden_scale 4-byte aligned");
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (!is_device_ptr(hidden, device) || !is_device_ptr(mask_idx, device) ||
      !is_device_ptr(hidden_q, device) || !is_device_ptr(hidden_scale, device) ||
      (csr && (!is_device_ptr(seq_offsets, device) || !is_device_ptr(mask_offsets, device))))
    return fail(MOSAIC_ERR_INVALID_ARG, "every array must be device memory of the current device");
  e = mosaic::quantize_masked_rows_e4m3_launch(hidden, L_tot, d, mask_idx, M,
                                               csr ? seq_offsets : nullptr,
                                               csr ? mask_offsets : nullptr, csr ? B : 0,
                                               hidden_q, hidden_scale,
                                               static_cast<cudaStream_t>(stream_ptr));
  if (e != cudaSuccess) return cuda_fail(e, "quantization launch");
  return MOSAIC_OK;
}

mosaic_status mosaic_quantize_rows_e4m3(const void* x, int64_t rows, int64_t d, void* q,
                                        float* scale, void* stream_ptr) {
  if (rows < 0 || d < 1) return fail(MOSAIC_ERR_INVALID_ARG, "rows < 0 or d < 1");
  if (d % 16 != 0) return fail(MOSAIC_ERR_UNSUPPORTED, "d must be a multiple of 16");
  if (rows >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "rows >= 2^31");
  if (rows == 0) return MOSAIC_OK;
  if (!x || !q || !scale) return fail(MOSAIC_ERR_INVALID_ARG, "NULL x, q or scale");
  if (!aligned16(x) || !aligned16(q) || reinterpret_cast<uintptr_t>(scale) % 4 != 0)
    return fail(MOSAIC_ERR_INVALID_ARG, "x and q must be 16-byte aligned, scale 4-byte aligned");
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (!is_device_ptr(x, device) || !is_device_ptr(q, device) || !is_device_ptr(scale, device))
    return fail(MOSAIC_ERR_INVALID_ARG, "x, q and scale must be device memory of the current device");
  e = mosaic::quantize_rows_e4m3_launch(x, rows, d, q, scale, static_cast<cudaStream_t>(stream_ptr));
  if (e != cudaSuccess) return cuda_fail(e, "quantization launch");
  return MOSAIC_OK;
}

int64_t mosaic_masked_sample_workspace_bytes(int64_t M, int64_t V, int64_t chunk_rows) {
  if (M < 0 || V < 1) return -1;
  const int64_t cr = (chunk_rows > 0 && chunk_rows < M) ? chunk_rows : M;
  const int64_t n_tiles = (V + mosaic::gather_gemm_block_n() - 1) / mosaic::gather_gemm_block_n();
  const int64_t ld = (n_tiles + 3) / 4 * 4;  // partials of one row, 16-byte aligned
  return 3 * cr * ld * 4;
}

mosaic_status mosaic_masked_sample(mosaic_handle* h, const void* hidden, int64_t L_tot, int64_t d,
                                   const int32_t* mask_idx, int64_t M,
                                   const int32_t* seq_offsets, const int32_t* mask_offsets,
                                   int32_t B, const void* W, int64_t V, int32_t* token,
                                   float* confidence, void* workspace, int64_t workspace_bytes,
                                   int64_t chunk_rows, void* stream_ptr) {
  if (!h) return fail(MOSAIC_ERR_INVALID_ARG, "NULL handle");
  if (M < 0) return fail(MOSAIC_ERR_INVALID_ARG, "M < 0");
  if (M >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "M >= 2^31");
  if ((seq_offsets == nullptr) != (mask_offsets == nullptr))
    return fail(MOSAIC_ERR_INVALID_ARG, "CSR mode needs both seq_offsets and mask_offsets");
  const bool csr = seq_offsets != nullptr;
  if (csr && B < 1) return fail(MOSAIC_ERR_INVALID_ARG, "CSR mode needs B >= 1");
  if (M == 0) return MOSAIC_OK;
  if (!hidden || !W || !mask_idx || !token || !confidence || !workspace)
    return fail(MOSAIC_ERR_INVALID_ARG, "NULL hidden, W, mask_idx, token, confidence or workspace");
  if (d < 1 || V < 1 || L_tot < 1) return fail(MOSAIC_ERR_INVALID_ARG, "d, V and L_tot must be >= 1");
  if (d % 8 != 0) return fail(MOSAIC_ERR_UNSUPPORTED, "d must be a multiple of 8 (16-byte rows)");
  if (L_tot >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "L_tot >= 2^31");
  if (V >= (1ll << 31) || d >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "V or d too large");
  if (!aligned16(hidden) || !aligned16(W) || !aligned16(workspace))
    return fail(MOSAIC_ERR_INVALID_ARG, "hidden, W and workspace must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(token) & 3u) || (reinterpret_cast<uintptr_t>(confidence) & 3u))
    return fail(MOSAIC_ERR_INVALID_ARG, "token and confidence must be 4-byte aligned");
  const int64_t need = mosaic_masked_sample_workspace_bytes(M, V, chunk_rows);
  if (workspace_bytes < need)
    return fail(MOSAIC_ERR_INVALID_ARG, "workspace of %lld bytes, %lld needed",
                static_cast<long long>(workspace_bytes), static_cast<long long>(need));
  cudaError_t e = cudaSetDevice(h->device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaSetDevice");
  if (!is_device_ptr(hidden, h->device) || !is_device_ptr(W, h->device) ||
      !is_device_ptr(mask_idx, h->device) || !is_device_ptr(token, h->device) ||
      !is_device_ptr(confidence, h->device) || !is_device_ptr(workspace, h->device) ||
      (csr && (!is_device_ptr(seq_offsets, h->device) || !is_device_ptr(mask_offsets, h->device))))
    return fail(MOSAIC_ERR_INVALID_ARG, "every array must be device memory of device %d", h->device);

  const int BM = mosaic::gather_gemm_block_m(), BN = mosaic::gather_gemm_block_n(),
            BK = mosaic::gather_gemm_block_k();
  const bool chunked = chunk_rows > 0 && chunk_rows < M;
  const int64_t cr = chunked ? chunk_rows : M;
  const int64_t n_tiles = (V + BN - 1) / BN;
  const int64_t m_tiles_max = (cr + BM - 1) / BM;
  if (m_tiles_max * n_tiles >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "too many tiles");
  const bool pair = m_tiles_max >= 2;
  const int cm = pair ? 2 : 1;
  CUtensorMap tm_w;
  if (!encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, V, d,
                 mosaic::gather_gemm_w_box_rows(pair), BK))
    return fail(MOSAIC_ERR_UNSUPPORTED, "tensor map for W rejected");
  const int64_t ld = (n_tiles + 3) / 4 * 4;
  float* part_max = static_cast<float*>(workspace);
  float* part_sum = part_max + cr * ld;
  int32_t* part_arg = reinterpret_cast<int32_t*>(part_sum + cr * ld);

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const int64_t n_chunks = (M + cr - 1) / cr;
  for (int64_t c = 0; c < n_chunks; ++c) {
    const int64_t rb = c * cr;
    const int64_t rows = (M - rb < cr) ? (M - rb) : cr;
    mosaic::GatherGemmParams p = {};
    p.hidden = hidden;
    p.idx = mask_idx;
    p.seq_offsets = csr ? seq_offsets : nullptr;
    p.mask_offsets = csr ? mask_offsets : nullptr;
    p.L_tot = L_tot;
    p.B = csr ? B : 0;
    p.M_total = static_cast<int32_t>(M);
    p.row_begin = static_cast<int32_t>(rb);
    p.rows = static_cast<int32_t>(rows);
    p.chunk_index = static_cast<int32_t>(c);
    p.V = static_cast<int32_t>(V);
    p.d = static_cast<int32_t>(d);
    p.k_blocks = static_cast<int32_t>((d + BK - 1) / BK);
    p.m_tiles = static_cast<int32_t>((rows + BM - 1) / BM);
    p.n_tiles = static_cast<int32_t>(n_tiles);
    p.cluster_m = cm;
    p.m_units = (p.m_tiles + cm - 1) / cm;
    p.group_u = pick_group_u(p.m_units, cm, d * 2);
    p.status = h->d_status;
    p.timeout_ns = h->timeout_ns;
    p.part_max = part_max;
    p.part_sum = part_sum;
    p.part_arg = part_arg;
    p.part_ld = static_cast<int32_t>(ld);
    const int grid = mosaic::gather_gemm_schedule(p, h->max_clusters_sample[pair ? 1 : 0]);
    e = mosaic::gather_gemm_launch_sample(tm_w, p, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "gather-GEMM (sampling) launch");
    e = mosaic::sample_reduce_launch(p, token, confidence, stream);
    if (e != cudaSuccess) return cuda_fail(e, "sampling reduction launch");
    h->launches += 2;
  }
  return MOSAIC_OK;
}

// ---------------------------------------------------------------------------------------------
// Allocation-free entry point. Its scratch (one status word per chunk) lives in this fixed
// device array instead of memory from cudaMalloc; host code must not use the array's name as a
// device address, so each device's address is looked up once with cudaGetSymbolAddress.
// ---------------------------------------------------------------------------------------------

static __device__ __align__(256) uint32_t g_noalloc_status[MOSAIC_NOALLOC_MAX_CHUNKS];

namespace {

struct NoallocDevice {
  bool ready = false;
  int num_sms = 0;
  int max_clusters[2][2] = {};
  uint32_t* status = nullptr;  // device address of g_noalloc_status on this device
};

constexpr int kMaxDevices = 64;
NoallocDevice g_noalloc_dev[kMaxDevices];
std::mutex g_noalloc_mutex;

// Once per device, with that device current: kernel attributes, occupancy, array address.
mosaic_status noalloc_setup(int device, NoallocDevice** out) {
  if (device < 0 || device >= kMaxDevices) return fail(MOSAIC_ERR_UNSUPPORTED, "device id %d", device);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  NoallocDevice& nd = g_noalloc_dev[device];
  if (!nd.ready) {
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, device);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
      return fail(MOSAIC_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                  device, prop.major, prop.minor);
    if (!encode_fn()) return fail(MOSAIC_ERR_CUDA, "cuTensorMapEncodeTiled entry point not found");
    for (int f32 = 0; f32 < 2; ++f32)
      for (int pair = 0; pair < 2; ++pair) {
        e = mosaic::gather_gemm_prepare(f32 != 0, pair != 0, &nd.max_clusters[f32][pair]);
        if (e != cudaSuccess)
          return cuda_fail(e, "kernel attributes (registers per thread) / cluster occupancy");
        if (nd.max_clusters[f32][pair] < 1) return fail(MOSAIC_ERR_CUDA, "kernel cannot be resident");
      }
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_noalloc_status);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress of the status array");
    nd.status = static_cast<uint32_t*>(ptr);
    nd.num_sms = prop.multiProcessorCount;
    nd.ready = true;
  }
  *out = &nd;
  return MOSAIC_OK;
}

}  // namespace

mosaic_status mosaic_masked_logits_noalloc(const void* hidden, int64_t L_tot, int64_t d,
                                           const int32_t* mask_idx, int64_t M,
                                           const int32_t* seq_offsets,
                                           const int32_t* mask_offsets, int32_t B,
                                           const void* W, int64_t V, void* out,
                                           mosaic_dtype out_dtype, int64_t chunk_rows,
                                           mosaic_chunk_cb cb, void* user,
                                           uint32_t* chunk_status, void* stream_ptr) {
  if (M < 0) return fail(MOSAIC_ERR_INVALID_ARG, "M < 0");
  if (M >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "M >= 2^31");
  if (out_dtype != MOSAIC_BF16 && out_dtype != MOSAIC_F32)
    return fail(MOSAIC_ERR_INVALID_ARG, "unknown out_dtype %d", static_cast<int>(out_dtype));
  if ((seq_offsets == nullptr) != (mask_offsets == nullptr))
    return fail(MOSAIC_ERR_INVALID_ARG, "CSR mode needs both seq_offsets and mask_offsets");
  const bool csr = seq_offsets != nullptr;
  if (csr && B < 1) return fail(MOSAIC_ERR_INVALID_ARG, "CSR mode needs B >= 1");
  const bool chunked = chunk_rows > 0 && chunk_rows < M;
  if (chunked && !cb) return fail(MOSAIC_ERR_INVALID_ARG, "chunking on (chunk_rows < M) needs a callback");
  if (M == 0) return MOSAIC_OK;
  if (!hidden || !W || !out || !mask_idx)
    return fail(MOSAIC_ERR_INVALID_ARG, "NULL hidden, W, out or mask_idx");
  if (d < 1 || V < 1 || L_tot < 1) return fail(MOSAIC_ERR_INVALID_ARG, "d, V and L_tot must be >= 1");
  if (d % 8 != 0) return fail(MOSAIC_ERR_UNSUPPORTED, "d must be a multiple of 8 (16-byte rows)");
  if (V % 8 != 0) return fail(MOSAIC_ERR_UNSUPPORTED, "V must be a multiple of 8 (16-byte rows)");
  if (L_tot >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "L_tot >= 2^31");
  if (V >= (1ll << 31) || d >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "V or d too large");
  if (!aligned16(hidden) || !aligned16(W) || !aligned16(out))
    return fail(MOSAIC_ERR_INVALID_ARG, "hidden, W and out must be 16-byte aligned");
  const int64_t cr = chunked ? chunk_rows : M;
  const int64_t n_chunks = (M + cr - 1) / cr;
  if (n_chunks > MOSAIC_NOALLOC_MAX_CHUNKS)
    return fail(MOSAIC_ERR_UNSUPPORTED,
                "%lld chunks exceed the %d status words of the allocation-free entry point; "
                "raise chunk_rows or use mosaic_masked_logits",
                static_cast<long long>(n_chunks), MOSAIC_NOALLOC_MAX_CHUNKS);

  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  NoallocDevice* nd = nullptr;
  mosaic_status st = noalloc_setup(device, &nd);
  if (st != MOSAIC_OK) return st;
  if (!is_device_ptr(hidden, device) || !is_device_ptr(W, device) ||
      !is_device_ptr(out, device) || !is_device_ptr(mask_idx, device) ||
      (csr && (!is_device_ptr(seq_offsets, device) || !is_device_ptr(mask_offsets, device))))
    return fail(MOSAIC_ERR_INVALID_ARG, "every array must be device memory of device %d", device);

  const bool f32 = out_dtype == MOSAIC_F32;
  const int BM = mosaic::gather_gemm_block_m(), BN = mosaic::gather_gemm_block_n(),
            BK = mosaic::gather_gemm_block_k();
  const int64_t n_tiles = (V + BN - 1) / BN;
  const int64_t m_tiles_max = (cr + BM - 1) / BM;
  if (m_tiles_max * n_tiles >= (1ll << 31)) return fail(MOSAIC_ERR_UNSUPPORTED, "too many tiles");
  const bool pair = m_tiles_max >= 2;
  const int cm = pair ? 2 : 1;
  CUtensorMap tm_w, tm_out;
  if (!encode_2d(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, W, V, d,
                 mosaic::gather_gemm_w_box_rows(pair), BK))
    return fail(MOSAIC_ERR_UNSUPPORTED, "tensor map for W rejected");

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  // The array keeps the previous call's words: clear the ones this call uses, in stream order.
  e = cudaMemsetAsync(nd->status, 0, static_cast<size_t>(n_chunks) * sizeof(uint32_t), stream);
  if (e != cudaSuccess) return cuda_fail(e, "clearing the status words");
  for (int64_t c = 0; c < n_chunks; ++c) {
    const int64_t rb = c * cr;
    const int64_t rows = (M - rb < cr) ? (M - rb) : cr;
    const CUtensorMapDataType odt = f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!encode_2d(&tm_out, odt, f32 ? 4 : 2, out, rows, V, BM, mosaic::gather_gemm_epi_cols(f32)))
      return fail(MOSAIC_ERR_UNSUPPORTED, "tensor map for out rejected");
    mosaic::GatherGemmParams p = {};  // fields a variant does not use stay null
    p.hidden = hidden;
    p.idx = mask_idx;
    p.seq_offsets = csr ? seq_offsets : nullptr;
    p.mask_offsets = csr ? mask_offsets : nullptr;
    p.L_tot = L_tot;
    p.B = csr ? B : 0;
    p.M_total = static_cast<int32_t>(M);
    p.row_begin = static_cast<int32_t>(rb);
    p.rows = static_cast<int32_t>(rows);
    p.chunk_index = static_cast<int32_t>(c);
    p.V = static_cast<int32_t>(V);
    p.d = static_cast<int32_t>(d);
    p.k_blocks = static_cast<int32_t>((d + BK - 1) / BK);
    p.m_tiles = static_cast<int32_t>((rows + BM - 1) / BM);
    p.n_tiles = static_cast<int32_t>(n_tiles);
    p.cluster_m = cm;
    p.m_units = (p.m_tiles + cm - 1) / cm;
    p.group_u = pick_group_u(p.m_units, cm, d * 2);
    p.status = nd->status + c;  // this chunk's word of the fixed array
    p.timeout_ns = 2000000000ull;
    const int grid = mosaic::gather_gemm_schedule(p, nd->max_clusters[f32 ? 1 : 0][pair ? 1 : 0]);
    e = mosaic::gather_gemm_launch(tm_w, tm_out, p, f32, grid, stream);
    if (e != cudaSuccess) return cuda_fail(e, "gather-GEMM launch");
    if (cb) cb(c, rb, rows, out, user);
  }
  if (!chunk_status) return MOSAIC_OK;
  e = cudaMemcpyAsync(chunk_status, nd->status, static_cast<size_t>(n_chunks) * sizeof(uint32_t),
                      cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "reading the status words");
  uint32_t any = 0;
  for (int64_t c = 0; c < n_chunks; ++c) any |= chunk_status[c];
  if (any & mosaic::MOSAIC_STATUS_TIMEOUT)
    return fail(MOSAIC_ERR_TIMEOUT, "a bounded wait inside the kernel ran out");
  if (any & mosaic::MOSAIC_STATUS_INDEX)
    return fail(MOSAIC_ERR_INDEX, "a mask index (or CSR offset) was outside its sequence");
  return MOSAIC_OK;
}

}  // extern "C"
