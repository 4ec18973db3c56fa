// Per-row E4M3 quantization for the FP8 variant of mask-only logits.
//
// The dLLM-Serve article "扩散大语言模型内存优化：从理论到系统设计" (section 5, extensions and
// future directions) names FP8 quantization of the logit computation as a next step without a
// scheme; this one scales each row by its own maximum magnitude: a = max |x|,
// scale = a / 448, codes = E4M3(x * (448 / a)) rounded to nearest even and clamped to +-448 (the
// largest finite E4M3 value), with both divisions and the multiply single IEEE fp32 operations,
// so the codes and scales are a deterministic function of the bf16 input. A row of zeros gets
// scale 0 and zero codes.
//
// One warp per row: the lanes stride the row in 16-byte pieces (8 bf16), reduce the maximum with
// shuffles, then convert the same pieces (8 codes, 8 bytes each) in a second pass over the row,
// which L1/L2 still hold. The masked form quantizes only the rows a logits call will read, in
// place in an [L_tot, d] code buffer.
#include <cuda_runtime.h>

#include <cstdint>

#include "gather_gemm.h"
#include "ptx.cuh"

namespace mosaic {

namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Rows to quantize: all rows of x (rows_map.idx == nullptr), or the hidden rows of the masked
// positions 0..n-1 given like the logits call's mask (flat: idx[i]; CSR: seq_offsets[b] + idx[i]
// for the sequence b whose mask_offsets range holds i). Positions whose row is out of range are
// skipped (the logits call reports them).
struct RowsMap {
  const int32_t* idx;
  const int32_t* seq_offsets;
  const int32_t* mask_offsets;
  int32_t B;
  int64_t L_tot;
};

__device__ __forceinline__ int64_t map_row(const RowsMap& m, int64_t i) {
  if (m.idx == nullptr) return i;
  const int32_t v = __ldg(m.idx + i);
  if (m.mask_offsets == nullptr) return (v >= 0 && v < m.L_tot) ? v : -1;
  int32_t lo = 0, hi = m.B;  // largest b with mask_offsets[b] <= i
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if (__ldg(m.mask_offsets + mid) <= i) lo = mid; else hi = mid;
  }
  const int64_t s0 = __ldg(m.seq_offsets + lo), s1 = __ldg(m.seq_offsets + lo + 1);
  const int64_t r = s0 + v;
  return (v >= 0 && s0 >= 0 && r < s1 && s1 <= m.L_tot) ? r : -1;
}

__global__ void __launch_bounds__(256) quantize_rows_e4m3_kernel(const uint4* __restrict__ x,
                                                                 int64_t n, int64_t d,
                                                                 uint2* __restrict__ q,
                                                                 float* __restrict__ scale,
                                                                 const RowsMap rows_map) {
  const int lane = threadIdx.x & 31;
  const int64_t i = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= n) return;  // whole warps leave together
  const int64_t row = map_row(rows_map, i);
  if (row < 0) return;
  const int64_t pieces = d / 8;
  const uint4* xr = x + row * pieces;
  float a = 0.0f;
  for (int64_t k = lane; k < pieces; k += 32) {
    const uint4 w = __ldg(xr + k);
    a = fmaxf(a, fmaxf(fmaxf(fabsf(bf16_lo(w.x)), fabsf(bf16_hi(w.x))),
                       fmaxf(fabsf(bf16_lo(w.y)), fabsf(bf16_hi(w.y)))));
    a = fmaxf(a, fmaxf(fmaxf(fabsf(bf16_lo(w.z)), fabsf(bf16_hi(w.z))),
                       fmaxf(fabsf(bf16_lo(w.w)), fabsf(bf16_hi(w.w)))));
  }
  for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  const float inv = a > 0.0f ? __fdiv_rn(448.0f, a) : 0.0f;
  if (lane == 0) scale[row] = a > 0.0f ? __fdiv_rn(a, 448.0f) : 0.0f;
  uint2* qr = q + row * pieces;
  for (int64_t k = lane; k < pieces; k += 32) {
    const uint4 w = __ldg(xr + k);
    const uint32_t c01 = e4m3x2_rn(__fmul_rn(bf16_lo(w.x), inv), __fmul_rn(bf16_hi(w.x), inv));
    const uint32_t c23 = e4m3x2_rn(__fmul_rn(bf16_lo(w.y), inv), __fmul_rn(bf16_hi(w.y), inv));
    const uint32_t c45 = e4m3x2_rn(__fmul_rn(bf16_lo(w.z), inv), __fmul_rn(bf16_hi(w.z), inv));
    const uint32_t c67 = e4m3x2_rn(__fmul_rn(bf16_lo(w.w), inv), __fmul_rn(bf16_hi(w.w), inv));
    qr[k] = make_uint2(c01 | (c23 << 16), c45 | (c67 << 16));
  }
}

}  // namespace

cudaError_t quantize_rows_e4m3_launch(const void* x, int64_t rows, int64_t d, void* q,
                                      float* scale, cudaStream_t stream) {
  return quantize_masked_rows_e4m3_launch(x, rows, d, nullptr, rows, nullptr, nullptr, 0, q, scale,
                                          stream);
}

cudaError_t quantize_masked_rows_e4m3_launch(const void* x, int64_t L_tot, int64_t d,
                                             const int32_t* idx, int64_t n,
                                             const int32_t* seq_offsets,
                                             const int32_t* mask_offsets, int32_t B, void* q,
                                             float* scale, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const int rows_per_block = 8;
  const int64_t blocks = (n + rows_per_block - 1) / rows_per_block;
  const RowsMap m{idx, seq_offsets, mask_offsets, B, L_tot};
  quantize_rows_e4m3_kernel<<<static_cast<unsigned>(blocks), 32 * rows_per_block, 0, stream>>>(
      static_cast<const uint4*>(x), n, d, static_cast<uint2*>(q), scale, m);
  return cudaGetLastError();
}

}  // namespace mosaic
