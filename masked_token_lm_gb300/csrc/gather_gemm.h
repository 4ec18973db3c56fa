// Internal interface between the C-ABI host layer and the gather-GEMM kernel.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace mosaic {

// Bits of the device status word.
constexpr uint32_t MOSAIC_STATUS_INDEX = 1u;    // a mask index / CSR offset was out of range
constexpr uint32_t MOSAIC_STATUS_TIMEOUT = 2u;  // a bounded wait gave up

struct GatherGemmParams {
  const void* hidden;           // bf16 [L_tot, d]
  const int32_t* idx;           // [M_total] mask indices (whole list, not just this chunk)
  const int32_t* seq_offsets;   // CSR [B+1] or nullptr
  const int32_t* mask_offsets;  // CSR [B+1] or nullptr
  int64_t L_tot;                // rows of H
  int32_t B;                    // sequences (CSR mode)
  int32_t M_total;              // all masked positions
  int32_t row_begin;            // first flat position of this chunk
  int32_t rows;                 // positions in this chunk
  int32_t chunk_index;
  int32_t V;
  int32_t d;
  int32_t k_blocks;             // ceil(d / BK)
  int32_t m_tiles, n_tiles;     // ceil(rows / BM), ceil(V / BN): BN-wide column panels
  int32_t cluster_m;            // 2: a CTA pair computes 256-row tiles (cta_group::2); 1: single
  int32_t m_units;              // ceil(m_tiles / cluster_m)
  int32_t group_u;              // M units per raster group
  // Work units (set by gather_gemm_schedule): a unit is one M unit times n_sub consecutive
  // panels (n_sub = 2 for a pair, 1 for a single CTA); n_wide = ceil(n_tiles / n_sub) unit
  // columns. Units [0, units_full) are whole; when the last round of the persistent schedule is
  // at most half full, its units are split into two single-panel units each, numbered
  // units_full .. units_total - 1.
  int32_t n_wide;
  int32_t units_full;
  int32_t units_total;
  uint32_t* status;             // device status word
  uint64_t timeout_ns;          // bound on any single wait
  // Sampling epilogue only: per (row, N tile) partials at row * part_ld + n_tile.
  float* part_max;              // max logit of the row within the N tile
  float* part_sum;              // sum over the tile's columns of exp(logit - part_max)
  int32_t* part_arg;            // first column of the maximum (-1: the row's index was bad)
  int32_t part_ld;
  // FP8 variant only: per-row scales of the E4M3 operands (hidden rows [L_tot], W rows [V]).
  const float* a_scale;
  const float* b_scale;
};

int gather_gemm_block_m();
int gather_gemm_block_n();
int gather_gemm_block_k();
int gather_gemm_block_k_fp8();  // E4M3 elements per K block
int gather_gemm_epi_cols(bool out_f32);
int gather_gemm_w_box_rows(bool pair);
// Fills p.n_wide / units_full / units_total from p.m_units, p.n_tiles and p.cluster_m for a grid
// of at most max_clusters clusters, and returns the grid size in CTAs.
int gather_gemm_schedule(GatherGemmParams& p, int max_clusters);
// Sets the kernel's shared-memory attribute and reports how many clusters fit at once.
cudaError_t gather_gemm_prepare(bool out_f32, bool pair, int* clusters);
// Same for the sampling epilogue.
cudaError_t gather_gemm_prepare_sample(bool pair, int* clusters);
// Gather-GEMM whose epilogue writes per-tile sampling partials instead of logits.
cudaError_t gather_gemm_launch_sample(const CUtensorMap& tm_w, const GatherGemmParams& p, int grid,
                                      cudaStream_t stream);
// Combine the partials of `rows` rows into token[r] and confidence[r].
cudaError_t sample_reduce_launch(const GatherGemmParams& p, int32_t* token, float* confidence,
                                 cudaStream_t stream);
cudaError_t gather_gemm_launch(const CUtensorMap& tm_w, const CUtensorMap& tm_out,
                               const GatherGemmParams& p, bool out_f32, int grid,
                               cudaStream_t stream);
// FP8 variant: E4M3 hidden rows and W (tensor map of bytes), p.a_scale / p.b_scale per row.
cudaError_t gather_gemm_prepare_fp8(bool out_f32, bool pair, int* clusters);
cudaError_t gather_gemm_launch_fp8(const CUtensorMap& tm_w, const CUtensorMap& tm_out,
                                   const GatherGemmParams& p, bool out_f32, int grid,
                                   cudaStream_t stream);
// Per-row E4M3 quantization of a bf16 [rows, d] matrix into codes [rows, d] and scales [rows].
cudaError_t quantize_rows_e4m3_launch(const void* x, int64_t rows, int64_t d, void* q,
                                      float* scale, cudaStream_t stream);
// The same for only the hidden rows of masked positions 0..n-1 (flat or CSR, as in the logits
// call); other rows of q / scale are left as they are, out-of-range positions are skipped.
cudaError_t quantize_masked_rows_e4m3_launch(const void* x, int64_t L_tot, int64_t d,
                                             const int32_t* idx, int64_t n,
                                             const int32_t* seq_offsets,
                                             const int32_t* mask_offsets, int32_t B, void* q,
                                             float* scale, cudaStream_t stream);

}  // namespace mosaic
