// Mask-only logits as one persistent, warp-specialised gather-GEMM kernel for sm_103a.
//
//   out[i, v] = sum_k H[row(i), k] * W[v, k]      (bf16 x bf16 -> fp32 accumulate)
//
// The operation is the "Mask-only Logits Kernel" of "Mosaic: Unlocking Long-Context Inference
// for Diffusion LLMs via Global Memory" (paper review, section 3, core component 1): it reads
// the hidden states of all tokens through the mask indices (indirect addressing), tiles the
// GEMM over the GPU's compute units and keeps the gathered rows on chip, so no gathered [M, d]
// buffer is ever written. The pages' kernel targeted RTX 3090 / A100; this one is designed for
// Blackwell instead:
//
//   warps 6..9  A gather: each of the 128 threads resolves 8 of the tile's mask indices to
//               hidden rows (index staging, once per tile) and, per K block, copies one 16-byte
//               piece of each of its 8 rows with cp.async into the 128-byte-swizzled A stage of
//               a STAGES-deep shared-memory ring (8 threads cover one 128-byte row segment).
//   warp 0      W stream: one thread issues a 2-D TMA load of the 256 x 64 W tile per K block.
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=256, K=16) into a
//               double-buffered TMEM accumulator (2 x 256 columns) and commits stage releases.
//   warps 2..5  epilogue: tcgen05.ld the accumulator, round to bf16 (or keep fp32), write
//               128-byte-swizzled staging tiles and TMA-store them; rows past the chunk are
//               clipped by the store's tensor map.
//
// The A rows are gathered with cp.async rather than TMA tile::gather4: measured on GB300, the
// 32 gather4 instructions a 128-row K block needs held the kernel to ~26 % of the tensor peak,
// while the same bytes through the load/store units keep the tensor pipe fed.
//
// Tiles are walked by a static persistent schedule: within a group of M tiles, N panels outer
// and M tiles inner, so each W panel is fetched from HBM once per group while the gathered A
// rows of the group stay in L2.
//
// Every wait is bounded (globaltimer); a wait that runs out records MOSAIC status bit 2, makes
// all roles stop, drains in-flight copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gather_gemm.h"
#include "ptx.cuh"

namespace mosaic {

namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;  // 64 bf16 = 128 B = one swizzle row
constexpr int UMMA_K = 16;
constexpr int STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;  // 16 KiB
constexpr int B_STAGE = BN * BK * 2;  // 32 KiB
constexpr int EPI_BUF = BM * 128;     // 128 rows x 128 B
constexpr int EPI_BUFS = 2;
constexpr int TMEM_COLS = 2 * BN;     // two accumulators
constexpr int EPI_WARP0 = 2;
constexpr int EPI_THREADS = 128;
constexpr int A_WARP0 = 6;
constexpr int A_THREADS = 128;
constexpr int NUM_THREADS = (A_WARP0 * 32) + A_THREADS;  // 320
constexpr int A_LAG = STAGES - 1;  // K blocks a gather thread keeps in flight before publishing

constexpr int SMEM_A_OFF = 0;
constexpr int SMEM_B_OFF = SMEM_A_OFF + STAGES * A_STAGE;
constexpr int SMEM_EPI_OFF = SMEM_B_OFF + STAGES * B_STAGE;
constexpr int SMEM_BAR_OFF = SMEM_EPI_OFF + EPI_BUFS * EPI_BUF;
// barriers: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr int SMEM_MISC_OFF = SMEM_BAR_OFF + NUM_BARS * 8;
constexpr int SMEM_USED = SMEM_MISC_OFF + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-B alignment of the base

static_assert(SMEM_BYTES <= 232448, "shared memory budget");

constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

struct Smem {
  uint8_t* base;
  __device__ uint32_t a(int s) const { return smem_u32(base + SMEM_A_OFF + s * A_STAGE); }
  __device__ uint32_t b(int s) const { return smem_u32(base + SMEM_B_OFF + s * B_STAGE); }
  __device__ uint32_t epi(int j) const { return smem_u32(base + SMEM_EPI_OFF + j * EPI_BUF); }
  __device__ uint32_t full(int s) const { return smem_u32(base + SMEM_BAR_OFF + s * 8); }
  __device__ uint32_t empty(int s) const {
    return smem_u32(base + SMEM_BAR_OFF + (STAGES + s) * 8);
  }
  __device__ uint32_t tfull(int j) const {
    return smem_u32(base + SMEM_BAR_OFF + (2 * STAGES + j) * 8);
  }
  __device__ uint32_t tempty(int j) const {
    return smem_u32(base + SMEM_BAR_OFF + (2 * STAGES + 2 + j) * 8);
  }
  __device__ uint32_t drain() const { return smem_u32(base + SMEM_BAR_OFF + (2 * STAGES + 4) * 8); }
  __device__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(base + SMEM_MISC_OFF); }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(base + SMEM_MISC_OFF + 4);
  }
  __device__ volatile int* epi_go() const {
    return reinterpret_cast<volatile int*>(base + SMEM_MISC_OFF + 8);
  }
};

// Bounded wait on an mbarrier phase. Returns false (after recording the timeout) if the wait
// ran out or another role already gave up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Smem& sm,
                                           const GatherGemmParams& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 63u) == 0) {
      if (*sm.abort_flag()) return false;
      if (globaltimer_ns() - t0 > p.timeout_ns) {
        *sm.abort_flag() = 1;
        atomicOr(p.status, MOSAIC_STATUS_TIMEOUT);
        return false;
      }
    }
  }
}

// Wait used while shutting down after an abort: fixed limit, no status side effects.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) break;  // 0.2 s
  }
}

// Hidden row of flat mask position i (0 <= i < M). Sets ok = false for an index outside its
// sequence or outside H; the returned row is then 0 (a safe address) and the output row is
// zero-filled by the epilogue.
__device__ __forceinline__ int32_t resolve_row(const GatherGemmParams& p, int32_t i, bool& ok) {
  const int32_t v = __ldg(p.idx + i);
  if (p.mask_offsets == nullptr) {
    ok = (v >= 0) && (static_cast<int64_t>(v) < p.L_tot);
    return ok ? v : 0;
  }
  // Largest b in [0, B) with mask_offsets[b] <= i (the sequence that owns position i).
  int32_t lo = 0, hi = p.B;
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if (__ldg(p.mask_offsets + mid) <= i) lo = mid; else hi = mid;
  }
  const int64_t s0 = __ldg(p.seq_offsets + lo);
  const int64_t s1 = __ldg(p.seq_offsets + lo + 1);
  const int64_t r = s0 + v;
  ok = (v >= 0) && (s0 >= 0) && (r < s1) && (s1 <= p.L_tot);
  return ok ? static_cast<int32_t>(r) : 0;
}

struct TileCoord {
  int m, n;
};

__device__ __forceinline__ TileCoord tile_coord(int t, const GatherGemmParams& p) {
  const int group_tiles = p.group_m * p.n_tiles;
  const int g = t / group_tiles;
  const int rem = t - g * group_tiles;
  const int m_first = g * p.group_m;
  const int gm = min(p.group_m, p.m_tiles - m_first);
  TileCoord c;
  c.n = rem / gm;
  c.m = m_first + (rem - c.n * gm);
  return c;
}

template <bool OUT_F32>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gather_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_out,
                       const GatherGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm;
  sm.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = p.m_tiles * p.n_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(sm.full(s), 1 + A_THREADS);  // W arrive.expect_tx + every gather thread
      mbar_init(sm.empty(s), 1);  // MMA commit
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(sm.tfull(j), 1);             // MMA commit
      mbar_init(sm.tempty(j), EPI_THREADS);  // every epilogue thread
    }
    mbar_init(sm.drain(), 1);
    *sm.abort_flag() = 0;
    fence_mbar_init();
    // Cross-check of the CSR offsets that the host cannot read: they must run from 0 to M.
    if (blockIdx.x == 0 && p.chunk_index == 0 && p.mask_offsets != nullptr) {
      if (__ldg(p.mask_offsets) != 0 || __ldg(p.mask_offsets + p.B) != p.M_total)
        atomicOr(p.status, MOSAIC_STATUS_INDEX);
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_out);
  }
  if (warp == 1) tmem_alloc<TMEM_COLS>(smem_u32(sm.tmem_slot()));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot();

  if (warp == 0) {
    // ---------------------------------------------------------------- W stream (TMA)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_normal();
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;  // K blocks issued (for the drain after an abort)
      bool alive = true;
      for (int t = blockIdx.x; t < num_tiles && alive; t += gridDim.x) {
        const TileCoord tc = tile_coord(t, p);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(sm.empty(stage), phase ^ 1u, sm, p)) { alive = false; break; }
          mbar_arrive_expect_tx(sm.full(stage), B_STAGE);
          tma_load_2d(sm.b(stage), &tm_w, kb * BK, tc.n * BN, sm.full(stage), pol_w);
          ++issued;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      if (!alive) {
        // Let every W load already issued land before the CTA can exit.
        for (int s = 0; s < STAGES; ++s) {
          const int64_t last = issued - 1 - ((issued - 1 - s) % STAGES + STAGES) % STAGES;
          if (issued > 0 && last >= 0)
            drain_wait(sm.full(s), static_cast<uint32_t>((last / STAGES) & 1));
        }
      }
    }
    __syncwarp();
  } else if (warp >= A_WARP0) {
    // ---------------------------------------------------------------- A gather (cp.async)
    const int at = threadIdx.x - A_WARP0 * 32;  // 0..127
    const int chunk = at & 7;                   // 16-byte piece of a 128-byte row segment
    const int row0 = at >> 3;                   // this thread's rows: row0 + 16 j, j = 0..7
    const uint64_t pol_a = policy_evict_last(); // gathered rows are re-read by every N tile
    const char* hbase = static_cast<const char*>(p.hidden) + chunk * 16;
    const int64_t row_bytes = static_cast<int64_t>(p.d) * 2;
    int64_t it = 0;  // K blocks issued by this thread across all of its tiles
    bool alive = true;
    for (int t = blockIdx.x; t < num_tiles && alive; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, p);
      // Index staging: resolve this thread's 8 rows once per tile. Rows past the chunk and
      // rows with a bad index are zero-filled (src size 0: no global read).
      const char* src[8];
      uint32_t valid = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int r = tc.m * BM + row0 + 16 * j;
        bool ok = false;
        int32_t row = 0;
        if (r < p.rows) row = resolve_row(p, p.row_begin + r, ok);
        src[j] = hbase + static_cast<int64_t>(row) * row_bytes;
        valid |= (ok ? 1u : 0u) << j;
      }
      for (int kb = 0; kb < p.k_blocks; ++kb) {
        // Publish the K block issued A_LAG iterations ago: its copies are complete, make them
        // visible to the tensor cores' (async-proxy) reads, then arrive on its full barrier.
        if (it >= A_LAG) {
          cp_async_wait<A_LAG - 1>();
          fence_proxy_async_smem();
          mbar_arrive(sm.full(static_cast<int>((it - A_LAG) % STAGES)));
        }
        const int stage = static_cast<int>(it % STAGES);
        const uint32_t phase = static_cast<uint32_t>((it / STAGES) & 1);
        if (!wait_phase(sm.empty(stage), phase ^ 1u, sm, p)) { alive = false; break; }
        const bool k_in = kb * BK + chunk * 8 < p.d;  // d % 8 == 0: pieces are all in or out
        const uint32_t a_stage = sm.a(stage);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int r = row0 + 16 * j;
          const uint32_t dst = a_stage + r * 128 + ((chunk ^ (r & 7)) << 4);
          const bool live = k_in && ((valid >> j) & 1u);
          // a zero-filling copy still names an address: keep it at the start of H
          cp_async_16(dst, live ? src[j] + static_cast<int64_t>(kb) * (BK * 2) : hbase,
                      live ? 16u : 0u, pol_a);
        }
        cp_async_commit();
        ++it;
      }
    }
    cp_async_wait<0>();
    if (alive) {
      fence_proxy_async_smem();
      for (int64_t q = (it > A_LAG ? it - A_LAG : 0); q < it; ++q)
        mbar_arrive(sm.full(static_cast<int>(q % STAGES)));
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool alive = true;
      bool issued_any = false;
      for (int t = blockIdx.x; t < num_tiles && alive; t += gridDim.x) {
        if (!wait_phase(sm.tempty(acc), acc_phase ^ 1u, sm, p)) { alive = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!wait_phase(sm.full(stage), phase, sm, p)) { alive = false; break; }
          tc_fence_after();
          const uint64_t a0 = smem_desc_sw128(sm.a(stage));
          const uint64_t b0 = smem_desc_sw128(sm.b(stage));
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            // advance the start address by k * 16 elements * 2 B = 32 B (2 in 16-B units)
            tc_mma_bf16(d_tmem, a0 + 2 * k, b0 + 2 * k, IDESC, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(sm.empty(stage));  // frees the stage once these MMAs have read it
          issued_any = true;
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!alive) break;
        tc_commit(sm.tfull(acc));  // accumulator complete
        if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
      }
      if (!alive && issued_any) {
        tc_commit(sm.drain());  // completes when every MMA issued above has finished
        drain_wait(sm.drain(), 0);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int et = threadIdx.x - EPI_WARP0 * 32;   // 0..127
    const int quad = warp & 3;                     // TMEM lane quadrant this warp may read
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    constexpr int COLS_PER_CHUNK = OUT_F32 ? 32 : 64;  // 128 B of output per row
    constexpr int CHUNKS = BN / COLS_PER_CHUNK;
    int acc = 0;
    uint32_t acc_phase = 0;
    int buf = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      const TileCoord tc = tile_coord(t, p);
      if (et == 0) *sm.epi_go() = wait_phase(sm.tfull(acc), acc_phase, sm, p) ? 1 : 0;
      named_bar_sync(1, EPI_THREADS);
      if (!*sm.epi_go()) break;
      tc_fence_after();
      const int r = tc.m * BM + row_in_tile;
      bool ok = true;
      if (r < p.rows) {
        resolve_row(p, p.row_begin + r, ok);
        if (!ok) atomicOr(p.status, MOSAIC_STATUS_INDEX);
      }
      const uint32_t t_acc = tmem_base + lane_base + static_cast<uint32_t>(acc * BN);
      const int n0 = tc.n * BN;
      for (int c = 0; c < CHUNKS; ++c) {
        uint32_t packed[32];
        if constexpr (OUT_F32) {
          tmem_ld_32x32b_x32(t_acc + c * 32, packed);
          tmem_wait_ld();
          if (!ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j) packed[j] = 0u;
          }
        } else {
          uint32_t v0[32], v1[32];
          tmem_ld_32x32b_x32(t_acc + c * 64, v0);
          tmem_ld_32x32b_x32(t_acc + c * 64 + 32, v1);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            packed[j] = pack_bf16x2(__uint_as_float(v0[2 * j]), __uint_as_float(v0[2 * j + 1]));
            packed[16 + j] =
                pack_bf16x2(__uint_as_float(v1[2 * j]), __uint_as_float(v1[2 * j + 1]));
          }
          if (!ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j) packed[j] = 0u;
          }
        }
        if (c == CHUNKS - 1) {
          // All columns of this accumulator are in registers: hand it back to the MMA warp.
          tc_fence_before();
          mbar_arrive(sm.tempty(acc));
        }
        // The staging buffer is free once the store issued from it two chunks ago has read it.
        if (et == 0) bulk_wait_group_read<EPI_BUFS - 1>();
        named_bar_sync(1, EPI_THREADS);
        const uint32_t dst = sm.epi(buf) + row_in_tile * 128;
        const int sw = row_in_tile & 7;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          st_shared_v4(dst + ((j ^ sw) << 4), packed[4 * j], packed[4 * j + 1], packed[4 * j + 2],
                       packed[4 * j + 3]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, EPI_THREADS);
        if (et == 0) {
          const int x = n0 + c * COLS_PER_CHUNK;
          if (x < p.V) {
            tma_store_2d(&tm_out, sm.epi(buf), x, tc.m * BM);
          }
          bulk_commit_group();
        }
        buf ^= 1;
      }
      if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
    }
    if (et == 0) bulk_wait_group_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<TMEM_COLS>(tmem_base);
}

}  // namespace

int gather_gemm_smem_bytes() { return SMEM_BYTES; }
int gather_gemm_block_m() { return BM; }
int gather_gemm_block_n() { return BN; }
int gather_gemm_block_k() { return BK; }
int gather_gemm_epi_cols(bool out_f32) { return out_f32 ? 32 : 64; }

cudaError_t gather_gemm_prepare(bool out_f32) {
  if (out_f32)
    return cudaFuncSetAttribute(gather_gemm_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  return cudaFuncSetAttribute(gather_gemm_kernel<false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

cudaError_t gather_gemm_launch(const CUtensorMap& tm_w, const CUtensorMap& tm_out,
                               const GatherGemmParams& p, bool out_f32, int grid,
                               cudaStream_t stream) {
  if (out_f32)
    gather_gemm_kernel<true><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(tm_w, tm_out, p);
  else
    gather_gemm_kernel<false><<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(tm_w, tm_out, p);
  return cudaGetLastError();
}

}  // namespace mosaic
