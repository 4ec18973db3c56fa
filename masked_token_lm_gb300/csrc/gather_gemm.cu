// Mask-only logits as one persistent, warp-specialised gather-GEMM kernel for sm_103a.
//
//   out[i, v] = sum_k H[row(i), k] * W[v, k]      (bf16 x bf16 -> fp32 accumulate)
//
// The operation is the "Mask-only Logits Kernel" of "Mosaic: Unlocking Long-Context Inference
// for Diffusion LLMs via Global Memory" (paper review, section 3, core component 1): it reads
// the hidden states of all tokens through the mask indices (indirect addressing), tiles the
// GEMM over the GPU's compute units and keeps the gathered rows on chip, so no gathered [M, d]
// buffer is ever written. The pages' kernel targeted RTX 3090 / A100; this one is designed for
// Blackwell instead.
//
// Roles (per CTA, 512 threads = 4 warpgroups; a warpgroup is 4 consecutive warps):
//   warp 0      W stream: one thread issues the 2-D TMA loads of the W rows of each K block.
//   warp 1      MMA issuer: one thread issues tcgen05.mma into two 256-column TMEM accumulator
//               slots and commits stage releases.
//   warp 2      relay: when a stage's gathered rows have landed, fences them into the async
//               proxy and reports the stage to the (leader's) full barrier.
//   warp 3      idle after the prologue.
//   warps 4..7  A gather: each of the 128 threads resolves 8 of the tile's mask indices to
//               hidden rows (index staging, once per tile) and, per K block, copies one 16-byte
//               piece of each of its 8 rows with cp.async into the 128-byte-swizzled A stage of
//               a 4-deep shared-memory ring (8 threads cover one 128-byte row segment).
//   warps 8..15 epilogue, two warps per TMEM lane quadrant, each half of them taking 128
//               columns of a slot: tcgen05.ld the accumulator into registers (rounded to bf16),
//               hand the slot back, then write 128-byte-swizzled staging tiles and TMA-store
//               them; rows past the chunk are clipped by the store's tensor map.
// The roles are grouped by warpgroup so that the pair kernels with bf16 output or sampling can
// move registers to the epilogue: right after the prologue, warpgroups 0-1 drop to 64 (72 when
// sampling) and warpgroups 2-3 rise to 192 (184) registers per thread (setmaxnreg acts on a
// whole warpgroup, each of whose warps executes the same instruction).
//
// PAIR = true (the normal case): two CTAs of a cluster form a pair that computes a 256 x 512
// unit: per K step two tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16), one per adjacent
// 256-column panel, each into its own TMEM slot, issued by the leader CTA. Each CTA gathers its
// own 128 A rows and loads its own 128-row half of each panel's W rows, so per K block an SM
// takes in 16 KiB of gathered rows and 32 KiB of W for 2 x 2^22 FLOP: 48 bytes per tensor-core
// cycle (a 256 x 256 unit needs 64 and measured ~81 % tensor-pipe busy; this form ~91 %).
// The leader's stage barriers collect the whole pair: its W expect_tx covers the boxes of both
// CTAs (each CTA's cta_group::2 TMA load reports its bytes there), and each CTA's relay reports
// its own gathered rows. Commits multicast to both CTAs. The slots are drained one after the
// other; the MMA issuer starts the next unit's slot-0 MMAs while slot 1 is still being read,
// holding up to 3 stages whose slot-1 MMAs it issues once that slot is free. With bf16 output
// the epilogue reads both slots (64 packed registers per panel and thread) and hands both back
// before it stores either, so slot 1 returns after two slot reads instead of after slot 0's
// stores; the stores then overlap the next unit's MMAs. The sampling epilogue likewise reads a
// whole slot (128 fp32 registers) before its arithmetic. PAIR = false runs 128 x 256 tiles on
// one CTA (problems with a single M tile), alternating the two slots.
//
// The A rows are gathered with cp.async rather than TMA tile::gather4: measured on GB300, the
// 32 gather4 instructions a 128-row K block needs held the kernel to ~26 % of the tensor peak,
// while the same bytes through the load/store units keep the tensor pipe fed.
//
// Units are walked by a static persistent schedule (one M tile per CTA of the pair, one unit
// column of panels): within a group of M units, unit columns outer and M units inner, so each W
// panel is fetched from HBM once per group while the gathered A rows of the group stay in L2.
// A last round that would keep at most half the clusters busy is split into single-panel units.
//
// Every wait is bounded (globaltimer); a wait that runs out records MOSAIC status bit 2, makes
// all roles stop, lets in-flight copies and MMAs finish, frees TMEM and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "gather_gemm.h"
#include "ptx.cuh"

namespace mosaic {

namespace {

constexpr int BM = 128;  // rows of D per CTA
constexpr int BN = 256;  // columns of one accumulator slot (one column panel)
// K block: 64 bf16 = 128-byte rows, stored with the 128-byte swizzle. (32 with the 64-byte
// swizzle and 8 stages computes the same bits but measured 17-24 % slower on GB300: the per-stage
// costs of the producers and the relay no longer fit in a 512-cycle K block.)
constexpr int BK = 64;
constexpr int ROW_BYTES = BK * 2;
constexpr int PIECES = ROW_BYTES / 16;  // 16-byte pieces per row of a K block
constexpr int UMMA_K = 16;
constexpr int A_STAGE = BM * BK * 2;  // 16 KiB
constexpr int EPI_BUF = BM * 128;     // 128 rows x 128 B
constexpr int EPI_BUFS = 2;           // one per epilogue half
constexpr int TMEM_COLS = 2 * BN;     // two accumulator slots
constexpr int STAGES = 4;
constexpr int B_STAGE = 2 * 128 * BK * 2;  // 32 KiB of W rows per stage (both forms)
constexpr int RELAY_WARP = 2;
constexpr int A_WARP0 = 4;            // warpgroup 1
constexpr int A_WARPS = 4;
constexpr int A_THREADS = 32 * A_WARPS;
constexpr int A_ROWS = BM * PIECES / A_THREADS;  // rows per gather thread (PIECES threads per row)
constexpr int EPI_WARP0 = 8;          // warpgroups 2 and 3: two warps per TMEM lane quadrant
constexpr int EPI_THREADS = 256;
constexpr int NUM_THREADS = 512;
// Registers per thread: REGS_LAUNCH at launch (the whole register file for one CTA of 512
// threads); kernels whose epilogue holds both slots then move 64 per thread from the producer
// warpgroups to the epilogue warpgroups.
constexpr int REGS_LAUNCH = 65536 / NUM_THREADS;  // 128
// Producers keep 64 (72 in the sampling kernel, whose gather code needs more to avoid spills);
// the epilogue gets the rest of the pool.
template <bool SAMPLE>
constexpr int kRegsLow = SAMPLE ? 72 : 64;
template <bool SAMPLE>
constexpr int kRegsHigh = 2 * REGS_LAUNCH - kRegsLow<SAMPLE>;
template <bool SAMPLE>
constexpr bool regs_ok() {
  return 2 * 128 * kRegsLow<SAMPLE> + 2 * 128 * kRegsHigh<SAMPLE> <= NUM_THREADS * REGS_LAUNCH &&
         kRegsLow<SAMPLE> % 8 == 0 && kRegsHigh<SAMPLE> % 8 == 0 && kRegsLow<SAMPLE> >= 24 &&
         kRegsHigh<SAMPLE> <= 256;
}
static_assert(regs_ok<false>() && regs_ok<true>(), "register split outside the launch's pool");
// The epilogue holds both slots of a pair unit (and the registers are split) when it writes
// bf16 logits: 2 panels x 128 columns x 2 B per thread fit in 64 + 64 registers. The sampling
// epilogue of a pair takes the split too: it reads a whole slot (128 fp32 registers) before
// handing it back and doing its arithmetic.
template <bool OUT_F32, bool PAIR, bool SAMPLE>
constexpr bool kHoldBoth = PAIR && !SAMPLE && !OUT_F32;
template <bool OUT_F32, bool PAIR, bool SAMPLE>
constexpr bool kRegSplit = PAIR && !OUT_F32;
constexpr int OFFS_CAP = 129;  // CSR offsets staged in shared memory when B + 1 <= OFFS_CAP

template <bool PAIR>
struct Cfg {
  // Panels per unit: a pair computes 256 x 512 (two N = 256 MMAs per K step, one per TMEM slot);
  // a single CTA computes 128 x 256, its two slots double-buffering successive tiles.
  static constexpr int NSUB = PAIR ? 2 : 1;
  static constexpr int B_BOX_ROWS = PAIR ? BN / 2 : BN;  // W rows per CTA per panel (one TMA box)
  static constexpr int B_BOX = B_BOX_ROWS * BK * 2;      // 16 or 32 KiB
  static_assert(NSUB * B_BOX == B_STAGE, "stage layout");
  static constexpr int SMEM_A_OFF = 0;
  static constexpr int SMEM_B_OFF = SMEM_A_OFF + STAGES * A_STAGE;
  static constexpr int SMEM_EPI_OFF = SMEM_B_OFF + STAGES * B_STAGE;
  static constexpr int SMEM_BAR_OFF = SMEM_EPI_OFF + EPI_BUFS * EPI_BUF;
  // full, empty, afull (peer gather -> relay), tfull[2], tempty[2], drain
  static constexpr int NUM_BARS = 3 * STAGES + 5;
  static constexpr int SMEM_MISC_OFF = (SMEM_BAR_OFF + NUM_BARS * 8 + 15) / 16 * 16;
  // misc: tmem slot, abort flag, epilogue go flag, pad; 16-byte relay signal slot
  static constexpr int SMEM_OFFS_OFF = SMEM_MISC_OFF + 32;  // seq_offsets, mask_offsets copies
  static constexpr int SMEM_BYTES = SMEM_OFFS_OFF + 2 * OFFS_CAP * 4 + 1024;  // + alignment slack
  // Arrivals per phase on the (leader's) full barrier: its W expect_tx and its relay's arrive
  // (the local gathered rows have landed and are fenced). The bytes it expects: W of both CTAs
  // and, for a pair, the 16-byte signal with which the peer's relay reports the peer's rows. On
  // the (leader's) tempty barrier: one arrive per CTA.
  static constexpr int FULL_COUNT = 2;
  static constexpr int TEMPTY_COUNT = PAIR ? 2 : 1;
  static constexpr int SIGNAL_BYTES = 16;
  // Bytes the (leader's) full barrier expects per stage of a unit with nsub panels.
  static __device__ __forceinline__ uint32_t w_tx(int nsub) {
    return PAIR ? static_cast<uint32_t>(nsub * 2 * B_BOX + SIGNAL_BYTES) : B_BOX;
  }
  static constexpr uint32_t IDESC = idesc_bf16_f32(PAIR ? 2 * BM : BM, BN);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

template <bool PAIR>
struct Smem {
  using C = Cfg<PAIR>;
  uint8_t* base;
  __device__ uint32_t a(int s) const { return smem_u32(base + C::SMEM_A_OFF + s * A_STAGE); }
  // W rows of panel j (0 .. NSUB-1) of stage s
  __device__ uint32_t b(int s, int j = 0) const {
    return smem_u32(base + C::SMEM_B_OFF + s * B_STAGE + j * C::B_BOX);
  }
  __device__ uint32_t epi(int j) const { return smem_u32(base + C::SMEM_EPI_OFF + j * EPI_BUF); }
  __device__ uint32_t bar(int i) const { return smem_u32(base + C::SMEM_BAR_OFF + i * 8); }
  __device__ uint32_t full(int s) const { return bar(s); }
  __device__ uint32_t empty(int s) const { return bar(STAGES + s); }
  __device__ uint32_t afull(int s) const { return bar(2 * STAGES + s); }
  __device__ uint32_t tfull(int j) const { return bar(3 * STAGES + j); }
  __device__ uint32_t tempty(int j) const { return bar(3 * STAGES + 2 + j); }
  __device__ uint32_t drain() const { return bar(3 * STAGES + 4); }
  __device__ uint32_t* tmem_slot() const {
    return reinterpret_cast<uint32_t*>(base + C::SMEM_MISC_OFF);
  }
  __device__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(base + C::SMEM_MISC_OFF + 4);
  }
  __device__ volatile int* epi_go() const {
    return reinterpret_cast<volatile int*>(base + C::SMEM_MISC_OFF + 8);
  }
  __device__ uint32_t signal_slot() const { return smem_u32(base + C::SMEM_MISC_OFF + 16); }
  __device__ int32_t* seq_offs() const { return reinterpret_cast<int32_t*>(base + C::SMEM_OFFS_OFF); }
  __device__ int32_t* mask_offs() const { return seq_offs() + OFFS_CAP; }
};

// Bounded wait on an mbarrier phase. Returns false (after recording the timeout) if the wait
// ran out or another role of this CTA already gave up. CLUSTER: acquire at cluster scope, for
// barriers the peer CTA arrives on with data to hand over.
template <bool CLUSTER, bool PAIR>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const Smem<PAIR>& sm,
                                           const GatherGemmParams& p) {
  auto probe = [&]() {
    return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (probe()) return true;
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

// Wait used while shutting down: fixed limit, no status side effects.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > 200000000ull) break;  // 0.2 s
  }
}

// CSR offsets as the index staging reads them: from shared memory when the batch is small
// enough to have been staged there at kernel start, else from global memory.
struct Offsets {
  const int32_t* seq;   // [B+1]
  const int32_t* mask;  // [B+1]
};

// Hidden row for flat mask position i (0 <= i < M) whose index value is v = idx[i]. Sets ok =
// false for an index outside its sequence or outside H; the returned row is then 0 (a safe
// address) and the output row is zero-filled.
__device__ __forceinline__ int32_t resolve_row(const GatherGemmParams& p, const Offsets& o,
                                               int32_t i, int32_t v, bool& ok) {
  if (p.mask_offsets == nullptr) {
    ok = (v >= 0) && (static_cast<int64_t>(v) < p.L_tot);
    return ok ? v : 0;
  }
  // Largest b in [0, B) with mask_offsets[b] <= i (the sequence that owns position i).
  int32_t lo = 0, hi = p.B;
  while (hi - lo > 1) {
    const int32_t mid = (lo + hi) >> 1;
    if (o.mask[mid] <= i) lo = mid; else hi = mid;
  }
  const int64_t s0 = o.seq[lo];
  const int64_t s1 = o.seq[lo + 1];
  const int64_t r = s0 + v;
  ok = (v >= 0) && (s0 >= 0) && (r < s1) && (s1 <= p.L_tot);
  return ok ? static_cast<int32_t>(r) : 0;
}

struct TileCoord {
  int m, n;
};

// Whole unit u = (cluster_m consecutive M tiles, one unit column of n_sub panels). Units are
// rastered in groups of group_u M units: unit columns outer, M units inner. CTA `rank` of the
// pair takes M tile mu * cluster_m + rank of the unit; c.n is the unit column.
__device__ __forceinline__ TileCoord unit_coord(int u, int rank, const GatherGemmParams& p) {
  const int group_units = p.group_u * p.n_wide;
  const int g = u / group_units;
  const int rem = u - g * group_units;
  const int mu_first = g * p.group_u;
  const int gm = min(p.group_u, p.m_units - mu_first);
  TileCoord c;
  c.n = rem / gm;
  c.m = (mu_first + (rem - c.n * gm)) * p.cluster_m + rank;
  return c;
}

// What unit u of the schedule computes: M tile m, panels panel0 .. panel0 + nsub - 1. Units at
// or past units_full are the halves of a split unit (one panel each). nsub = 0 for the empty
// half of a unit column that has a single panel (odd n_tiles): every role skips it.
struct Unit {
  int m, panel0, nsub;
};

template <bool PAIR>
__device__ __forceinline__ Unit unit_of(int u, int rank, const GatherGemmParams& p) {
  int base = u, half = 0;
  const bool split = u >= p.units_full;
  if (split) {
    const int h = u - p.units_full;
    base = p.units_full + (h >> 1);
    half = h & 1;
  }
  const TileCoord c = unit_coord(base, rank, p);
  Unit t;
  t.m = c.m;
  t.panel0 = c.n * Cfg<PAIR>::NSUB + half;
  t.nsub = min(split ? 1 : Cfg<PAIR>::NSUB, max(p.n_tiles - t.panel0, 0));
  return t;
}

// Greedy-sampling fold of 64 fp32 logits v[off .. off + 63], the columns n0 + c0 + j of this
// thread's row half (only those with c0 + j < valid count, unless the block lies inside V): the
// running maximum m, its first column a and the sum s of exp(x - m), rescaled when the maximum
// grows. exp(x - m) = 2^(x log2(e) - m log2(e)): one FMA and one ex2 per column.
constexpr float SAMPLE_LOG2E = 1.4426950408889634f;
template <int N>
__device__ __forceinline__ void sample_fold64(const uint32_t (&v)[N], int off, int c0, int valid,
                                              int n0, float& m, float& s, int& a) {
  const bool inside = valid >= c0 + 64;
  float bm = -INFINITY;
#pragma unroll
  for (int j = 0; j < 64; ++j)
    if (inside || c0 + j < valid) bm = fmaxf(bm, __uint_as_float(v[off + j]));
  if (bm > m) {  // a new maximum: its first column, and the sum rescaled to it
    int ba = 0;
#pragma unroll
    for (int j = 63; j >= 0; --j)
      if (__uint_as_float(v[off + j]) == bm && (inside || c0 + j < valid)) ba = j;
    s *= ex2_approx((m - bm) * SAMPLE_LOG2E);
    m = bm;
    a = n0 + c0 + ba;
  }
  const float mL = m * SAMPLE_LOG2E;
#pragma unroll
  for (int j = 0; j < 64; ++j)
    if (inside || c0 + j < valid)
      s += ex2_approx(fmaf(__uint_as_float(v[off + j]), SAMPLE_LOG2E, -mL));
}

// Merge the other row half's (m1, s1, a1) into this half's (m, s, a). This half's columns come
// first, so an equal maximum keeps its index.
__device__ __forceinline__ void sample_merge(float& m, float& s, int& a, float m1, float s1,
                                             int a1) {
  if (m1 > m) {
    s = s * ex2_approx((m - m1) * SAMPLE_LOG2E) + s1;
    m = m1;
    a = a1;
  } else if (s1 > 0.0f) {
    s += s1 * ex2_approx((m1 - m) * SAMPLE_LOG2E);
  }
}

// FP8: E4M3 operands (per-row scales applied in the epilogue): a K block is then 128 elements of
// the same 128-byte rows, and the MMA is kind::f8f6f4 (K = 32 per instruction, 4 per K block).
template <bool OUT_F32, bool PAIR, bool SAMPLE, bool FP8 = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gather_gemm_kernel(const __grid_constant__ CUtensorMap tm_w,
                       const __grid_constant__ CUtensorMap tm_out,
                       const GatherGemmParams p) {
  using C = Cfg<PAIR>;
  static_assert(!(FP8 && SAMPLE), "the sampling epilogue takes bf16 operands");
  constexpr int BKE = FP8 ? ROW_BYTES : BK;   // elements per K block
  constexpr int EPP = FP8 ? 16 : 8;           // elements per 16-byte piece
  constexpr uint32_t IDESC = FP8 ? idesc_e4m3_f32(PAIR ? 2 * BM : BM, BN) : C::IDESC;
  constexpr bool HOLD = kHoldBoth<OUT_F32, PAIR, SAMPLE>;
  constexpr bool SPLIT = kRegSplit<OUT_F32, PAIR, SAMPLE>;
  extern __shared__ uint8_t smem_raw[];
  Smem<PAIR> sm;
  sm.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;
  const int unit0 = static_cast<int>(blockIdx.x) / p.cluster_m;
  const int unit_stride = static_cast<int>(gridDim.x) / p.cluster_m;
  const int num_units = p.units_total;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(sm.full(s), C::FULL_COUNT);  // used in the leader (or the single CTA)
      mbar_init(sm.empty(s), 1);             // MMA commit (multicast to both CTAs of a pair)
      mbar_init(sm.afull(s), A_THREADS);     // gather threads (hardware arrive on landing)
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(sm.tfull(j), 1);                 // MMA commit
      mbar_init(sm.tempty(j), C::TEMPTY_COUNT);  // epilogue (of both CTAs of a pair)
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
  // Index staging, part 1: small CSR batches keep their offsets in shared memory.
  const bool offs_in_smem = p.mask_offsets != nullptr && p.B + 1 <= OFFS_CAP;
  if (offs_in_smem) {
    for (int i = threadIdx.x; i <= p.B; i += NUM_THREADS) {
      sm.seq_offs()[i] = __ldg(p.seq_offsets + i);
      sm.mask_offs()[i] = __ldg(p.mask_offsets + i);
    }
  }
  if (warp == 1) tmem_alloc<TMEM_COLS, PAIR>(smem_u32(sm.tmem_slot()));
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The peer arrives on this CTA's barriers: wait until both CTAs have initialised theirs.
  if (PAIR) cluster_sync();
  const uint32_t tmem_base = *sm.tmem_slot();
  const Offsets offs = offs_in_smem ? Offsets{sm.seq_offs(), sm.mask_offs()}
                                    : Offsets{p.seq_offsets, p.mask_offsets};
  // Barriers that both CTAs of a pair report to live in the leader.
  auto full_c = [&](int s) { return PAIR ? mapa_shared(sm.full(s), 0) : sm.full(s); };
  auto tempty_c = [&](int j) { return PAIR ? mapa_shared(sm.tempty(j), 0) : sm.tempty(j); };

  if (warp < EPI_WARP0) {
    // Producer warpgroups 0 and 1: every warp executes this one instruction, then the
    // roles split.
    if constexpr (SPLIT) setmaxnreg_dec<kRegsLow<SAMPLE>>();
    if (warp == 0) {
      // ---------------------------------------------------------------- W stream (TMA)
      if (lane == 0) {
        const uint64_t pol_w = policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0;
        for (int u = unit0; u < num_units; u += unit_stride) {
          const Unit t = unit_of<PAIR>(u, rank, p);
          if (t.nsub == 0) continue;
          bool alive = true;
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!wait_phase<false>(sm.empty(stage), phase ^ 1u, sm, p)) { alive = false; break; }
            if constexpr (PAIR) {
              // Per panel, this CTA loads its 128-row half of the panel's 256 W rows. The leader
              // expects the halves of both CTAs; each load lands in its own CTA's shared memory
              // and reports its bytes to the leader's barrier.
              if (leader) mbar_arrive_expect_tx(sm.full(stage), C::w_tx(t.nsub));
              for (int j = 0; j < t.nsub; ++j)
                tma_load_2d_pair(sm.b(stage, j), &tm_w, kb * BKE,
                                 (t.panel0 + j) * BN + rank * C::B_BOX_ROWS, full_c(stage), pol_w);
            } else {
              mbar_arrive_expect_tx(sm.full(stage), C::w_tx(1));
              tma_load_2d(sm.b(stage), &tm_w, kb * BKE, t.panel0 * BN, sm.full(stage), pol_w);
            }
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          if (!alive) break;
        }
      }
      __syncwarp();
    } else if (warp >= A_WARP0 && warp < A_WARP0 + A_WARPS) {
      // ---------------------------------------------------------------- A gather (cp.async)
      // The gather warps' instruction stream is on the critical path (they issue every copy of
      // the gathered rows), so the per-K-block work is kept to the copies themselves: addresses
      // advance by a constant, destinations and byte counts are fixed per tile.
      const int at = threadIdx.x - A_WARP0 * 32;    // 0 .. A_THREADS-1
      const int chunk = at % PIECES;                // 16-byte piece of a row segment
      const int row0 = at / PIECES;                 // rows row0 + ROW_STEP * j
      constexpr int ROW_STEP = A_THREADS / PIECES;
      const uint64_t pol_a = policy_evict_last();   // gathered rows are re-read by every N tile
      const char* hbase = static_cast<const char*>(p.hidden) + chunk * 16;
      const int64_t row_bytes = static_cast<int64_t>(p.d) * (FP8 ? 1 : 2);
      const int k_full = p.d / BKE;                 // K blocks with every piece inside d
      const bool tail_in = chunk * EPP < p.d % BKE; // this piece in the partial last K block
      // The swizzle of TMA and of the MMA descriptors: the piece index (address bits 4..) is
      // XORed with address bits 7.. of the row start (64-byte rows: (row / 2) % 4; 128: row % 8).
      uint32_t dst_off[A_ROWS];
#pragma unroll
      for (int j = 0; j < A_ROWS; ++j) {
        const int r = row0 + ROW_STEP * j;
        dst_off[j] = r * ROW_BYTES + ((chunk ^ ((r * ROW_BYTES >> 7) & (PIECES - 1))) << 4);
      }
      int stage = 0;
      uint32_t phase = 0;
      bool alive = true;
      // Index staging, part 2: the mask indices of a tile are loaded one tile ahead (they land
      // while the previous tile's K loop runs) and resolved to rows at the tile's start.
      int32_t vnext[A_ROWS];
      auto load_idx = [&](int u, int32_t (&v)[A_ROWS]) {
        const Unit t = unit_of<PAIR>(u, rank, p);
#pragma unroll
        for (int j = 0; j < A_ROWS; ++j) {
          const int r = t.m * BM + row0 + ROW_STEP * j;
          v[j] = r < p.rows ? __ldg(p.idx + p.row_begin + r) : 0;
        }
      };
      if (unit0 < num_units) load_idx(unit0, vnext);
      for (int u = unit0; u < num_units && alive; u += unit_stride) {
        const Unit tc = unit_of<PAIR>(u, rank, p);
        int32_t v[A_ROWS];
#pragma unroll
        for (int j = 0; j < A_ROWS; ++j) v[j] = vnext[j];
        if (u + unit_stride < num_units) load_idx(u + unit_stride, vnext);
        if (tc.nsub == 0) continue;
        // Rows past the chunk and rows with a bad index are zero-filled: 0 source bytes (no read)
        // from row 0 of H, an address that stays inside H for every full K block.
        const char* src[A_ROWS];
        uint32_t bytes[A_ROWS];
#pragma unroll
        for (int j = 0; j < A_ROWS; ++j) {
          const int r = tc.m * BM + row0 + ROW_STEP * j;
          bool ok = false;
          int32_t row = 0;
          if (r < p.rows) row = resolve_row(p, offs, p.row_begin + r, v[j], ok);
          src[j] = hbase + static_cast<int64_t>(row) * row_bytes;
          bytes[j] = ok ? 16u : 0u;
        }
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          int go = 1;
          if (lane == 0) go = wait_phase<false>(sm.empty(stage), phase ^ 1u, sm, p) ? 1 : 0;
          go = __shfl_sync(0xffffffffu, go, 0);
          if (!go) { alive = false; break; }
          const uint32_t a_stage = sm.a(stage);
          if (kb < k_full) {
#pragma unroll
            for (int j = 0; j < A_ROWS; ++j) cp_async_16(a_stage + dst_off[j], src[j], bytes[j], pol_a);
          } else {  // partial last K block: pieces past d are zero-filled, named at the start of H
#pragma unroll
            for (int j = 0; j < A_ROWS; ++j)
              cp_async_16(a_stage + dst_off[j], tail_in ? src[j] : hbase, tail_in ? bytes[j] : 0u, pol_a);
          }
#pragma unroll
          for (int j = 0; j < A_ROWS; ++j) src[j] += BK * 2;
          // Publish without waiting: the arrive on afull happens when these copies have landed;
          // the relay then fences them into the async proxy for the tensor cores.
          cp_async_arrive_noinc(sm.afull(stage));
          if (++stage == STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      cp_async_wait<0>();
    } else if (warp == RELAY_WARP) {
      // ---------------------------------------------------------------- relay
      if (lane == 0) {
        // Once a stage's gathered rows have landed (every gather thread's hardware arrive on
        // afull), fence them into the async proxy and report the stage: in the leader (or a single
        // CTA) by a local arrive on full; in the peer of a pair through the async proxy, with a
        // 16-byte shared-to-shared bulk copy whose complete_tx lands on the leader's full barrier
        // (a cluster-scope release arrive instead cost ~0.8 us per K block). Keeping the fence
        // here keeps it off the MMA issuer, the kernel's critical thread.
        const uint32_t dst = PAIR ? mapa_shared(sm.signal_slot(), 0) : 0;
        int stage = 0;
        uint32_t phase = 0;
        bool alive = true;
        for (int u = unit0; u < num_units && alive; u += unit_stride) {
          if (unit_of<PAIR>(u, rank, p).nsub == 0) continue;
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!wait_phase<false>(sm.afull(stage), phase, sm, p)) { alive = false; break; }
            fence_proxy_async_smem();
            if (leader) mbar_arrive(sm.full(stage));
            else bulk_copy_s2s_cluster(dst, sm.signal_slot(), C::SIGNAL_BYTES, full_c(stage));
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
        }
      }
      __syncwarp();
    } else if (warp == 1) {
      // ---------------------------------------------------------------- MMA issuer
      if (lane == 0 && leader) {
        int stage = 0;
        uint32_t phase = 0;
        uint32_t tphase = 0;  // bit j: parity of the current use of accumulator slot j
        int slot_next = 0;    // single CTA: tiles alternate between the two slots
        bool alive = true;
        bool issued_any = false;
        // The 4 MMAs of one K block of panel j (W rows b(st, j)) into accumulator slot `slot`.
        auto mma_kblock = [&](int st, int kb, int slot, int j) {
          const uint64_t a0 = smem_desc_kmajor<ROW_BYTES>(sm.a(st));
          const uint64_t b0 = smem_desc_kmajor<ROW_BYTES>(sm.b(st, j));
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(slot * BN);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            // advance the start address by k * 16 elements * 2 B = 32 B (2 in 16-B units)
            if constexpr (FP8)
              tc_mma_e4m3<PAIR>(d_tmem, a0 + 2 * k, b0 + 2 * k, IDESC, (kb | k) != 0 ? 1u : 0u);
            else
              tc_mma_bf16<PAIR>(d_tmem, a0 + 2 * k, b0 + 2 * k, IDESC, (kb | k) != 0 ? 1u : 0u);
          }
        };
        for (int u = unit0; u < num_units && alive; u += unit_stride) {
          const Unit t = unit_of<PAIR>(u, rank, p);
          if (t.nsub == 0) continue;
          const int s0 = PAIR ? 0 : slot_next;
          if (!PAIR) slot_next ^= 1;
          if (!wait_phase<PAIR>(sm.tempty(s0), ((tphase >> s0) & 1u) ^ 1u, sm, p)) { alive = false; break; }
          tc_fence_after();
          // Two panels (pair): slot 1 may still be draining the previous unit's second panel. The
          // slot-0 MMAs run ahead meanwhile, holding up to STAGES - 1 stages whose slot-1 MMAs are
          // issued (oldest first) as soon as the slot is free.
          const uint32_t s1_parity = ((tphase >> 1) & 1u) ^ 1u;
          bool s1_free = t.nsub < 2;
          int held = 0;
          auto flush_held = [&](int kb_end) {
            int hs = stage - held;
            if (hs < 0) hs += STAGES;
            for (int i = 0; i < held; ++i) {
              mma_kblock(hs, kb_end - held + i, 1, 1);
              tc_commit<PAIR>(sm.empty(hs));  // frees the stage once these MMAs have read it
              if (++hs == STAGES) hs = 0;
            }
            held = 0;
          };
          for (int kb = 0; kb < p.k_blocks; ++kb) {
            if (!wait_phase<PAIR>(sm.full(stage), phase, sm, p)) { alive = false; break; }
            tc_fence_after();
            mma_kblock(stage, kb, s0, 0);
            issued_any = true;
            if (!s1_free) {
              if (held < STAGES - 1 && !mbar_test_wait_cluster(sm.tempty(1), s1_parity)) {
                ++held;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                continue;
              }
              if (!wait_phase<PAIR>(sm.tempty(1), s1_parity, sm, p)) { alive = false; break; }
              tc_fence_after();
              s1_free = true;
              flush_held(kb);
            }
            if (t.nsub == 2) mma_kblock(stage, kb, 1, 1);
            tc_commit<PAIR>(sm.empty(stage));
            if (++stage == STAGES) { stage = 0; phase ^= 1u; }
          }
          if (!alive) break;
          tc_commit<PAIR>(sm.tfull(s0));  // slot s0 complete
          if (t.nsub == 2) {
            if (!s1_free) {  // fewer K blocks than the stages the slot-0 MMAs may run ahead
              if (!wait_phase<PAIR>(sm.tempty(1), s1_parity, sm, p)) { alive = false; break; }
              tc_fence_after();
              flush_held(p.k_blocks);
            }
            tc_commit<PAIR>(sm.tfull(1));
          }
          tphase ^= (1u << s0) | (t.nsub == 2 ? 2u : 0u);
        }
        if (issued_any) {
          // Completes when every MMA issued above (and the arrives it triggers) has finished.
          tc_commit_local<PAIR>(sm.drain());
          drain_wait(sm.drain(), 0);
        }
      }
      __syncwarp();
    }
  } else {
    if constexpr (SPLIT) setmaxnreg_inc<kRegsHigh<SAMPLE>>();  // epilogue warpgroups 2 and 3
    // ---------------------------------------------------------------- epilogue
    // Two warps per TMEM lane quadrant: warp w may read lanes 32 * (w % 4) .. + 31, and the
    // warps of half h = 0 / 1 take columns h * 128 .. + 127 of the accumulator slot. Each half
    // stages its output through its own 128-byte-swizzled buffer and TMA-stores it.
    const int et = threadIdx.x - EPI_WARP0 * 32;   // 0 .. EPI_THREADS-1
    const int half = et / (EPI_THREADS / 2);
    const int gt = et % (EPI_THREADS / 2);         // thread within the half
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const uint32_t stage_buf = sm.epi(half);
    const uint32_t bar_half = 2 + half;           // named barrier of this half's 128 threads
    uint32_t tphase = 0;  // bit j: parity of the current use of accumulator slot j
    int slot_next = 0;    // single CTA: tiles alternate between the two slots
    bool go = true;
    // One 128-byte row segment of this thread's output row into the half's staging buffer, then
    // one TMA store of the buffer (rows past the chunk are clipped by the tensor map).
    auto stage_store = [&](const uint32_t (&w)[32], int x, int m_tile) {
      if (gt == 0) bulk_wait_group_read<0>();  // the buffer's previous store has read it
      __syncwarp();  // the named barriers are warp-aligned: reconverge after the one-lane wait
      named_bar_sync(bar_half, EPI_THREADS / 2);
      const uint32_t dst = stage_buf + row_in_tile * 128;
      const int sw = row_in_tile & 7;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        st_shared_v4(dst + ((j ^ sw) << 4), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
      fence_proxy_async_smem();
      named_bar_sync(bar_half, EPI_THREADS / 2);
      if (gt == 0) {
        if (x < p.V && m_tile < p.m_tiles) tma_store_2d(&tm_out, stage_buf, x, m_tile * BM);
        bulk_commit_group();
      }
    };
    // One epilogue thread waits (bounded) until accumulator slot `slot` holds a finished panel
    // and tells the others through shared memory; false when the wait ran out.
    auto acquire_slot = [&](int slot) -> bool {
      if (et == 0)
        *sm.epi_go() = wait_phase<false>(sm.tfull(slot), (tphase >> slot) & 1u, sm, p) ? 1 : 0;
      __syncwarp();  // lane 0 of this warp waited alone; the barrier below is warp-aligned
      named_bar_sync(1, EPI_THREADS);
      if (!*sm.epi_go()) return false;
      tc_fence_after();
      tphase ^= 1u << slot;
      return true;
    };
    // All TMEM reads of the slot are done in every epilogue thread: hand it back to the MMA issuer.
    auto release_slot = [&](int slot) {
      tc_fence_before();
      named_bar_sync(1, EPI_THREADS);
      if (et == 0) {
        if (PAIR) mbar_arrive_cluster(tempty_c(slot)); else mbar_arrive(sm.tempty(slot));
      }
    };
    for (int u = unit0; u < num_units && go; u += unit_stride) {
      const Unit tc = unit_of<PAIR>(u, rank, p);
      if (tc.nsub == 0) continue;
      // The row this thread stores is the same for every panel of the unit.
      const int r = tc.m * BM + row_in_tile;
      bool ok = true;
      float sa = 0.0f;  // FP8: scale of this output row's hidden row
      if (r < p.rows) {
        const int32_t hr = resolve_row(p, offs, p.row_begin + r, __ldg(p.idx + p.row_begin + r), ok);
        if (!ok && half == 0) atomicOr(p.status, MOSAIC_STATUS_INDEX);
        if constexpr (FP8) sa = __ldg(p.a_scale + hr);
      }
      // FP8: the 4 column scales from column c (a multiple of 4; V % 8 == 0, so a group of 4 is
      // either inside V or past it), times the row's scale.
      auto col_scales = [&](int c, float* s4) {
        const float4 w = c < p.V ? __ldg(reinterpret_cast<const float4*>(p.b_scale + c))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        s4[0] = sa * w.x; s4[1] = sa * w.y; s4[2] = sa * w.z; s4[3] = sa * w.w;
      };
      // FP8 with bf16 out: W's column scales from column c0, applied to 64 rounded, packed
      // values (a second bf16 rounding).
      auto scale_cols = [&](uint32_t (&w32)[32], int c0) {
#pragma unroll
        for (int g = 0; g < 16; ++g) {
          const int c = c0 + 4 * g;
          const float4 w = c < p.V ? __ldg(reinterpret_cast<const float4*>(p.b_scale + c))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
          uint32_t& a = w32[2 * g];
          uint32_t& b = w32[2 * g + 1];
          a = pack_bf16x2(__uint_as_float(a << 16) * w.x, __uint_as_float(a & 0xffff0000u) * w.y);
          b = pack_bf16x2(__uint_as_float(b << 16) * w.z, __uint_as_float(b & 0xffff0000u) * w.w);
        }
      };
      if constexpr (SAMPLE && PAIR) {
        // Sampling epilogue of a pair: per panel, this row's maximum, its first column and the
        // sum of exp(x - max) over the half's valid columns, from the fp32 accumulators. Each
        // slot is read whole (128 registers) and handed back before its arithmetic; the two
        // halves of the row are merged for both panels at the end of the unit, through shared
        // memory.
        const int col_h = half * (BN / 2);  // first slot column of this half
        float pm[2], ps[2];
        int pa[2];
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {
          if (jp < tc.nsub && go) {
            if (!acquire_slot(jp)) {
              go = false;
            } else {
              const uint32_t t_acc = tmem_base + lane_base + static_cast<uint32_t>(jp * BN + col_h);
              uint32_t v[128];
#pragma unroll
              for (int q = 0; q < 8; ++q)
                tmem_ld_32x32b_x16(t_acc + q * 16, *reinterpret_cast<uint32_t(*)[16]>(v + q * 16));
              tmem_wait_ld();
              release_slot(jp);
              const int n0 = tc.panel0 * BN + jp * BN + col_h;  // first output column of this half
              const int valid = p.V - n0;  // columns of this half inside V (all when >= 128)
              float m = -INFINITY, sum = 0.0f;
              int a = 0;
              sample_fold64(v, 0, 0, valid, n0, m, sum, a);
              sample_fold64(v, 64, 64, valid, n0, m, sum, a);
              pm[jp] = m;
              ps[jp] = sum;
              pa[jp] = a;
            }
          }
        }
        if (!go) break;
        float* xm = reinterpret_cast<float*>(sm.base + Cfg<PAIR>::SMEM_EPI_OFF);  // [2][BM]
        float* xs = xm + 2 * BM;
        int* xa = reinterpret_cast<int*>(xs + 2 * BM);
        if (half == 1) {
#pragma unroll
          for (int jp = 0; jp < 2; ++jp) {
            if (jp < tc.nsub) {
              xm[jp * BM + row_in_tile] = pm[jp];
              xs[jp * BM + row_in_tile] = ps[jp];
              xa[jp * BM + row_in_tile] = pa[jp];
            }
          }
        }
        named_bar_sync(1, EPI_THREADS);  // the exchange above before the reads below
        if (half == 0) {
#pragma unroll
          for (int jp = 0; jp < 2; ++jp) {
            if (jp < tc.nsub) {
              float m = pm[jp], sum = ps[jp];
              int a = pa[jp];
              sample_merge(m, sum, a, xm[jp * BM + row_in_tile], xs[jp * BM + row_in_tile],
                           xa[jp * BM + row_in_tile]);
              if (r < p.rows && tc.m < p.m_tiles) {
                const int64_t o = static_cast<int64_t>(r) * p.part_ld + tc.panel0 + jp;
                p.part_max[o] = m;
                p.part_sum[o] = sum;
                p.part_arg[o] = ok ? a : -1;
              }
            }
          }
        }
      } else if constexpr (HOLD) {
        // bf16 out, CTA pair: both panels of the unit are read out of TMEM (rounded and packed,
        // 64 registers per panel) and both slots handed back before any store, so the MMA
        // issuer gets slot 1 back two slot reads after the unit's last MMA; the four stores
        // below then overlap the next unit's MMAs. 8-column TMEM loads keep the live registers
        // within the epilogue's share (192).
        uint32_t pk[2][2][32];
        const int col_h = half * (BN / 2);  // first slot column of this half
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {
          if (jp < tc.nsub && go) {
            if (!acquire_slot(jp)) {
              go = false;
            } else {
              const uint32_t t_acc = tmem_base + lane_base + static_cast<uint32_t>(jp * BN + col_h);
#pragma unroll
              for (int q = 0; q < 16; ++q) {
                uint32_t v[8];
                tmem_ld_32x32b_x8(t_acc + q * 8, v);
                tmem_wait_ld();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  if constexpr (FP8)  // the row's scale here; the columns' at the store
                    pk[jp][q >> 3][(q & 7) * 4 + j] = pack_bf16x2(__uint_as_float(v[2 * j]) * sa,
                                                                  __uint_as_float(v[2 * j + 1]) * sa);
                  else
                    pk[jp][q >> 3][(q & 7) * 4 + j] =
                        pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                }
              }
              release_slot(jp);
            }
          }
        }
        if (!go) break;
#pragma unroll
        for (int jp = 0; jp < 2; ++jp) {
          if (jp < tc.nsub) {
            if (!ok) {
#pragma unroll
              for (int j = 0; j < 32; ++j) { pk[jp][0][j] = 0u; pk[jp][1][j] = 0u; }
            }
            const int n0 = tc.panel0 * BN + jp * BN + col_h;  // first output column of this half
            if constexpr (FP8) scale_cols(pk[jp][0], n0);
            stage_store(pk[jp][0], n0, tc.m);
            if constexpr (FP8) scale_cols(pk[jp][1], n0 + 64);
            stage_store(pk[jp][1], n0 + 64, tc.m);
          }
        }
      } else {
        for (int jp = 0; jp < tc.nsub; ++jp) {
          // Panel jp of the unit sits in slot jp (pair) or in the tile's slot (single CTA).
          const int slot = PAIR ? jp : slot_next;
          if (!PAIR) slot_next ^= 1;
          if (!acquire_slot(slot)) { go = false; break; }
          const int col_h = half * (BN / 2);  // first slot column of this half
          const uint32_t t_acc = tmem_base + lane_base + static_cast<uint32_t>(slot * BN + col_h);
          const int n0 = tc.panel0 * BN + jp * BN + col_h;  // first output column of this half
          if constexpr (SAMPLE) {
            // Sampling epilogue of a single CTA: this row's maximum, its first column and the sum
            // of exp(x - max) over the half's valid columns (fp32 logits straight from TMEM), in
            // two blocks of 64 columns; the slot is handed back right after the second block's
            // TMEM read, before its arithmetic. The two halves of the row are then merged through
            // shared memory.
            float m = -INFINITY, s = 0.0f;
            int a = 0;
            const int valid = p.V - n0;  // columns of this half inside V (all when >= 128)
            uint32_t v[64];
            auto load64 = [&](int c0) {
#pragma unroll
              for (int q = 0; q < 4; ++q)
                tmem_ld_32x32b_x16(t_acc + c0 + q * 16, *reinterpret_cast<uint32_t(*)[16]>(v + q * 16));
              tmem_wait_ld();
            };
            load64(0);
            sample_fold64(v, 0, 0, valid, n0, m, s, a);
            load64(64);
            release_slot(slot);
            sample_fold64(v, 0, 64, valid, n0, m, s, a);
            float* xm = reinterpret_cast<float*>(sm.base + Cfg<PAIR>::SMEM_EPI_OFF);
            float* xs = xm + BM;
            int* xa = reinterpret_cast<int*>(xs + BM);
            if (half == 1) { xm[row_in_tile] = m; xs[row_in_tile] = s; xa[row_in_tile] = a; }
            named_bar_sync(1, EPI_THREADS);  // the exchange above before the reads below
            if (half == 0) {
              sample_merge(m, s, a, xm[row_in_tile], xs[row_in_tile], xa[row_in_tile]);
              if (r < p.rows && tc.m < p.m_tiles) {
                const int64_t o = static_cast<int64_t>(r) * p.part_ld + tc.panel0 + jp;
                p.part_max[o] = m;
                p.part_sum[o] = s;
                p.part_arg[o] = ok ? a : -1;
              }
            }
          } else if constexpr (OUT_F32) {
            // fp32 out: 4 chunks of 32 columns (128 B per row), the slot released after the last load
            for (int c = 0; c < BN / 2 / 32; ++c) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(t_acc + c * 32, v);
              tmem_wait_ld();
              if constexpr (FP8) {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                  float s4[4];
                  col_scales(n0 + c * 32 + 4 * g, s4);
#pragma unroll
                  for (int e = 0; e < 4; ++e)
                    v[4 * g + e] = __float_as_uint(__uint_as_float(v[4 * g + e]) * s4[e]);
                }
              }
              if (!ok) {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0u;
              }
              if (c == BN / 2 / 32 - 1) release_slot(slot);
              stage_store(v, n0 + c * 32, tc.m);
            }
          } else {
            // bf16 out: the half's 128 columns go to registers (rounded and packed) before any
            // store, so the slot is handed back after 4 TMEM loads rather than after the stores.
            uint32_t packed[2][32];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              uint32_t v[16];
              tmem_ld_32x32b_x16(t_acc + q * 16, v);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                if constexpr (FP8)  // the row's scale here; the columns' after the slot is free
                  packed[q >> 2][(q & 3) * 8 + j] = pack_bf16x2(__uint_as_float(v[2 * j]) * sa,
                                                                __uint_as_float(v[2 * j + 1]) * sa);
                else
                  packed[q >> 2][(q & 3) * 8 + j] =
                      pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
              }
            }
            release_slot(slot);
            if (!ok) {
#pragma unroll
              for (int j = 0; j < 32; ++j) { packed[0][j] = 0u; packed[1][j] = 0u; }
            }
            if constexpr (FP8) scale_cols(packed[0], n0);
            stage_store(packed[0], n0, tc.m);
            if constexpr (FP8) scale_cols(packed[1], n0 + 64);
            stage_store(packed[1], n0 + 64, tc.m);
          }
        }  // panels of the unit
      }
    }
    if (gt == 0) bulk_wait_group_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  const bool aborted = *sm.abort_flag() != 0;
  // No CTA leaves (or frees TMEM the leader's MMAs write) while its peer still works.
  if (PAIR) cluster_sync();
  if (aborted) {  // loads issued just before giving up: let them land before the CTA exits
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 100000ull) {
    }
  }
  tc_fence_after();
  if (warp == 1) tmem_dealloc<TMEM_COLS, PAIR>(tmem_base);
}

template <bool F32, bool PAIR>
cudaLaunchConfig_t launch_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = Cfg<PAIR>::SMEM_BYTES;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = PAIR ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <bool F32, bool PAIR, bool SAMPLE = false, bool FP8 = false>
cudaError_t prepare_one(int* clusters) {
  cudaError_t e = cudaFuncSetAttribute(gather_gemm_kernel<F32, PAIR, SAMPLE, FP8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Cfg<PAIR>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if constexpr (kRegSplit<F32, PAIR, SAMPLE>) {
    // The register split assumes exactly REGS_LAUNCH registers per thread at launch: with
    // fewer, the epilogue's increase would wait for registers that never come free. Refuse.
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, gather_gemm_kernel<F32, PAIR, SAMPLE, FP8>);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != REGS_LAUNCH || fa.maxThreadsPerBlock < NUM_THREADS)
      return cudaErrorInvalidConfiguration;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config<F32, PAIR>((PAIR ? 2 : 1) * 64, nullptr, attr);
  return cudaOccupancyMaxActiveClusters(clusters, gather_gemm_kernel<F32, PAIR, SAMPLE, FP8>,
                                        &cfg);
}

template <bool F32, bool PAIR, bool SAMPLE = false, bool FP8 = false>
cudaError_t launch_one(const CUtensorMap& tm_w, const CUtensorMap& tm_out,
                       const GatherGemmParams& p, int grid, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = launch_config<F32, PAIR>(grid, stream, attr);
  return cudaLaunchKernelEx(&cfg, gather_gemm_kernel<F32, PAIR, SAMPLE, FP8>, tm_w, tm_out, p);
}

// One warp per row: lane l combines the row's partials of N tiles l, l + 32, ... (partials are
// stored row by row, so the warp's reads are contiguous), then the warp combines the lanes. The
// maximum goes to the smallest column among equal values (columns of different tiles are
// disjoint and ordered like the tiles), so ties go to the smallest v; the order of the sums is
// fixed, so results do not depend on chunking or timing.
__global__ void sample_reduce_kernel(const GatherGemmParams p, int32_t* token, float* confidence) {
  const int lane = threadIdx.x & 31;
  const int r = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
  if (r >= p.rows) return;  // whole warps leave together
  const float* pm = p.part_max + static_cast<int64_t>(r) * p.part_ld;
  const float* ps = p.part_sum + static_cast<int64_t>(r) * p.part_ld;
  const int32_t* pa = p.part_arg + static_cast<int64_t>(r) * p.part_ld;
  float m = -INFINITY;
  int a = 0x7fffffff;
  bool bad = false;
  for (int n = lane; n < p.n_tiles; n += 32) {
    const float x = pm[n];
    const int g = pa[n];
    bad |= g < 0;
    if (x > m || (x == m && g < a)) { m = x; a = g; }
  }
  for (int off = 16; off > 0; off >>= 1) {
    const float xo = __shfl_xor_sync(0xffffffffu, m, off);
    const int go = __shfl_xor_sync(0xffffffffu, a, off);
    if (xo > m || (xo == m && go < a)) { m = xo; a = go; }
  }
  bad = __any_sync(0xffffffffu, bad);
  float s = 0.0f;
  for (int n = lane; n < p.n_tiles; n += 32) s += ps[n] * expf(pm[n] - m);
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) {
    token[p.row_begin + r] = bad ? -1 : a;
    confidence[p.row_begin + r] = bad ? 0.0f : 1.0f / s;
  }
}

}  // namespace

int gather_gemm_block_m() { return BM; }
int gather_gemm_block_n() { return BN; }
int gather_gemm_block_k() { return BK; }
int gather_gemm_block_k_fp8() { return ROW_BYTES; }
int gather_gemm_epi_cols(bool out_f32) { return out_f32 ? 32 : 64; }
int gather_gemm_w_box_rows(bool pair) {
  return pair ? Cfg<true>::B_BOX_ROWS : Cfg<false>::B_BOX_ROWS;
}

int gather_gemm_schedule(GatherGemmParams& p, int max_clusters) {
  const int nsub = p.cluster_m == 2 ? Cfg<true>::NSUB : Cfg<false>::NSUB;
  p.n_wide = (p.n_tiles + nsub - 1) / nsub;
  const int64_t units = static_cast<int64_t>(p.m_units) * p.n_wide;
  p.units_full = p.units_total = static_cast<int32_t>(units);
  const int64_t P = max_clusters > 0 ? max_clusters : 1;
  if (nsub > 1) {
    // A last round that keeps at most half of the clusters busy is run as twice as many
    // single-panel units instead, so that every cluster shares it.
    const int64_t rounds = (units + P - 1) / P;
    const int64_t last = units - (rounds - 1) * P;
    if (units > 0 && 2 * last <= P) {
      p.units_full = static_cast<int32_t>((rounds - 1) * P);
      p.units_total = static_cast<int32_t>(p.units_full + 2 * last);
    }
  }
  const int64_t clusters = p.units_total < P ? p.units_total : P;
  return static_cast<int>(clusters * p.cluster_m);
}

cudaError_t gather_gemm_prepare_sample(bool pair, int* clusters) {
  return pair ? prepare_one<false, true, true>(clusters) : prepare_one<false, false, true>(clusters);
}

cudaError_t gather_gemm_launch_sample(const CUtensorMap& tm_w, const GatherGemmParams& p, int grid,
                                      cudaStream_t stream) {
  // the sampling epilogue stores no logits: tm_w stands in for the unused output map
  return p.cluster_m == 2 ? launch_one<false, true, true>(tm_w, tm_w, p, grid, stream)
                          : launch_one<false, false, true>(tm_w, tm_w, p, grid, stream);
}

cudaError_t sample_reduce_launch(const GatherGemmParams& p, int32_t* token, float* confidence,
                                 cudaStream_t stream) {
  const int threads = 256;  // 8 rows per block
  const int blocks = (p.rows + threads / 32 - 1) / (threads / 32);
  sample_reduce_kernel<<<blocks, threads, 0, stream>>>(p, token, confidence);
  return cudaGetLastError();
}

cudaError_t gather_gemm_prepare_fp8(bool out_f32, bool pair, int* clusters) {
  if (out_f32)
    return pair ? prepare_one<true, true, false, true>(clusters)
                : prepare_one<true, false, false, true>(clusters);
  return pair ? prepare_one<false, true, false, true>(clusters)
              : prepare_one<false, false, false, true>(clusters);
}

cudaError_t gather_gemm_launch_fp8(const CUtensorMap& tm_w, const CUtensorMap& tm_out,
                                   const GatherGemmParams& p, bool out_f32, int grid,
                                   cudaStream_t stream) {
  const bool pair = p.cluster_m == 2;
  if (out_f32)
    return pair ? launch_one<true, true, false, true>(tm_w, tm_out, p, grid, stream)
                : launch_one<true, false, false, true>(tm_w, tm_out, p, grid, stream);
  return pair ? launch_one<false, true, false, true>(tm_w, tm_out, p, grid, stream)
              : launch_one<false, false, false, true>(tm_w, tm_out, p, grid, stream);
}

cudaError_t gather_gemm_prepare(bool out_f32, bool pair, int* clusters) {
  if (out_f32) return pair ? prepare_one<true, true>(clusters) : prepare_one<true, false>(clusters);
  return pair ? prepare_one<false, true>(clusters) : prepare_one<false, false>(clusters);
}

cudaError_t gather_gemm_launch(const CUtensorMap& tm_w, const CUtensorMap& tm_out,
                               const GatherGemmParams& p, bool out_f32, int grid,
                               cudaStream_t stream) {
  const bool pair = p.cluster_m == 2;
  if (out_f32)
    return pair ? launch_one<true, true>(tm_w, tm_out, p, grid, stream)
                : launch_one<true, false>(tm_w, tm_out, p, grid, stream);
  return pair ? launch_one<false, true>(tm_w, tm_out, p, grid, stream)
              : launch_one<false, false>(tm_w, tm_out, p, grid, stream);
}

}  // namespace mosaic
