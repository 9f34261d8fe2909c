// dllm_lmhead.cu -- the LM head fused with the statistics pass (sm_103a).
//
// mlx-arsenal "dLLM block decoding" (the statistics of the logits) and
// mojo-dllm manual, "The GPU path": the LM head's output rows are only ever
// consumed by the row statistics, so the logits z = h W^T need not reach
// HBM.  logits tile = hidden tile (128 tokens x d) x weight tile (bn ids x
// d)^T on the 5th-generation tensor cores: TMA brings 64-wide K slabs of both
// into a shared-memory ring of up to 16 stages filling the CTA's shared memory
// (128-byte swizzle), one thread issues
// tcgen05.mma (kind::f16, bf16 in, fp32 accumulate) into one of two TMEM
// accumulators (128 lanes x 256 columns each, bn of them used), and two
// warpgroups of epilogue warps read each finished accumulator back with
// tcgen05.ld -- thread i of warp w holds token 32 (w % 4) + i, warpgroup g the
// tile's 32-column chunks c = g (mod 2) -- and fold the logits into that
// token's running statistics (max, sum 2^y, sum 2^y y, first argmax, best
// Gumbel score), the same state the statistics kernels keep.  CTA c owns a
// contiguous range of vocabulary tiles for every token tile; a finish kernel
// combines the per-token partials (one per CTA and warpgroup) and writes x0,
// prob and entropy.
//
// Waits are bounded (a clock64 deadline of about a second, then a fault code
// in the workspace), the TMEM allocation is released before every exit, and
// the optional fp32 logits output exists for validation.
#include <cuda.h>  // CUtensorMap and its enums (types only; the encoder comes from the driver at run time)
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/dllmcommit.h"
#include "dllm_stats_kernels.cuh"

namespace dllm {

constexpr int kLhBM = 128;                       // tokens per tile (the MMA's M)
constexpr int kLhMaxBN = 256;                    // vocabulary ids per tile (the MMA's N), chosen per call
constexpr int kLhBK = 64;                        // K per stage: one 128-byte swizzle row of bf16
constexpr int kLhUK = 16;                        // K of one tcgen05.mma.kind::f16
constexpr int kLhMaxStages = 16;
constexpr int kLhATile = kLhBM * kLhBK * 2;      // 16 KB: a full 128-row hidden tile
constexpr int kLhEpiGroups = 2;                  // epilogue warpgroups: group g reads the chunks c = g (mod 2)
constexpr int kLhEpiWarps = 4 * kLhEpiGroups;    // warp w reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31
// Warp w issues on scheduler w % 4; the warps of the tile's first 32 tokens
// (0 and 4) are the busiest when there are few tokens, so the TMA and MMA
// warps sit on schedulers 2 and 3 (warps 8 and 9 have no role).
constexpr int kLhTmaWarp = kLhEpiWarps + 2;
constexpr int kLhMmaWarp = kLhEpiWarps + 3;
constexpr int kLhThreads = (kLhEpiWarps + 4) * 32;
constexpr int kLhTmemCols = 2 * kLhMaxBN;        // two accumulators, at columns 0 and 256
// Dynamic shared memory: the ring, plus 1 KB to align it, plus slack for the
// MMA's reads of a hidden tile's unused rows past the last stage (a full
// tile less the rows the box brings).  kLhSmem is the most a CTA may ask for
// (227 KB less the static barriers).
constexpr int kLhSmem = 227 * 1024 - 1024;

// Instruction descriptor of tcgen05.mma.kind::f16: fp32 accumulator
// (bits 4-5 = 1), bf16 A and B (bits 7-9, 10-12 = 1), both K-major (bits 15,
// 16 = 0), N / 8 in bits 17-22, M / 16 in bits 24-28.
constexpr uint32_t lh_idesc(int bn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(bn >> 3) << 17) |
         (static_cast<uint32_t>(kLhBM >> 4) << 24);
}

struct LmHeadParams {
  CUtensorMap tm_h;        // hidden (T, d) bf16, box 64 x a_rows, 128-byte swizzle
  CUtensorMap tm_w;        // weight (V, d) bf16, box 64 x bn, 128-byte swizzle
  int64_t T, V, d;
  int32_t n_k;             // d / 64
  int32_t n_t;             // token tiles
  int32_t n_v;             // vocabulary tiles
  int32_t P;               // CTAs
  int32_t a_rows;          // hidden rows one TMA box brings: min(128, T rounded up to 8)
  int32_t a_bytes;         // their share of a stage, rounded up to 1024 bytes (the swizzle atom)
  int32_t bn;              // vocabulary ids per tile: a multiple of 16 in [64, 256]
  int32_t b_bytes;         // bn 128 bytes (a multiple of 1024)
  uint32_t idesc;          // lh_idesc(bn)
  int32_t slabs;           // 64-wide K slabs per stage (1 or 2): a stage reads that many consecutive
                           // 128-byte pieces of every weight row together
  int32_t stages;          // ring stages of slabs (a_bytes + b_bytes)
  float temperature;
  PhiloxSchedule keys;
  int32_t n_sup;
  int32_t sup[DLLM_MAX_SUPPRESS];
  Partial* partials;       // (n_t * 128, kLhEpiGroups P): token-major, one per CTA and epilogue group
  float* logits;           // (T, V) fp32 or nullptr
  int64_t logits_stride;
  int32_t* fault;
};

// Shared-memory matrix descriptor of a K-major tile with 128-byte rows in
// the 128-byte swizzle (what TMA writes with CU_TENSOR_MAP_SWIZZLE_128B):
// start address / 16 in bits 0-13, the leading byte offset (not used by this
// layout) 16 B, the stride byte offset between 8-row groups 1024 B in bits
// 32-45, descriptor version 1 in bits 46-47, swizzle mode 2 (128 B) in bits
// 61-63.  Within the 128-byte row, the k-th 16-element slice starts 32 k
// bytes further.
__device__ __forceinline__ uint64_t lh_desc(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ void lh_tma_load(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void lh_mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void lh_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void lh_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void lh_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread).
__device__ __forceinline__ void lh_tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// A bounded wait: false after the deadline or once the CTA aborted.
__device__ __forceinline__ bool lh_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

__device__ __forceinline__ void lh_fail(const LmHeadParams& p, volatile int32_t* abort_flag, int32_t code) {
  if (!*abort_flag) {
    atomicExch(p.fault, code);
    *abort_flag = 1;
  }
}

// Per-token running statistics of one epilogue thread (raw logits).
struct LhAcc {
  float m, Z, S2;
  int32_t idx;
  float best_s, best_z;
  int32_t best_v;
};

template <bool GUMBEL>
__global__ void __launch_bounds__(kLhThreads, 1) lm_head_kernel(const __grid_constant__ LmHeadParams p) {
  extern __shared__ __align__(1024) uint8_t lh_smem[];
  __shared__ __align__(8) uint64_t full_bar[kLhMaxStages], empty_bar[kLhMaxStages], accf_bar[2], acce_bar[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int32_t abort_flag_s;
  __shared__ int32_t sup_s[DLLM_MAX_SUPPRESS];  // the suppressed ids (parameter-space reads with a
                                                // run-time index are slow)
  volatile int32_t* abort_flag = &abort_flag_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t ring = (smem_addr(lh_smem) + 1023u) & ~1023u;
  const int vt0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.n_v / p.P);
  const int vt1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.n_v / p.P);
  const int nvt = vt1 - vt0;
  const int n_my = nvt * p.n_t;  // tiles in order: token tile outer, vocabulary tile inner

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&accf_bar[b]), 1);
      mbar_init(smem_addr(&acce_bar[b]), kLhEpiWarps);
    }
    abort_flag_s = 0;
    fence_mbar_init();
  }
  for (int q = threadIdx.x; q < p.n_sup; q += blockDim.x) sup_s[q] = p.sup[q];
  if (warp == kLhMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                 "r"(kLhTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  lh_fence_before();
  __syncthreads();
  lh_fence_after();
  const uint32_t tmem = tmem_slot;
  if (warp != kLhTmaWarp) pdl_wait();  // (the TMA warp waits once it has requested the first weight slabs)
  pdl_launch_dependents();

  if (warp == kLhTmaWarp) {
    if (lane == 0) {
      // Stage q holds K slabs (q mod per_tile) p.slabs .. of this CTA's tile q / per_tile.
      const int per_tile = p.n_k / p.slabs;
      const int total = n_my * per_tile;
      const int pre = total < p.stages ? total : p.stages;
      const uint32_t stage_bytes = static_cast<uint32_t>(p.slabs * (p.a_bytes + p.b_bytes));
      const uint32_t tx = static_cast<uint32_t>(p.slabs * (p.a_rows * kLhBK * 2 + p.b_bytes));
      auto load = [&](int q, int s, bool hidden, bool weight) {
        const int i = q / per_tile, k = (q % per_tile) * p.slabs;
        const int tt = i / nvt, vt = vt0 + i % nvt;
        const uint32_t bar = smem_addr(&full_bar[s]);
        for (int j = 0; j < p.slabs; ++j) {
          const uint32_t sub = ring + static_cast<uint32_t>(s) * stage_bytes + static_cast<uint32_t>(j * (p.a_bytes + p.b_bytes));
          if (hidden) lh_tma_load(sub, &p.tm_h, (k + j) * kLhBK, tt * kLhBM, bar);
          if (weight) lh_tma_load(sub + static_cast<uint32_t>(p.a_bytes), &p.tm_w, (k + j) * kLhBK, vt * p.bn, bar);
        }
      };
      // The weight is not written by the preceding kernel in the stream, so
      // the first stages' weight slabs are requested before the grid
      // dependency resolves (the ring fills while the previous call
      // finishes); their hidden slabs only after it.
      for (int q = 0; q < pre; ++q) {
        mbar_arrive_expect_tx(smem_addr(&full_bar[q]), tx);
        load(q, q, false, true);
      }
      pdl_wait();
      for (int q = 0; q < pre; ++q) load(q, q, true, false);
      int s = pre == p.stages ? 0 : pre;
      uint32_t ph = pre == p.stages ? 1u : 0u;
      for (int q = pre; q < total && !*abort_flag; ++q) {
        if (!lh_wait(smem_addr(&empty_bar[s]), ph ^ 1u, abort_flag)) {
          lh_fail(p, abort_flag, kFaultEmptyWait);
          break;
        }
        mbar_arrive_expect_tx(smem_addr(&full_bar[s]), tx);
        load(q, s, true, true);
        if (++s == p.stages) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == kLhMmaWarp) {
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      for (int i = 0; i < n_my && !*abort_flag; ++i) {
        const int buf = i & 1;
        const uint32_t aph = static_cast<uint32_t>((i >> 1) & 1);
        if (!lh_wait(smem_addr(&acce_bar[buf]), aph ^ 1u, abort_flag)) {
          lh_fail(p, abort_flag, kFaultEmptyWait);
          break;
        }
        lh_fence_after();
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(buf * kLhMaxBN);
        for (int k = 0; k < p.n_k; k += p.slabs) {
          if (!lh_wait(smem_addr(&full_bar[s]), ph, abort_flag)) {
            lh_fail(p, abort_flag, kFaultFullWait);
            break;
          }
          lh_fence_after();
          for (int j = 0; j < p.slabs; ++j) {
            const uint32_t a = ring + static_cast<uint32_t>((s * p.slabs + j) * (p.a_bytes + p.b_bytes));
            const uint32_t b = a + static_cast<uint32_t>(p.a_bytes);
#pragma unroll
            for (int kk = 0; kk < kLhBK / kLhUK; ++kk)
              lh_mma(d_tmem, lh_desc(a + kk * 32), lh_desc(b + kk * 32), p.idesc, (k + j) != 0 || kk != 0 ? 1u : 0u);
          }
          lh_commit(smem_addr(&empty_bar[s]));  // the stage is free once these MMAs have read it
          if (++s == p.stages) {
            s = 0;
            ph ^= 1u;
          }
        }
        lh_commit(smem_addr(&accf_bar[buf]));  // the accumulator is complete
      }
    }
  } else if (warp < kLhEpiWarps) {
    // Epilogue: thread (warp, lane) owns token row 32 (warp % 4) + lane of the
    // tile, and the tile's 32-column chunks c = warp / 4 (mod kLhEpiGroups).
    const int ew = warp & 3, half = warp >> 2;
    const float t = p.temperature;
    const float t_ln2 = t * kLn2;
    LhAcc acc;
    for (int i = 0; i < n_my; ++i) {
      const int tt = i / nvt, vt = vt0 + i % nvt;
      const int buf = i & 1;
      const uint32_t aph = static_cast<uint32_t>((i >> 1) & 1);
      if (vt == vt0) {
        acc.m = kMInit;
        acc.Z = 0.0f;
        acc.S2 = 0.0f;
        acc.idx = 0x7FFFFFFF;
        acc.best_s = kNegInf;
        acc.best_z = 0.0f;
        acc.best_v = 0x7FFFFFFF;
      }
      // warp-uniform: the TMEM loads below are .sync.aligned
      const bool ok = __all_sync(0xFFFFFFFFu, lh_wait(smem_addr(&accf_bar[buf]), aph, abort_flag));
      if (!ok) {
        if (lane == 0) lh_fail(p, abort_flag, kFaultFullWait);
        break;
      }
      lh_fence_after();
      const int64_t token = static_cast<int64_t>(tt) * kLhBM + ew * 32 + lane;
      const uint64_t row_lo_hi = static_cast<uint64_t>(token);
      // A warp whose 32 TMEM lanes hold no token (a tile of fewer than 128
      // tokens) only hands the accumulator back; chunks past V are skipped.
      const int64_t ids = std::min<int64_t>(p.bn, p.V - static_cast<int64_t>(vt) * p.bn);
      const int n_chunks = token - lane < p.T ? static_cast<int>((ids + 31) / 32) : 0;
#pragma unroll 1
      for (int c = half; c < n_chunks; c += kLhEpiGroups) {
        uint32_t r[32];
        // (the last chunk of a tile may reach past bn: those columns are in
        // the 256-column slot but hold no id of this tile, and are masked)
        lh_tmem_ld32(tmem + (static_cast<uint32_t>(ew * 32) << 16) + static_cast<uint32_t>(buf * kLhMaxBN + c * 32), r);
        const int64_t v0 = static_cast<int64_t>(vt) * p.bn + c * 32;
        const int64_t vend = std::min<int64_t>(p.V, static_cast<int64_t>(vt + 1) * p.bn);
        const int lim = static_cast<int>(std::min<int64_t>(32, vend - v0));  // columns holding ids (1 .. 32)
        if (p.logits && token < p.T) {
          float* out = p.logits + token * p.logits_stride + v0;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < lim) out[j] = __uint_as_float(r[j]);
        }
        // Columns with no id (past the tile or V) or a suppressed id, as bits.
        uint32_t absent = lim >= 32 ? 0u : ~((1u << lim) - 1u);
        for (int q = 0; q < p.n_sup; ++q) {
          const int64_t off = sup_s[q] - v0;
          if (off >= 0 && off < 32) absent |= 1u << off;
        }
        // Every index below is a compile-time constant, so z stays in registers.
        float z[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) z[j] = fminf(fmaxf(__uint_as_float(r[j]), kSentinel), kTopClamp);  // NaN -> -2^100
        if (absent != 0u) {  // warp-uniform and rare: a tile's last chunk, or a suppressed id
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if ((absent >> j) & 1u) z[j] = kAbsent;
        }
        float cm[4] = {kMInit, kMInit, kMInit, kMInit};
#pragma unroll
        for (int j = 0; j < 32; ++j) cm[j & 3] = fmaxf(cm[j & 3], z[j]);
        const float cmax = fmaxf(fmaxf(cm[0], cm[1]), fmaxf(cm[2], cm[3]));
        if (cmax > acc.m) {  // rescale to the new running max (shift between exponent references)
          const float d = ref_shift(exp_ref(acc.m), exp_ref(cmax));
          const float f = ex2_approx(d);
          acc.S2 = f * fmaf(d, acc.Z, acc.S2);
          acc.Z *= f;
          acc.m = cmax;
          uint32_t eq = 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) eq |= (z[j] == cmax ? 1u : 0u) << j;
          acc.idx = static_cast<int32_t>(v0 + (__ffs(eq) - 1));  // strictly larger than every earlier value
        }
        // The chunk's sums in packed pairs on two independent chains, then
        // added to the row's: y = z log2 e - ref, ref = RU(m log2 e), sum 2^y,
        // sum 2^y y.
        {
          const float nmc = -exp_ref(acc.m);
          const uint64_t nmc2 = pack2(nmc, nmc), l2e2 = pack2(kLog2e, kLog2e);
          uint64_t Za = 0, Sa = 0, Zb = 0, Sb = 0;
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            acc_pair2<false>(Za, Sa, z[j], z[j + 1], nmc2, l2e2, 0);
            acc_pair2<false>(Zb, Sb, z[j + 2], z[j + 3], nmc2, l2e2, 0);
          }
          float z0, z1, s0, s1;
          unpack2(add2(Za, Zb), z0, z1);
          unpack2(add2(Sa, Sb), s0, s1);
          acc.Z += z0 + z1;
          acc.S2 += s0 + s1;
        }
        if (GUMBEL) {
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint4 o = philox4x32_10(static_cast<uint32_t>((v0 >> 2) + g), static_cast<uint32_t>(row_lo_hi),
                                          static_cast<uint32_t>(row_lo_hi >> 32), 0u, p.keys);
            const uint32_t w4[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = 4 * g + e;
              // g = -ln(-ln u) <= -ln(1 - u): the exact score is evaluated only
              // where this bound (with a margin for the rounding of lg2.approx
              // and the fmaf) reaches the best score so far.
              const float w1 = __fsub_rn(1.0f, uniform_from_bits(w4[e]));
              const float bound = fmaf(t_ln2, -lg2_approx(w1), z[j] + fmaf(fabsf(z[j]), 1e-6f, 1e-3f));
              if (z[j] <= kAbsent || bound < acc.best_s) continue;
              const float sc = gumbel_score(z[j], t, w4[e]);
              if (sc > acc.best_s) {
                acc.best_s = sc;
                acc.best_v = static_cast<int32_t>(v0 + j);
                acc.best_z = z[j];
              }
            }
          }
        }
      }
      lh_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&acce_bar[buf]));
      if (vt == vt1 - 1 && token < p.T) {
        Partial q;
        q.m = acc.m;
        q.Z = acc.Z;
        q.S2 = acc.S2;
        q.idx = acc.idx;
        q.best_s = acc.best_s;
        q.best_z = acc.best_z;
        q.best_v = acc.best_v;
        q.m2 = kMInit;
        store_partial(p.partials + token * (kLhEpiGroups * p.P) + kLhEpiGroups * blockIdx.x + half, q);
      }
    }
  }
  // Every MMA has completed (the epilogue waited for each accumulator) or the
  // CTA aborted; release the TMEM.
  lh_fence_before();
  __syncthreads();
  if (warp == kLhMmaWarp) {
    lh_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kLhTmemCols) : "memory");
  }
}

// One warp per token: combine the CTAs' partials, finish the row.
template <bool GUMBEL>
__global__ void __launch_bounds__(256) lm_head_finish_kernel(const __grid_constant__ StatsParams sp, int32_t P,
                                                              const Partial* __restrict__ partials) {
  constexpr int MODE = GUMBEL ? kModeSample : 0;
  pdl_wait();
  pdl_launch_dependents();
  const int64_t token = blockIdx.x * static_cast<int64_t>(8) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= sp.T) return;
  Partial tot = empty_partial();
  for (int k = lane; k < P; k += 32) part_combine<MODE>(tot, load_partial(partials + token * P + k), 1.0f);
  tot = warp_combine<MODE>(tot, 1.0f);
  if (lane == 0) finish_row(sp, token, row_out<MODE>(sp, tot), RowPre());
}

}  // namespace dllm

namespace {

using namespace dllm;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// A 2-D bf16 tensor map of rows x cols (cols contiguous) with a box of
// box_rows x 64 columns in the 128-byte swizzle; rows past the end read as 0.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t stride_elems, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride_elems) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kLhBK), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct LhDevice {
  int sms = 0;
  cudaError_t err = cudaSuccess;
};
LhDevice g_lh[64];
std::once_flag g_lh_once[64];

const LhDevice* lh_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::call_once(g_lh_once[dev], [dev]() {
    LhDevice& d = g_lh[dev];
    d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    for (const void* k : {reinterpret_cast<const void*>(&lm_head_kernel<false>),
                          reinterpret_cast<const void*>(&lm_head_kernel<true>)})
      if (d.err == cudaSuccess) d.err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kLhSmem);
    if (d.err != cudaSuccess) (void)cudaGetLastError();  // report through the status, leave no sticky error
  });
  return g_lh[dev].err == cudaSuccess ? &g_lh[dev] : nullptr;
}

// The tile width: the multiple of 16 in [64, 256] that minimises the ids the
// busiest CTA handles, ceil(ceil(V / bn) / P) bn with P = min(SMs, tiles);
// ties go to the wider tile.
int32_t lh_tile_width(int64_t sms, int64_t V) {
  int32_t best = kLhMaxBN;
  int64_t best_cost = INT64_MAX;
  for (int32_t bn = kLhMaxBN; bn >= 64; bn -= 16) {
    const int64_t tiles = (V + bn - 1) / bn;
    const int64_t P = std::min<int64_t>(sms, tiles);
    const int64_t cost = (tiles + P - 1) / P * bn;
    if (cost < best_cost) {
      best_cost = cost;
      best = bn;
    }
  }
  return best;
}

dllm_status lh_launch(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, kernel, args) == cudaSuccess ? DLLM_OK : DLLM_ERR_CUDA;
}

}  // namespace

extern "C" {

size_t dllm_lm_head_stats_workspace_size(int64_t T, int64_t V, int64_t d) {
  (void)d;
  if (T <= 0 || V <= 0) return 256;
  const LhDevice* dev = lh_device();
  const int64_t sms = dev ? dev->sms : 1024;
  const int64_t P = std::min<int64_t>(sms, (V + 63) / 64);   // the most CTAs any tile width uses
  const int64_t n_t = (T + kLhBM - 1) / kLhBM;
  return 256 + static_cast<size_t>(n_t * kLhBM * P * kLhEpiGroups) * sizeof(Partial);
}

dllm_status dllm_lm_head_stats(const void* hidden, int64_t T, int64_t d, int64_t hidden_stride, const void* weight,
                               int64_t V, int64_t weight_stride, float temperature, uint64_t key,
                               const int32_t* suppress_ids, int32_t n_suppress, int32_t* x0, float* prob,
                               float* entropy, float* logits, int64_t logits_stride, void* workspace,
                               size_t workspace_bytes, dllm_stream_t stream) {
  if (T < 0 || V < 1 || V > INT32_MAX || d < 1) return DLLM_ERR_INVALID_ARGUMENT;
  if (!(temperature >= 0.0f) || !(temperature <= 0x1p+64f)) return DLLM_ERR_INVALID_ARGUMENT;
  if (hidden_stride < d || weight_stride < d || (logits && logits_stride < V)) return DLLM_ERR_INVALID_ARGUMENT;
  if (n_suppress < 0 || (n_suppress > 0 && !suppress_ids)) return DLLM_ERR_INVALID_ARGUMENT;
  if (n_suppress > DLLM_MAX_SUPPRESS) return DLLM_ERR_UNSUPPORTED;
  std::vector<int32_t> sup(suppress_ids, suppress_ids + n_suppress);
  for (int32_t id : sup)
    if (id < 0 || id >= V) return DLLM_ERR_INVALID_ARGUMENT;
  std::sort(sup.begin(), sup.end());
  sup.erase(std::unique(sup.begin(), sup.end()), sup.end());
  if (static_cast<int64_t>(sup.size()) >= V) return DLLM_ERR_INVALID_ARGUMENT;
  if (T == 0) return DLLM_OK;
  if (!hidden || !weight || !x0 || !prob || !entropy) return DLLM_ERR_INVALID_ARGUMENT;
  // TMA: 16-byte aligned bases and row strides; K in whole 64-wide slabs.
  // A hidden box covers only the rows that exist (a tile of fewer than 128
  // tokens leaves the rest of the A tile stale in shared memory: the MMA's
  // output rows past T are garbage and never read; each row depends only on
  // its own A row).
  if (d % kLhBK != 0 || (reinterpret_cast<uintptr_t>(hidden) & 15u) || (reinterpret_cast<uintptr_t>(weight) & 15u) ||
      (hidden_stride * 2) % 16 != 0 || (weight_stride * 2) % 16 != 0 || T > (static_cast<int64_t>(1) << 31))
    return DLLM_ERR_UNSUPPORTED;
  const LhDevice* dev = lh_device();
  if (!dev) return DLLM_ERR_CUDA;
  const int32_t bn = lh_tile_width(dev->sms, V);
  const int64_t P = std::min<int64_t>(dev->sms, (V + bn - 1) / bn);
  const int64_t n_t = (T + kLhBM - 1) / kLhBM;
  const size_t need = 256 + static_cast<size_t>(n_t * kLhBM * P * kLhEpiGroups) * sizeof(Partial);
  if (!workspace || workspace_bytes < need) return DLLM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return DLLM_ERR_INVALID_ARGUMENT;

  LmHeadParams p;
  std::memset(&p, 0, sizeof(p));
  const int32_t a_rows = T >= kLhBM ? kLhBM : static_cast<int32_t>((T + 7) / 8 * 8);
  if (!make_map(&p.tm_h, hidden, T, d, hidden_stride, static_cast<uint32_t>(a_rows)) ||
      !make_map(&p.tm_w, weight, V, d, weight_stride, static_cast<uint32_t>(bn)))
    return DLLM_ERR_CUDA;
  p.a_rows = a_rows;
  p.a_bytes = (a_rows * kLhBK * 2 + 1023) / 1024 * 1024;
  p.bn = bn;
  p.b_bytes = bn * kLhBK * 2;
  p.idesc = lh_idesc(bn);

  p.T = T;
  p.V = V;
  p.d = d;
  p.n_k = static_cast<int32_t>(d / kLhBK);
  p.slabs = 1;  // two measured no faster on GB300 (the limit is the bytes in flight, not DRAM locality)
  const int32_t slack = kLhATile - p.a_bytes + 1024;
  p.stages = std::min(kLhMaxStages, (kLhSmem - slack) / (p.slabs * (p.a_bytes + p.b_bytes)));
  const size_t smem = static_cast<size_t>(p.stages) * p.slabs * (p.a_bytes + p.b_bytes) + slack;
  p.n_t = static_cast<int32_t>(n_t);
  p.n_v = static_cast<int32_t>((V + bn - 1) / bn);
  p.P = static_cast<int32_t>(P);
  p.temperature = temperature;
  uint32_t k0 = static_cast<uint32_t>(key), k1 = static_cast<uint32_t>(key >> 32);
  for (int r = 0; r < 10; ++r) {
    p.keys.k[r][0] = k0;
    p.keys.k[r][1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  p.n_sup = static_cast<int32_t>(sup.size());
  for (size_t i = 0; i < sup.size(); ++i) p.sup[i] = sup[i];
  uint8_t* w = static_cast<uint8_t*>(workspace);
  p.fault = reinterpret_cast<int32_t*>(w);
  p.partials = reinterpret_cast<Partial*>(w + 256);
  p.logits = logits;
  p.logits_stride = logits_stride;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool gumbel = temperature > 0.0f;
  void* args[] = {&p};
  dllm_status st = lh_launch(gumbel ? reinterpret_cast<const void*>(&lm_head_kernel<true>)
                                    : reinterpret_cast<const void*>(&lm_head_kernel<false>),
                             dim3(static_cast<unsigned>(P)), dim3(kLhThreads), smem, s, args);
  if (st != DLLM_OK) return st;

  StatsParams sp;
  std::memset(&sp, 0, sizeof(sp));
  sp.T = T;
  sp.V = V;
  sp.L = T;
  sp.scale = 1.0f;
  sp.ln_veff = static_cast<float>(std::log(static_cast<double>(V - static_cast<int64_t>(sup.size()))));
  sp.x0 = x0;
  sp.prob = prob;
  sp.entropy = entropy;
  sp.fault = p.fault;
  int32_t P32 = p.P * kLhEpiGroups;  // partials per token
  const Partial* parts = p.partials;
  void* fargs[] = {&sp, &P32, &parts};
  return lh_launch(gumbel ? reinterpret_cast<const void*>(&lm_head_finish_kernel<true>)
                          : reinterpret_cast<const void*>(&lm_head_finish_kernel<false>),
                   dim3(static_cast<unsigned>((T + 7) / 8)), dim3(256), 0, s, fargs);
}

}  // extern "C"
