// dllm_stats.cu -- the statistics pass (and the fused commit step) on sm_103a.
//
// What it computes (mlx-arsenal "dLLM block decoding", "What mlx-arsenal
// ships": token_stats; mojo-dllm manual, "Row statistics on the device"): for
// every logit row, the proposal x0 (first argmax, or Gumbel-max), its
// probability and the entropy of the softmax over the non-suppressed ids.
//
// How (one pass over HBM, persistent grid):
//   * The T rows are cut into units of chunk_vec 16-byte vectors; the U units
//     are dealt to the P CTAs in contiguous, equal ranges, so every CTA reads
//     the same number of bytes whatever the shape (few long rows or many).
//   * In each CTA one producer thread streams its units into a shared-memory
//     ring with cp.async.bulk (TMA bulk copies), one mbarrier per stage; eight
//     consumer warps read each unit from shared memory.
//   * Each consumer thread keeps an online softmax state: running max m,
//     Z = sum 2^y and S2 = sum 2^y y with y = (z - m) log2 e (packed fp32x2
//     accumulators), rescaled when the max grows; entropy = ln Z - S2 ln 2 / Z.
//     The first index of the max is located only when the max grows.
//   * Gumbel-max: one Philox4x32-10 call per four ids; a bound on the noise
//     from the largest uniform of each 16-byte vector lets most vectors skip
//     the two logarithms; the warp shares its best score to tighten the bound.
//   * A row that spans CTAs is combined by whichever CTA contributes last
//     (atomic arrival count, no waiting); in the fused commit step the CTA that
//     finishes the last row of a batch row then runs that row's commit rule.
#include <cuda_runtime.h>

#include <cstdint>

#include "dllm_stats.cuh"

namespace dllm {

struct Acc {
  float m;
  uint64_t Z2;      // two partial sums of 2^y
  uint64_t S2;      // two partial sums of 2^y y
  float negm;
  int32_t idx;
  float best_s;
  int32_t best_v;
  float best_z;
};

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

constexpr float kMInit = -0x1p+121f;  // below every sanitized value
constexpr float kTopClamp = 0x1p+100f;
constexpr uint32_t kTopBf16x2 = 0x71807180u;  // two bf16 2^100

__device__ __forceinline__ void acc_init(Acc& a) {
  a.m = kMInit;
  a.Z2 = 0;
  a.S2 = 0;
  a.negm = -kMInit;
  a.idx = 0x7FFFFFFF;
  a.best_s = -__int_as_float(0x7F800000);
  a.best_v = 0x7FFFFFFF;
  a.best_z = 0.0f;
}

// Raise the running max to mnew (> a.m): Z' = c Z, S2' = c (S2 + d Z),
// c = 2^d, d = (m - mnew) log2 e.
__device__ __forceinline__ void acc_rescale(Acc& a, float mnew) {
  const float d = (a.m - mnew) * kLog2e;
  const float c = ex2_approx(d);
  const uint64_t d2 = pack2(d, d), c2 = pack2(c, c);
  a.S2 = mul2(c2, fma2(d2, a.Z2, a.S2));
  a.Z2 = mul2(a.Z2, c2);
  a.m = mnew;
  a.negm = -mnew;
}

// Adds two sanitized logits (already <= a.m) to the sums.
__device__ __forceinline__ void acc_pair(Acc& a, float z0, float z1) {
  const uint64_t d2 = add2(pack2(z0, z1), pack2(a.negm, a.negm));
  const uint64_t y2 = mul2(d2, pack2(kLog2e, kLog2e));
  float y0, y1;
  unpack2(y2, y0, y1);
  const uint64_t e2 = pack2(ex2_approx(y0), ex2_approx(y1));
  a.Z2 = add2(a.Z2, e2);
  a.S2 = fma2(e2, y2, a.S2);
}

__device__ __forceinline__ float sanitize(float z) {
  return fminf(fmaxf(z, kSentinel), kTopClamp);  // fmaxf drops a NaN operand
}

// Combines b into a (a and b may cover any id sets).
template <bool GUMBEL>
__device__ __forceinline__ void part_combine(Partial& a, const Partial& b) {
  const float m = fmaxf(a.m, b.m);
  const float da = (a.m - m) * kLog2e, db = (b.m - m) * kLog2e;
  const float ca = ex2_approx(da), cb = ex2_approx(db);
  const float Z = ca * a.Z + cb * b.Z;
  const float S2 = ca * fmaf(da, a.Z, a.S2) + cb * fmaf(db, b.Z, b.S2);
  int32_t idx = a.idx;
  if (b.m > a.m || (b.m == a.m && b.idx < a.idx)) idx = b.idx;
  a.m = m;
  a.Z = Z;
  a.S2 = S2;
  a.idx = idx;
  if (GUMBEL) {
    if (b.best_s > a.best_s || (b.best_s == a.best_s && b.best_v < a.best_v)) {
      a.best_s = b.best_s;
      a.best_v = b.best_v;
      a.best_z = b.best_z;
    }
  }
}

__device__ __forceinline__ Partial acc_to_partial(const Acc& a) {
  Partial p;
  float z0, z1, s0, s1;
  unpack2(a.Z2, z0, z1);
  unpack2(a.S2, s0, s1);
  p.m = a.m;
  p.Z = z0 + z1;
  p.S2 = s0 + s1;
  p.idx = a.idx;
  p.best_s = a.best_s;
  p.best_z = a.best_z;
  p.best_v = a.best_v;
  p.pad = 0;
  return p;
}

template <bool GUMBEL>
__device__ __forceinline__ Partial shfl_partial(const Partial& p, int o) {
  Partial q;
  q.m = __shfl_xor_sync(0xFFFFFFFFu, p.m, o);
  q.Z = __shfl_xor_sync(0xFFFFFFFFu, p.Z, o);
  q.S2 = __shfl_xor_sync(0xFFFFFFFFu, p.S2, o);
  q.idx = __shfl_xor_sync(0xFFFFFFFFu, p.idx, o);
  if (GUMBEL) {
    q.best_s = __shfl_xor_sync(0xFFFFFFFFu, p.best_s, o);
    q.best_z = __shfl_xor_sync(0xFFFFFFFFu, p.best_z, o);
    q.best_v = __shfl_xor_sync(0xFFFFFFFFu, p.best_v, o);
  } else {
    q.best_s = p.best_s;
    q.best_z = p.best_z;
    q.best_v = p.best_v;
  }
  q.pad = 0;
  return q;
}

__device__ __forceinline__ void store_partial(Partial* dst, const Partial& p) {
  const int4* s = reinterpret_cast<const int4*>(&p);
  int4* d = reinterpret_cast<int4*>(dst);
  __stcg(d, s[0]);
  __stcg(d + 1, s[1]);
}

__device__ __forceinline__ Partial load_partial(const Partial* src) {
  Partial p;
  int4* d = reinterpret_cast<int4*>(&p);
  const int4* s = reinterpret_cast<const int4*>(src);
  d[0] = __ldcg(s);
  d[1] = __ldcg(s + 1);
  return p;
}

// Writes x0, prob and entropy of one row from its full reduction.
template <bool GUMBEL>
__device__ __forceinline__ void finalize_row(const StatsParams& p, int64_t row, const Partial& r) {
  const int32_t x0 = GUMBEL ? r.best_v : r.idx;
  const float zx = GUMBEL ? r.best_z : r.m;
  const float prob = ex2_approx((zx - r.m) * kLog2e) / r.Z;
  float H = logf(r.Z) - r.S2 * kLn2 / r.Z;
  H = fminf(fmaxf(H, 0.0f), p.ln_veff);
  p.x0[row] = x0;
  p.prob[row] = prob;
  p.entropy[row] = H;
}

__device__ __forceinline__ int64_t unit_start(int64_t c, int64_t U, int64_t P) { return (c * U) / P; }
// The CTA whose range holds unit u: the largest c with unit_start(c) <= u.
__device__ __forceinline__ int64_t cta_of_unit(int64_t u, int64_t U, int64_t P) {
  return ((u + 1) * P + U - 1) / U - 1;
}

struct SharedCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  Partial warp_part[kConsumerWarps];
  Partial result;
  uint64_t rule_red64[kConsumerWarps];
  int32_t rule_red32[4 * kConsumerWarps];
  float warp_best[kConsumerWarps];
  int32_t abort_flag;
  int32_t flag;            // broadcast of per-segment decisions
};

// Bounded wait used by the consumers: gives up when the CTA has aborted.
__device__ __forceinline__ bool consumer_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

template <bool BF16, bool GUMBEL>
__global__ void __launch_bounds__(kThreads, 2) stats_kernel(const __grid_constant__ StatsParams p) {
  extern __shared__ __align__(128) uint8_t dsmem[];
  __shared__ SharedCtl ctl;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t c = blockIdx.x;
  const int64_t u_begin = unit_start(c, p.U, p.P);
  const int64_t u_end = unit_start(c + 1, p.U, p.P);
  const int64_t n_units = u_end - u_begin;
  const int stages = p.stages;
  const uint32_t chunk_bytes = static_cast<uint32_t>(p.chunk_vec) * 16u;
  const uint32_t ring = smem_addr(dsmem);

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_addr(&ctl.full[s]), 1);
      mbar_init(smem_addr(&ctl.empty[s]), kConsumerWarps);
    }
    ctl.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Inputs may be written by the previous kernel in the stream.
  pdl_wait();
  pdl_launch_dependents();

  volatile int32_t* abort_flag = &ctl.abort_flag;

  if (warp == kConsumerWarps) {
    // ---------------- producer: one thread issues the bulk copies ----------------
    if (lane == 0) {
      int64_t issued = 0;
      for (int64_t i = 0; i < n_units; ++i) {
        const int slot = static_cast<int>(i % stages);
        if (i >= stages) {
          const uint32_t par = static_cast<uint32_t>((i / stages - 1) & 1);
          if (!mbar_wait_bounded(smem_addr(&ctl.empty[slot]), par) || *abort_flag) {
            if (!*abort_flag) {
              atomicExch(p.fault, kFaultEmptyWait);
              *abort_flag = 1;
            }
            break;
          }
        }
        const int64_t u = u_begin + i;
        const int64_t row = u / p.K, uk = u - row * p.K;
        const int64_t v0 = uk * p.chunk_vec;
        int64_t nv = p.nvec - v0;
        nv = nv < p.chunk_vec ? nv : p.chunk_vec;
        nv = nv > 0 ? nv : 0;
        const uint32_t bar = smem_addr(&ctl.full[slot]);
        if (nv > 0) {
          const uint32_t bytes = static_cast<uint32_t>(nv) * 16u;
          mbar_arrive_expect_tx(bar, bytes);
          bulk_copy_g2s(ring + slot * chunk_bytes, p.logits + row * p.row_bytes + v0 * 16, bytes, bar);
        } else {
          mbar_arrive(bar);
        }
        issued = i + 1;
      }
      // Drain: every issued copy must land before the CTA may exit.
      const uint64_t t0 = global_timer_ns();
      for (int64_t i = (issued > stages ? issued - stages : 0); i < issued; ++i) {
        const int slot = static_cast<int>(i % stages);
        const uint32_t par = static_cast<uint32_t>((i / stages) & 1);
        while (!mbar_try_wait(smem_addr(&ctl.full[slot]), par)) {
          if (global_timer_ns() - t0 > kWaitLimitNs) {
            atomicExch(p.fault, kFaultDrainWait);
            i = issued;
            break;
          }
        }
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte vector
  const float t = p.temperature;
  const float t_ln2 = t * kLn2;

  RuleScratch rs;
  rs.keys = reinterpret_cast<uint64_t*>(dsmem + static_cast<size_t>(stages) * chunk_bytes);
  rs.flags = reinterpret_cast<uint8_t*>(rs.keys + kFusedSortCap);
  rs.red64 = ctl.rule_red64;
  rs.red32 = ctl.rule_red32;
  rs.cap = kFusedSortCap;

  Acc acc;
  acc_init(acc);
  float warp_best = -__int_as_float(0x7F800000);
  int64_t cur_row = -1, seg_uk0 = 0;
  bool first_segment = true;

  // Reduces the consumers' states of the current segment and publishes it:
  // finalize directly, or as a partial for a row shared with other CTAs.
  auto flush = [&](int64_t row, int64_t uk0, int64_t uk1) {
    Partial part = acc_to_partial(acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Partial q = shfl_partial<GUMBEL>(part, o);
      part_combine<GUMBEL>(part, q);
    }
    if (lane == 0) ctl.warp_part[warp] = part;
    named_sync(1, kConsumers);
    int32_t run_rule_b = -1;
    if (tid == 0) {
      Partial r = ctl.warp_part[0];
      for (int w = 1; w < kConsumerWarps; ++w) part_combine<GUMBEL>(r, ctl.warp_part[w]);
      bool done = false;
      if (!*abort_flag) {
        if (uk0 == 0 && uk1 == p.K - 1) {
          finalize_row<GUMBEL>(p, row, r);
          done = true;
        } else {
          const int64_t slot = 2 * c + (first_segment ? 0 : 1);
          store_partial(p.partials + slot, r);
          __threadfence();
          const int32_t add = static_cast<int32_t>(uk1 - uk0 + 1);
          const int32_t old = atomicAdd(p.row_count + row, add);
          if (old + add == p.K) {
            // last contributor: combine every partial of the row, in CTA order
            __threadfence();
            const int64_t c0 = cta_of_unit(row * p.K, p.U, p.P);
            const int64_t c1 = cta_of_unit(row * p.K + p.K - 1, p.U, p.P);
            Partial tot = load_partial(
                p.partials + 2 * c0 + ((unit_start(c0, p.U, p.P) < row * p.K) ? 1 : 0));
            for (int64_t cc = c0 + 1; cc <= c1; ++cc) {
              const Partial q = load_partial(p.partials + 2 * cc);
              part_combine<GUMBEL>(tot, q);
            }
            p.row_count[row] = 0;
            finalize_row<GUMBEL>(p, row, tot);
            done = true;
          }
        }
        if (done && p.fused) {
          __threadfence();
          const int64_t b = row / p.L;
          const int32_t old = atomicAdd(p.batch_count + b, 1);
          if (old == p.L - 1) run_rule_b = static_cast<int32_t>(b);
        }
      }
      ctl.flag = run_rule_b;
    }
    named_sync(1, kConsumers);
    run_rule_b = ctl.flag;
    if (run_rule_b >= 0) {
      __threadfence();
      run_rule<kConsumers, 1>(p.rule, run_rule_b, rs, tid);
      if (tid == 0) p.batch_count[run_rule_b] = 0;
    }
    first_segment = false;
  };

  for (int64_t i = 0; i < n_units; ++i) {
    const int slot = static_cast<int>(i % stages);
    const uint32_t par = static_cast<uint32_t>((i / stages) & 1);
    const int64_t u = u_begin + i;
    const int64_t row = u / p.K, uk = u - row * p.K;
    if (row != cur_row) {
      if (cur_row >= 0) flush(cur_row, seg_uk0, p.K - 1);
      acc_init(acc);
      warp_best = -__int_as_float(0x7F800000);
      cur_row = row;
      seg_uk0 = uk;
    }
    const int64_t v_unit = uk * p.chunk_vec;  // first vector of the unit
    int64_t nv = p.nvec - v_unit;
    nv = nv < p.chunk_vec ? nv : p.chunk_vec;
    // suppressed ids inside this unit (CTA-uniform)
    const int64_t id_lo = v_unit * EPV;
    const int64_t id_hi = (uk == p.K - 1) ? p.V : (v_unit + nv) * EPV;
    bool unit_has_sup = false;
    for (int s = 0; s < p.n_sup; ++s) unit_has_sup |= (p.sup[s] >= id_lo && p.sup[s] < id_hi);

    if (!*abort_flag && !consumer_wait(smem_addr(&ctl.full[slot]), par, abort_flag)) {
      if (!*abort_flag) {
        atomicExch(p.fault, kFaultFullWait);
        *abort_flag = 1;
      }
    }
    const uint32_t base = ring + slot * chunk_bytes;
    // The trip count is the same for every consumer thread (warp-collective
    // operations below need all 32 lanes); lanes past the unit's end idle.
    for (int64_t vb = 0; vb < nv; vb += kConsumers) {
      const int64_t vi = vb + tid;
      const bool valid = vi < nv;
      const uint4 q = valid ? lds128(base + static_cast<uint32_t>(vi) * 16u) : make_uint4(0, 0, 0, 0);
      const int64_t v0 = (v_unit + vi) * EPV;
      float z[EPV];
      if (BF16) {
        uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) w[j] = bmax2(w[j], kSentinelBf16x2);
        // clamp the top at 2^100 (min of bf16 pairs)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t r;
          asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(w[j]), "r"(kTopBf16x2));
          w[j] = r;
        }
        if (unit_has_sup) {
          for (int s = 0; s < p.n_sup; ++s) {
            const int64_t off = p.sup[s] - v0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (off == 2 * j) w[j] = (w[j] & 0xFFFF0000u) | kAbsentBf16;
              if (off == 2 * j + 1) w[j] = (w[j] & 0x0000FFFFu) | (kAbsentBf16 << 16);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          z[2 * j] = bf16lo(w[j]);
          z[2 * j + 1] = bf16hi(w[j]);
        }
      } else {
        z[0] = sanitize(__uint_as_float(q.x));
        z[1] = sanitize(__uint_as_float(q.y));
        z[2] = sanitize(__uint_as_float(q.z));
        z[3] = sanitize(__uint_as_float(q.w));
        if (unit_has_sup) {
          for (int s = 0; s < p.n_sup; ++s) {
            const int64_t off = p.sup[s] - v0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              if (off == j) z[j] = kAbsent;
          }
        }
      }
      float vmax = z[0];
#pragma unroll
      for (int j = 1; j < EPV; ++j) vmax = fmaxf(vmax, z[j]);
      if (valid) {
        if (vmax > acc.m) {
          acc_rescale(acc, vmax);
          if (!GUMBEL) {
#pragma unroll
            for (int j = EPV - 1; j >= 0; --j)
              if (z[j] == vmax) acc.idx = static_cast<int32_t>(v0 + j);
          }
        }
#pragma unroll
        for (int j = 0; j < EPV; j += 2) acc_pair(acc, z[j], z[j + 1]);
      }

      if (GUMBEL) {
        // Philox words of ids v0 .. v0 + EPV - 1 (v0 is a multiple of 4)
        uint32_t r[EPV];
        const uint32_t row_lo = static_cast<uint32_t>(row), row_hi = static_cast<uint32_t>(static_cast<uint64_t>(row) >> 32);
#pragma unroll
        for (int h = 0; h < EPV / 4; ++h) {
          const uint4 o = philox4x32_10(static_cast<uint32_t>((v0 >> 2) + h), row_lo, row_hi, 0u, p.key);
          r[4 * h + 0] = o.x;
          r[4 * h + 1] = o.y;
          r[4 * h + 2] = o.z;
          r[4 * h + 3] = o.w;
        }
        uint32_t rmax = r[0];
#pragma unroll
        for (int j = 1; j < EPV; ++j) rmax = max(rmax, r[j]);
        // g = -ln(-ln u) <= -ln(1 - u) for every id of the vector; the margin
        // covers the fp32 rounding of ln_p, lg2.approx and the final fmaf.
        const float w1 = __fsub_rn(1.0f, uniform_from_bits(rmax));
        const float gbound = -lg2_approx(w1);
        const float bound = fmaf(t_ln2, gbound, vmax + fmaf(fabsf(vmax), 1e-6f, 1e-3f));
        const bool survive = valid && !(bound < warp_best);
        bool updated = false;
        if (survive) {
#pragma unroll
          for (int j = 0; j < EPV; ++j) {
            const float s = gumbel_score(z[j], t, r[j]);
            if (s > acc.best_s) {
              acc.best_s = s;
              acc.best_v = static_cast<int32_t>(v0 + j);
              acc.best_z = z[j];
              updated = true;
            }
          }
        }
        if (__any_sync(0xFFFFFFFFu, updated)) {
          float wb = acc.best_s;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) wb = fmaxf(wb, __shfl_xor_sync(0xFFFFFFFFu, wb, o));
          warp_best = fmaxf(warp_best, wb);
        }
      }
    }
    // Release the stage: one arrival per consumer warp.
    __syncwarp();
    if (lane == 0 && !*abort_flag) mbar_arrive(smem_addr(&ctl.empty[slot]));

    // Elements after the last full vector of the row (V * size % 16 != 0).
    if (uk == p.K - 1 && p.tail > 0 && tid < p.tail && !*abort_flag) {
      const int64_t v = p.nvec * EPV + tid;
      const uint8_t* rowp = p.logits + row * p.row_bytes;
      float z;
      if (BF16) {
        const uint16_t bits = __ldg(reinterpret_cast<const uint16_t*>(rowp) + v);
        z = __uint_as_float(static_cast<uint32_t>(bits) << 16);
      } else {
        z = __ldg(reinterpret_cast<const float*>(rowp) + v);
      }
      z = sanitize(z);
      for (int s = 0; s < p.n_sup; ++s)
        if (p.sup[s] == v) z = kAbsent;
      if (z > acc.m) {
        acc_rescale(acc, z);
        acc.idx = static_cast<int32_t>(v);
      }
      {
        const float y = (z - acc.m) * kLog2e;
        const float e = ex2_approx(y);
        acc.Z2 = add2(acc.Z2, pack2(e, 0.0f));
        acc.S2 = fma2(pack2(e, 0.0f), pack2(y, 0.0f), acc.S2);
      }
      if (GUMBEL) {
        const uint4 o = philox4x32_10(static_cast<uint32_t>(v >> 2), static_cast<uint32_t>(row),
                                      static_cast<uint32_t>(static_cast<uint64_t>(row) >> 32), 0u, p.key);
        const int w = static_cast<int>(v & 3);
        const uint32_t word = w == 0 ? o.x : (w == 1 ? o.y : (w == 2 ? o.z : o.w));
        const float s = gumbel_score(z, t, word);
        if (s > acc.best_s) {
          acc.best_s = s;
          acc.best_v = static_cast<int32_t>(v);
          acc.best_z = z;
        }
      }
    }
  }
  if (cur_row >= 0) {
    const int64_t last_u = u_end - 1;
    flush(cur_row, seg_uk0, last_u - cur_row * p.K);
  }
}

// Explicit instantiations used by the launcher.
template __global__ void stats_kernel<false, false>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, false>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<false, true>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, true>(const __grid_constant__ StatsParams);

const void* stats_kernel_ptr(bool bf16, bool gumbel) {
  if (bf16) return gumbel ? reinterpret_cast<const void*>(&stats_kernel<true, true>)
                          : reinterpret_cast<const void*>(&stats_kernel<true, false>);
  return gumbel ? reinterpret_cast<const void*>(&stats_kernel<false, true>)
                : reinterpret_cast<const void*>(&stats_kernel<false, false>);
}

}  // namespace dllm
