// dllm_stats_kernels.cuh -- the statistics pass (and the fused commit step) on
// sm_103a: the kernel templates.  dllm_stats_{greedy,sample,margin}.cu
// instantiate them per mode, in parallel translation units.
//
// What it computes (mlx-arsenal "dLLM block decoding", "What mlx-arsenal
// ships": token_stats; mojo-dllm manual, "Row statistics on the device"): for
// every logit row, the proposal x0 (first argmax, or Gumbel-max), its
// probability and the entropy of the softmax over the non-suppressed ids.
//
// How (one pass over HBM):
//   * Rows are cut into units of chunk_vec 16-byte vectors.  In each CTA one
//     producer thread streams its units into a shared-memory ring with
//     cp.async.bulk (TMA bulk copies), one mbarrier per stage; eight consumer
//     warps read each unit from shared memory.
//   * Each consumer thread keeps an online softmax state of the scaled logits
//     z' = fp32(z s) (s = 1 unless the caller scales them): running max m of
//     the raw logits, Z = sum 2^y and S2 = sum 2^y y with y = z' log2 e - ref
//     and ref = RU(m' log2 e), the product rounded up (packed fp32x2
//     accumulators, one fused multiply-add per pair); entropy = ln Z - S2
//     ln 2 / Z.  The lanes of a warp share one running max (the warp's, by
//     redux.sync), so the sums are rescaled only when it grows.  Decisions
//     (argmax, ties, Gumbel scores) compare the scaled values z' themselves.
//   * Consumer::consume streams a (row, vector range) segment: full units in
//     a loop specialised on the vectors each thread holds, the ragged last
//     unit after it, with warp-uniform control flow.
//   * Rows whose maximum the streaming pass cannot resolve exactly (|ref| >=
//     2^28, or no logit above the no-mass sentinel -2^100) are recomputed by
//     one warp from the logits as they are (exotic_row).
//     The first index of the max is located once per row, from the first
//     vector that holds the thread's max (in the plain greedy mode recorded
//     only by the lanes that hold a new warp max); the largest value outside
//     that element (the runner-up of the margin confidence) comes with it.
//   * Gumbel-max: one Philox4x32-10 call per four ids (rounds 0 and 1 folded
//     per row); a bound on the noise
//     from the largest uniform of each 16-byte vector lets most vectors skip
//     the two logarithms; the warp shares its best score to tighten the bound.
//   * Many rows (persistent kernel): the units are dealt to the CTAs in equal
//     contiguous ranges; a row shared by several CTAs is combined by the one
//     that contributes last (atomic arrival count, no waiting), its warp 0
//     loading the partials in parallel.
//   * Few rows (cluster kernel): one thread-block cluster per row, each CTA a
//     contiguous slice; the CTAs' partials are combined through distributed
//     shared memory by rank 0.
//   * Short batch rows whose inputs are ready early (batch-row kernel): one
//     cluster per batch row, each CTA whole rows; rank 0 gathers their
//     partials through distributed shared memory and decides the rule in
//     shared memory before the grid dependency, so only stores follow it.
//   * Fused commit step: the thread that finalizes a row also makes the row's
//     threshold / edit decision and canvas update; the last row of a batch row
//     applies the forced commit when nothing passed (or, for the sorting rules,
//     its CTA runs the whole rule).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "dllm_stats.cuh"

namespace dllm {

struct Acc {
  float m;          // running max of the raw logits
  uint64_t Z2;      // two partial sums of 2^y
  uint64_t S2;      // two partial sums of 2^y y
  float nref;       // -ref, ref = RU(m' log2 e): minus the exponent reference of m
  int32_t idx;      // first index of m among the tail elements (greedy)
  float vm;         // greedy: z' of the thread's recorded max (its first
                    // occurrence among the thread's full vectors; in the
                    // plain greedy mode recorded only when it was the warp's
                    // new max, so a thread may hold no record of its own max)
  int32_t vv;       // first id of the first vector holding vm, -1 if none
  uint32_t bw[4];   // that vector's sanitized words
  float m2o;        // max of z' over the thread's other full vectors; after
                    // resolve_index, the thread's runner-up
  float vm_tail;    // z' of the thread's tail element, if any (greedy)
  float best_s;
  int32_t best_v;
  float best_z;
};

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Below every sanitized value (kAbsent is -2^110), and finite after scaling
// by the largest logit scale (256): -2^120.
constexpr float kMInit = -0x1p+112f;
constexpr float kExoticRef = 0x1p+28f;  // rows whose |ref| reaches this take exotic_row
constexpr float kTopClamp = 0x1p+100f;
constexpr uint32_t kTopBf16x2 = 0x71807180u;  // two bf16 2^100
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ void acc_init(Acc& a) {
  a.m = kMInit;
  a.Z2 = 0;
  a.S2 = 0;
  a.nref = 0x1.fffffep+127f;   // the reference of "no max yet": every rescale from it gives 0
  a.idx = 0x7FFFFFFF;
  a.vm = kMInit;
  a.vv = -1;
  a.bw[0] = a.bw[1] = a.bw[2] = a.bw[3] = 0u;
  a.vm_tail = kMInit;
  a.best_s = kNegInf;
  a.best_v = 0x7FFFFFFF;
  a.best_z = 0.0f;
}

// The exponent reference of a running max m' (a scaled logit): ref =
// RU(m' log2 e), the product rounded up.  A term is 2^(z' log2 e - ref) with
// z' log2 e - ref formed exactly and rounded once (one fused multiply-add),
// so every term is at most 1 and the sums stay finite for any logit; the
// max's own term is 2^(m' log2 e - ref), in (2^-ulp(ref), 1].  Rescales and
// combines shift by differences of these references, so sums built against
// different maxima agree on their scale.
__device__ __forceinline__ float exp_ref(float ms) { return __fmul_ru(ms, kLog2e); }

// z' = fp32(z s) in the scaled modes, z itself otherwise.
template <bool SCALED>
__device__ __forceinline__ float scaled(float z, float s) { return SCALED ? __fmul_rn(z, s) : z; }

// The shift from reference `from` to reference `to` (>= from), clamped to
// [-256, 0] (2^-256 is 0 in fp32): the clamp keeps it finite when a
// reference sits at the end of the fp32 range.
__device__ __forceinline__ float ref_shift(float from, float to) {
  return fminf(fmaxf(from - to, -256.0f), 0.0f);
}

// Raise the running max to mnew (> a.m): Z' = f Z, S2' = f (S2 + d Z),
// f = 2^d, d = ref(m) - ref(mnew).
template <bool SCALED>
__device__ __forceinline__ void acc_rescale(Acc& a, float mnew, float s) {
  const float rn = exp_ref(scaled<SCALED>(mnew, s));
  const float d = ref_shift(-a.nref, rn);
  const float c = ex2_approx(d);
  const uint64_t d2 = pack2(d, d), c2 = pack2(c, c);
  a.S2 = mul2(c2, fma2(d2, a.Z2, a.S2));
  a.Z2 = mul2(a.Z2, c2);
  a.m = mnew;
  a.nref = -rn;
}

__device__ __forceinline__ float sanitize(float z) {
  return fminf(fmaxf(z, kSentinel), kTopClamp);  // fmaxf drops a NaN operand
}

// fp32 bits: NaN and values <= -2^100 -> -2^100 (fmaxf drops a NaN operand).
__device__ __forceinline__ uint32_t sanitize_low_bits(uint32_t b) {
  return __float_as_uint(fmaxf(__uint_as_float(b), kSentinel));
}
__device__ __forceinline__ uint32_t clamp_top_bits(uint32_t b) {
  return __float_as_uint(fminf(__uint_as_float(b), kTopClamp));
}
__device__ __forceinline__ uint32_t bmin2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Adds two sanitized logits (<= m) to the sums (Z2, S2): z' = fp32(z s) in
// the scaled modes (one packed multiply; s2 holds s twice), y = z' log2 e -
// ref in one fused multiply-add per pair (l2e2 holds log2 e twice, nref2
// holds -ref twice, ref = exp_ref(m')), 2^y and 2^y y.
template <bool SCALED>
__device__ __forceinline__ void acc_pair2(uint64_t& Z2, uint64_t& S2, float z0, float z1, uint64_t nref2,
                                          uint64_t l2e2, uint64_t s2) {
  const uint64_t zz = SCALED ? mul2(pack2(z0, z1), s2) : pack2(z0, z1);
  const uint64_t y2 = fma2(zz, l2e2, nref2);
  float y0, y1;
  unpack2(y2, y0, y1);
  const uint64_t e2 = pack2(ex2_approx(y0), ex2_approx(y1));
  Z2 = add2(Z2, e2);
  S2 = fma2(e2, y2, S2);
}

// Combines b into a (a and b may cover any id sets; m is the raw max the
// sums are taken against, the argmax is decided on the scaled maxima
// fp32(m s), ties to the lower id).  The runner-up of the union is the larger
// of the winner's runner-up and the loser's largest scaled value: its max,
// or, for a part that holds no id of its m (idx unset: a lane whose values
// all lie below its warp's max), the value its m2 carries.
template <int MODE>
__device__ __forceinline__ void part_combine(Partial& a, const Partial& b, float s) {
  constexpr bool GUMBEL = mode_sample(MODE), RUNNER = mode_runner(MODE), SCALED = mode_scaled(MODE);
  const float m = fmaxf(a.m, b.m);
  const float sa = scaled<SCALED>(a.m, s), sb = scaled<SCALED>(b.m, s);
  const float ra = exp_ref(sa), rb = exp_ref(sb), r = fmaxf(ra, rb);   // r = exp_ref(m')
  const float da = ref_shift(ra, r), db = ref_shift(rb, r);
  const float ca = ex2_approx(da), cb = ex2_approx(db);
  const float Z = ca * a.Z + cb * b.Z;
  const float S2 = ca * fmaf(da, a.Z, a.S2) + cb * fmaf(db, b.Z, b.S2);
  const bool b_wins = sb > sa || (sb == sa && b.idx < a.idx);
  if (RUNNER) {
    const float ta = a.idx == 0x7FFFFFFF ? a.m2 : sa, tb = b.idx == 0x7FFFFFFF ? b.m2 : sb;
    a.m2 = b_wins ? fmaxf(b.m2, ta) : fmaxf(a.m2, tb);
  }
  a.m = m;
  a.Z = Z;
  a.S2 = S2;
  a.idx = b_wins ? b.idx : a.idx;
  if (GUMBEL) {
    if (b.best_s > a.best_s || (b.best_s == a.best_s && b.best_v < a.best_v)) {
      a.best_s = b.best_s;
      a.best_v = b.best_v;
      a.best_z = b.best_z;
    }
  }
}

__device__ __forceinline__ Partial empty_partial() {
  Partial p;
  p.m = kMInit;
  p.Z = 0.0f;
  p.S2 = 0.0f;
  p.idx = 0x7FFFFFFF;
  p.best_s = kNegInf;
  p.best_z = 0.0f;
  p.best_v = 0x7FFFFFFF;
  p.m2 = kMInit;
  return p;
}

// RUNNER: the thread tracked a runner-up (else m2 is not carried, so the
// field holds no register through the streaming loop).
template <bool RUNNER>
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
  p.m2 = RUNNER ? a.m2o : kMInit;
  return p;
}

template <int MODE>
__device__ __forceinline__ Partial shfl_partial(const Partial& p, int o) {
  constexpr bool GUMBEL = mode_sample(MODE), RUNNER = mode_runner(MODE);
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
  q.m2 = RUNNER ? __shfl_xor_sync(0xFFFFFFFFu, p.m2, o) : p.m2;
  return q;
}

template <int MODE>
__device__ __forceinline__ Partial warp_combine(Partial part, float s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const Partial q = shfl_partial<MODE>(part, o);
    part_combine<MODE>(part, q, s);
  }
  return part;
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

// Reads a Partial held in the shared memory of CTA `rank` of this cluster.
__device__ __forceinline__ Partial load_partial_dsmem(const Partial* local, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
  Partial p;
  uint32_t* w = reinterpret_cast<uint32_t*>(&p);
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(remote)
               : "memory");
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "r"(remote + 16u)
               : "memory");
  return p;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// The row's candidate flag and current canvas token, when already loaded.
struct RowPre {
  bool have = false;
  bool cand = false;
  int32_t tok = 0;
};

__device__ __forceinline__ RowPre load_row_pre(const StatsParams& p, int64_t row) {
  RowPre pre;
  if (!p.fused) return pre;
  const int64_t b = row / p.L, l = row - b * p.L;
  pre.cand = is_candidate(p.rule, b, l, &pre.tok);
  pre.have = true;
  return pre;
}

__device__ __forceinline__ unsigned long long atom_add_acq_rel(unsigned long long* a, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(a), "l"(v) : "memory");
  return old;
}

// x0, prob and entropy of one row from its full reduction.  exotic: the
// row's maximum is outside what the streaming pass resolves (see exotic_row).
struct RowOut {
  int32_t x0, argmax;
  float prob, H, margin;
  bool exotic;
};

// prob = x0's term over Z (its exponent formed exactly as the sums formed
// it); entropy = ln Z - S2 ln 2 / Z clamped to [0, ln |A|].  The margin's
// runner-up is the largest z' without x0: the row's runner-up when x0 is the
// argmax, else the max itself.
template <int MODE>
__device__ __forceinline__ RowOut row_out(const StatsParams& p, const Partial& r) {
  constexpr bool GUMBEL = mode_sample(MODE), RUNNER = mode_runner(MODE), SCALED = mode_scaled(MODE);
  RowOut o;
  o.x0 = GUMBEL ? r.best_v : r.idx;
  o.argmax = r.idx;
  const float ms = scaled<SCALED>(r.m, p.scale);                // the scaled max m'
  const float ref = exp_ref(ms);
  o.exotic = !(fabsf(ref) < kExoticRef);
  const float ytop = fmaf(ms, kLog2e, -ref);                      // the max's own exponent
  // best_z is the raw logit of x0: its exponent as the sums formed it
  const float yx = GUMBEL ? fmaf(scaled<SCALED>(r.best_z, p.scale), kLog2e, -ref) : ytop;
  o.prob = ex2_approx(yx) / r.Z;
  const float H = logf(r.Z) - r.S2 * kLn2 / r.Z;
  o.H = fminf(fmaxf(H, 0.0f), p.ln_veff);
  o.margin = 0.0f;
  if (RUNNER) {
    const float r2 = (!GUMBEL || r.best_v == r.idx) ? r.m2 : ms;   // a scaled logit
    o.margin = o.prob - ex2_approx(fmaf(r2, kLog2e, -ref)) / r.Z;
  }
  return o;
}

// The statistics of a row whose maximum the streaming pass does not resolve
// exactly: |RU(m' log2 e)| >= 2^28 (logits beyond about 1.8e8 / s in magnitude,
// +inf included, where the fp32 spacing of the reference exceeds 16), or no
// logit above the no-mass sentinel (NaN, -inf or finite values <= -2^100
// only).  One warp recomputes the row from the logits as they are, reading
// them again: a NaN has no mass, +inf entries share the mass equally, every
// finite logit takes the ordinary softmax ("dLLM block decoding", What
// mlx-arsenal ships: token_stats is NaN-safe), and a row with no mass at all
// gives the uniform limit.  Model output never holds such rows; this path
// costs two or three extra reads of the row by one warp.
template <bool BF16, int MODE>
__device__ __noinline__ RowOut exotic_row(const StatsParams& p, int64_t row, int lane) {
  constexpr bool GUMBEL = mode_sample(MODE), RUNNER = mode_runner(MODE), SCALED = mode_scaled(MODE);
  constexpr int32_t kNone = 0x7FFFFFFF;
  const float s = SCALED ? p.scale : 1.0f;
  const float t = p.temperature;
  const uint8_t* rowp = p.logits + row * p.row_bytes;
  const int32_t V = static_cast<int32_t>(p.V);
  const int32_t n_sup = p.n_sup;
  // z' of id v: NaN -> -inf, else fp32(z s)
  auto zl = [&](int32_t v) -> float {
    float z;
    if (BF16)
      z = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(rowp) + v)) << 16);
    else
      z = __ldg(reinterpret_cast<const float*>(rowp) + v);
    if (isnan(z)) return kNegInf;
    return SCALED ? __fmul_rn(z, s) : z;
  };
  // Walks this lane's ids v = lane, lane + 32, ... of the token set (the
  // sorted suppress list is stepped through alongside, one read per id it holds).
  auto for_each = [&](auto&& fn) {
    int32_t si = 0;
    int32_t next = n_sup > 0 ? p.sup[0] : kNone;
    for (int64_t vv = lane; vv < V; vv += 32) {
      const int32_t v = static_cast<int32_t>(vv);
      while (next < v) next = (++si < n_sup) ? p.sup[si] : kNone;
      if (next == v) continue;
      fn(v, zl(v));
    }
  };
  // Pass 1: the max M of z' over the token set and its first id (with no
  // mass anywhere, M = -inf and the id is the set's first).
  float M = kNegInf;
  int32_t am = kNone;
  for_each([&](int32_t v, float z) {
    if (am == kNone || z > M) {
      M = z;
      am = v;
    }
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float M2 = __shfl_xor_sync(0xFFFFFFFFu, M, o);
    const int32_t a2 = __shfl_xor_sync(0xFFFFFFFFu, am, o);
    if (a2 != kNone && (am == kNone || M2 > M || (M2 == M && a2 < am))) {
      M = M2;
      am = a2;
    }
  }
  const float veff = static_cast<float>(p.V - n_sup);
  RowOut o;
  o.exotic = false;
  o.argmax = am;
  o.x0 = am;
  o.margin = 0.0f;
  if (M == kNegInf) {  // the uniform limit; every Gumbel score is -inf, so x0 is the first id too
    o.prob = 1.0f / veff;
    o.H = p.ln_veff;
    if (RUNNER) o.margin = veff >= 2.0f ? 0.0f : o.prob;
    return o;
  }
  if (M == -kNegInf) {  // the +inf entries share the mass; the first of them is x0 and has the top score
    int32_t n_inf = 0;
    for_each([&](int32_t, float z) { n_inf += z == M ? 1 : 0; });
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) n_inf += __shfl_xor_sync(0xFFFFFFFFu, n_inf, k);
    o.prob = 1.0f / static_cast<float>(n_inf);
    o.H = fminf(static_cast<float>(log(static_cast<double>(n_inf))), p.ln_veff);
    if (RUNNER) o.margin = n_inf >= 2 ? 0.0f : o.prob;
    return o;
  }
  // Finite M.  Pass 2: Z = sum 2^y, S2 = sum 2^y y, y = (z' - M) log2 e
  // (accumulated in double), and the Gumbel-max sample: an id can beat the
  // argmax's score only if z' + 17 t >= M - 3 t (every noise value g of the
  // sampler lies in [-3, 17]), so only those ids get a score.
  const uint32_t row_lo = static_cast<uint32_t>(row);
  const uint32_t row_hi = static_cast<uint32_t>(static_cast<uint64_t>(row) >> 32);
  const float floor_s = fmaf(t, -3.0f, M);
  double Z = 0.0, S2 = 0.0;
  float bs = kNegInf, bz = 0.0f;
  int32_t bv = kNone;
  for_each([&](int32_t v, float z) {
    const float y = (z - M) * kLog2e;
    if (y > -200.0f) {
      const float e = ex2_approx(y);
      Z += static_cast<double>(e);
      S2 += static_cast<double>(e) * static_cast<double>(y);
    }
    if (GUMBEL && fmaf(t, 17.0f, z) >= floor_s) {
      const uint4 w4 = philox4x32_10(static_cast<uint32_t>(v >> 2), row_lo, row_hi, 0u, p.keys);
      const int k = v & 3;
      const uint32_t word = k == 0 ? w4.x : (k == 1 ? w4.y : (k == 2 ? w4.z : w4.w));
      const float sc = gumbel_score(z, t, word);
      if (bv == kNone || sc > bs) {   // ids rise in a lane: a strict > keeps the first of equal scores
        bs = sc;
        bv = v;
        bz = z;
      }
    }
  });
#pragma unroll
  for (int k = 16; k > 0; k >>= 1) {
    Z += __shfl_xor_sync(0xFFFFFFFFu, Z, k);
    S2 += __shfl_xor_sync(0xFFFFFFFFu, S2, k);
    if (GUMBEL) {
      const float s2 = __shfl_xor_sync(0xFFFFFFFFu, bs, k);
      const int32_t v2 = __shfl_xor_sync(0xFFFFFFFFu, bv, k);
      const float z2 = __shfl_xor_sync(0xFFFFFFFFu, bz, k);
      if (v2 != kNone && (bv == kNone || s2 > bs || (s2 == bs && v2 < bv))) {
        bs = s2;
        bv = v2;
        bz = z2;
      }
    }
  }
  if (GUMBEL) o.x0 = bv;
  const float zx = GUMBEL ? bz : M;
  o.prob = static_cast<float>(static_cast<double>(ex2_approx((zx - M) * kLog2e)) / Z);
  const double H = log(Z) - S2 * 0.6931471805599453 / Z;
  o.H = fminf(fmaxf(static_cast<float>(H), 0.0f), p.ln_veff);
  if (RUNNER) {
    // Pass 3: the runner-up, the largest z' over the token set without x0.
    float r2 = kNegInf;
    const int32_t x0 = o.x0;
    for_each([&](int32_t v, float z) {
      if (v != x0) r2 = fmaxf(r2, z);
    });
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) r2 = fmaxf(r2, __shfl_xor_sync(0xFFFFFFFFu, r2, k));
    const float y2 = (r2 - M) * kLog2e;
    const double p2 = y2 > -200.0f ? static_cast<double>(ex2_approx(y2)) / Z : 0.0;
    o.margin = static_cast<float>(static_cast<double>(o.prob) - p2);
  }
  return o;
}

// Writes x0, prob and entropy of one row and, in the fused step, makes the
// row's own commit / edit decisions.  Run by one thread.  Returns the batch
// row whose sorting rule this CTA must now run, or -1.
inline __device__ int32_t finish_row(const StatsParams& p, int64_t row, const RowOut& o, RowPre pre) {
  const int32_t x0 = o.x0;
  const float prob = o.prob, H = o.H;
  p.x0[row] = x0;
  p.prob[row] = prob;
  p.entropy[row] = H;
  if (p.margin) p.margin[row] = o.margin;
  if (p.argmax) p.argmax[row] = o.argmax;
  if (!p.fused) return -1;

  const RuleArgs& a = p.rule;
  const int64_t b = row / p.L, l = row - b * p.L;
  const bool per_row = a.rule == kRuleThreshold || a.rule == kRuleNone;
  unsigned long long inc = 1ull;
  if (per_row) {
    if (!pre.have) pre = load_row_pre(p, row);
    const bool cand = pre.cand;
    const int32_t tok = pre.tok;
    const float c = nan_to(prob, kNegInf);
    bool commit = false, edit = false;
    if (a.rule == kRuleThreshold && cand) commit = a.strict ? (c > a.tau) : (c >= a.tau);
    if (a.edit && !cand) edit = (x0 != tok) && (c > a.tau_edit);
    if (a.commit) a.commit[row] = commit ? 1 : 0;
    if (a.edit_mask) a.edit_mask[row] = edit ? 1 : 0;
    if ((commit || edit) && a.canvas) a.canvas[b * a.canvas_stride + a.canvas_offset + l] = x0;
    if (cand && a.rule == kRuleThreshold) atomicMax(p.batch_forced + b, ~desc_key(c, l));
    inc |= (cand ? 1ull << 16 : 0ull) | (commit ? 1ull << 32 : 0ull) | (edit ? 1ull << 48 : 0ull);
  }
  // One release-acquire arrival per row: this row's writes become visible to
  // whichever thread sees the batch row complete.
  const unsigned long long tot = atom_add_acq_rel(p.batch_packed + b, inc) + inc;
  if (static_cast<int64_t>(tot & 0xFFFFull) != p.L) return -1;
  p.batch_packed[b] = 0ull;
  if (!per_row) return static_cast<int32_t>(b);
  // Last row of the batch row: force one commit if candidates exist and none passed.
  const int32_t n_cand = static_cast<int32_t>((tot >> 16) & 0xFFFFull);
  int32_t n_commit = static_cast<int32_t>((tot >> 32) & 0xFFFFull);
  const int32_t n_edit = static_cast<int32_t>((tot >> 48) & 0xFFFFull);
  if (a.rule == kRuleThreshold && n_cand > 0 && n_commit == 0) {
    const unsigned long long key = ~__ldcg(p.batch_forced + b);
    const int64_t lf = static_cast<int64_t>(key & 0xFFFFFFFFull);
    if (a.commit) a.commit[b * p.L + lf] = 1;
    if (a.canvas) a.canvas[b * a.canvas_stride + a.canvas_offset + lf] = __ldcg(p.x0 + b * p.L + lf);
    n_commit = 1;
  }
  if (a.rule == kRuleThreshold) p.batch_forced[b] = 0ull;
  if (a.counts) {
    a.counts[3 * b + 0] = n_cand;
    a.counts[3 * b + 1] = n_commit;
    a.counts[3 * b + 2] = n_edit;
  }
  return -1;
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
  int32_t abort_flag;
  int32_t flag;
  int32_t flag2;
  uint32_t cta_best;   // running best Gumbel score of the CTA's current row (order-preserving bits)
};

// Bounded wait used by the consumers: sleeps in hardware until the copy
// lands; gives up when the CTA has aborted or the deadline passes.
__device__ __forceinline__ bool consumer_wait(uint32_t bar, uint32_t parity, volatile int32_t* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

// Position in the shared-memory ring: stage index and mbarrier phase parity.
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance(int stages) {
    if (++slot == stages) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// The consumers' wait for a ring stage once the first try failed: bounded,
// and it gives up at once when the CTA has aborted; a wait that runs out
// records the fault and aborts the CTA (the loops then run to their end
// without waiting, and nothing is written).
static __device__ __noinline__ void wait_unit_slow(const StatsParams& p, SharedCtl& ctl, int slot, uint32_t phase) {
  volatile int32_t* abort_flag = &ctl.abort_flag;
  if (!*abort_flag && !consumer_wait(smem_addr(&ctl.full[slot]), phase, abort_flag)) {
    if (!*abort_flag) {
      atomicExch(p.fault, kFaultFullWait);
      *abort_flag = 1;
    }
  }
}

struct VecWords {
  uint32_t w[4];
};
struct GumbelWords {
  uint32_t w[8];
};

struct GumbelBest {
  float s;
  int32_t v;
  float z;   // the raw (unscaled) logit of v
};

// Exact Gumbel scores of the elements of one vector that can still beat
// max(floor, best.s): each element's own bound z + t (-ln(1 - u)) (plus
// margin) gates the two logarithms.  Out of line: it runs for few vectors, and
// keeping it out of the streaming loop keeps that loop small.
template <bool BF16>
__device__ __noinline__ GumbelBest gumbel_exact(GumbelBest best, VecWords vw, GumbelWords r, int32_t v0, float t,
                                                float t_ln2, float floor, float s) {
  constexpr int EPV = BF16 ? 8 : 4;
#pragma unroll 1
  for (int e = 0; e < EPV; ++e) {
    const uint32_t word = vw.w[BF16 ? (e >> 1) : e];
    const float zr = BF16 ? ((e & 1) ? bf16hi(word) : bf16lo(word)) : __uint_as_float(word);
    const float z = __fmul_rn(zr, s);
    const uint32_t re = r.w[e];
    const float w1 = __fsub_rn(1.0f, uniform_from_bits(re));
    const float bound = fmaf(t_ln2, -lg2_approx(w1), z + fmaf(fabsf(z), 1e-6f, 1e-3f));
    if (bound < floor || bound < best.s) continue;
    const float sc = gumbel_score(z, t, re);
    if (sc > best.s) {
      best.s = sc;
      best.v = v0 + e;
      best.z = zr;   // the raw logit
    }
  }
  return best;
}

// Consumer-side state of one CTA.
template <bool BF16, int MODE>
struct Consumer {
  static constexpr bool GUMBEL = mode_sample(MODE);    // a Gumbel-max sample
  static constexpr bool GREEDY = mode_argmax(MODE);    // the first argmax
  static constexpr bool RUNNER = mode_runner(MODE);    // and its runner-up
  static constexpr bool SCALED = mode_scaled(MODE);    // logit scale s != 1
  static constexpr int EPV = BF16 ? 8 : 4;  // elements per 16-byte vector
  const StatsParams& p;
  SharedCtl& ctl;
  uint32_t ring, chunk_bytes;
  int tid, warp, lane;
  float t, t_ln2;
  float s;          // logit scale
  uint64_t s2;      // (s, s)
  uint64_t l2e2;    // (log2 e, log2 e)
  Acc acc;
  float warp_best;

  __device__ Consumer(const StatsParams& p_, SharedCtl& ctl_, uint32_t ring_, uint32_t chunk_bytes_)
      : p(p_), ctl(ctl_), ring(ring_), chunk_bytes(chunk_bytes_) {
    tid = threadIdx.x;
    warp = tid >> 5;
    lane = tid & 31;
    t = p.temperature;
    t_ln2 = t * kLn2;
    s = SCALED ? p.scale : 1.0f;
    s2 = pack2(s, s);
    l2e2 = pack2(kLog2e, kLog2e);
    reset();
  }

  // Per-row reset of the thread's state (the CTA-wide best is cleared at the
  // start of the kernel and at the end of every flush, before a barrier).
  __device__ void reset() {
    acc_init(acc);
    if (RUNNER) acc.m2o = kMInit;
    warp_best = kNegInf;
    sup_restart();
  }

  static constexpr int kVPT = 1024 / kConsumers;  // vectors per thread in the largest unit
  static constexpr uint32_t kAbsentWord = BF16 ? 0xF680F680u : 0xF6800000u;  // -2^110 in every lane

  // Streams vectors [vb, ve) of global row `row` from the ring: units of
  // p.chunk_vec vectors from vb, the last one ragged when the range is not a
  // multiple; an empty range is one empty unit (a row with no full vector).
  // Every consumer thread runs it, and its control flow is warp-uniform: the
  // full units run in a loop specialised on the vectors each thread holds.
  __device__ __forceinline__ void consume(RingPos& rc, int64_t row, int64_t vb, int64_t ve) {
    const int32_t n = static_cast<int32_t>(ve - vb);
    int32_t v = static_cast<int32_t>(vb);
    if (p.chunk_vec == 1024)
      v = full_units<4>(rc, row, v, n / 1024);
    else if (p.chunk_vec == 512)
      v = full_units<2>(rc, row, v, n / 512);
    else
      v = full_units<1>(rc, row, v, n / 256);
    const int32_t rest = static_cast<int32_t>(ve) - v;
    if (rest > 0 || n == 0) {
      const bool sup = has_sup(static_cast<uint32_t>(v) * EPV, static_cast<uint32_t>(v + rest) * EPV);
      wait_stage(rc);
      unit_t<kVPT, false>(ring + rc.slot * chunk_bytes, row, v, rest, sup);
      release_stage(rc);
      rc.advance(p.stages);
    }
  }

  template <int NPT>
  __device__ __forceinline__ int32_t full_units(RingPos& rc, int64_t row, int32_t v, int32_t nfull) {
    constexpr int32_t CV = NPT * kConsumers;
    for (int32_t i = 0; i < nfull; ++i, v += CV) {
      const bool sup = has_sup(static_cast<uint32_t>(v) * EPV, static_cast<uint32_t>(v + CV) * EPV);
      wait_stage(rc);
      unit_t<NPT, true>(ring + rc.slot * chunk_bytes, row, v, CV, sup);
      release_stage(rc);
      rc.advance(p.stages);
    }
    return v;
  }

  // Waits for the unit at ring position r (fast path: every lane sees the
  // phase complete at the first try).
  __device__ __forceinline__ void wait_stage(const RingPos& r) {
    const bool ok = mbar_try_wait(smem_addr(&ctl.full[r.slot]), r.phase);
    if (!__all_sync(0xFFFFFFFFu, ok)) wait_unit_slow(p, ctl, r.slot, r.phase);
  }

  // The warp is done with the unit at ring position r.
  __device__ __forceinline__ void release_stage(const RingPos& r) {
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&ctl.empty[r.slot]));
  }

  // Thread tid holds vectors tid, tid + 256, ... (NPT of them; FULL: all of
  // them exist).  All loads are issued first, the unit's max comes from one
  // max tree (bf16x2 for bf16), the running state is rescaled once without
  // branching, and the sums run on two independent accumulator pairs.
  template <int NPT, bool FULL>
  __device__ __forceinline__ void unit_t(uint32_t base, int64_t row, int32_t v_unit, int32_t nv,
                                         bool unit_has_sup) {
    uint32_t w[NPT][4];
    bool valid[NPT];
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      const int32_t vi = j * kConsumers + tid;
      valid[j] = FULL || vi < nv;
      const uint4 q = valid[j] ? lds128(base + static_cast<uint32_t>(vi) * 16u)
                               : make_uint4(kAbsentWord, kAbsentWord, kAbsentWord, kAbsentWord);
      w[j][0] = q.x;
      w[j][1] = q.y;
      w[j][2] = q.z;
      w[j][3] = q.w;
    }
    // NaN and values <= -2^100 -> -2^100 (the top clamp is applied below,
    // only when the unit holds a value above 2^100).
#pragma unroll
    for (int j = 0; j < NPT; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) w[j][k] = BF16 ? bmax2(w[j][k], kSentinelBf16x2) : sanitize_low_bits(w[j][k]);
    const int32_t id0 = (v_unit + tid) * EPV;  // first id of vector j = 0; vector j adds j * 256 * EPV
    if (__any_sync(0xFFFFFFFFu, unit_has_sup)) {   // the same in every thread
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
        const int32_t v0 = id0 + j * kConsumers * EPV;
        for (int i = 0; i < p.n_sup; ++i) {
          const int32_t off = p.sup[i] - v0;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (BF16) {
              if (off == 2 * k) w[j][k] = (w[j][k] & 0xFFFF0000u) | kAbsentBf16;
              if (off == 2 * k + 1) w[j][k] = (w[j][k] & 0x0000FFFFu) | (kAbsentBf16 << 16);
            } else if (off == k) {
              w[j][k] = __float_as_uint(kAbsent);
            }
          }
        }
      }
    }
    // The plain greedy mode on a full unit needs only the unit's max: one
    // max tree over all its words; the lanes holding a new warp max look for
    // its first vector (rare after the first units: a lane's value below the
    // warp's max can be neither the row's max nor its first index).  The
    // other modes keep every vector's max (the Gumbel bound, the runner-up).
    constexpr bool LEAN = GREEDY && !RUNNER && !GUMBEL && FULL;
    float vmax[NPT];
    float umax;
    if (LEAN) {
      umax = unit_max(w);
    } else {
#pragma unroll
      for (int j = 0; j < NPT; ++j) vmax[j] = valid[j] ? vector_max(w[j]) : kMInit;
      umax = vmax[0];
#pragma unroll
      for (int j = 1; j < NPT; ++j) umax = fmaxf(umax, vmax[j]);
    }
    if (__any_sync(0xFFFFFFFFu, umax > kTopClamp)) {  // rare: +inf or huge logits count as 2^100
#pragma unroll
      for (int j = 0; j < NPT; ++j) {
#pragma unroll
        for (int k = 0; k < 4; ++k) w[j][k] = BF16 ? bmin2(w[j][k], kTopBf16x2) : clamp_top_bits(w[j][k]);
        if (!LEAN) vmax[j] = fminf(vmax[j], kTopClamp);
      }
      umax = fminf(umax, kTopClamp);
    }
    // The warp's running max: every lane's sums take its reference, so they
    // are rescaled only when it grows (every lane of the warp is here).
    const float wmax = warp_max_f32(umax);
    const bool grow = __any_sync(0xFFFFFFFFu, wmax > acc.m);
    float vms[NPT];
    if (LEAN) {
#pragma unroll
      for (int j = 0; j < NPT; ++j) vms[j] = 0.0f;   // unused: no per-vector bound in this mode
      if (grow) {
        // The scaling is monotone: the scaled warp max is the largest scaled
        // value, and a lane holds it when its scaled unit max equals it.
        const float wms = scaled<SCALED>(wmax, s);
        if (scaled<SCALED>(umax, s) == wms && wms > scaled<SCALED>(acc.m, s)) {
          bool found = false;
#pragma unroll
          for (int j = 0; j < NPT; ++j) {
            const bool hit = !found && scaled<SCALED>(vector_max(w[j]), s) == wms;
            if (hit) {
              found = true;
              acc.vm = wms;
              acc.vv = id0 + j * kConsumers * EPV;
#pragma unroll
              for (int k = 0; k < 4; ++k) acc.bw[k] = w[j][k];
            }
          }
        }
      }
    } else {
      // Maxima of the scaled logits z' = z s (the scaling is monotone, so the
      // max of the scaled elements is the scaled max, bit for bit).
#pragma unroll
      for (int j = 0; j < NPT; ++j) vms[j] = !SCALED ? vmax[j] : ((FULL || valid[j]) ? __fmul_rn(vmax[j], s) : kMInit);
      if (GREEDY) {
      // The first vector holding this thread's max (ids increase with j and
      // from unit to unit, so a strict > keeps the earliest), kept with its
      // words; the element inside it is located once per row.  Every other
      // vector's max feeds the runner-up.
#pragma unroll
        for (int j = 0; j < NPT; ++j) {
          const bool better = vms[j] > acc.vm;
          if (RUNNER) acc.m2o = fmaxf(acc.m2o, better ? acc.vm : vms[j]);
          acc.vm = better ? vms[j] : acc.vm;
          acc.vv = better ? id0 + j * kConsumers * EPV : acc.vv;
#pragma unroll
          for (int k = 0; k < 4; ++k) acc.bw[k] = better ? w[j][k] : acc.bw[k];
        }
      }
    }
    gumbel_and_sums<NPT, FULL>(w, valid, vms, wmax, grow, row, id0);
  }

  // The rescale, the sums and (Gumbel modes) the samples of one unit's
  // vectors; vms[j] is vector j's scaled max (unused in the lean mode),
  // wmax the warp's max over the unit, grow whether it is above some lane's
  // running max (a lane already above it keeps its reference).
  template <int NPT, bool FULL>
  __device__ __forceinline__ void gumbel_and_sums(uint32_t (&w)[NPT][4], const bool (&valid)[NPT],
                                                  const float (&vms)[NPT], float wmax, bool grow, int64_t row,
                                                  int32_t id0) {
    if (grow) acc_rescale<SCALED>(acc, fmaxf(acc.m, wmax), s);
    const uint64_t nmc2 = pack2(acc.nref, acc.nref);
    uint64_t Zb = 0, Sb = 0;
#pragma unroll
    for (int j = 0; j < NPT; ++j) {
      if (!FULL && !valid[j]) continue;
#pragma unroll
      for (int e = 0; e < EPV; e += 4) {
        acc_pair2<SCALED>(acc.Z2, acc.S2, elem(w[j], e), elem(w[j], e + 1), nmc2, l2e2, s2);
        acc_pair2<SCALED>(Zb, Sb, elem(w[j], e + 2), elem(w[j], e + 3), nmc2, l2e2, s2);
      }
    }
    acc.Z2 = add2(acc.Z2, Zb);
    acc.S2 = add2(acc.S2, Sb);

    if (GUMBEL) {
      const PhiloxRow pr = philox_row(static_cast<uint32_t>(row),
                                      static_cast<uint32_t>(static_cast<uint64_t>(row) >> 32), p.keys);
      // The pruning floor: the best score any warp of the CTA has seen in
      // this row (a lower bound of the row's winning score; the same in every
      // lane of the warp).
      warp_best = fmaxf(warp_best, key_float(*reinterpret_cast<volatile uint32_t*>(&ctl.cta_best)));
      constexpr int PAIR = NPT >= 2 ? 2 : 1;
#pragma unroll
      for (int j0 = 0; j0 < NPT; j0 += PAIR) {
        GumbelWords r[PAIR];
        bool survive[PAIR];
        // Philox words of the vectors j0 .. j0 + PAIR - 1, generated together
#pragma unroll
        for (int q = 0; q < PAIR; ++q) {
          const int32_t v0 = id0 + (j0 + q) * kConsumers * EPV;
#pragma unroll
          for (int h = 0; h < EPV / 4; ++h) {
            const uint4 o = philox4x32_10_row(static_cast<uint32_t>(v0 >> 2) + h, pr, p.keys);
            r[q].w[4 * h + 0] = o.x;
            r[q].w[4 * h + 1] = o.y;
            r[q].w[4 * h + 2] = o.z;
            r[q].w[4 * h + 3] = o.w;
          }
        }
#pragma unroll
        for (int q = 0; q < PAIR; ++q) {
          const int j = j0 + q;
          uint32_t rmax = r[q].w[0];
#pragma unroll
          for (int e = 1; e < EPV; ++e) rmax = max(rmax, r[q].w[e]);
          // g = -ln(-ln u) <= -ln(1 - u) for every id of the vector; the
          // margin covers the fp32 rounding of ln_p, lg2.approx and the fmaf.
          const float w1 = __fsub_rn(1.0f, uniform_from_bits(rmax));
          const float bound = fmaf(t_ln2, -lg2_approx(w1), vms[j] + fmaf(fabsf(vms[j]), 1e-6f, 1e-3f));
          survive[q] = (FULL || valid[j]) && !(bound < warp_best);
        }
#pragma unroll
        for (int q = 0; q < PAIR; ++q) {
          const int j = j0 + q;
          if (__any_sync(0xFFFFFFFFu, survive[q])) {
            bool updated = false;
            if (survive[q]) {
              VecWords vw;
#pragma unroll
              for (int k = 0; k < 4; ++k) vw.w[k] = w[j][k];
              GumbelBest b{acc.best_s, acc.best_v, acc.best_z};
              b = gumbel_exact<BF16>(b, vw, r[q], id0 + j * kConsumers * EPV, t, t_ln2, warp_best, s);
              updated = b.s > acc.best_s;
              acc.best_s = b.s;
              acc.best_v = b.v;
              acc.best_z = b.z;
            }
            if (__any_sync(0xFFFFFFFFu, updated)) {
              float wb = acc.best_s;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) wb = fmaxf(wb, __shfl_xor_sync(0xFFFFFFFFu, wb, o));
              if (wb > warp_best) {
                warp_best = wb;
                if (lane == 0) atomicMax(&ctl.cta_best, float_key(wb));
              }
            }
          }
        }
      }
    }
  }

  __device__ __forceinline__ static float key_float(uint32_t k) {
    // inverse of float_key
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
  }

  // Element e of a 16-byte vector held as four 32-bit words.
  __device__ __forceinline__ static float elem(const uint32_t (&v)[4], int e) {
    if (BF16) return (e & 1) ? bf16hi(v[e >> 1]) : bf16lo(v[e >> 1]);
    return __uint_as_float(v[e]);
  }

  // The max of all elements of a unit's vectors (sanitized words).
  template <int NPT>
  __device__ __forceinline__ static float unit_max(const uint32_t (&w)[NPT][4]) {
    if (BF16) {
      uint32_t m[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) m[k] = w[0][k];
#pragma unroll
      for (int j = 1; j < NPT; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) m[k] = bmax2(m[k], w[j][k]);
      const uint32_t t = bmax2(bmax2(m[0], m[1]), bmax2(m[2], m[3]));
      return fmaxf(bf16lo(t), bf16hi(t));
    }
    float m[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) m[k] = __uint_as_float(w[0][k]);
#pragma unroll
    for (int j = 1; j < NPT; ++j)
#pragma unroll
      for (int k = 0; k < 4; ++k) m[k] = fmaxf(m[k], __uint_as_float(w[j][k]));
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
  }

  __device__ __forceinline__ static float vector_max(const uint32_t (&v)[4]) {
    if (BF16) {
      const uint32_t m = bmax2(bmax2(v[0], v[1]), bmax2(v[2], v[3]));
      return fmaxf(bf16lo(m), bf16hi(m));
    }
    return fmaxf(fmaxf(__uint_as_float(v[0]), __uint_as_float(v[1])),
                 fmaxf(__uint_as_float(v[2]), __uint_as_float(v[3])));
  }

  // Elements after the last full vector of `row` (V * size % 16 != 0); one
  // element per thread tid < p.tail.
  __device__ void tail(int64_t row) {
    if (p.tail <= 0 || tid >= p.tail) return;
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
    for (int i = 0; i < p.n_sup; ++i)
      if (p.sup[i] == v) z = kAbsent;
    const float zs = SCALED ? __fmul_rn(z, s) : z;
    if (z > acc.m) acc_rescale<SCALED>(acc, z, s);
    acc.idx = static_cast<int32_t>(v);  // one tail element per thread
    acc.vm_tail = zs;
    const float y = fmaf(zs, kLog2e, acc.nref);
    const float e = ex2_approx(y);
    acc.Z2 = add2(acc.Z2, pack2(e, 0.0f));
    acc.S2 = fma2(pack2(e, 0.0f), pack2(y, 0.0f), acc.S2);
    if (GUMBEL) {
      const uint4 o = philox4x32_10(static_cast<uint32_t>(v >> 2), static_cast<uint32_t>(row),
                                    static_cast<uint32_t>(static_cast<uint64_t>(row) >> 32), 0u, p.keys);
      const int w = static_cast<int>(v & 3);
      const uint32_t word = w == 0 ? o.x : (w == 1 ? o.y : (w == 2 ? o.z : o.w));
      const float sc = gumbel_score(zs, t, word);
      if (sc > acc.best_s) {
        acc.best_s = sc;
        acc.best_v = static_cast<int32_t>(v);
        acc.best_z = z;   // the raw logit (prob forms its exponent as the sums did)
      }
    }
  }

  // Greedy x0 bookkeeping: the first id holding this thread's max acc.m.  It
  // is in the best full vector (whose sanitized words the thread kept; its
  // ids are below every tail element) unless the tail element is larger.
  // The thread's runner-up is the largest of its other vectors' maxima, the
  // best vector's other elements and the tail element, whichever is not idx.
  __device__ void resolve_index() {
    if (!GREEDY) return;
    int32_t idx = 0x7FFFFFFF;
    float r2 = RUNNER ? acc.m2o : kMInit;
    const float ms = SCALED ? __fmul_rn(acc.m, s) : acc.m;   // the thread's scaled max
    if (acc.vv >= 0 && acc.vm == ms) {
      bool found = false;
#pragma unroll
      for (int e = 0; e < EPV; ++e) {
        const float ze = SCALED ? __fmul_rn(elem(acc.bw, e), s) : elem(acc.bw, e);
        if (!found && ze == acc.vm) {
          idx = acc.vv + e;
          found = true;
        } else if (RUNNER) {
          r2 = fmaxf(r2, ze);
        }
      }
      if (RUNNER) r2 = fmaxf(r2, acc.vm_tail);
    } else if (acc.vm_tail == ms && acc.m > kMInit) {
      idx = acc.idx;
      if (RUNNER) r2 = fmaxf(r2, acc.vm);
    } else if (RUNNER) {
      // None of the thread's ids holds the max its sums are taken against
      // (the warp's): all of them are "other" ids, and the runner-up field
      // carries the largest (see part_combine).
      r2 = fmaxf(acc.vm, acc.vm_tail);
    }
    acc.idx = idx;
    acc.m2o = r2;
  }

  // Whether suppressed ids fall in [lo, hi) (the same answer in every
  // thread).  The loops ask for ranges of one row in increasing order, so a
  // cursor walks the sorted list: one parameter read per suppressed id per
  // row, not one per range (an indexed parameter read costs hundreds of
  // cycles).  reset() restarts it for the next row.
  int32_t sup_i;
  uint32_t sup_next;   // ids are below V <= 2^31 - 1, and unit ends below 2^31 + 2^13
  __device__ void sup_restart() {
    sup_i = 0;
    sup_next = p.n_sup > 0 ? static_cast<uint32_t>(p.sup[0]) : 0xFFFFFFFFu;
  }
  __device__ bool has_sup(uint32_t lo, uint32_t hi) {
    while (sup_next < lo) sup_next = (++sup_i < p.n_sup) ? static_cast<uint32_t>(p.sup[sup_i]) : 0xFFFFFFFFu;
    return sup_next < hi;
  }

  // The CTA's reduction of all consumer states; valid in thread 0.  When
  // every lane of a warp holds the same max (the usual case: the lanes share
  // the warp's running max), the warp's combine is plain sums and the least
  // index, bit for bit what part_combine gives for equal maxima.
  __device__ Partial cta_reduce() {
    Partial part = acc_to_partial<RUNNER>(acc);
    if (!GUMBEL && !RUNNER && __all_sync(0xFFFFFFFFu, part.m == __shfl_sync(0xFFFFFFFFu, part.m, 0))) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        part.Z = part.Z + __shfl_xor_sync(0xFFFFFFFFu, part.Z, o);
        part.S2 = part.S2 + __shfl_xor_sync(0xFFFFFFFFu, part.S2, o);
      }
      part.idx = static_cast<int32_t>(__reduce_min_sync(0xFFFFFFFFu, static_cast<uint32_t>(part.idx)));
    } else {
      part = warp_combine<MODE>(part, s);
    }
    if (lane == 0) ctl.warp_part[warp] = part;
    named_sync(1, kConsumers);
    Partial r = empty_partial();
    if (warp == 0) {
      if (lane < kConsumerWarps) r = ctl.warp_part[lane];
#pragma unroll
      for (int o = kConsumerWarps / 2; o > 0; o >>= 1) {
        const Partial q = shfl_partial<MODE>(r, o);
        part_combine<MODE>(r, q, s);
      }
    }
    return r;
  }

  // Runs the sorting rule of batch row b in this CTA's consumer warps.
  __device__ void rule_if_needed(int32_t b, uint8_t* rule_smem) {
    if (b < 0) return;
    RuleScratch rs;
    rs.keys = reinterpret_cast<uint64_t*>(rule_smem);
    rs.flags = rule_smem + static_cast<size_t>(kFusedSortCap) * 8;
    rs.red64 = ctl.rule_red64;
    rs.red32 = ctl.rule_red32;
    rs.cap = kFusedSortCap;
    __threadfence();
    run_rule<kConsumers, 1>(p.rule, b, rs, tid);
  }
};

// Producer: issues the bulk copies of this CTA's n units in order; next(src,
// bytes) yields each unit's global address and size.  Returns when every
// issued copy has landed (or, after a fault, when the drain deadline passes).
// drop_first (tests only): the first unit's copy is not issued and its stage
// not arrived on, so the consumers' bounded wait for it runs out.
template <typename Next>
__device__ void produce(const StatsParams& p, SharedCtl& ctl, uint32_t ring, uint32_t chunk_bytes, int64_t n,
                        Next next, bool drop_first = false) {
  volatile int32_t* abort_flag = &ctl.abort_flag;
  const int stages = p.stages;
  RingPos r;
  int64_t issued = 0;
  for (int64_t i = 0; i < n; ++i) {
    if (i >= stages) {  // wait until the consumers released this stage's previous unit
      if (!mbar_wait_bounded(smem_addr(&ctl.empty[r.slot]), r.phase ^ 1u) || *abort_flag) {
        if (!*abort_flag) {
          atomicExch(p.fault, kFaultEmptyWait);
          *abort_flag = 1;
        }
        break;
      }
    }
    const uint8_t* src;
    uint32_t bytes;
    next(src, bytes);
    const uint32_t bar = smem_addr(&ctl.full[r.slot]);
    if (i == 0 && drop_first) {
      // nothing issued, nothing arrived: this stage never completes
    } else if (bytes > 0) {
      mbar_arrive_expect_tx(bar, bytes);
      bulk_copy_g2s(ring + r.slot * chunk_bytes, src, bytes, bar);
    } else {
      mbar_arrive(bar);
    }
    issued = i + 1;
    r.advance(stages);
  }
  // Drain: the last (up to `stages`) issued copies must land before exit.
  const long long t0 = clock64();
  for (int64_t i = (issued > stages ? issued - stages : 0); i < issued; ++i) {
    if (i == 0 && drop_first) continue;   // never issued
    const int slot = static_cast<int>(i % stages);
    const uint32_t par = static_cast<uint32_t>((i / stages) & 1);
    while (!mbar_try_wait_sleep(smem_addr(&ctl.full[slot]), par, kSleepHintNs)) {
      if (clock64() - t0 > kWaitLimitCycles) {
        atomicExch(p.fault, kFaultDrainWait);
        return;
      }
    }
  }
}

__device__ __forceinline__ void init_barriers(SharedCtl& ctl, int stages) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_addr(&ctl.full[s]), 1);
      mbar_init(smem_addr(&ctl.empty[s]), kConsumerWarps);
    }
    ctl.abort_flag = 0;
    ctl.cta_best = float_key(-__int_as_float(0x7F800000));
    fence_mbar_init();
  }
}


// CTAs per SM each kernel is compiled for: three for the plain greedy mode
// (its per-thread state fits 72 registers without spilling, and three rings
// of 64 KB fit the SM's shared memory), two for the modes that track more.
__host__ __device__ constexpr int min_ctas_per_sm(int mode) { return mode == 0 ? 3 : 2; }

// ---------------------------------------------------------------------------
// Persistent kernel: many rows.  CTA c owns units [c U / P, (c+1) U / P).
// ---------------------------------------------------------------------------
template <bool BF16, int MODE>
__global__ void __launch_bounds__(kThreads, min_ctas_per_sm(MODE)) stats_kernel(const __grid_constant__ StatsParams p) {
  extern __shared__ __align__(128) uint8_t dsmem[];
  __shared__ SharedCtl ctl;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int64_t c = blockIdx.x;
  const int64_t u_begin = unit_start(c, p.U, p.P);
  const int64_t u_end = unit_start(c + 1, p.U, p.P);
  const int64_t n_units = u_end - u_begin;
  const uint32_t chunk_bytes = static_cast<uint32_t>(p.chunk_vec) * 16u;
  const uint32_t ring = smem_addr(dsmem);

  pdl_launch_dependents();   // the next kernel may launch now: it waits for this one before reading its outputs
  init_barriers(ctl, p.stages);
  __syncthreads();
  if (!p.early) pdl_wait();   // inputs may come from the previous kernel in the stream

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      int64_t prow = u_begin / p.K, puk = u_begin - prow * p.K;
      produce(p, ctl, ring, chunk_bytes, n_units, [&](const uint8_t*& src, uint32_t& bytes) {
        const int64_t v0 = puk * p.chunk_vec;
        int64_t nv = p.nvec - v0;
        nv = nv < p.chunk_vec ? nv : p.chunk_vec;
        nv = nv > 0 ? nv : 0;
        src = p.logits + prow * p.row_bytes + v0 * 16;
        bytes = static_cast<uint32_t>(nv) * 16u;
        if (++puk == p.K) {
          puk = 0;
          ++prow;
        }
      }, p.test_drop != 0 && blockIdx.x == 0);
    }
    return;
  }

  Consumer<BF16, MODE> con(p, ctl, ring, chunk_bytes);
  uint8_t* rule_smem = dsmem + static_cast<size_t>(p.stages) * chunk_bytes;
  volatile int32_t* abort_flag = &ctl.abort_flag;
  bool first_segment = true;
  bool waited = !p.early;

  auto flush = [&](int64_t row, int64_t uk0, int64_t uk1) {
    if (!waited) {
      pdl_wait();  // nothing is written before the previous kernel has finished
      waited = true;
    }
    con.resolve_index();
    const Partial r = con.cta_reduce();
    if (tid == 0) {
      int32_t action = 0;  // 0 nothing, 1 finish r, 2 combine the row's partials
      if (!*abort_flag) {
        if (uk0 == 0 && uk1 == p.K - 1) {
          ctl.result = r;
          action = 1;
        } else {
          const int64_t slot = 2 * c + (first_segment ? 0 : 1);
          store_partial(p.partials + slot, r);
          __threadfence();
          const int32_t add = static_cast<int32_t>(uk1 - uk0 + 1);
          if (atomicAdd(p.row_count + row, add) + add == p.K) {
            __threadfence();
            action = 2;
          }
        }
      }
      ctl.flag = action;
    }
    named_sync(1, kConsumers);
    const int32_t action = ctl.flag;
    if (action == 2 && warp == 0) {
      // last contributor: warp 0 loads the row's partials in parallel
      const int64_t c0 = cta_of_unit(row * p.K, p.U, p.P);
      const int64_t c1 = cta_of_unit(row * p.K + p.K - 1, p.U, p.P);
      const bool c0_tail = unit_start(c0, p.U, p.P) < row * p.K;
      Partial tot = empty_partial();
      for (int64_t cb = c0; cb <= c1; cb += 32) {
        const int64_t cc = cb + lane;
        Partial q = empty_partial();
        if (cc <= c1) q = load_partial(p.partials + 2 * cc + ((cc == c0 && c0_tail) ? 1 : 0));
        part_combine<MODE>(tot, q, p.scale);
      }
      tot = warp_combine<MODE>(tot, p.scale);
      if (lane == 0) {
        p.row_count[row] = 0;
        ctl.result = tot;
      }
    }
    if (warp == 0) {
      __syncwarp();   // ctl.result, when lane 0 of this warp wrote it
      int32_t rule_b = -1;
      if (action != 0) {
        RowOut o = row_out<MODE>(p, ctl.result);
        if (__shfl_sync(0xFFFFFFFFu, o.exotic ? 1 : 0, 0)) o = exotic_row<BF16, MODE>(p, row, lane);
        if (lane == 0) rule_b = finish_row(p, row, o, RowPre());
      }
      if (lane == 0) {
        ctl.flag2 = rule_b;
        ctl.cta_best = float_key(kNegInf);  // the next row starts with no pruning floor
      }
    }
    named_sync(1, kConsumers);
    con.rule_if_needed(ctl.flag2, rule_smem);
    first_segment = false;
  };

  // Row segments: units [uk0, uk1) of one row each.
  RingPos rc;
  for (int64_t u = u_begin; u < u_end;) {
    const int64_t row = u / p.K, uk0 = u - row * p.K;
    const int64_t uk1 = (u_end - row * p.K) < p.K ? (u_end - row * p.K) : p.K;
    con.reset();
    const int64_t ve = uk1 * p.chunk_vec;
    con.consume(rc, row, uk0 * p.chunk_vec, ve < p.nvec ? ve : p.nvec);
    if (uk1 == p.K && !*abort_flag) con.tail(row);
    flush(row, uk0, uk1 - 1);
    u = row * p.K + uk1;
  }
}

// ---------------------------------------------------------------------------
// Cluster kernel: few rows.  Cluster `row` of p.cluster CTAs reduces one row;
// CTA rank k owns vectors [k nvec / S, (k+1) nvec / S) (and rank S-1 the
// tail).  Rank 0 combines the CTAs' partials through distributed shared
// memory and finishes the row.
// ---------------------------------------------------------------------------
template <bool BF16, int MODE>
__global__ void __launch_bounds__(kThreads, min_ctas_per_sm(MODE)) stats_cluster_kernel(const __grid_constant__ StatsParams p) {
  extern __shared__ __align__(128) uint8_t dsmem[];
  __shared__ SharedCtl ctl;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int S = p.cluster;
  const uint32_t rank = cluster_rank();
  const int64_t row = blockIdx.x / S;
  const int64_t vb = (static_cast<int64_t>(rank) * p.nvec) / S;
  const int64_t ve = (static_cast<int64_t>(rank + 1) * p.nvec) / S;
  const int64_t n_units = (ve - vb + p.chunk_vec - 1) / p.chunk_vec;
  const uint32_t chunk_bytes = static_cast<uint32_t>(p.chunk_vec) * 16u;
  const uint32_t ring = smem_addr(dsmem);

  pdl_launch_dependents();   // the next kernel may launch now: it waits for this one before reading its outputs
  init_barriers(ctl, p.stages);
  __syncthreads();
  if (!p.early) pdl_wait();

  int32_t rule_b = -1;
  if (warp == kConsumerWarps) {
    if (lane == 0) {
      int64_t pv = vb;
      produce(p, ctl, ring, chunk_bytes, n_units, [&](const uint8_t*& src, uint32_t& bytes) {
        int64_t nv = ve - pv;
        nv = nv < p.chunk_vec ? nv : p.chunk_vec;
        src = p.logits + row * p.row_bytes + pv * 16;
        bytes = static_cast<uint32_t>(nv) * 16u;
        pv += p.chunk_vec;
      }, p.test_drop != 0 && blockIdx.x == 0);
    }
    __syncwarp();
    cluster_sync_all();  // partials published
    // second barrier: rank 0 has read them (rank 0 itself only arrives)
    if (rank == 0)
      cluster_arrive();
    else
      cluster_sync_all();
    return;
  }

  Consumer<BF16, MODE> con(p, ctl, ring, chunk_bytes);
  // Rank 0 finishes the row; its candidate flag and canvas token are loaded
  // now so they are at hand then (after the grid dependency in early mode).
  RowPre pre;
  // In early mode the candidate mask is an input like the logits; only a
  // canvas (which steps rewrite) waits for the previous kernel.
  const bool reads_canvas = p.rule.canvas != nullptr && (p.rule.edit || p.rule.cand == nullptr);
  if (rank == 0 && tid == 0 && (!p.early || !reads_canvas)) pre = load_row_pre(p, row);
  RingPos rc;
  con.consume(rc, row, vb, ve);
  if (rank == static_cast<uint32_t>(S - 1) && !ctl.abort_flag) con.tail(row);
  con.resolve_index();
  const Partial r = con.cta_reduce();
  if (tid == 0) ctl.result = r;
  __syncwarp();
  cluster_sync_all();
  if (rank == 0) {
    // Read the cluster's partials, then release the other CTAs at once (they
    // exit and free their SM slots while rank 0 finishes the row).
    Partial tot = empty_partial();
    if (warp == 0)
      for (int k = lane; k < S; k += 32) part_combine<MODE>(tot, load_partial_dsmem(&ctl.result, k), p.scale);
    __syncwarp();
    cluster_arrive();
    RowOut o{};
    if (warp == 0) {
      o = row_out<MODE>(p, warp_combine<MODE>(tot, p.scale));
      if (__shfl_sync(0xFFFFFFFFu, o.exotic ? 1 : 0, 0)) o = exotic_row<BF16, MODE>(p, row, lane);
    }
    // Everything above touched only this cluster's own memory.  In early mode
    // the wait for the previous kernel comes here, so that only the row's
    // writes (outputs, canvas, batch-row counters) follow that kernel's end.
    if (p.early) {
      pdl_wait();
      if (tid == 0 && !pre.have) pre = load_row_pre(p, row);
    }
    if (tid == 0) rule_b = ctl.abort_flag ? -1 : finish_row(p, row, o, pre);
  } else {
    __syncwarp();
    cluster_sync_all();
    return;
  }
  {
    if (tid == 0) ctl.flag2 = rule_b;
    named_sync(1, kConsumers);
    con.rule_if_needed(ctl.flag2, dsmem + static_cast<size_t>(p.stages) * chunk_bytes);
  }
}

// ---------------------------------------------------------------------------
// Batch-row kernel: the fused step when the inputs are ready before the
// previous kernel ends (DLLM_FLAG_INPUTS_READY) and batch rows are short.
// Cluster b of p.cluster CTAs takes batch row b; CTA rank k reduces rows
// [k L / S, (k+1) L / S) of it, each whole, one after the other, and keeps
// their partials in shared memory.  Rank 0 gathers the L partials through
// distributed shared memory, finishes every row and runs the batch row's
// rule on shared-memory copies of the statistics, so that no CTA depends on
// another through global memory: after the grid dependency it only loads
// the canvas (when a rule needs it) and stores.  (The row-cluster kernel
// instead publishes each row with a release-acquire atomic, which puts two
// L2 round trips into every step's serial chain.)
// ---------------------------------------------------------------------------
// A row's inputs to the rule, as rank 0 holds them in shared memory.
struct SharedRowSrc {
  const float* c;
  const float* h;
  const int32_t* x;
  const uint8_t* cd;
  const int32_t* tk;
  __device__ bool cand(int64_t l, int32_t* tok) const {
    *tok = tk[l];
    return cd[l] != 0;
  }
  __device__ float conf(int64_t l) const { return c[l]; }
  __device__ float entropy(int64_t l) const { return h[l]; }
  __device__ int32_t x0(int64_t l) const { return x[l]; }
};

// The rule's decisions kept in shared memory (bit 0 commit, bit 1 edit; the
// counts in three ints), to be stored once the grid dependency allows.
struct SharedEmit {
  uint8_t* flags;
  int32_t* cnt;
  __device__ void operator()(int64_t l, bool commit, bool edit, int32_t) const {
    flags[l] = static_cast<uint8_t>((commit ? 1 : 0) | (edit ? 2 : 0));
  }
  __device__ void counts(int n_cand, int n_commit, int n_edit) const {
    cnt[0] = n_cand;
    cnt[1] = n_commit;
    cnt[2] = n_edit;
  }
};

template <bool BF16, int MODE>
__global__ void __launch_bounds__(kThreads, min_ctas_per_sm(MODE)) stats_batch_kernel(const __grid_constant__ StatsParams p) {
  extern __shared__ __align__(128) uint8_t dsmem[];
  __shared__ SharedCtl ctl;
  __shared__ Partial row_part[kBatchMaxRowsPerCta];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int S = p.cluster;
  const uint32_t rank = cluster_rank();
  const int64_t b = blockIdx.x / S;
  const int64_t L = p.L;
  const int64_t l0 = (static_cast<int64_t>(rank) * L) / S;
  const int64_t l1 = (static_cast<int64_t>(rank + 1) * L) / S;
  const int64_t n_units = (l1 - l0) * p.K;
  const uint32_t chunk_bytes = static_cast<uint32_t>(p.chunk_vec) * 16u;
  const uint32_t ring = smem_addr(dsmem);

  pdl_launch_dependents();   // the next kernel may launch now: it waits for this one before reading its outputs
  init_barriers(ctl, p.stages);
  __syncthreads();
  if (!p.early) pdl_wait();

  if (warp == kConsumerWarps) {
    if (lane == 0) {
      int64_t prow = b * L + l0, puk = 0;
      produce(p, ctl, ring, chunk_bytes, n_units, [&](const uint8_t*& src, uint32_t& bytes) {
        const int64_t v0 = puk * p.chunk_vec;
        int64_t nv = p.nvec - v0;
        nv = nv < p.chunk_vec ? nv : p.chunk_vec;
        nv = nv > 0 ? nv : 0;
        src = p.logits + prow * p.row_bytes + v0 * 16;
        bytes = static_cast<uint32_t>(nv) * 16u;
        if (++puk == p.K) {
          puk = 0;
          ++prow;
        }
      }, p.test_drop != 0 && blockIdx.x == 0);
    }
    __syncwarp();
    cluster_sync_all();  // row partials published
    if (rank == 0)
      cluster_arrive();
    else
      cluster_sync_all();  // rank 0 has read them
    return;
  }

  Consumer<BF16, MODE> con(p, ctl, ring, chunk_bytes);
  volatile int32_t* abort_flag = &ctl.abort_flag;
  // When no canvas is read, the candidate flags come from the candidate mask
  // (or none), an input like the logits: rank 0 loads its row's flag now, so
  // that the load's latency hides behind the stream.
  const RuleArgs& a = p.rule;
  const bool reads_canvas = a.canvas != nullptr && (a.edit || a.cand == nullptr);
  bool pre_cand = false;
  if (rank == 0 && tid < L && !reads_canvas) {
    int32_t unused_tok;   // 0: no canvas is read
    pre_cand = is_candidate(a, b, tid, &unused_tok);
  }
  RingPos rc;
  for (int64_t j = 0; j < l1 - l0; ++j) {
    const int64_t row = b * L + l0 + j;
    con.reset();
    con.consume(rc, row, 0, p.nvec);
    if (!*abort_flag) con.tail(row);
    con.resolve_index();
    const Partial r = con.cta_reduce();
    if (tid == 0) {
      row_part[j] = r;
      ctl.cta_best = float_key(kNegInf);  // the next row starts with no pruning floor
    }
    named_sync(1, kConsumers);  // warp_part is free again before the next row's reduction
  }
  __syncwarp();
  cluster_sync_all();
  if (rank != 0) {
    __syncwarp();
    cluster_sync_all();
    return;
  }

  // Rank 0.  Every bulk copy of this CTA has landed (the producer drained
  // before the cluster barrier), so the ring holds the rule's inputs now.
  float* s_conf = reinterpret_cast<float*>(dsmem);
  float* s_ent = s_conf + kBatchMaxL;
  int32_t* s_x0 = reinterpret_cast<int32_t*>(s_ent + kBatchMaxL);
  int32_t* s_tok = s_x0 + kBatchMaxL;
  uint8_t* s_cand = reinterpret_cast<uint8_t*>(s_tok + kBatchMaxL);
  uint8_t* s_exotic = s_cand + kBatchMaxL;
  RowOut o{};
  const int64_t t = tid;   // the row this thread finishes (L <= kConsumers)
  if (t < L) {
    const int64_t k = ((t + 1) * S + L - 1) / L - 1;   // the CTA whose range holds row t
    const int64_t j = t - (k * L) / S;
    o = row_out<MODE>(p, load_partial_dsmem(&row_part[j], static_cast<uint32_t>(k)));
    s_exotic[t] = o.exotic ? 1 : 0;
  }
  named_sync(1, kConsumers);
  cluster_arrive();   // the other CTAs may exit: their partials are read
  // Rows the streaming pass does not resolve are recomputed, a warp each.
  for (int64_t e = warp; e < L; e += kConsumerWarps) {
    if (!s_exotic[e]) continue;
    const RowOut q = exotic_row<BF16, MODE>(p, b * L + e, lane);
    if (lane == 0) {
      s_conf[e] = q.prob;
      s_ent[e] = q.H;
      s_x0[e] = q.x0;
      s_tok[e] = q.argmax;
      s_cand[e] = 0;
      *reinterpret_cast<float*>(s_exotic + kBatchMaxL + 4 * e) = q.margin;
    }
  }
  named_sync(1, kConsumers);
  if (t < L && o.exotic) {
    o.prob = s_conf[t];
    o.H = s_ent[t];
    o.x0 = s_x0[t];
    o.argmax = s_tok[t];
    o.margin = *reinterpret_cast<const float*>(s_exotic + kBatchMaxL + 4 * t);
  }
  named_sync(1, kConsumers);
  if (*abort_flag) return;   // a wait ran out (the fault is recorded): write nothing
  // The rule's inputs and decisions.  When the candidates come from the
  // candidate mask (an input like the logits), the whole rule is decided
  // before the grid dependency and only stores follow it; when a canvas
  // supplies candidates or tokens (rewritten by the step before), the canvas
  // is read, and the rule decided, after it.
  uint8_t* s_flags = s_exotic;               // reused: the exotic marks are consumed
  int32_t* s_cnt = reinterpret_cast<int32_t*>(s_exotic + kBatchMaxL);
  RuleScratch rs;
  rs.keys = reinterpret_cast<uint64_t*>(dsmem + static_cast<size_t>(p.stages) * chunk_bytes);
  rs.flags = dsmem + static_cast<size_t>(p.stages) * chunk_bytes + static_cast<size_t>(kFusedSortCap) * 8;
  rs.red64 = ctl.rule_red64;
  rs.red32 = ctl.rule_red32;
  rs.cap = kFusedSortCap;
  auto decide = [&]() {
    int32_t tok = 0;
    bool cand = false;
    if (t < L) {
      cand = reads_canvas ? is_candidate(a, b, t, &tok) : pre_cand;
      s_conf[t] = o.prob;
      s_ent[t] = o.H;
      s_x0[t] = o.x0;
      s_tok[t] = tok;
      s_cand[t] = cand ? 1 : 0;
    }
    named_sync(1, kConsumers);
    run_rule_src<kConsumers, 1>(a, b, rs, tid, SharedRowSrc{s_conf, s_ent, s_x0, s_cand, s_tok},
                                SharedEmit{s_flags, s_cnt});
  };
  if (!reads_canvas) decide();
  if (p.early) pdl_wait();
  if (reads_canvas) decide();
  if (t < L) {
    const int64_t row = b * L + t;
    p.x0[row] = o.x0;
    p.prob[row] = o.prob;
    p.entropy[row] = o.H;
    if (p.margin) p.margin[row] = o.margin;
    if (p.argmax) p.argmax[row] = o.argmax;
    const uint8_t f = s_flags[t];
    if (a.commit) a.commit[row] = f & 1;
    if (a.edit_mask) a.edit_mask[row] = (f >> 1) & 1;
    if (f != 0 && a.canvas) a.canvas[b * a.canvas_stride + a.canvas_offset + t] = o.x0;
  }
  if (tid == 0 && a.counts) {
    a.counts[3 * b + 0] = s_cnt[0];
    a.counts[3 * b + 1] = s_cnt[1];
    a.counts[3 * b + 2] = s_cnt[2];
  }
}

// Kernel entry of (dtype, mode, grid kind) as a launchable pointer.
template <bool BF16, int MODE>
const void* stats_entry(int kind) {
  if (kind == kGridCluster) return reinterpret_cast<const void*>(&stats_cluster_kernel<BF16, MODE>);
  if (kind == kGridBatch) return reinterpret_cast<const void*>(&stats_batch_kernel<BF16, MODE>);
  return reinterpret_cast<const void*>(&stats_kernel<BF16, MODE>);
}

}  // namespace dllm
