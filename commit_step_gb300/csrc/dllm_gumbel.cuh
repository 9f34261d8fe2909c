// dllm_gumbel.cuh -- the Gumbel-max noise of the statistics pass (device).
//
// The noise of id v in global row `row` is fixed bit for bit:
//   r = Philox4x32-10(counter (v >> 2, row lo, row hi, 0), key (lo, hi))[v & 3]
//   u = (2 (r >> 9) + 1) 2^-24           (exact in fp32, 0 < u < 1)
//   g = -ln_p(-ln_p(u))                  (standard Gumbel)
//   s = fmaf(t, g, z)
// argmax_v s_v samples softmax(z / t): the Gumbel-max trick LLaDA applies at
// temperature > 0 (mojo-dllm manual, "The loop LLaDA uses"; mlx-arsenal "dLLM
// block decoding", "What mlx-arsenal ships": sampling with an explicit key).
//
// Philox4x32-10 is written from Salmon et al., "Parallel random numbers: as
// easy as 1, 2, 3" (SC'11).  ln_p is this project's fp32 logarithm: split
// x = 2^e m with m in (sqrt(1/2), sqrt(2)], then ln m = 2 atanh(s),
// s = (m - 1)/(m + 1), from the odd series s + s^3/3 + ... + s^11/11.  Every
// step is an explicitly rounded fp32 operation, so any IEEE implementation
// of the same steps gives the same bits.
#pragma once

#include <cstdint>

namespace dllm {

struct PhiloxKey {
  uint32_t k0, k1;
};

// The key of each of the ten rounds: round i uses (k0 + i 0x9E3779B9,
// k1 + i 0xBB67AE85) mod 2^32.  Computed once per launch on the host.
struct PhiloxSchedule {
  uint32_t k[10][2];
};

__device__ __forceinline__ void mulhilo(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
  uint64_t p;
  asm("mul.wide.u32 %0, %1, %2;" : "=l"(p) : "r"(a), "r"(b));
  lo = static_cast<uint32_t>(p);
  hi = static_cast<uint32_t>(p >> 32);
}

// Ten Philox rounds on (c0, c1, c2, c3) with a precomputed key schedule.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               const PhiloxSchedule& ks) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    uint32_t hi0, lo0, hi1, lo1;
    mulhilo(0xD2511F53u, c0, hi0, lo0);
    mulhilo(0xCD9E8D57u, c2, hi1, lo1);
    const uint32_t n0 = hi1 ^ c1 ^ ks.k[round][0];
    const uint32_t n2 = hi0 ^ c3 ^ ks.k[round][1];
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
  }
  return make_uint4(c0, c1, c2, c3);
}

// The same generator for counters (x, row lo, row hi, 0) of one row.  The
// words other than x enter only the first two rounds, and there only through
// values that depend on the row alone; those are computed once per row, and
// rounds 0 and 1 take five instructions instead of eight.
struct PhiloxRow {
  uint32_t k01;   // round 0, key word 1
  uint32_t a1k;   // round 0 output word 1, xor round 1 key word 0
  uint32_t b0k;   // high word of round 1's first product, xor round 1 key word 1
  uint32_t b1;    // low word of round 1's first product: round 1 output word 3
};

__device__ __forceinline__ PhiloxRow philox_row(uint32_t lo, uint32_t hi, const PhiloxSchedule& ks) {
  uint32_t h1, l1, h0, l0;
  mulhilo(0xCD9E8D57u, hi, h1, l1);           // round 0, second product (counter word 2 = hi)
  const uint32_t a0 = h1 ^ lo ^ ks.k[0][0];   // round 0 output word 0
  mulhilo(0xD2511F53u, a0, h0, l0);           // round 1, first product
  PhiloxRow r;
  r.k01 = ks.k[0][1];
  r.a1k = l1 ^ ks.k[1][0];
  r.b0k = h0 ^ ks.k[1][1];
  r.b1 = l0;
  return r;
}

__device__ __forceinline__ uint4 philox4x32_10_row(uint32_t x, const PhiloxRow& pr, const PhiloxSchedule& ks) {
  uint32_t h0, l0, h1, l1;
  mulhilo(0xD2511F53u, x, h0, l0);            // round 0, first product (counter word 0 = x)
  const uint32_t c2 = h0 ^ pr.k01;            // round 0 output word 2 (counter word 3 is 0)
  mulhilo(0xCD9E8D57u, c2, h1, l1);           // round 1, second product
  uint32_t c0 = h1 ^ pr.a1k, c1 = l1, c3 = pr.b1;
  uint32_t d2 = pr.b0k ^ l0;                  // round 1 output word 2 (round 0 output word 3 is l0)
#pragma unroll
  for (int round = 2; round < 10; ++round) {
    uint32_t hi0, lo0, hi1, lo1;
    mulhilo(0xD2511F53u, c0, hi0, lo0);
    mulhilo(0xCD9E8D57u, d2, hi1, lo1);
    const uint32_t n0 = hi1 ^ c1 ^ ks.k[round][0];
    const uint32_t n2 = hi0 ^ c3 ^ ks.k[round][1];
    c0 = n0;
    c1 = lo1;
    d2 = n2;
    c3 = lo0;
  }
  return make_uint4(c0, c1, d2, c3);
}

// u = (2 (r >> 9) + 1) 2^-24, built exactly: 1 + k 2^-23 minus (1 - 2^-24)
// (the subtraction is exact by Sterbenz's lemma).
__device__ __forceinline__ float uniform_from_bits(uint32_t r) {
  const float one_plus = __uint_as_float(0x3F800000u | (r >> 9));
  return __fsub_rn(one_plus, 0x1.fffffep-1f);
}

__device__ __forceinline__ float ln_p(float x) {
  const uint32_t bits = __float_as_uint(x);
  int e = static_cast<int>(bits >> 23) - 127;
  float m = __uint_as_float((bits & 0x007FFFFFu) | 0x3F800000u);
  if (m > 0x1.6a09e6p+0f) {  // sqrt(2) in fp32
    m = __fmul_rn(m, 0.5f);
    e += 1;
  }
  const float s = __fdiv_rn(__fsub_rn(m, 1.0f), __fadd_rn(m, 1.0f));
  const float s2 = __fmul_rn(s, s);
  float poly = 0x1.745d18p-4f;                  // 1/11
  poly = __fmaf_rn(poly, s2, 0x1.c71c72p-4f);   // 1/9
  poly = __fmaf_rn(poly, s2, 0x1.24924ap-3f);   // 1/7
  poly = __fmaf_rn(poly, s2, 0x1.99999ap-3f);   // 1/5
  poly = __fmaf_rn(poly, s2, 0x1.555556p-2f);   // 1/3
  const float s3 = __fmul_rn(s, s2);
  const float atanh_s = __fmaf_rn(s3, poly, s);
  return __fmaf_rn(__int2float_rn(e), 0x1.62e430p-1f, __fmul_rn(2.0f, atanh_s));
}

// The Gumbel score of an element whose Philox word is r.
__device__ __forceinline__ float gumbel_score(float z, float t, uint32_t r) {
  const float u = uniform_from_bits(r);
  const float E = -ln_p(u);
  const float g = -ln_p(E);
  return __fmaf_rn(t, g, z);
}

}  // namespace dllm
