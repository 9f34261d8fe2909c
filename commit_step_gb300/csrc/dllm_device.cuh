// dllm_device.cuh -- device helpers shared by the libdllmcommit kernels
// (sm_103a): PTX wrappers for the bulk-copy pipeline, bounded mbarrier waits,
// packed fp32 arithmetic, order-preserving float keys and reductions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace dllm {

// Fault codes a kernel writes into the workspace fault word.
enum : int32_t {
  kFaultNone = 0,
  kFaultFullWait = 1,   // a consumer gave up waiting for a bulk copy
  kFaultEmptyWait = 2,  // the producer gave up waiting for a free stage
  kFaultDrainWait = 3,  // the final drain of in-flight copies gave up
};

// A bulk-copy wait that has not completed after this many SM clock cycles
// (about 1 s at 2 GHz) is treated as a fault: the kernel records it and stops
// instead of waiting forever.  The SM-local cycle counter is cheap to read,
// unlike the global timer.
constexpr long long kWaitLimitCycles = 2000ll * 1000ll * 1000ll;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread sleeps in hardware until the phase
// completes or about `hint_ns` pass, instead of spinning and taking issue
// slots from the warps that share its scheduler.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

constexpr uint32_t kSleepHintNs = 200;  // one hardware sleep before the deadline is checked again

// Waits for the phase with the given parity to complete.  Gives up after
// kWaitLimitCycles and returns false; the caller records the fault and stops.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

// One bulk (non-tensor) copy global -> shared, completion counted in bytes on
// the mbarrier.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Programmatic dependent launch.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

// Named barrier among the first `count` threads of the CTA (warps 0..count/32-1).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// The largest of the 32 lanes' values (NaN-free), in every lane; every lane
// of the warp takes part.
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (sm_100+): one instruction for two lanes of arithmetic.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// bf16x2 max; a NaN operand yields the other operand.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Order-preserving map of a float onto uint32 (a < b  <=>  key(a) < key(b)),
// with -0 folded onto +0 so equal values tie.
__device__ __forceinline__ uint32_t float_key(float x) {
  uint32_t b = __float_as_uint(x);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inverse of float_key.
__device__ __forceinline__ float key_to_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Exact sums of entropies (the entropy-bound rule, the stopping criterion):
// fixed point with 40 fractional bits, q(h) = floor(min(max(h, 0), 64) 2^40),
// NaN counting as 64.  The clamped value times 2^40 is exact in fp32 (a
// power-of-two scaling) and below 2^46, so the conversion is exact and sums
// of up to 2^16 values stay below 2^62; integer sums agree in any order.
__device__ __forceinline__ long long fixed_q(float h) {
  const float c = isnan(h) ? 64.0f : fminf(fmaxf(h, 0.0f), 64.0f);
  return __float2ll_rz(c * 0x1p+40f);
}

// A bound compared with such a sum S: S <= bound <=> S <= floor(bound 2^40);
// -1 for a negative bound; bounds above 2^22 (beyond any sum) count as 2^22.
__device__ __forceinline__ long long fixed_bound(float bound) {
  if (bound < 0.0f) return -1;
  return __float2ll_rz(fminf(bound, 0x1p+22f) * 0x1p+40f);
}

// The streaming statistics read NaN and values <= -2^100 as this sentinel and
// clamp values above 2^100 to 2^100; in every row they finish themselves
// (maximum within about 1.8e8 of zero) that reading equals the plain softmax,
// and other rows are recomputed from the logits as they are.
constexpr float kSentinel = -0x1p+100f;
// Suppressed ids become this (no mass, never chosen).  Its product with the
// largest exponent scale (256 log2 e) stays finite, so 2^y y is 0, not NaN.
constexpr float kAbsent = -0x1p+110f;
constexpr uint32_t kSentinelBf16x2 = 0xF180F180u;  // two bf16 -2^100
constexpr uint32_t kAbsentBf16 = 0xF680u;           // bf16 -2^110
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

}  // namespace dllm
