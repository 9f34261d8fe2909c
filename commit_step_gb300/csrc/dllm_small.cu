// dllm_small.cu -- the standalone commit-rule, edit and schedule kernels.
//
// One CTA per batch row runs the rule (dllm_rules.cuh); the edit rule and the
// transfer schedule are element-wise.  Sources: mlx-arsenal "dLLM block
// decoding", "What mlx-arsenal ships" (threshold_transfer, topk_transfer,
// factor_transfer, entropy_bound_transfer, edit_transfer, transfer_schedule)
// and "Token editing (LLaDA2.1)"; mojo-dllm manual, "The loop LLaDA uses"
// (even per-step quotas).
#include <cuda_runtime.h>

#include <cstdint>

#include "dllm_device.cuh"
#include "dllm_rules.cuh"

namespace dllm {

template <int NT>
__global__ void __launch_bounds__(NT) rules_kernel(const __grid_constant__ RuleArgs a, int32_t cap) {
  extern __shared__ __align__(16) uint8_t dsmem[];
  __shared__ uint64_t red64[NT / 32];
  __shared__ int32_t red32[4 * (NT / 32)];
  pdl_wait();
  pdl_launch_dependents();
  RuleScratch s;
  s.keys = reinterpret_cast<uint64_t*>(dsmem);
  s.flags = dsmem + static_cast<size_t>(cap) * 8;
  s.red64 = red64;
  s.red32 = red32;
  s.cap = cap;
  run_rule<NT, 0>(a, blockIdx.x, s, threadIdx.x);
}

__global__ void edit_kernel(const int32_t* __restrict__ x0, const float* __restrict__ prob,
                            const int32_t* __restrict__ tokens, const uint8_t* __restrict__ editable,
                            int64_t n, float tau_edit, uint8_t* __restrict__ edit) {
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float p = nan_to(prob[i], -__int_as_float(0x7F800000));
    edit[i] = (editable[i] != 0 && x0[i] != tokens[i] && p > tau_edit) ? 1 : 0;
  }
}

__global__ void schedule_kernel(const int32_t* __restrict__ counts, int64_t B, int32_t steps,
                                int32_t* __restrict__ quotas) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t total = B * steps;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = i / steps;
    const int32_t s = static_cast<int32_t>(i - b * steps);
    const int32_t n = counts[b] > 0 ? counts[b] : 0;
    quotas[i] = n / steps + (s < n % steps ? 1 : 0);
  }
}

const void* rules_kernel_ptr(int nt) {
  switch (nt) {
    case 128: return reinterpret_cast<const void*>(&rules_kernel<128>);
    case 256: return reinterpret_cast<const void*>(&rules_kernel<256>);
    case 512: return reinterpret_cast<const void*>(&rules_kernel<512>);
    default: return reinterpret_cast<const void*>(&rules_kernel<1024>);
  }
}
const void* edit_kernel_ptr() { return reinterpret_cast<const void*>(&edit_kernel); }
const void* schedule_kernel_ptr() { return reinterpret_cast<const void*>(&schedule_kernel); }

}  // namespace dllm
