// dllm_stats_dispatch.cu -- the launchable statistics kernel of each
// (dtype, mode, grid kind); the kernels live in one translation unit per
// tracking family, so they compile in parallel.
#include "dllm_stats.cuh"

namespace dllm {

const void* stats_kernel_ptr_greedy(bool bf16, int mode, bool cluster);
const void* stats_kernel_ptr_greedy_scaled(bool bf16, int mode, bool cluster);
const void* stats_kernel_ptr_sample(bool bf16, int mode, bool cluster);
const void* stats_kernel_ptr_sample_scaled(bool bf16, int mode, bool cluster);
const void* stats_kernel_ptr_margin(bool bf16, int mode, bool cluster);
const void* stats_kernel_ptr_margin_scaled(bool bf16, int mode, bool cluster);

const void* stats_kernel_ptr(bool bf16, int mode, bool cluster) {
  const bool scaled = mode_scaled(mode);
  switch (mode & 7) {
    case 0:
    case 4:
      return scaled ? stats_kernel_ptr_greedy_scaled(bf16, mode, cluster) : stats_kernel_ptr_greedy(bf16, mode, cluster);
    case 1:
    case 3:
      return scaled ? stats_kernel_ptr_sample_scaled(bf16, mode, cluster) : stats_kernel_ptr_sample(bf16, mode, cluster);
    case 7:
      return scaled ? stats_kernel_ptr_margin_scaled(bf16, mode, cluster) : stats_kernel_ptr_margin(bf16, mode, cluster);
    default:
      return nullptr;
  }
}

}  // namespace dllm
