// dllm_stats_dispatch.cu -- the launchable statistics kernel of each
// (dtype, mode, grid kind); the kernels live in one translation unit per
// tracking family, so they compile in parallel.
#include "dllm_stats.cuh"

namespace dllm {

const void* stats_kernel_ptr_greedy(bool bf16, int mode, int kind);
const void* stats_kernel_ptr_greedy_scaled(bool bf16, int mode, int kind);
const void* stats_kernel_ptr_sample(bool bf16, int mode, int kind);
const void* stats_kernel_ptr_sample_scaled(bool bf16, int mode, int kind);
const void* stats_kernel_ptr_margin(bool bf16, int mode, int kind);
const void* stats_kernel_ptr_margin_scaled(bool bf16, int mode, int kind);

const void* stats_kernel_ptr(bool bf16, int mode, int kind) {
  const bool scaled = mode_scaled(mode);
  switch (mode & 7) {
    case 0:
    case 4:
      return scaled ? stats_kernel_ptr_greedy_scaled(bf16, mode, kind) : stats_kernel_ptr_greedy(bf16, mode, kind);
    case 1:
    case 3:
      return scaled ? stats_kernel_ptr_sample_scaled(bf16, mode, kind) : stats_kernel_ptr_sample(bf16, mode, kind);
    case 7:
      return scaled ? stats_kernel_ptr_margin_scaled(bf16, mode, kind) : stats_kernel_ptr_margin(bf16, mode, kind);
    default:
      return nullptr;
  }
}

}  // namespace dllm
