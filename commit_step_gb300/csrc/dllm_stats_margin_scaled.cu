// dllm_stats_margin_scaled.cu -- the statistics kernels of Gumbel-max rows
// with their argmax and its runner-up (mode 7), on scaled logits.
#include "dllm_stats_kernels.cuh"

namespace dllm {

template __global__ void stats_kernel<false, 15>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 15>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 15>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 15>(const __grid_constant__ StatsParams);

const void* stats_kernel_ptr_margin_scaled(bool bf16, int mode, bool cluster) {
  switch (mode) {
    case 15: return bf16 ? stats_entry<true, 15>(cluster) : stats_entry<false, 15>(cluster);
    default: return nullptr;
  }
}

}  // namespace dllm
