// dllm_stats_margin.cu -- the statistics kernels of Gumbel-max rows with their
// argmax and its runner-up (mode 7).
#include "dllm_stats_kernels.cuh"

namespace dllm {

template __global__ void stats_kernel<false, 7>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 7>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<false, 7>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 7>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 7>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<true, 7>(const __grid_constant__ StatsParams);

const void* stats_kernel_ptr_margin(bool bf16, int mode, int kind) {
  switch (mode) {
    case 7: return bf16 ? stats_entry<true, 7>(kind) : stats_entry<false, 7>(kind);
    default: return nullptr;
  }
}

}  // namespace dllm
