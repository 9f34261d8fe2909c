// dllm_stats_greedy.cu -- the statistics kernels of greedy rows, with and
// without the runner-up of the margin (modes 0, 4).
#include "dllm_stats_kernels.cuh"

namespace dllm {

template __global__ void stats_kernel<false, 0>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 0>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<false, 0>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 0>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 0>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<true, 0>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<false, 4>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 4>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<false, 4>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 4>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 4>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<true, 4>(const __grid_constant__ StatsParams);

const void* stats_kernel_ptr_greedy(bool bf16, int mode, int kind) {
  switch (mode) {
    case 0: return bf16 ? stats_entry<true, 0>(kind) : stats_entry<false, 0>(kind);
    case 4: return bf16 ? stats_entry<true, 4>(kind) : stats_entry<false, 4>(kind);
    default: return nullptr;
  }
}

}  // namespace dllm
