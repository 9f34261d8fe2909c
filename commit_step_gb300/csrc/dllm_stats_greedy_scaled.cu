// dllm_stats_greedy_scaled.cu -- the statistics kernels of greedy rows, with
// and without the runner-up of the margin (modes 0, 4), on scaled logits.
#include "dllm_stats_kernels.cuh"

namespace dllm {

template __global__ void stats_kernel<false, 8>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 8>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<false, 8>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 8>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 8>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<true, 8>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<false, 12>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 12>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<false, 12>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 12>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 12>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<true, 12>(const __grid_constant__ StatsParams);

const void* stats_kernel_ptr_greedy_scaled(bool bf16, int mode, int kind) {
  switch (mode) {
    case 8: return bf16 ? stats_entry<true, 8>(kind) : stats_entry<false, 8>(kind);
    case 12: return bf16 ? stats_entry<true, 12>(kind) : stats_entry<false, 12>(kind);
    default: return nullptr;
  }
}

}  // namespace dllm
