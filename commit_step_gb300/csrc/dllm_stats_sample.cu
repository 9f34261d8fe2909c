// dllm_stats_sample.cu -- the statistics kernels of Gumbel-max rows: the
// sample alone and the sample with its row's argmax (modes 1, 3).
#include "dllm_stats_kernels.cuh"

namespace dllm {

template __global__ void stats_kernel<false, 1>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 1>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<false, 1>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 1>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 1>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<true, 1>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<false, 3>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 3>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<false, 3>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 3>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 3>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<true, 3>(const __grid_constant__ StatsParams);

const void* stats_kernel_ptr_sample(bool bf16, int mode, int kind) {
  switch (mode) {
    case 1: return bf16 ? stats_entry<true, 1>(kind) : stats_entry<false, 1>(kind);
    case 3: return bf16 ? stats_entry<true, 3>(kind) : stats_entry<false, 3>(kind);
    default: return nullptr;
  }
}

}  // namespace dllm
