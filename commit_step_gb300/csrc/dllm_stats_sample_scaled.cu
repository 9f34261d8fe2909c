// dllm_stats_sample_scaled.cu -- the statistics kernels of Gumbel-max rows:
// the sample alone and the sample with its row's argmax (modes 1, 3), on
// scaled logits.
#include "dllm_stats_kernels.cuh"

namespace dllm {

template __global__ void stats_kernel<false, 9>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 9>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<false, 9>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 9>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 9>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<true, 9>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<false, 11>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<false, 11>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<false, 11>(const __grid_constant__ StatsParams);
template __global__ void stats_kernel<true, 11>(const __grid_constant__ StatsParams);
template __global__ void stats_cluster_kernel<true, 11>(const __grid_constant__ StatsParams);
template __global__ void stats_batch_kernel<true, 11>(const __grid_constant__ StatsParams);

const void* stats_kernel_ptr_sample_scaled(bool bf16, int mode, int kind) {
  switch (mode) {
    case 9: return bf16 ? stats_entry<true, 9>(kind) : stats_entry<false, 9>(kind);
    case 11: return bf16 ? stats_entry<true, 11>(kind) : stats_entry<false, 11>(kind);
    default: return nullptr;
  }
}

}  // namespace dllm
