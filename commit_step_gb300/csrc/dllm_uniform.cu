// dllm_uniform.cu -- the helpers of uniform-noise decoding on the device.
//
// mlx-arsenal "dLLM block decoding", function table (uniform_canvas, renoise,
// StableConfidentStopping) and "Uniform-noise decoding (DiffusionGemma)": the
// canvas starts as uniformly random tokens, the positions a step does not
// accept are re-noised, and a row stops for good once its argmax canvas is
// stable and confident; stopped rows stay frozen.  All three are element- or
// row-wise and tiny next to the statistics pass.
#include <cuda_runtime.h>

#include <cstdint>

#include "dllm_device.cuh"
#include "dllm_gumbel.cuh"

namespace dllm {

// canvas[b, j] = floor(r V / 2^32), r = Philox4x32-10(counter (j >> 2, b lo,
// b hi, 1), key) word j & 3: one Philox call per four tokens.
__global__ void uniform_canvas_kernel(const __grid_constant__ PhiloxSchedule ks, int64_t B, int64_t N, uint32_t V,
                                      int32_t* __restrict__ canvas, int64_t stride) {
  pdl_wait();
  pdl_launch_dependents();
  const int64_t groups = (N + 3) / 4;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < B * groups;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = i / groups, g = i - b * groups;
    const uint4 r = philox4x32_10(static_cast<uint32_t>(g), static_cast<uint32_t>(b),
                                  static_cast<uint32_t>(static_cast<uint64_t>(b) >> 32), 1u, ks);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t j = 4 * g + k;
      if (j < N) canvas[b * stride + j] = static_cast<int32_t>((static_cast<uint64_t>(w[k]) * V) >> 32);
    }
  }
}

// out[b, j] = accepted[b, j] ? sample[b, j] : noise[b, j] (accepted == nullptr:
// sample everywhere), except in rows with frozen[b] != 0, which keep out.
__global__ void renoise_kernel(const int32_t* __restrict__ sample, const uint8_t* __restrict__ accepted,
                               const int32_t* __restrict__ noise, const uint8_t* __restrict__ frozen, int64_t B,
                               int64_t N, int32_t* out) {
  pdl_wait();
  pdl_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < B * N;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    if (frozen && frozen[i / N]) continue;
    out[i] = (!accepted || accepted[i]) ? sample[i] : noise[i];
  }
}

constexpr int kStopThreads = 256;

// One call of the stopping criterion, one CTA per batch row b: the row is
// stable when its argmax canvas equals prev (count[b] >= 0 says prev holds
// a canvas); count[b] counts consecutive stable calls; the row is confident
// when its mean entropy is below the threshold, decided exactly in the fixed
// point of fixed_q (sum_l q(H_l) < L q(threshold): integer sums, so any order
// gives the same answer).  prev takes the canvas; stop[b] = count >=
// stability and confident; done[b] |= stop[b].
__global__ void __launch_bounds__(kStopThreads) stop_kernel(const int32_t* __restrict__ argmax,
                                                             const float* __restrict__ entropy, int64_t L,
                                                             int32_t stability, float threshold, int32_t* prev,
                                                             int32_t* count, uint8_t* stop, uint8_t* done) {
  __shared__ long long part[kStopThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int64_t b = blockIdx.x;
  const int32_t* a = argmax + b * L;
  int32_t* pv = prev + b * L;
  const float* e = entropy + b * L;
  int diff = 0;
  long long sum = 0;
  for (int64_t l = threadIdx.x; l < L; l += kStopThreads) {
    const int32_t v = a[l];
    diff |= v != pv[l] ? 1 : 0;
    pv[l] = v;
    sum += fixed_q(e[l]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = sum;
  const int any_diff = __syncthreads_or(diff);
  if (threadIdx.x == 0) {
    long long total = 0;
    for (int w = 0; w < kStopThreads / 32; ++w) total += part[w];
    const int32_t c = count[b];
    const int32_t nc = (c >= 0 && !any_diff) ? c + 1 : 0;
    count[b] = nc;
    const bool confident = total < static_cast<long long>(L) * fixed_q(threshold);
    const uint8_t st = (nc >= stability && confident) ? 1 : 0;
    if (stop) stop[b] = st;
    if (done && st) done[b] = 1;
  }
}

// The rest of one uniform-noise step after the statistics, one CTA per batch
// row b, in one launch -- the same results as uniform_canvas (key), renoise
// with the done flags as frozen rows, renoise of the argmax (accepted ==
// nullptr, same frozen rows) and the stopping criterion, in that order:
//   if !done[b]: canvas[b, j] = accepted ? sample : noise(j); argmax[b, j] = step_argmax[b, j]
//   then the criterion on argmax[b, :] and entropy[b, :] (prev, count), done[b] |= stop.
__global__ void __launch_bounds__(kStopThreads) uniform_update_kernel(
    const __grid_constant__ PhiloxSchedule ks, const int32_t* __restrict__ sample,
    const uint8_t* __restrict__ accepted, const int32_t* __restrict__ step_argmax, const float* __restrict__ entropy,
    int64_t N, uint32_t V, int32_t stability, float threshold, int32_t* canvas, int32_t* argmax, int32_t* prev,
    int32_t* count, uint8_t* done) {
  __shared__ long long part[kStopThreads / 32];
  pdl_wait();
  pdl_launch_dependents();
  const int64_t b = blockIdx.x;
  const bool frozen = done[b] != 0;
  const int64_t base = b * N;
  int diff = 0;
  long long sum = 0;
  // thread t takes groups of four consecutive positions: one Philox call each
  for (int64_t g = threadIdx.x; g * 4 < N; g += kStopThreads) {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    if (!frozen) {
      const uint4 r = philox4x32_10(static_cast<uint32_t>(g), static_cast<uint32_t>(b),
                                    static_cast<uint32_t>(static_cast<uint64_t>(b) >> 32), 1u, ks);
      w[0] = r.x;
      w[1] = r.y;
      w[2] = r.z;
      w[3] = r.w;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t j = 4 * g + k;
      if (j >= N) break;
      int32_t am = argmax[base + j];
      if (!frozen) {
        const int32_t noise = static_cast<int32_t>((static_cast<uint64_t>(w[k]) * V) >> 32);
        canvas[base + j] = accepted[base + j] ? sample[base + j] : noise;
        am = step_argmax[base + j];
        argmax[base + j] = am;
      }
      diff |= am != prev[base + j] ? 1 : 0;
      prev[base + j] = am;
      sum += fixed_q(entropy[base + j]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = sum;
  const int any_diff = __syncthreads_or(diff);
  if (threadIdx.x == 0) {
    long long total = 0;
    for (int wi = 0; wi < kStopThreads / 32; ++wi) total += part[wi];
    const int32_t c = count[b];
    const int32_t nc = (c >= 0 && !any_diff) ? c + 1 : 0;
    count[b] = nc;
    const bool confident = total < static_cast<long long>(N) * fixed_q(threshold);
    if (nc >= stability && confident) done[b] = 1;
  }
}

const void* uniform_canvas_kernel_ptr() { return reinterpret_cast<const void*>(&uniform_canvas_kernel); }
const void* uniform_update_kernel_ptr() { return reinterpret_cast<const void*>(&uniform_update_kernel); }
const void* renoise_kernel_ptr() { return reinterpret_cast<const void*>(&renoise_kernel); }
const void* stop_kernel_ptr() { return reinterpret_cast<const void*>(&stop_kernel); }

}  // namespace dllm
