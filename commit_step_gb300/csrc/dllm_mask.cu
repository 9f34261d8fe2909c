// dllm_mask.cu -- block_causal_mask on the device.
//
// mlx-arsenal "dLLM block decoding", "What mlx-arsenal ships" (the attention
// helper) and "Mask conventions": the mask block-diffusion models are trained
// with -- bidirectional inside a block, causal across blocks, blocks aligned
// on absolute positions -- as an additive mask (0 attend, -inf blocked), or as
// the 0/1 keep mask that boolean-mask runtimes read.
//
// Row i of the mask (query at absolute position q_offset + i) attends to the
// keys j < jlim = (floor((q_offset + i) / block_len) + 1) block_len -
// k_offset, so each row is one run of "attend" and one run of "blocked".
// Block b of the grid writes chunk c of row i (b = i * chunks_per_row + c),
// kMaskChunkVec 16-byte vectors with consecutive threads on consecutive
// vectors; the blocks running at once therefore cover one contiguous window
// of rows and the writes reach DRAM in address order, as a plain fill's do.
// Pure HBM writes.
#include <cuda_runtime.h>

#include <cstdint>

#include "dllm_device.cuh"

namespace dllm {

constexpr int kMaskThreads = 256;
constexpr int kMaskChunkVec = 4 * kMaskThreads;   // vectors per block: 16 KiB

// ES: element size (4 fp32, 2 bf16, 1 uint8).  attend_bits / block_bits: the
// element's bit pattern for an allowed / a blocked pair.  vec: rows are
// 16-byte aligned (base and stride), so whole vectors can be stored; the
// elements past a row's last whole vector (all of them when vec is 0) are
// stored one by one by the block holding the row's last chunk.
template <int ES>
__global__ void __launch_bounds__(kMaskThreads) mask_kernel(int64_t Lq, int64_t Lk, int64_t q_offset,
                                                             int64_t k_offset, int64_t block_len, uint8_t* out,
                                                             int64_t row_bytes, uint32_t attend_bits,
                                                             uint32_t block_bits, int vec, int64_t chunks_per_row) {
  constexpr int EPV = 16 / ES;
  pdl_wait();
  pdl_launch_dependents();
  const int64_t nvec = vec ? Lk / EPV : 0;  // whole vectors of a row
  const int64_t total = Lq * chunks_per_row;
  for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
    const int64_t i = b / chunks_per_row;
    const int64_t c = b - i * chunks_per_row;
    int64_t jlim = ((q_offset + i) / block_len + 1) * block_len - k_offset;
    jlim = jlim < 0 ? 0 : (jlim > Lk ? Lk : jlim);
    uint8_t* row = out + i * row_bytes;
#pragma unroll
    for (int k = 0; k < kMaskChunkVec / kMaskThreads; ++k) {
      const int64_t v = c * kMaskChunkVec + k * kMaskThreads + threadIdx.x;
      if (v < nvec) {
        const int64_t j0 = v * EPV;
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t word = 0;
#pragma unroll
          for (int e = 0; e < 4 / ES; ++e) {
            const int64_t j = j0 + q * (4 / ES) + e;
            word |= (j < jlim ? attend_bits : block_bits) << (8 * ES * e);
          }
          w[q] = word;
        }
        *reinterpret_cast<uint4*>(row + j0 * ES) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    if (c == chunks_per_row - 1) {
      for (int64_t j = nvec * EPV + threadIdx.x; j < Lk; j += kMaskThreads) {
        const uint32_t bits = j < jlim ? attend_bits : block_bits;
        if (ES == 4) *reinterpret_cast<uint32_t*>(row + j * 4) = bits;
        if (ES == 2) *reinterpret_cast<uint16_t*>(row + j * 2) = static_cast<uint16_t>(bits);
        if (ES == 1) row[j] = static_cast<uint8_t>(bits);
      }
    }
  }
}

int mask_chunk_vec() { return kMaskChunkVec; }
int mask_threads() { return kMaskThreads; }

const void* mask_kernel_ptr(int es) {
  if (es == 4) return reinterpret_cast<const void*>(&mask_kernel<4>);
  if (es == 2) return reinterpret_cast<const void*>(&mask_kernel<2>);
  return reinterpret_cast<const void*>(&mask_kernel<1>);
}

}  // namespace dllm
