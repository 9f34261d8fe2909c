// dllm_stats.cuh -- parameters shared by the statistics kernel and its host
// launcher.
#pragma once

#include <cstdint>

#include "../../include/dllmcommit.h"
#include "dllm_gumbel.cuh"
#include "dllm_rules.cuh"

namespace dllm {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;  // threads that reduce the logits
constexpr int kThreads = kConsumers + 32;        // plus one warp that issues the bulk copies
constexpr int kMaxStages = 16;
constexpr int kRingBytes = 64 * 1024;
constexpr int kFusedSortCap = 1024;              // largest L the fused sorting rules take
constexpr int kMaxCtasPerSm = 4;
constexpr int kBatchMaxL = 256;            // L the batch-row kernel takes (one consumer thread per row)
constexpr int kBatchMaxRowsPerCta = 16;    // rows one of its CTAs reduces (L <= 16 S)

// What a row's pass tracks, as bits: kModeSample, a Gumbel-max sample
// (else the greedy argmax); kModeArgmax, the first argmax beside a sample;
// kModeRunner, the runner-up of the argmax (the margin output); kModeScaled,
// a logit scale other than 1 (the unscaled kernels carry no scaling
// arithmetic at all).  The tracking modes built: greedy (0), greedy +
// runner-up (4), sample (1), sample + argmax (3), sample + argmax + runner-up
// (7), each with and without kModeScaled.
enum : int { kModeSample = 1, kModeArgmax = 2, kModeRunner = 4, kModeScaled = 8, kModeSlots = 16 };

__host__ __device__ constexpr bool mode_sample(int m) { return (m & kModeSample) != 0; }
__host__ __device__ constexpr bool mode_argmax(int m) { return !mode_sample(m) || (m & kModeArgmax) != 0; }
__host__ __device__ constexpr bool mode_runner(int m) { return (m & kModeRunner) != 0; }
__host__ __device__ constexpr bool mode_scaled(int m) { return (m & kModeScaled) != 0; }
__host__ __device__ constexpr bool mode_built(int m) {
  return (m & 7) == 0 || (m & 7) == 4 || (m & 7) == 1 || (m & 7) == 3 || (m & 7) == 7;
}

// Grid kinds of the statistics kernel: the persistent grid (many rows), a
// cluster per row (few rows), a cluster per batch row (few short batch rows
// whose inputs are ready early).
enum : int { kGridPersistent = 0, kGridCluster = 1, kGridBatch = 2 };

// Launchable statistics kernels, one per (dtype, mode, grid kind); defined
// in dllm_stats_{greedy,sample,margin}{,_scaled}.cu.
const void* stats_kernel_ptr(bool bf16, int mode, int kind);

// Partial reduction of one row segment, in scaled logits z' = z s: max m,
// Z = sum 2^y and S2 = sum 2^y y with y = (z' - m) log2(e), the first index
// of m, the best Gumbel score with its id and scaled logit, and m2, the
// largest z' of the segment without the element at idx (the runner-up).
struct alignas(16) Partial {
  float m, Z, S2;
  int32_t idx;
  float best_s, best_z;
  int32_t best_v;
  float m2;
};

struct StatsParams {
  const uint8_t* logits;
  int32_t cluster;          // CTAs per row in the cluster kernel (0: persistent kernel)
  int32_t early;            // logits are ready before the previous kernel ends: load before the grid dependency
  int32_t test_drop;        // test only: CTA 0 does not issue its first unit's copy (its consumers' wait runs out)
  int64_t row_bytes;        // row stride in bytes (multiple of 16)
  int64_t T, V, L;
  int64_t nvec;             // full 16-byte vectors per row
  int32_t tail;             // elements after the last full vector
  int32_t chunk_vec;        // vectors per unit (256, 512 or 1024)
  int64_t K, U;             // units per row, units in all
  int32_t P;                // CTAs in the grid
  int32_t stages;           // ring stages
  float temperature;
  float scale;              // logit scale s: every statistic is of z' = fp32(z s)
  PhiloxSchedule keys;      // Philox round keys of the caller's key
  int32_t n_sup;
  int32_t sup[DLLM_MAX_SUPPRESS];  // sorted, distinct
  float ln_veff;
  int32_t* x0;
  float* prob;
  float* entropy;
  float* margin;            // (T) or nullptr: prob(x0) - prob(runner-up)
  int32_t* argmax;          // (T) or nullptr: first id of the largest z'
  int32_t* fault;
  int32_t* row_count;       // (T) contributions that arrived, split rows only
  // (B) per batch row, four 16-bit fields: rows finished | candidates | commits | edits
  unsigned long long* batch_packed;
  unsigned long long* batch_forced;  // (B) max of ~ranking key over candidates: the forced commit
  Partial* partials;        // (2 P)
  int32_t fused;
  RuleArgs rule;
};

}  // namespace dllm
