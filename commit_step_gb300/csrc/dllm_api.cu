// dllm_api.cu -- the C ABI of libdllmcommit (include/dllmcommit.h): argument
// validation, launch planning, workspace layout and kernel launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/dllmcommit.h"
#include "dllm_stats.cuh"

namespace dllm {
const void* rules_kernel_ptr(int nt);
const void* edit_kernel_ptr();
const void* schedule_kernel_ptr();
const void* uniform_canvas_kernel_ptr();
const void* renoise_kernel_ptr();
const void* stop_kernel_ptr();
const void* uniform_update_kernel_ptr();
const void* mask_kernel_ptr(int es);
int mask_chunk_vec();
int mask_threads();
}  // namespace dllm

namespace {

using namespace dllm;

constexpr int kMaxDevices = 64;
constexpr size_t kStatsSmemMax = static_cast<size_t>(kRingBytes) + kFusedSortCap * 9;

struct DeviceInfo {
  int sms = 0;
  // Per kernel variant, index bf16 * kModeSlots + mode: CTAs per SM of
  // stats_kernel, and co-resident clusters of stats_cluster_kernel per
  // cluster size 1, 2, 4, 8, 16.
  int occ[2 * kModeSlots] = {};
  int clusters[2 * kModeSlots][5] = {};
  int batch_clusters[2 * kModeSlots][5] = {};   // co-resident clusters of stats_batch_kernel per size
  cudaError_t err = cudaSuccess;
};

DeviceInfo g_dev[kMaxDevices];
std::once_flag g_once[kMaxDevices];

const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::call_once(g_once[dev], [dev]() {
    DeviceInfo& d = g_dev[dev];
    d.err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    for (int v = 0; v < 2 * kModeSlots && d.err == cudaSuccess; ++v) {
      if (!mode_built(v % kModeSlots)) continue;
      const void* k = stats_kernel_ptr(v >= kModeSlots, v % kModeSlots, kGridPersistent);
      d.err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kStatsSmemMax));
      if (d.err != cudaSuccess) break;
      int n = 0;
      d.err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kThreads, kStatsSmemMax);
      d.occ[v] = std::max(1, std::min(n, kMaxCtasPerSm));
    }
    for (int kind : {kGridCluster, kGridBatch}) {
      for (int v = 0; v < 2 * kModeSlots && d.err == cudaSuccess; ++v) {
        if (!mode_built(v % kModeSlots)) continue;
        const void* k = stats_kernel_ptr(v >= kModeSlots, v % kModeSlots, kind);
        d.err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kStatsSmemMax));
        if (d.err == cudaSuccess) d.err = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        for (int e = 0; e < 5 && d.err == cudaSuccess; ++e) {
          const int S = 1 << e;
          cudaLaunchConfig_t cfg{};
          cfg.gridDim = dim3(S * 64);
          cfg.blockDim = dim3(kThreads);
          cfg.dynamicSmemBytes = kStatsSmemMax;
          cudaLaunchAttribute attr[1];
          attr[0].id = cudaLaunchAttributeClusterDimension;
          attr[0].val.clusterDim.x = S;
          attr[0].val.clusterDim.y = 1;
          attr[0].val.clusterDim.z = 1;
          cfg.attrs = attr;
          cfg.numAttrs = 1;
          int n = 0;
          if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();  // an unsupported size only rules that size out
            n = 0;
          }
          (kind == kGridCluster ? d.clusters : d.batch_clusters)[v][e] = n;
        }
      }
    }
    for (int nt : {128, 256, 512, 1024}) {
      if (d.err != cudaSuccess) break;
      d.err = cudaFuncSetAttribute(rules_kernel_ptr(nt), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   DLLM_MAX_SORT_L * 9);
    }
  });
  const DeviceInfo* d = &g_dev[dev];
  return d->err == cudaSuccess ? d : nullptr;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct WsLayout {
  size_t fault = 0, partials = 0, row_count = 0, batch_packed = 0, batch_forced = 0, total = 0;
};

// Fault word, then the partials (a size fixed per device), then the counters.
// Counters of every shape share one region that only ever holds counters, and
// every successful call returns the counters it used to zero, so a workspace
// serves calls of any shape in turn.
WsLayout ws_layout(int64_t B, int64_t L, int sms) {
  WsLayout w;
  w.fault = 0;
  w.partials = 256;
  w.row_count = w.partials + static_cast<size_t>(2) * sms * kMaxCtasPerSm * sizeof(Partial);
  w.batch_packed = align_up(w.row_count + static_cast<size_t>(B * L) * 4, 8);
  w.batch_forced = w.batch_packed + static_cast<size_t>(B) * 8;
  w.total = align_up(w.batch_forced + static_cast<size_t>(B) * 8, 256);
  return w;
}

struct StatsPlan {
  int64_t nvec, K, U;
  int32_t tail, chunk_vec, P, stages, cluster;
  int32_t kind;   // kGridPersistent, kGridCluster or kGridBatch
};

int chunk_for(int64_t vectors_per_cta) {
  int chunk = 1024;
  while (chunk > 256 && static_cast<int64_t>(4) * chunk > vectors_per_cta) chunk >>= 1;
  return chunk;
}

// Few rows: one cluster of S CTAs per row, the largest S whose whole grid is
// co-resident (one wave) and leaves each CTA at least 128 vectors.  Many
// rows: the persistent grid over equal unit ranges.
StatsPlan plan_stats(const DeviceInfo& d, int variant, int64_t T, int64_t V, int esize, bool overlap) {
  StatsPlan pl{};
  pl.nvec = (V * esize) / 16;
  pl.tail = static_cast<int32_t>(V - pl.nvec * (16 / esize));
  // A call that overlaps the previous launch (DLLM_FLAG_INPUTS_READY) sizes
  // its cluster grid to a quarter of the co-resident CTAs, so that several
  // steps stream at once while earlier ones finish their rows; rows too many
  // for a cluster grid that small take the whole budget before falling back
  // to the persistent grid.
  const int ctas = d.sms * d.occ[variant];
  const int budgets[2] = {overlap ? std::max(1, ctas / 4) : ctas, ctas};
  for (int bi = 0; bi < 2; ++bi)
  for (int e = 4; e >= 1; --e) {
    const int S = 1 << e;
    if (T <= d.clusters[variant][e] && T * S <= budgets[bi] && pl.nvec >= static_cast<int64_t>(S) * 128) {
      pl.cluster = S;
      pl.kind = kGridCluster;
      // slices are equal by construction: favour few, large copies
      const int64_t slice = pl.nvec / S;
      pl.chunk_vec = slice >= 768 ? 1024 : (slice >= 384 ? 512 : 256);
      pl.stages = std::min(kMaxStages, kRingBytes / (pl.chunk_vec * 16));
      pl.P = static_cast<int32_t>(T * S);
      pl.K = 0;
      pl.U = 0;
      return pl;
    }
  }
  const int64_t total_vec = T * std::max<int64_t>(pl.nvec, 1);
  pl.cluster = 0;
  pl.kind = kGridPersistent;
  pl.chunk_vec = chunk_for(total_vec / std::max(ctas, 1));
  pl.stages = std::min(kMaxStages, kRingBytes / (pl.chunk_vec * 16));
  pl.K = pl.nvec > 0 ? (pl.nvec + pl.chunk_vec - 1) / pl.chunk_vec : 1;
  pl.U = T * pl.K;
  pl.P = static_cast<int32_t>(std::min<int64_t>(pl.U, ctas));
  return pl;
}

// The fused step on few short batch rows whose inputs are ready early
// (where the few-rows plan took a cluster per row): one cluster of S CTAs
// per batch row, S the largest power of two <= min(16, L) whose clusters can
// be resident, each CTA taking at most kBatchMaxRowsPerCta whole rows.
bool plan_batch(const DeviceInfo& d, int variant, int64_t B, int64_t L, StatsPlan& pl) {
  if (L > kBatchMaxL || B > INT32_MAX / 16) return false;
  for (int e = 4; e >= 0; --e) {
    const int S = 1 << e;
    if (S > L || d.batch_clusters[variant][e] <= 0) continue;
    if ((L + S - 1) / S > kBatchMaxRowsPerCta) return false;
    pl.kind = kGridBatch;
    pl.cluster = S;
    pl.chunk_vec = pl.nvec >= 3 * 1024 ? 1024 : (pl.nvec >= 3 * 512 ? 512 : 256);
    pl.stages = std::min(kMaxStages, kRingBytes / (pl.chunk_vec * 16));
    pl.K = pl.nvec > 0 ? (pl.nvec + pl.chunk_vec - 1) / pl.chunk_vec : 1;
    pl.U = 0;
    pl.P = static_cast<int32_t>(B * S);
    return true;
  }
  return false;
}

dllm_status launch(const void* kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void** args,
                   int cluster = 0) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  if (cluster > 0) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cfg.attrs = attr;
  return cudaLaunchKernelExC(&cfg, kernel, args) == cudaSuccess ? DLLM_OK : DLLM_ERR_CUDA;
}

int esize_of(dllm_dtype dt) { return dt == DLLM_BF16 ? 2 : 4; }

// a * b for a, b >= 0, or -1 when the product does not fit in int64 (such a
// shape cannot describe memory; the entry points reject it before any other
// arithmetic on it).
int64_t checked_mul(int64_t a, int64_t b) {
  if (a < 0 || b < 0) return -1;
  if (a == 0 || b == 0) return 0;
  return a > INT64_MAX / b ? -1 : a * b;
}

// Shared validation of the statistics arguments; fills the suppress list.
dllm_status check_stats(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V, int64_t row_stride,
                        float temperature, const int32_t* sup, int32_t n_sup, const int32_t* x0, const float* prob,
                        const float* entropy, std::vector<int32_t>& sorted_sup) {
  if (B < 0 || L < 0 || V < 1 || V > INT32_MAX || row_stride < V) return DLLM_ERR_INVALID_ARGUMENT;
  if (dt != DLLM_F32 && dt != DLLM_BF16) return DLLM_ERR_INVALID_ARGUMENT;
  // the logits' byte extent T * row_stride * size must be representable
  if (checked_mul(checked_mul(checked_mul(B, L), row_stride), 4) < 0) return DLLM_ERR_INVALID_ARGUMENT;
  // (0, 2^64]: the streaming pass reads NaN as -2^100, and at these
  // temperatures no noise lifts such an entry above a real logit's score.
  if (!(temperature >= 0.0f) || !(temperature <= 0x1p+64f)) return DLLM_ERR_INVALID_ARGUMENT;
  if (n_sup < 0 || (n_sup > 0 && !sup)) return DLLM_ERR_INVALID_ARGUMENT;
  if (n_sup > DLLM_MAX_SUPPRESS) return DLLM_ERR_UNSUPPORTED;
  sorted_sup.assign(sup, sup + n_sup);
  for (int32_t id : sorted_sup)
    if (id < 0 || id >= V) return DLLM_ERR_INVALID_ARGUMENT;
  std::sort(sorted_sup.begin(), sorted_sup.end());
  sorted_sup.erase(std::unique(sorted_sup.begin(), sorted_sup.end()), sorted_sup.end());
  if (static_cast<int64_t>(sorted_sup.size()) >= V) return DLLM_ERR_INVALID_ARGUMENT;  // empty token set
  if (B * L == 0) return DLLM_OK;
  if (!logits || !x0 || !prob || !entropy) return DLLM_ERR_INVALID_ARGUMENT;
  const int es = esize_of(dt);
  if ((reinterpret_cast<uintptr_t>(logits) & 15u) != 0 || (row_stride * es) % 16 != 0) return DLLM_ERR_UNSUPPORTED;
  return DLLM_OK;
}

// The round keys of Philox4x32-10 for a 64-bit key: round i uses
// (lo + i 0x9E3779B9, hi + i 0xBB67AE85) mod 2^32.
PhiloxSchedule philox_schedule(uint64_t key) {
  PhiloxSchedule ks;
  uint32_t k0 = static_cast<uint32_t>(key), k1 = static_cast<uint32_t>(key >> 32);
  for (int r = 0; r < 10; ++r) {
    ks.k[r][0] = k0;
    ks.k[r][1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return ks;
}

// The extended statistics options, resolved (dllm_stats_ex or the defaults).
struct StatsOpts {
  float scale = 1.0f;
  float* margin = nullptr;
  int32_t* argmax = nullptr;
};

dllm_status resolve_ex(const dllm_stats_ex* ex, StatsOpts& o) {
  o = StatsOpts();
  if (!ex) return DLLM_OK;
  if (!(ex->logit_scale > 0.0f) || !(ex->logit_scale <= 256.0f)) return DLLM_ERR_INVALID_ARGUMENT;
  o.scale = ex->logit_scale;
  o.margin = ex->margin;
  o.argmax = ex->argmax;
  return DLLM_OK;
}

dllm_status run_stats(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V, int64_t row_stride,
                      float temperature, uint64_t key, const std::vector<int32_t>& sup, int32_t* x0, float* prob,
                      float* entropy, const RuleArgs* rule, void* ws, size_t ws_bytes, cudaStream_t s,
                      bool early = false, const StatsOpts& opt = StatsOpts(), bool test_drop = false) {
  const DeviceInfo* d = device_info();
  if (!d) return DLLM_ERR_CUDA;
  const bool bf16 = dt == DLLM_BF16, gumbel = temperature > 0.0f;
  // Track only what the outputs need: the argmax beside a sample when the
  // argmax or the margin is asked for, the runner-up only for the margin.
  int mode = gumbel ? kModeSample : 0;
  if (gumbel && (opt.margin || opt.argmax)) mode |= kModeArgmax;
  if (opt.margin) mode |= kModeRunner;
  if (opt.scale != 1.0f) mode |= kModeScaled;
  const int es = esize_of(dt);
  const int64_t T = B * L;
  const WsLayout lay = ws_layout(B, L, d->sms);
  if (!ws || ws_bytes < lay.total) return DLLM_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 15u) != 0) return DLLM_ERR_INVALID_ARGUMENT;
  const int variant = (bf16 ? kModeSlots : 0) + mode;
  StatsPlan pl = plan_stats(*d, variant, T, V, es, early);
  // Inputs ready early, a rule to run and short batch rows: one cluster per
  // batch row, so the step's rule needs no global atomics after the wait.
  // Taken where the plan was a cluster per row (few rows), or where each of
  // its CTAs would stream at most 1 MiB (a small step, whose serial chain
  // matters more than how many CTAs stream it).
  if (early && rule) {
    StatsPlan bp = pl;
    if (plan_batch(*d, variant, B, L, bp) &&
        (pl.kind == kGridCluster || T * V * es <= static_cast<int64_t>(bp.P) * (1 << 20)))
      pl = bp;
  }

  StatsParams p{};
  p.logits = static_cast<const uint8_t*>(logits);
  p.cluster = pl.cluster;
  p.early = early ? 1 : 0;
  p.test_drop = test_drop ? 1 : 0;
  p.row_bytes = row_stride * es;
  p.T = T;
  p.V = V;
  p.L = L;
  p.nvec = pl.nvec;
  p.tail = pl.tail;
  p.chunk_vec = pl.chunk_vec;
  p.K = pl.K;
  p.U = pl.U;
  p.P = pl.P;
  p.stages = pl.stages;
  p.temperature = temperature;
  p.scale = opt.scale;
  p.keys = philox_schedule(key);
  p.n_sup = static_cast<int32_t>(sup.size());
  for (size_t i = 0; i < sup.size(); ++i) p.sup[i] = sup[i];
  p.ln_veff = static_cast<float>(std::log(static_cast<double>(V - static_cast<int64_t>(sup.size()))));
  p.x0 = x0;
  p.prob = prob;
  p.entropy = entropy;
  p.margin = opt.margin;
  p.argmax = opt.argmax;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.fault = reinterpret_cast<int32_t*>(w + lay.fault);
  p.row_count = reinterpret_cast<int32_t*>(w + lay.row_count);
  p.batch_packed = reinterpret_cast<unsigned long long*>(w + lay.batch_packed);
  p.batch_forced = reinterpret_cast<unsigned long long*>(w + lay.batch_forced);
  p.partials = reinterpret_cast<Partial*>(w + lay.partials);
  p.fused = rule ? 1 : 0;
  if (rule) p.rule = *rule;
  const size_t smem = static_cast<size_t>(pl.stages) * pl.chunk_vec * 16 + (rule ? kFusedSortCap * 9 : 0);
  void* args[] = {&p};
  if (pl.kind != kGridPersistent)
    return launch(stats_kernel_ptr(bf16, mode, pl.kind), dim3(pl.P), dim3(kThreads), smem, s, args, pl.cluster);
  return launch(stats_kernel_ptr(bf16, mode, kGridPersistent), dim3(pl.P), dim3(kThreads), smem, s, args);
}

int next_pow2(int64_t x) {
  int n = 1;
  while (n < x) n <<= 1;
  return n;
}

dllm_status check_rule_tail(int64_t B, int64_t L, const int32_t* x0, const int32_t* canvas, int64_t canvas_stride,
                            int64_t canvas_offset) {
  if ((x0 == nullptr) != (canvas == nullptr)) return DLLM_ERR_INVALID_ARGUMENT;
  if (canvas) {
    if (canvas_offset < 0 || canvas_stride < 0) return DLLM_ERR_INVALID_ARGUMENT;
    if (B > 1 && canvas_stride < canvas_offset + L) return DLLM_ERR_INVALID_ARGUMENT;
  }
  return DLLM_OK;
}

dllm_status run_rule_kernel(const RuleArgs& a, int64_t B, int64_t L, cudaStream_t s) {
  const DeviceInfo* d = device_info();
  if (!d) return DLLM_ERR_CUDA;
  const bool sorting = a.rule == kRuleTopk || a.rule == kRuleFactor || a.rule == kRuleEntropyBound;
  int cap = 0, nt = 128;
  if (sorting) {
    if (L > DLLM_MAX_SORT_L) return DLLM_ERR_UNSUPPORTED;
    cap = next_pow2(L);
    nt = std::min(1024, std::max(128, cap / 2));
  } else {
    nt = L >= 1024 ? 1024 : (L >= 512 ? 512 : (L >= 256 ? 256 : 128));
  }
  RuleArgs args_copy = a;
  int32_t cap_arg = cap;
  void* args[] = {&args_copy, &cap_arg};
  return launch(rules_kernel_ptr(nt), dim3(static_cast<unsigned>(B)), dim3(nt), static_cast<size_t>(cap) * 9, s, args);
}

dllm_status rule_entry(int32_t kind, const float* conf, const uint8_t* cand, int64_t B, int64_t L, float tau,
                       int strict, const int32_t* k, float factor, float gamma, uint8_t* commit, const int32_t* x0,
                       int32_t* canvas, int64_t canvas_stride, int64_t canvas_offset, cudaStream_t s) {
  if (B < 0 || L < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (B > INT32_MAX || L > INT32_MAX) return DLLM_ERR_UNSUPPORTED;
  if (B * L == 0) return DLLM_OK;
  if (!conf || !cand || !commit) return DLLM_ERR_INVALID_ARGUMENT;
  if (kind == kRuleTopk && !k) return DLLM_ERR_INVALID_ARGUMENT;
  if (std::isnan(tau) || std::isnan(factor) || std::isnan(gamma)) return DLLM_ERR_INVALID_ARGUMENT;
  dllm_status st = check_rule_tail(B, L, x0, canvas, canvas_stride, canvas_offset);
  if (st != DLLM_OK) return st;
  RuleArgs a{};
  a.rule = kind;
  a.strict = strict ? 1 : 0;
  a.tau = tau;
  a.factor = factor;
  a.gamma = gamma;
  a.k = k;
  a.conf = conf;
  a.entropy = conf;
  a.cand = cand;
  a.commit = commit;
  a.x0 = x0;
  a.canvas = canvas;
  a.canvas_stride = canvas_stride;
  a.canvas_offset = canvas_offset;
  a.L = L;
  return run_rule_kernel(a, B, L, s);
}

// Scratch of dllm_token_stats_noalloc: one fixed array per GPU that loads the
// library.  Host code must not use `g_noalloc_scratch` as an address (it is a
// host-side stand-in); the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_noalloc_scratch[DLLM_NOALLOC_SCRATCH_BYTES];

struct NoallocSlot {
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
NoallocSlot g_noalloc[kMaxDevices];
std::once_flag g_noalloc_once[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
void* noalloc_scratch(cudaError_t* err) {
  int dev = 0;
  if ((*err = cudaGetDevice(&dev)) != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::call_once(g_noalloc_once[dev], [dev]() {
    void* p = nullptr;
    g_noalloc[dev].err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    g_noalloc[dev].ptr = g_noalloc[dev].err == cudaSuccess ? p : nullptr;
  });
  *err = g_noalloc[dev].err;
  return g_noalloc[dev].ptr;
}

// The checks of dllm_commit_step, and the rule arguments and options they
// resolve (shared by the device- and host-buffer entry points).
struct CommitCall {
  std::vector<int32_t> sup;
  RuleArgs a{};
  StatsOpts opt;
  bool early = false;
  bool test_drop = false;
};

dllm_status commit_check(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V, int64_t row_stride,
                         float temperature, const int32_t* suppress_ids, int32_t n_suppress, int32_t* x0, float* prob,
                         float* entropy, const dllm_commit_params* cp, CommitCall& c) {
  dllm_status st = check_stats(logits, dt, B, L, V, row_stride, temperature, suppress_ids, n_suppress, x0, prob,
                               entropy, c.sup);
  if (st != DLLM_OK) return st;
  if (!cp) return DLLM_ERR_INVALID_ARGUMENT;
  if (cp->rule < DLLM_RULE_NONE || cp->rule > DLLM_RULE_ENTROPY_BOUND) return DLLM_ERR_INVALID_ARGUMENT;
  if (B * L == 0) return DLLM_OK;
  if (B > INT32_MAX || L > 65535) return DLLM_ERR_UNSUPPORTED;  // per-batch-row counters are 16-bit
  if (cp->rule != DLLM_RULE_NONE && !cp->commit) return DLLM_ERR_INVALID_ARGUMENT;
  if (cp->rule == DLLM_RULE_TOPK && !cp->k) return DLLM_ERR_INVALID_ARGUMENT;
  if (cp->edit && !cp->edit_mask) return DLLM_ERR_INVALID_ARGUMENT;
  if (!cp->cand && !cp->canvas) return DLLM_ERR_INVALID_ARGUMENT;
  if (std::isnan(cp->tau) || std::isnan(cp->factor) || std::isnan(cp->gamma) || std::isnan(cp->tau_edit))
    return DLLM_ERR_INVALID_ARGUMENT;
  const bool sorting = cp->rule == DLLM_RULE_TOPK || cp->rule == DLLM_RULE_FACTOR || cp->rule == DLLM_RULE_ENTROPY_BOUND;
  if (sorting && L > kFusedSortCap) return DLLM_ERR_UNSUPPORTED;
  if (cp->canvas) {
    if (cp->canvas_offset < 0 || cp->canvas_stride < 0) return DLLM_ERR_INVALID_ARGUMENT;
    if (B > 1 && cp->canvas_stride < cp->canvas_offset + L) return DLLM_ERR_INVALID_ARGUMENT;
  }
  RuleArgs& a = c.a;
  a.rule = cp->rule;
  a.strict = cp->strict ? 1 : 0;
  a.tau = cp->tau;
  a.factor = cp->factor;
  a.gamma = cp->gamma;
  a.k = cp->k;
  a.conf = prob;
  a.entropy = entropy;
  a.cand = cp->cand;
  a.mask_id = cp->mask_id;
  a.edit = cp->edit ? 1 : 0;
  a.tau_edit = cp->tau_edit;
  a.x0 = x0;
  a.commit = cp->commit;
  a.edit_mask = cp->edit ? cp->edit_mask : nullptr;
  a.canvas = cp->canvas;
  a.canvas_stride = cp->canvas_stride;
  a.canvas_offset = cp->canvas_offset;
  a.counts = cp->counts;
  a.L = L;
  if (cp->flags & ~static_cast<int32_t>(DLLM_FLAG_INPUTS_READY | DLLM_FLAG_TEST_DROP_COPY))
    return DLLM_ERR_INVALID_ARGUMENT;
  if (resolve_ex(cp->ex, c.opt) != DLLM_OK) return DLLM_ERR_INVALID_ARGUMENT;
  c.early = (cp->flags & DLLM_FLAG_INPUTS_READY) != 0;
  c.test_drop = (cp->flags & DLLM_FLAG_TEST_DROP_COPY) != 0;
  return DLLM_OK;
}

}  // namespace

extern "C" {

const char* dllm_status_string(dllm_status status) {
  switch (status) {
    case DLLM_OK: return "DLLM_OK";
    case DLLM_ERR_INVALID_ARGUMENT: return "DLLM_ERR_INVALID_ARGUMENT: a shape, pointer, value or alignment is wrong";
    case DLLM_ERR_UNSUPPORTED: return "DLLM_ERR_UNSUPPORTED: valid, but outside what this library version handles";
    case DLLM_ERR_WORKSPACE: return "DLLM_ERR_WORKSPACE: workspace missing or too small";
    case DLLM_ERR_CUDA: return "DLLM_ERR_CUDA: a CUDA launch or query failed";
    case DLLM_ERR_DEVICE: return "DLLM_ERR_DEVICE: a kernel reported a fault";
  }
  return "unknown dllm_status";
}

const char* dllm_version(void) { return "libdllmcommit 0.1.0 (sm_103a)"; }

size_t dllm_token_stats_workspace_size(int64_t B, int64_t L, int64_t V, dllm_dtype dt) {
  (void)V;
  (void)dt;
  if (B < 0 || L < 0) return 0;
  const int64_t T = checked_mul(B, L);
  if (T < 0 || T > (static_cast<int64_t>(1) << 56) || B > (static_cast<int64_t>(1) << 56)) return 0;
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 160;  // no device: size for the largest part the library targets
  return ws_layout(B, L, sms).total;
}

dllm_status dllm_token_stats(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V, int64_t row_stride,
                             float temperature, uint64_t key, const int32_t* suppress_ids, int32_t n_suppress,
                             int32_t* x0, float* prob, float* entropy, void* workspace, size_t workspace_bytes,
                             dllm_stream_t stream) {
  std::vector<int32_t> sup;
  dllm_status st = check_stats(logits, dt, B, L, V, row_stride, temperature, suppress_ids, n_suppress, x0, prob,
                               entropy, sup);
  if (st != DLLM_OK || B * L == 0) return st;
  return run_stats(logits, dt, B, L, V, row_stride, temperature, key, sup, x0, prob, entropy, nullptr, workspace,
                   workspace_bytes, reinterpret_cast<cudaStream_t>(stream));
}

dllm_status dllm_token_stats_ex(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V,
                                int64_t row_stride, float temperature, uint64_t key, const int32_t* suppress_ids,
                                int32_t n_suppress, const dllm_stats_ex* ex, int32_t* x0, float* prob,
                                float* entropy, void* workspace, size_t workspace_bytes, dllm_stream_t stream) {
  std::vector<int32_t> sup;
  dllm_status st = check_stats(logits, dt, B, L, V, row_stride, temperature, suppress_ids, n_suppress, x0, prob,
                               entropy, sup);
  if (st != DLLM_OK) return st;
  StatsOpts opt;
  st = resolve_ex(ex, opt);
  if (st != DLLM_OK || B * L == 0) return st;
  return run_stats(logits, dt, B, L, V, row_stride, temperature, key, sup, x0, prob, entropy, nullptr, workspace,
                   workspace_bytes, reinterpret_cast<cudaStream_t>(stream), false, opt);
}

dllm_status dllm_threshold_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L, float tau,
                                    int strict, uint8_t* commit, const int32_t* x0, int32_t* canvas,
                                    int64_t canvas_stride, int64_t canvas_offset, dllm_stream_t stream) {
  return rule_entry(kRuleThreshold, conf, cand, B, L, tau, strict, nullptr, 0.f, 0.f, commit, x0, canvas,
                    canvas_stride, canvas_offset, reinterpret_cast<cudaStream_t>(stream));
}

dllm_status dllm_topk_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L, const int32_t* k,
                               uint8_t* commit, const int32_t* x0, int32_t* canvas, int64_t canvas_stride,
                               int64_t canvas_offset, dllm_stream_t stream) {
  return rule_entry(kRuleTopk, conf, cand, B, L, 0.f, 0, k, 0.f, 0.f, commit, x0, canvas, canvas_stride,
                    canvas_offset, reinterpret_cast<cudaStream_t>(stream));
}

dllm_status dllm_factor_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L, float factor,
                                 uint8_t* commit, const int32_t* x0, int32_t* canvas, int64_t canvas_stride,
                                 int64_t canvas_offset, dllm_stream_t stream) {
  return rule_entry(kRuleFactor, conf, cand, B, L, 0.f, 0, nullptr, factor, 0.f, commit, x0, canvas, canvas_stride,
                    canvas_offset, reinterpret_cast<cudaStream_t>(stream));
}

dllm_status dllm_entropy_bound_transfer(const float* entropy, const uint8_t* cand, int64_t B, int64_t L, float gamma,
                                        uint8_t* commit, const int32_t* x0, int32_t* canvas, int64_t canvas_stride,
                                        int64_t canvas_offset, dllm_stream_t stream) {
  return rule_entry(kRuleEntropyBound, entropy, cand, B, L, 0.f, 0, nullptr, 0.f, gamma, commit, x0, canvas,
                    canvas_stride, canvas_offset, reinterpret_cast<cudaStream_t>(stream));
}

dllm_status dllm_edit_transfer(const int32_t* x0, const float* prob, const int32_t* tokens, const uint8_t* editable,
                               int64_t B, int64_t L, float tau_edit, uint8_t* edit, dllm_stream_t stream) {
  if (B < 0 || L < 0 || std::isnan(tau_edit)) return DLLM_ERR_INVALID_ARGUMENT;
  const int64_t n = checked_mul(B, L);
  if (n < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (n == 0) return DLLM_OK;
  if (!x0 || !prob || !tokens || !editable || !edit) return DLLM_ERR_INVALID_ARGUMENT;
  const DeviceInfo* d = device_info();
  if (!d) return DLLM_ERR_CUDA;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, static_cast<int64_t>(d->sms) * 8);
  void* args[] = {const_cast<int32_t**>(&x0), const_cast<float**>(&prob), const_cast<int32_t**>(&tokens),
                  const_cast<uint8_t**>(&editable), const_cast<int64_t*>(&n), &tau_edit, &edit};
  return launch(edit_kernel_ptr(), dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                reinterpret_cast<cudaStream_t>(stream), args);
}

dllm_status dllm_transfer_schedule(const int32_t* counts, int64_t B, int32_t steps, int32_t* quotas,
                                   dllm_stream_t stream) {
  if (B < 0 || steps <= 0 || checked_mul(B, steps) < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (B == 0) return DLLM_OK;
  if (!counts || !quotas) return DLLM_ERR_INVALID_ARGUMENT;
  const DeviceInfo* d = device_info();
  if (!d) return DLLM_ERR_CUDA;
  const int64_t total = B * steps;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, static_cast<int64_t>(d->sms) * 8);
  void* args[] = {const_cast<int32_t**>(&counts), &B, &steps, &quotas};
  return launch(schedule_kernel_ptr(), dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                reinterpret_cast<cudaStream_t>(stream), args);
}

dllm_status dllm_linear_temperature(int32_t remaining, int32_t num_steps, float t_min, float t_max,
                                    float* temperature) {
  if (!temperature || num_steps <= 0 || remaining < 0 || remaining > num_steps) return DLLM_ERR_INVALID_ARGUMENT;
  if (!(t_min > 0.0f) || !(t_max >= t_min) || std::isinf(t_max)) return DLLM_ERR_INVALID_ARGUMENT;
  const double frac = static_cast<double>(remaining) / static_cast<double>(num_steps);
  *temperature = static_cast<float>(static_cast<double>(t_min) + (static_cast<double>(t_max) - t_min) * frac);
  return DLLM_OK;
}

dllm_status dllm_uniform_canvas(int64_t B, int64_t N, int64_t V, uint64_t key, int32_t* canvas,
                                int64_t canvas_stride, dllm_stream_t stream) {
  if (B < 0 || N < 0 || V <= 0 || V > INT32_MAX || canvas_stride < N) return DLLM_ERR_INVALID_ARGUMENT;
  if (checked_mul(B, canvas_stride) < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (B * N == 0) return DLLM_OK;
  if (!canvas) return DLLM_ERR_INVALID_ARGUMENT;
  const DeviceInfo* d = device_info();
  if (!d) return DLLM_ERR_CUDA;
  PhiloxSchedule ks = philox_schedule(key);
  uint32_t v32 = static_cast<uint32_t>(V);
  const int64_t work = B * ((N + 3) / 4);
  const int64_t blocks = std::min<int64_t>((work + 255) / 256, static_cast<int64_t>(d->sms) * 8);
  void* args[] = {&ks, &B, &N, &v32, &canvas, &canvas_stride};
  return launch(uniform_canvas_kernel_ptr(), dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                reinterpret_cast<cudaStream_t>(stream), args);
}

dllm_status dllm_renoise(const int32_t* sample, const uint8_t* accepted, const int32_t* noise, const uint8_t* frozen,
                         int64_t B, int64_t N, int32_t* out, dllm_stream_t stream) {
  if (B < 0 || N < 0 || checked_mul(B, N) < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (B * N == 0) return DLLM_OK;
  if (!sample || !out || (accepted && !noise)) return DLLM_ERR_INVALID_ARGUMENT;
  const DeviceInfo* d = device_info();
  if (!d) return DLLM_ERR_CUDA;
  const int64_t blocks = std::min<int64_t>((B * N + 255) / 256, static_cast<int64_t>(d->sms) * 8);
  void* args[] = {const_cast<int32_t**>(&sample), const_cast<uint8_t**>(&accepted), const_cast<int32_t**>(&noise),
                  const_cast<uint8_t**>(&frozen), &B, &N, &out};
  return launch(renoise_kernel_ptr(), dim3(static_cast<unsigned>(blocks)), dim3(256), 0,
                reinterpret_cast<cudaStream_t>(stream), args);
}

dllm_status dllm_stable_confident_stop(const int32_t* argmax, const float* entropy, int64_t B, int64_t L,
                                       int32_t stability_threshold, float confidence_threshold, int32_t* prev,
                                       int32_t* count, uint8_t* stop, uint8_t* done, dllm_stream_t stream) {
  if (B < 0 || L <= 0 || L > (static_cast<int64_t>(1) << 16) || stability_threshold < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (!(confidence_threshold >= 0.0f && confidence_threshold <= 64.0f)) return DLLM_ERR_INVALID_ARGUMENT;
  if (B == 0) return DLLM_OK;
  if (B > INT32_MAX || !argmax || !entropy || !prev || !count) return DLLM_ERR_INVALID_ARGUMENT;
  void* args[] = {const_cast<int32_t**>(&argmax), const_cast<float**>(&entropy), &L, &stability_threshold,
                  &confidence_threshold, &prev, &count, &stop, &done};
  return launch(stop_kernel_ptr(), dim3(static_cast<unsigned>(B)), dim3(256), 0,
                reinterpret_cast<cudaStream_t>(stream), args);
}

dllm_status dllm_uniform_update(const int32_t* sample, const uint8_t* accepted, const int32_t* step_argmax,
                                const float* entropy, int64_t B, int64_t N, int64_t V, uint64_t noise_key,
                                int32_t stability_threshold, float confidence_threshold, int32_t* canvas,
                                int32_t* argmax, int32_t* prev, int32_t* count, uint8_t* done, dllm_stream_t stream) {
  if (B < 0 || N <= 0 || N > (static_cast<int64_t>(1) << 16) || V <= 0 || V > INT32_MAX || stability_threshold < 0)
    return DLLM_ERR_INVALID_ARGUMENT;
  if (!(confidence_threshold >= 0.0f && confidence_threshold <= 64.0f)) return DLLM_ERR_INVALID_ARGUMENT;
  if (B == 0) return DLLM_OK;
  if (B > INT32_MAX || !sample || !accepted || !step_argmax || !entropy || !canvas || !argmax || !prev || !count ||
      !done)
    return DLLM_ERR_INVALID_ARGUMENT;
  PhiloxSchedule ks = philox_schedule(noise_key);
  uint32_t v32 = static_cast<uint32_t>(V);
  void* args[] = {&ks, const_cast<int32_t**>(&sample), const_cast<uint8_t**>(&accepted),
                  const_cast<int32_t**>(&step_argmax), const_cast<float**>(&entropy), &N, &v32,
                  &stability_threshold, &confidence_threshold, &canvas, &argmax, &prev, &count, &done};
  return launch(uniform_update_kernel_ptr(), dim3(static_cast<unsigned>(B)), dim3(256), 0,
                reinterpret_cast<cudaStream_t>(stream), args);
}

dllm_status dllm_block_causal_mask(int64_t Lq, int64_t Lk, int64_t q_offset, int64_t k_offset, int64_t block_len,
                                   dllm_mask_kind kind, void* out, int64_t row_stride, dllm_stream_t stream) {
  if (Lq < 0 || Lk < 0 || q_offset < 0 || k_offset < 0 || block_len <= 0 || row_stride < Lk)
    return DLLM_ERR_INVALID_ARGUMENT;
  if (kind != DLLM_MASK_F32 && kind != DLLM_MASK_BF16 && kind != DLLM_MASK_KEEP_U8) return DLLM_ERR_INVALID_ARGUMENT;
  if (q_offset > INT64_MAX / 2 - Lq || k_offset > INT64_MAX / 2 - Lk || block_len > INT64_MAX / 4)
    return DLLM_ERR_INVALID_ARGUMENT;
  if (checked_mul(checked_mul(Lq, row_stride), 4) < 0) return DLLM_ERR_INVALID_ARGUMENT;  // byte extent
  if (Lq * Lk == 0) return DLLM_OK;
  if (!out) return DLLM_ERR_INVALID_ARGUMENT;
  const DeviceInfo* d = device_info();
  if (!d) return DLLM_ERR_CUDA;
  const int es = kind == DLLM_MASK_F32 ? 4 : (kind == DLLM_MASK_BF16 ? 2 : 1);
  uint32_t attend = kind == DLLM_MASK_KEEP_U8 ? 1u : 0u;
  uint32_t blocked = kind == DLLM_MASK_F32 ? 0xFF800000u : (kind == DLLM_MASK_BF16 ? 0xFF80u : 0u);
  int64_t row_bytes = row_stride * es;
  int vec = ((reinterpret_cast<uintptr_t>(out) & 15u) == 0 && row_bytes % 16 == 0) ? 1 : 0;
  // one block per chunk of mask_chunk_vec() vectors of a row (one per row
  // when rows are not vector-aligned); the kernel's block loop covers a
  // grid capped below the launch limit
  const int64_t nvec = vec ? Lk / (16 / es) : 0;
  int64_t chunks_per_row = (nvec + mask_chunk_vec() - 1) / mask_chunk_vec();
  if (chunks_per_row < 1) chunks_per_row = 1;
  const int64_t blocks = std::min<int64_t>(Lq * chunks_per_row, int64_t{1} << 30);
  uint8_t* o = static_cast<uint8_t*>(out);
  void* args[] = {&Lq, &Lk, &q_offset, &k_offset, &block_len, &o, &row_bytes, &attend, &blocked, &vec,
                  &chunks_per_row};
  return launch(mask_kernel_ptr(es), dim3(static_cast<unsigned>(blocks)), dim3(mask_threads()), 0,
                reinterpret_cast<cudaStream_t>(stream), args);
}

dllm_status dllm_block_ranges(int64_t P, int64_t gen_len, int64_t block_len, int align, int64_t* ranges, int64_t cap,
                              int64_t* n_out) {
  if (P < 0 || gen_len < 0 || block_len <= 0 || cap < 0 || !n_out) return DLLM_ERR_INVALID_ARGUMENT;
  if (cap > 0 && !ranges) return DLLM_ERR_INVALID_ARGUMENT;
  if (P > INT64_MAX - gen_len) return DLLM_ERR_INVALID_ARGUMENT;
  const int64_t first = align ? (P / block_len) * block_len : P;
  const int64_t stop = P + gen_len;
  const int64_t n = gen_len == 0 ? 0 : (stop - first + block_len - 1) / block_len;
  for (int64_t i = 0; i < n && i < cap; ++i) {
    const int64_t start = first + i * block_len;
    ranges[2 * i] = start;
    ranges[2 * i + 1] = std::min(start + block_len, stop);
  }
  *n_out = n;
  return n > cap ? DLLM_ERR_WORKSPACE : DLLM_OK;
}

dllm_status dllm_commit_step(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V, int64_t row_stride,
                             float temperature, uint64_t key, const int32_t* suppress_ids, int32_t n_suppress,
                             int32_t* x0, float* prob, float* entropy, const dllm_commit_params* cp, void* workspace,
                             size_t workspace_bytes, dllm_stream_t stream) {
  CommitCall c;
  const dllm_status st = commit_check(logits, dt, B, L, V, row_stride, temperature, suppress_ids, n_suppress, x0, prob,
                                      entropy, cp, c);
  if (st != DLLM_OK || B * L == 0) return st;
  return run_stats(logits, dt, B, L, V, row_stride, temperature, key, c.sup, x0, prob, entropy, &c.a, workspace,
                   workspace_bytes, reinterpret_cast<cudaStream_t>(stream), c.early, c.opt, c.test_drop);
}

dllm_status dllm_commit_step_host(const void* host_logits, void* dev_logits, dllm_dtype dt, int64_t B, int64_t L,
                                  int64_t V, float temperature, uint64_t key, const int32_t* suppress_ids,
                                  int32_t n_suppress, const dllm_commit_params* cp, void* dev_out, void* host_out,
                                  void* workspace, size_t workspace_bytes, dllm_stream_t stream) {
  if (!cp || B < 0 || L < 0 || V < 1 || checked_mul(B, L) < 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (B * L == 0) return DLLM_OK;
  if (!host_logits || !dev_logits || !dev_out || !host_out) return DLLM_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(dev_out) & 3u) != 0) return DLLM_ERR_INVALID_ARGUMENT;
  if (dt != DLLM_F32 && dt != DLLM_BF16) return DLLM_ERR_INVALID_ARGUMENT;
  const int64_t T = B * L;
  if (T > INT64_MAX / V / esize_of(dt)) return DLLM_ERR_INVALID_ARGUMENT;
  int32_t* x0 = static_cast<int32_t*>(dev_out);
  float* prob = reinterpret_cast<float*>(x0 + T);
  float* entropy = prob + T;
  dllm_commit_params p = *cp;
  if (p.rule != DLLM_RULE_NONE) p.commit = reinterpret_cast<uint8_t*>(entropy + T);
  CommitCall c;
  const dllm_status st = commit_check(dev_logits, dt, B, L, V, V, temperature, suppress_ids, n_suppress, x0, prob,
                                      entropy, &p, c);
  if (st != DLLM_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(dev_logits, host_logits, static_cast<size_t>(T * V * esize_of(dt)), cudaMemcpyHostToDevice,
                      s) != cudaSuccess)
    return DLLM_ERR_CUDA;
  const dllm_status rs = run_stats(dev_logits, dt, B, L, V, V, temperature, key, c.sup, x0, prob, entropy, &c.a,
                                   workspace, workspace_bytes, s, c.early, c.opt);
  if (rs != DLLM_OK) return rs;
  const size_t out_bytes = static_cast<size_t>(T) * (p.rule != DLLM_RULE_NONE ? 13 : 12);
  return cudaMemcpyAsync(host_out, dev_out, out_bytes, cudaMemcpyDeviceToHost, s) == cudaSuccess ? DLLM_OK
                                                                                                   : DLLM_ERR_CUDA;
}

dllm_status dllm_token_stats_noalloc(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V,
                                     int64_t row_stride, float temperature, uint64_t key, const int32_t* suppress_ids,
                                     int32_t n_suppress, int32_t* x0, float* prob, float* entropy,
                                     dllm_stream_t stream) {
  std::vector<int32_t> sup;
  dllm_status st = check_stats(logits, dt, B, L, V, row_stride, temperature, suppress_ids, n_suppress, x0, prob,
                               entropy, sup);
  if (st != DLLM_OK || B * L == 0) return st;
  const DeviceInfo* d = device_info();
  if (!d) return DLLM_ERR_CUDA;
  const size_t need = ws_layout(B, L, d->sms).total;
  if (need > DLLM_NOALLOC_SCRATCH_BYTES) return DLLM_ERR_UNSUPPORTED;  // shape too large for the fixed scratch
  cudaError_t err = cudaSuccess;
  void* scratch = noalloc_scratch(&err);
  if (!scratch) return DLLM_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents: clear the fault word and
  // the counters this call relies on starting at zero.
  if (cudaMemsetAsync(scratch, 0, need, s) != cudaSuccess) return DLLM_ERR_CUDA;
  return run_stats(logits, dt, B, L, V, row_stride, temperature, key, sup, x0, prob, entropy, nullptr, scratch,
                   DLLM_NOALLOC_SCRATCH_BYTES, s);
}

dllm_status dllm_noalloc_fault(dllm_stream_t stream, int32_t* fault) {
  if (!fault) return DLLM_ERR_INVALID_ARGUMENT;
  cudaError_t err = cudaSuccess;
  void* scratch = noalloc_scratch(&err);
  if (!scratch) return DLLM_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DLLM_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DLLM_ERR_CUDA;
  if (v != 0 && cudaMemsetAsync(scratch, 0, sizeof(int32_t), s) != cudaSuccess) return DLLM_ERR_CUDA;
  *fault = v;
  return DLLM_OK;
}

dllm_status dllm_workspace_fault(void* workspace, dllm_stream_t stream, int32_t* fault) {
  if (!workspace || !fault) return DLLM_ERR_INVALID_ARGUMENT;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return DLLM_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DLLM_ERR_CUDA;
  if (v != 0 && cudaMemsetAsync(workspace, 0, sizeof(int32_t), s) != cudaSuccess) return DLLM_ERR_CUDA;
  *fault = v;
  return DLLM_OK;
}

}  // extern "C"
