// dllm_rules.cuh -- the commit rules of one batch row, run by NT threads.
//
// Sources (page, section):
//   mlx-arsenal "dLLM block decoding": "What mlx-arsenal ships" (the
//   threshold, top-k, factor, entropy-bound and edit rules), "Deviations from
//   the references" (stable ranking, the forced token is the earliest maximal
//   one, no factor off-by-one), "Token editing (LLaDA2.1)".
//   mlxcel "Block Diffusion": "Samplers and Reveal Policies" (forced progress,
//   at least one accepted under the entropy bound).
//
// Ranking keys are 64-bit: (order-preserving score bits << 32) | position, so
// a plain ascending sort gives "best first, ties to the lower position".
// Confidences rank descending with NaN as -inf; entropies rank ascending with
// NaN as +inf.  The factor product and the entropy prefix sum are evaluated in
// double with explicitly rounded operations, in ranking order.
#pragma once

#include <cstdint>

#include "dllm_device.cuh"

namespace dllm {

enum RuleKind : int32_t { kRuleNone = 0, kRuleThreshold = 1, kRuleTopk = 2, kRuleFactor = 3, kRuleEntropyBound = 4 };

struct RuleArgs {
  int32_t rule;
  int32_t strict;
  float tau, factor, gamma;
  const int32_t* k;        // (B,) top-k quotas
  const float* conf;       // (B, L) confidence (threshold / top-k / factor)
  const float* entropy;    // (B, L) entropy (entropy bound)
  const uint8_t* cand;     // (B, L) or nullptr: cand = canvas token == mask_id
  int32_t mask_id;
  int32_t edit;            // also apply the edit rule with editable = !cand
  float tau_edit;
  const int32_t* x0;       // (B, L) proposals (canvas update / edit)
  uint8_t* commit;         // (B, L)
  uint8_t* edit_mask;      // (B, L) when edit
  int32_t* canvas;         // nullable
  int64_t canvas_stride, canvas_offset;
  int32_t* counts;         // (B, 3) or nullptr
  int64_t L;
};

constexpr uint64_t kNoKey = ~0ull;

__device__ __forceinline__ float nan_to(float x, float v) { return x != x ? v : x; }

__device__ __forceinline__ uint64_t desc_key(float c, int64_t l) {
  const float cc = nan_to(c, -__int_as_float(0x7F800000));
  return (static_cast<uint64_t>(~float_key(cc)) << 32) | static_cast<uint32_t>(l);
}

__device__ __forceinline__ uint64_t asc_key(float h, int64_t l) {
  const float hh = nan_to(h, __int_as_float(0x7F800000));
  return (static_cast<uint64_t>(float_key(hh)) << 32) | static_cast<uint32_t>(l);
}

// Synchronisation among the NT threads running a rule: a named barrier when
// they are a subset of the CTA, __syncthreads when they are all of it.
template <int NT, int BAR>
__device__ __forceinline__ void rsync() {
  if (BAR == 0)
    __syncthreads();
  else
    named_sync(BAR, NT);
}

// Exclusive prefix sum of one int64 per thread over the NT threads (in
// thread order).  Uses s.red64; all NT threads must call it.
template <int NT, int BAR>
__device__ __forceinline__ long long rule_excl_scan(long long v, const struct RuleScratch& s, int tid);

struct RuleScratch {
  uint64_t* keys;     // capacity `cap` keys (power of two)
  uint8_t* flags;     // capacity `cap` bytes
  uint64_t* red64;    // NT/32 entries
  int32_t* red32;     // 4 * NT/32 entries
  int32_t cap;
};

template <int NT, int BAR>
__device__ __forceinline__ uint64_t rule_min_u64(uint64_t v, const RuleScratch& s, int tid) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
    v = w < v ? w : v;
  }
  rsync<NT, BAR>();
  if ((tid & 31) == 0) s.red64[tid >> 5] = v;
  rsync<NT, BAR>();
  v = s.red64[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) v = s.red64[w] < v ? s.red64[w] : v;
  return v;
}

// Sums of up to four int32 counters over the NT threads.
template <int NT, int BAR>
__device__ __forceinline__ int4 rule_sum4(int4 v, const RuleScratch& s, int tid) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xFFFFFFFFu, v.x, o);
    v.y += __shfl_xor_sync(0xFFFFFFFFu, v.y, o);
    v.z += __shfl_xor_sync(0xFFFFFFFFu, v.z, o);
    v.w += __shfl_xor_sync(0xFFFFFFFFu, v.w, o);
  }
  rsync<NT, BAR>();
  if ((tid & 31) == 0) {
    s.red32[4 * (tid >> 5) + 0] = v.x;
    s.red32[4 * (tid >> 5) + 1] = v.y;
    s.red32[4 * (tid >> 5) + 2] = v.z;
    s.red32[4 * (tid >> 5) + 3] = v.w;
  }
  rsync<NT, BAR>();
  int4 t = make_int4(0, 0, 0, 0);
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    t.x += s.red32[4 * w + 0];
    t.y += s.red32[4 * w + 1];
    t.z += s.red32[4 * w + 2];
    t.w += s.red32[4 * w + 3];
  }
  return t;
}

// Ascending bitonic sort of n (a power of two) keys in shared memory.
// Compare-exchange steps whose partners are 32 or more apart go through
// shared memory with a barrier each; the steps below 32 of every stage run in
// registers with warp shuffles (element e lives in thread e mod NT, so
// partners e ^ j with j < 32 are lanes of the same warp).  Every lane of every
// warp takes part in the shuffles: lanes past n carry dummy keys, which (n
// being a power of two) only ever meet each other.
template <int NT, int BAR>
__device__ __forceinline__ void bitonic_sort(uint64_t* keys, int n, int tid) {
  const int lane = tid & 31;
  for (int size = 2; size <= n; size <<= 1) {
    int stride = size >> 1;
    for (; stride >= 32; stride >>= 1) {
      rsync<NT, BAR>();
      for (int i = tid; i < (n >> 1); i += NT) {
        const int lo = 2 * i - (i & (stride - 1));
        const int hi = lo + stride;
        const bool up = (lo & size) == 0;
        const uint64_t a = keys[lo], b = keys[hi];
        if ((a > b) == up) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
    }
    rsync<NT, BAR>();
    for (int r = 0; r * NT < n; ++r) {
      const int e = r * NT + tid;
      uint64_t v = e < n ? keys[e] : kNoKey;
      const bool up = (e & size) == 0;
      for (int j = stride; j > 0; j >>= 1) {
        const uint64_t w = __shfl_xor_sync(0xFFFFFFFFu, v, j);
        const bool keep_min = ((lane & j) == 0) == up;
        v = keep_min ? (w < v ? w : v) : (w > v ? w : v);
      }
      if (e < n) keys[e] = v;
    }
  }
  rsync<NT, BAR>();
}

__device__ __forceinline__ bool is_candidate(const RuleArgs& a, int64_t b, int64_t l, int32_t* tok_out) {
  const int64_t i = b * a.L + l;
  int32_t tok = 0;  // the canvas token matters only to the edit rule and to a missing mask
  if (a.canvas && (a.edit || !a.cand)) tok = a.canvas[b * a.canvas_stride + a.canvas_offset + l];
  *tok_out = tok;
  if (a.cand) return __ldcg(a.cand + i) != 0;
  return tok == a.mask_id;
}

template <int NT, int BAR>
__device__ __forceinline__ long long rule_excl_scan(long long v, const RuleScratch& s, int tid) {
  const int lane = tid & 31, w = tid >> 5;
  long long x = v;  // inclusive scan within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s.red64[w] = static_cast<uint64_t>(x);
  rsync<NT, BAR>();
  long long off = 0;
  for (int k = 0; k < w; ++k) off += static_cast<long long>(s.red64[k]);
  rsync<NT, BAR>();
  return off + x - v;
}

// The inputs of one batch row's rule as global memory holds them (written by
// other CTAs of the same kernel, so read through L2 with ld.global.cg).
struct GlobalRowSrc {
  const RuleArgs& a;
  int64_t b;
  __device__ bool cand(int64_t l, int32_t* tok) const { return is_candidate(a, b, l, tok); }
  __device__ float conf(int64_t l) const { return __ldcg(a.conf + b * a.L + l); }
  __device__ float entropy(int64_t l) const { return __ldcg(a.entropy + b * a.L + l); }
  __device__ int32_t x0(int64_t l) const { return a.x0 ? __ldcg(a.x0 + b * a.L + l) : 0; }
};

// Where a rule's decisions go: the masks, the canvas and the counts of
// RuleArgs in global memory.
struct GlobalEmit {
  const RuleArgs& a;
  int64_t b;
  __device__ void operator()(int64_t l, bool commit, bool edit, int32_t x0) const {
    const int64_t i = b * a.L + l;
    if (a.commit) a.commit[i] = commit ? 1 : 0;
    if (a.edit_mask) a.edit_mask[i] = edit ? 1 : 0;
    if ((commit || edit) && a.canvas && a.x0) a.canvas[b * a.canvas_stride + a.canvas_offset + l] = x0;
  }
  __device__ void counts(int n_cand, int n_commit, int n_edit) const {
    a.counts[3 * b + 0] = n_cand;
    a.counts[3 * b + 1] = n_commit;
    a.counts[3 * b + 2] = n_edit;
  }
};

// Runs the rule of batch row b on the inputs `src` gives (candidate flag and
// canvas token, confidence, entropy, proposal per position) and hands each
// position's commit / edit decision, and (when RuleArgs asks for counts) the
// batch row's counts from thread 0, to `emit`.  All NT threads must call it.
template <int NT, int BAR, typename Src, typename Emit>
__device__ void run_rule_src(const RuleArgs& a, int64_t b, const RuleScratch& s, int tid, const Src& src,
                             const Emit& emit) {
  const int64_t L = a.L;
  const int64_t base = b * L;
  int32_t n_commit_forced = 0;
  uint64_t forced = kNoKey;
  int64_t n_take = 0;      // sorting rules: commit the first n_take ranked keys
  int n_cand_total = 0;

  if (a.rule == kRuleThreshold || a.rule == kRuleNone) {
    int any_pass = 0, n_cand = 0;
    uint64_t best = kNoKey;
    for (int64_t l = tid; l < L; l += NT) {
      int32_t tok;
      if (!src.cand(l, &tok)) continue;
      ++n_cand;
      if (a.rule == kRuleThreshold) {
        const float c = nan_to(src.conf(l), -__int_as_float(0x7F800000));
        const bool pass = a.strict ? (c > a.tau) : (c >= a.tau);
        any_pass |= pass ? 1 : 0;
        const uint64_t key = desc_key(c, l);
        best = key < best ? key : best;
      }
    }
    const int4 t = rule_sum4<NT, BAR>(make_int4(n_cand, any_pass, 0, 0), s, tid);
    n_cand_total = t.x;
    if (a.rule == kRuleThreshold) {
      best = rule_min_u64<NT, BAR>(best, s, tid);
      if (t.x > 0 && t.y == 0) forced = best;
    }
  } else {
    int n = 1;
    while (n < L) n <<= 1;
    // n <= s.cap is guaranteed by the host
    int n_cand = 0;
    for (int64_t l = tid; l < n; l += NT) {
      uint64_t key = kNoKey;
      if (l < L) {
        int32_t tok;
        if (src.cand(l, &tok)) {
          ++n_cand;
          key = (a.rule == kRuleEntropyBound) ? asc_key(src.entropy(l), l) : desc_key(src.conf(l), l);
        }
      }
      s.keys[l] = key;
    }
    n_cand_total = rule_sum4<NT, BAR>(make_int4(n_cand, 0, 0, 0), s, tid).x;
    bitonic_sort<NT, BAR>(s.keys, n, tid);
    if (a.rule == kRuleTopk) {
      const int32_t kb = __ldcg(a.k + b);
      n_take = kb < 0 ? 0 : (kb > n_cand_total ? n_cand_total : kb);
    } else if (a.rule == kRuleFactor) {
      // first rank i whose (i+1)(1 - c_(i)) exceeds f, in double
      uint64_t first_fail = static_cast<uint64_t>(n_cand_total);
      for (int i = tid; i < n_cand_total; i += NT) {
        const int64_t l = static_cast<int64_t>(s.keys[i] & 0xFFFFFFFFu);
        const double c = nan_to(src.conf(l), -__int_as_float(0x7F800000));
        const double lhs = __dmul_rn(static_cast<double>(i + 1), __dsub_rn(1.0, c));
        if (!(lhs <= static_cast<double>(a.factor))) {
          first_fail = static_cast<uint64_t>(i) < first_fail ? static_cast<uint64_t>(i) : first_fail;
        }
      }
      n_take = static_cast<int64_t>(rule_min_u64<NT, BAR>(first_fail, s, tid));
    } else {  // entropy bound: exact fixed-point prefix sums of the ranking, in parallel
      // Each thread takes a contiguous run of ranks; the entropy of a rank is
      // read back from its key.  S_i (the sum of the ranks before i) never
      // decreases, so the ranks within the bound are a prefix: count them.
      const long long bound = fixed_bound(a.gamma);
      const int per = (n_cand_total + NT - 1) / NT;
      const int i0 = tid * per < n_cand_total ? tid * per : n_cand_total;
      const int i1 = i0 + per < n_cand_total ? i0 + per : n_cand_total;
      long long run = 0;
      for (int i = i0; i < i1; ++i) run += fixed_q(key_to_float(static_cast<uint32_t>(s.keys[i] >> 32)));
      long long S = rule_excl_scan<NT, BAR>(run, s, tid);
      int within = 0;
      for (int i = i0; i < i1; ++i) {
        within += S <= bound ? 1 : 0;
        S += fixed_q(key_to_float(static_cast<uint32_t>(s.keys[i] >> 32)));
      }
      n_take = rule_sum4<NT, BAR>(make_int4(within, 0, 0, 0), s, tid).x;
    }
    if (a.rule != kRuleTopk && n_cand_total > 0 && n_take < 1) n_take = 1;
    // flags[l] = 1 for the first n_take ranked candidates
    for (int64_t l = tid; l < L; l += NT) s.flags[l] = 0;
    rsync<NT, BAR>();
    for (int64_t i = tid; i < n_take; i += NT) s.flags[s.keys[i] & 0xFFFFFFFFu] = 1;
    rsync<NT, BAR>();
  }

  // The masks and the canvas update.
  int n_commit = 0, n_edit = 0;
  for (int64_t l = tid; l < L; l += NT) {
    int32_t tok;
    const bool cand = src.cand(l, &tok);
    bool commit = false;
    if (a.rule == kRuleThreshold) {
      if (cand) {
        const float c = nan_to(src.conf(l), -__int_as_float(0x7F800000));
        commit = a.strict ? (c > a.tau) : (c >= a.tau);
        if (forced != kNoKey && static_cast<int64_t>(forced & 0xFFFFFFFFu) == l) commit = true;
      }
    } else if (a.rule != kRuleNone) {
      commit = s.flags[l] != 0;
    }
    bool edit = false;
    const int32_t x0 = src.x0(l);
    if (a.edit && !cand) {
      const float p = nan_to(src.conf(l), -__int_as_float(0x7F800000));
      edit = (x0 != tok) && (p > a.tau_edit);
    }
    emit(l, commit, edit, x0);
    n_commit += commit ? 1 : 0;
    n_edit += edit ? 1 : 0;
  }
  (void)n_commit_forced;
  if (a.counts) {
    const int4 t = rule_sum4<NT, BAR>(make_int4(n_commit, n_edit, 0, 0), s, tid);
    if (tid == 0) emit.counts(n_cand_total, t.x, t.y);
  }
  rsync<NT, BAR>();
}

// The rule of batch row b on its inputs in global memory, written there.
template <int NT, int BAR>
__device__ void run_rule(const RuleArgs& a, int64_t b, const RuleScratch& s, int tid) {
  run_rule_src<NT, BAR>(a, b, s, tid, GlobalRowSrc{a, b}, GlobalEmit{a, b});
}

}  // namespace dllm
