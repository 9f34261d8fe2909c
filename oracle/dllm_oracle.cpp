// dllm_oracle.cpp -- plain CPU oracle of the diffusion-LM commit step.
//
// TEST INFRASTRUCTURE ONLY: the slow, obviously correct reference the GPU
// library is checked against.  Only the tests, the smoke check and the bench's
// CPU-baseline leg load it.  It shares no code with the GPU library.
//
// Sources (page title, section):
//   [ARS]  "dLLM block decoding" research notes (mlx-arsenal): "The pattern",
//          "What mlx-arsenal ships" (function table), "Reference loop",
//          "Token editing (LLaDA2.1)", "Deviations from the references".
//   [MOJO] mojo-dllm manual: "The loop LLaDA uses"; "The GPU path", paragraph
//          "Row statistics on the device".
//   [MLXC] "Block Diffusion" (mlxcel manual): "Samplers and Reveal Policies".
//
// Every floating-point statistic is computed in double, two passes per row.
// The Gumbel score is an fp32 value by definition (see gumbel_score), so the
// oracle computes it in fp32 with explicit fused multiply-adds; build with
// -ffp-contract=off so no other operation is fused.
//
// Parity pins (the tests): worked examples per rule, closed forms for the
// statistics, invariants, brute force on tiny inputs, Philox against
// PyTorch's independent header-only engine, ln_p against the true logarithm
// within its derived bound, and a chi-square check of Gumbel-max sampling.

#include "dllm_oracle.h"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <limits>
#include <thread>
#include <vector>
#if defined(__linux__)
#include <sched.h>
#endif

namespace {

// ---------------------------------------------------------------------------
// Philox4x32-10, from its definition in Salmon et al., "Parallel random
// numbers: as easy as 1, 2, 3" (SC'11): ten rounds of two 32x32->64
// multiplies; the key is bumped by the Weyl constants between rounds.
// ---------------------------------------------------------------------------
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

void philox(const uint32_t in[4], const uint32_t key_in[2], uint32_t out[4]) {
  uint32_t x0 = in[0], x1 = in[1], x2 = in[2], x3 = in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    const uint64_t prod0 = static_cast<uint64_t>(kPhiloxM0) * x0;
    const uint64_t prod1 = static_cast<uint64_t>(kPhiloxM1) * x2;
    const uint32_t hi0 = static_cast<uint32_t>(prod0 >> 32), lo0 = static_cast<uint32_t>(prod0);
    const uint32_t hi1 = static_cast<uint32_t>(prod1 >> 32), lo1 = static_cast<uint32_t>(prod1);
    const uint32_t y0 = hi1 ^ x1 ^ k0;
    const uint32_t y1 = lo1;
    const uint32_t y2 = hi0 ^ x3 ^ k1;
    const uint32_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

// ---------------------------------------------------------------------------
// ln_p: the project's fp32 natural log.  x = 2^e * m with m in
// (sqrt(1/2), sqrt(2)]; ln m = 2 atanh(s), s = (m-1)/(m+1), |s| <= 0.1716,
// atanh(s) = s + s^3/3 + s^5/5 + ... + s^11/11 (the next term is below
// 2^-33 |s|).  ln x = e*ln2 + 2 atanh(s).  Valid for positive normal x, the
// only inputs the Gumbel transform produces.
// ---------------------------------------------------------------------------
float ln_p(float x) {
  uint32_t bits;
  std::memcpy(&bits, &x, 4);
  int e = static_cast<int>(bits >> 23) - 127;
  const uint32_t mbits = (bits & 0x007FFFFFu) | 0x3F800000u;
  float m;
  std::memcpy(&m, &mbits, 4);
  if (m > 0x1.6a09e6p+0f) {  // sqrt(2) rounded to fp32: fold m into (sqrt(1/2), sqrt(2)]
    m = m * 0.5f;
    e += 1;
  }
  const float s = (m - 1.0f) / (m + 1.0f);
  const float s2 = s * s;
  // Series coefficients 1/11, 1/9, 1/7, 1/5, 1/3 rounded to fp32.
  float poly = 0x1.745d18p-4f;
  poly = std::fma(poly, s2, 0x1.c71c72p-4f);
  poly = std::fma(poly, s2, 0x1.24924ap-3f);
  poly = std::fma(poly, s2, 0x1.99999ap-3f);
  poly = std::fma(poly, s2, 0x1.555556p-2f);
  const float s3 = s * s2;
  const float atanh_s = std::fma(s3, poly, s);
  return std::fma(static_cast<float>(e), 0x1.62e430p-1f /* ln 2 in fp32 */, 2.0f * atanh_s);
}

// Gumbel-perturbed score of id v in global row `row` (fp32 by definition):
//   r = Philox4x32-10(counter = (v >> 2, row_lo, row_hi, 0), key = (key_lo, key_hi))[v & 3]
//   u = (2 (r >> 9) + 1) 2^-24            exact, u in (0, 1)
//   g = -ln_p(-ln_p(u))                   standard Gumbel noise
//   s = fmaf(t, g, z)
// argmax_v s_v is a sample of softmax(z / t): the Gumbel-max trick LLaDA
// applies before its argmax ([MOJO] "The loop LLaDA uses"; [ARS] token_stats
// "greedy or Gumbel-max sampling with an explicit key").
float gumbel_score(float z, float t, uint64_t key, int64_t row, int64_t v) {
  const uint32_t ctr[4] = {static_cast<uint32_t>(static_cast<uint64_t>(v) >> 2),
                           static_cast<uint32_t>(static_cast<uint64_t>(row)),
                           static_cast<uint32_t>(static_cast<uint64_t>(row) >> 32), 0u};
  const uint32_t k[2] = {static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32)};
  uint32_t out[4];
  philox(ctr, k, out);
  const uint32_t r = out[v & 3];
  const float u = static_cast<float>(2u * (r >> 9) + 1u) * 0x1p-24f;
  const float E = -ln_p(u);
  const float g = -ln_p(E);
  return std::fma(t, g, z);
}

// A logit as the statistics see it: bf16 widens exactly to fp32 and a NaN
// counts as -inf (no probability mass, [ARS] token_stats "NaN-safe").  Every
// other value, however large, is the logit itself: finite logits go through
// the ordinary softmax, and +inf entries (if any) share the mass (the limit
// of the softmax as those logits grow together).
inline float load_logit(const void* base, int dtype, int64_t idx) {
  float z;
  if (dtype == 1) {
    const uint32_t b = static_cast<uint32_t>(static_cast<const uint16_t*>(base)[idx]) << 16;
    std::memcpy(&z, &b, 4);
  } else {
    z = static_cast<const float*>(base)[idx];
  }
  if (std::isnan(z)) return -std::numeric_limits<float>::infinity();
  return z;
}

struct RowOut {
  int32_t x0;
  double prob;
  double entropy;
  double margin;   // prob(x0) - prob(runner-up)
  int32_t argmax;  // first id of the largest scaled logit
};

// The logit of id v as the statistics see it: sanitised (load_logit), then
// scaled by the caller's fp32 factor s in one fp32 multiplication (a product
// beyond the fp32 range is +-inf; a logit with no mass keeps none).  s = 1
// leaves the logit as it is; s = 1/T gives the temperature-scaled logits the
// uniform-noise loop of "dLLM block decoding" (section "Uniform-noise
// decoding (DiffusionGemma)") measures its entropy on and samples from.
inline float scaled_logit(const void* logits, int dtype, int64_t idx, float s) {
  const float z = load_logit(logits, dtype, idx);
  if (z == -std::numeric_limits<float>::infinity()) return z;
  return z * s;
}

// token_stats for one row.  [ARS] "What mlx-arsenal ships" and "Deviations":
// per position the proposal x0, its probability and the entropy, computed
// without NaN trouble, by argmax or by Gumbel-max with a caller key; the
// suppressed ids take no part in the softmax.  [MOJO] "Row statistics on the
// device": the row max, sum exp(z - max) and sum exp(z - max)(z - max) give
// both numbers; the argmax tie rule keeps the smallest id; the argmax has
// p = 1 / sum; the largest logit at any other id gives the runner-up whose
// probability topk_margin subtracts.
RowOut stats_row(const void* logits, int dtype, int64_t row_off, int64_t V, int64_t grow,
                 float t, uint64_t key, float s, const std::vector<uint8_t>& absent, int64_t v_eff) {
  const double inf = std::numeric_limits<double>::infinity();
  auto zl = [&](int64_t v) { return scaled_logit(logits, dtype, row_off + v, s); };
  // Pass 1: the max over the token set A (ids not suppressed) and its first id.
  float m = -std::numeric_limits<float>::infinity();
  int64_t first_max = -1;
  for (int64_t v = 0; v < V; ++v) {
    if (absent[v]) continue;
    const float z = zl(v);
    if (first_max < 0 || z > m) {
      m = z;
      first_max = v;
    }
  }
  // x0: lowest id in A maximizing z (greedy) or the Gumbel score (t > 0).
  int64_t x0 = first_max;
  if (t > 0.0f) {
    float best = 0.0f;
    x0 = -1;
    for (int64_t v = 0; v < V; ++v) {
      if (absent[v]) continue;
      const float sc = gumbel_score(zl(v), t, key, grow, v);
      if (x0 < 0 || sc > best) {
        best = sc;
        x0 = v;
      }
    }
  }
  // The runner-up: the largest logit over A without x0 (-inf if A = {x0}).
  float r = -std::numeric_limits<float>::infinity();
  bool have_r = false;
  for (int64_t v = 0; v < V; ++v) {
    if (absent[v] || v == x0) continue;
    r = have_r ? std::max(r, zl(v)) : zl(v);
    have_r = true;
  }
  RowOut out{static_cast<int32_t>(x0), 0.0, 0.0, 0.0, static_cast<int32_t>(first_max)};
  const double log_veff = std::log(static_cast<double>(v_eff));
  if (m == -std::numeric_limits<float>::infinity()) {
    // No mass anywhere (every logit NaN or -inf): the uniform limit over A.
    out.prob = 1.0 / static_cast<double>(v_eff);
    out.entropy = log_veff;
    out.margin = out.prob - (have_r ? out.prob : 0.0);
    return out;
  }
  if (m == std::numeric_limits<float>::infinity()) {
    // The +inf entries share the mass equally; every finite logit has none.
    int64_t n_inf = 0;
    for (int64_t v = 0; v < V; ++v)
      if (!absent[v] && zl(v) == m) ++n_inf;
    const double share = 1.0 / static_cast<double>(n_inf);
    out.prob = zl(x0) == m ? share : 0.0;
    out.margin = out.prob - ((have_r && r == m) ? share : 0.0);
    out.entropy = std::min(std::log(static_cast<double>(n_inf)), log_veff);
    return out;
  }
  // Pass 2: Z = sum exp(z - m), S = sum exp(z - m)(z - m); -inf terms add 0.
  const double md = m;
  double Z = 0.0, S = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    if (absent[v]) continue;
    const double z = zl(v);
    if (z == -inf) continue;
    const double d = z - md;
    const double e = std::exp(d);
    Z += e;
    S += e * d;
  }
  const double zx0 = zl(x0);
  out.prob = zx0 == -inf ? 0.0 : std::exp(zx0 - md) / Z;
  const double p_r = (have_r && r != -std::numeric_limits<float>::infinity()) ? std::exp(double(r) - md) / Z : 0.0;
  out.margin = out.prob - p_r;
  // H = -sum p log p = log Z - S / Z, clamped to its range [0, log |A|].
  double H = std::log(Z) - S / Z;
  H = std::min(std::max(H, 0.0), log_veff);
  out.entropy = H;
  return out;
}

// A confidence as the rules see it: NaN ranks as -inf.
inline float conf_of(float c) { return std::isnan(c) ? -std::numeric_limits<float>::infinity() : c; }
// An entropy as the entropy-bound rule sees it: NaN ranks as +inf.
inline float ent_of(float h) { return std::isnan(h) ? std::numeric_limits<float>::infinity() : h; }

// Entropies in the exact sums of the entropy-bound rule and the stopping
// criterion: fixed point with 40 fractional bits, q(h) = floor(min(max(h, 0),
// 64) 2^40), NaN counting as 64.  Exact: the clamped value times 2^40 is an
// integer-or-fraction fp32 value below 2^46 whose floor converts exactly, and
// sums of at most 2^16 of them stay below 2^62.
int64_t fixed_q(float h) {
  const float c = std::isnan(h) ? 64.0f : std::min(std::max(h, 0.0f), 64.0f);
  return static_cast<int64_t>(std::floor(static_cast<double>(c) * 1099511627776.0));
}

// A bound compared with such a sum: S <= bound <=> S <= floor(bound 2^40)
// (S is an integer); -1 for a negative bound (nothing is within it); bounds
// above 2^22 (more than any sum reaches) count as 2^22.
int64_t fixed_bound(float bound) {
  if (bound < 0.0f) return -1;
  return static_cast<int64_t>(std::floor(static_cast<double>(std::min(bound, 4194304.0f)) * 1099511627776.0));
}

// Candidate positions of batch row b, ranked by descending confidence.  The
// sort is stable: among equal confidences the smaller position ranks first
// ([ARS] "Deviations", the paragraph on ties).
std::vector<int64_t> rank_desc(const float* conf, const uint8_t* cand, int64_t b, int64_t L) {
  std::vector<int64_t> pos;
  for (int64_t l = 0; l < L; ++l)
    if (cand[b * L + l]) pos.push_back(l);
  std::stable_sort(pos.begin(), pos.end(), [&](int64_t a, int64_t c) {
    return conf_of(conf[b * L + a]) > conf_of(conf[b * L + c]);
  });
  return pos;
}

int resolve_threads(int n) {
  if (n > 0) return n;
  return orc_default_threads();
}

}  // namespace

extern "C" {

int orc_default_threads(void) {
#if defined(__linux__)
  cpu_set_t set;
  if (sched_getaffinity(0, sizeof(set), &set) == 0) {
    const int c = CPU_COUNT(&set);
    if (c > 0) return c;
  }
#endif
  const unsigned h = std::thread::hardware_concurrency();
  return h ? static_cast<int>(h) : 1;
}

void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  philox(ctr, key, out);
}

float orc_ln_p(float x) { return ln_p(x); }

void orc_ln_p_many(const float* x, int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = ln_p(x[i]);
}

float orc_gumbel_score(float z, float temperature, uint64_t key, int64_t row, int64_t v) {
  return gumbel_score(z, temperature, key, row, v);
}

int orc_token_stats_ex(const void* logits, int dtype, int64_t n_rows, int64_t V, int64_t row_stride,
                       const int64_t* row_ids, float temperature, uint64_t key, float logit_scale,
                       const int32_t* suppress_ids, int32_t n_suppress,
                       int32_t* x0, double* prob, double* entropy, double* margin, int32_t* argmax,
                       int n_threads) {
  if (n_rows < 0 || V <= 0 || row_stride < V || (dtype != 0 && dtype != 1)) return -1;
  if (!(temperature >= 0.0f) || n_suppress < 0) return -1;
  if (!(logit_scale > 0.0f) || !(logit_scale <= 256.0f)) return -1;
  if (n_rows == 0) return 0;
  if (!logits || !x0 || !prob || !entropy) return -1;
  std::vector<uint8_t> absent(static_cast<size_t>(V), 0);
  for (int32_t i = 0; i < n_suppress; ++i) {
    if (suppress_ids[i] < 0 || suppress_ids[i] >= V) return -1;
    absent[suppress_ids[i]] = 1;
  }
  int64_t v_eff = 0;
  for (int64_t v = 0; v < V; ++v) v_eff += absent[v] ? 0 : 1;
  if (v_eff == 0) return -1;  // an empty token set has no distribution

  const int nt = static_cast<int>(std::min<int64_t>(resolve_threads(n_threads), n_rows));
  auto work = [&](int tid) {
    for (int64_t r = tid; r < n_rows; r += nt) {
      const int64_t grow = row_ids ? row_ids[r] : r;
      const RowOut o = stats_row(logits, dtype, r * row_stride, V, grow, temperature, key, logit_scale, absent, v_eff);
      x0[r] = o.x0;
      prob[r] = o.prob;
      entropy[r] = o.entropy;
      if (margin) margin[r] = o.margin;
      if (argmax) argmax[r] = o.argmax;
    }
  };
  if (nt <= 1) {
    work(0);
  } else {
    std::vector<std::thread> pool;
    for (int i = 0; i < nt; ++i) pool.emplace_back(work, i);
    for (auto& th : pool) th.join();
  }
  return 0;
}

int orc_token_stats(const void* logits, int dtype, int64_t n_rows, int64_t V, int64_t row_stride,
                    const int64_t* row_ids, float temperature, uint64_t key,
                    const int32_t* suppress_ids, int32_t n_suppress,
                    int32_t* x0, double* prob, double* entropy, int n_threads) {
  return orc_token_stats_ex(logits, dtype, n_rows, V, row_stride, row_ids, temperature, key, 1.0f, suppress_ids,
                            n_suppress, x0, prob, entropy, nullptr, nullptr, n_threads);
}

// threshold_transfer.  [ARS] function table: a candidate commits when its
// confidence reaches tau (exceeds it in strict mode); a row where nobody
// qualifies commits exactly one.  [ARS] "Deviations": that one is the earliest
// of the maximal confidences.  [MLXC] "Samplers and Reveal Policies": the
// forced commit is what makes every step progress.
int orc_threshold_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L,
                           float tau, int strict, uint8_t* commit) {
  if (B < 0 || L < 0) return -1;
  for (int64_t b = 0; b < B; ++b) {
    bool any_cand = false, any_pass = false;
    int64_t best = -1;
    for (int64_t l = 0; l < L; ++l) {
      const int64_t i = b * L + l;
      commit[i] = 0;
      if (!cand[i]) continue;
      any_cand = true;
      const float c = conf_of(conf[i]);
      const bool pass = strict ? (c > tau) : (c >= tau);
      if (pass) {
        commit[i] = 1;
        any_pass = true;
      }
      if (best < 0 || c > conf_of(conf[b * L + best])) best = l;
    }
    if (any_cand && !any_pass) commit[b * L + best] = 1;
  }
  return 0;
}

// topk_transfer.  [ARS] function table: each row commits its k best
// candidates, with its own k.  [MOJO] "The loop LLaDA uses": this is LLaDA's
// low-confidence remasking.  k is clamped to [0, number of candidates].
int orc_topk_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L,
                      const int32_t* k, uint8_t* commit) {
  if (B < 0 || L < 0) return -1;
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t l = 0; l < L; ++l) commit[b * L + l] = 0;
    const std::vector<int64_t> order = rank_desc(conf, cand, b, L);
    const int64_t kk = std::min<int64_t>(std::max<int64_t>(k[b], 0), static_cast<int64_t>(order.size()));
    for (int64_t i = 0; i < kk; ++i) commit[b * L + order[i]] = 1;
  }
  return 0;
}

// factor_transfer.  [ARS] function table: the longest prefix of the ranking
// with (i+1)(1 - c_(i)) <= f, c_(i) the i-th largest confidence; [ARS]
// "Deviations": the Fast-dLLM off-by-one is not reproduced.  The product is
// evaluated in double, and a row with candidates commits at least one.
int orc_factor_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L,
                        float factor, uint8_t* commit) {
  if (B < 0 || L < 0) return -1;
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t l = 0; l < L; ++l) commit[b * L + l] = 0;
    const std::vector<int64_t> order = rank_desc(conf, cand, b, L);
    const int64_t n_cand = static_cast<int64_t>(order.size());
    int64_t n = 0;
    while (n < n_cand) {
      const double c = conf_of(conf[b * L + order[n]]);
      const double lhs = static_cast<double>(n + 1) * (1.0 - c);
      if (!(lhs <= static_cast<double>(factor))) break;
      ++n;
    }
    if (n_cand > 0) n = std::max<int64_t>(n, 1);
    for (int64_t i = 0; i < n; ++i) commit[b * L + order[i]] = 1;
  }
  return 0;
}

// entropy_bound_transfer.  [ARS] function table: rank by ascending entropy
// and take the longest prefix whose members satisfy sum_{j<i} H_(j) <= gamma.
// [MLXC] "Samplers and Reveal Policies": the rule always accepts one position
// or more.  The pages fix no precision for the sum: it is taken exactly, in
// the fixed point of fixed_q (40 fractional bits), and compared exactly with
// gamma.
int orc_entropy_bound_transfer(const float* entropy, const uint8_t* cand, int64_t B, int64_t L,
                               float gamma, uint8_t* commit) {
  if (B < 0 || L < 0 || L > (static_cast<int64_t>(1) << 16) || std::isnan(gamma)) return -1;
  for (int64_t b = 0; b < B; ++b) {
    std::vector<int64_t> order;
    for (int64_t l = 0; l < L; ++l) {
      commit[b * L + l] = 0;
      if (cand[b * L + l]) order.push_back(l);
    }
    std::stable_sort(order.begin(), order.end(), [&](int64_t a, int64_t c) {
      return ent_of(entropy[b * L + a]) < ent_of(entropy[b * L + c]);
    });
    const int64_t n_cand = static_cast<int64_t>(order.size());
    // The prefix sums are exact in the fixed point of fixed_q, compared
    // exactly with gamma (fixed_bound).
    const int64_t gamma_q = fixed_bound(gamma);
    int64_t prefix = 0;   // sum of q(H) over the entropies ranked before position i
    int64_t n = 0;
    while (n < n_cand && prefix <= gamma_q) {
      prefix += fixed_q(ent_of(entropy[b * L + order[n]]));
      ++n;
    }
    if (n_cand > 0) n = std::max<int64_t>(n, 1);
    for (int64_t i = 0; i < n; ++i) commit[b * L + order[i]] = 1;
  }
  return 0;
}

// edit_transfer.  [ARS] function table and "Token editing (LLaDA2.1)": an
// already decoded (editable) position is rewritten with the proposal when the
// proposal differs from the current token and its probability is strictly
// above tau_edit.
int orc_edit_transfer(const int32_t* x0, const float* prob, const int32_t* tokens,
                      const uint8_t* editable, int64_t n, float tau_edit, uint8_t* edit) {
  if (n < 0) return -1;
  for (int64_t i = 0; i < n; ++i) {
    const float p = conf_of(prob[i]);
    edit[i] = (editable[i] && x0[i] != tokens[i] && p > tau_edit) ? 1 : 0;
  }
  return 0;
}

// transfer_schedule.  [ARS] function table: a (B, steps) table of per-step
// quotas in LLaDA's linear style; [MOJO] "The loop LLaDA uses": a block's
// masked count is divided evenly among its steps.  The remainder goes to the
// first steps; a negative count is treated as zero.
int orc_transfer_schedule(const int32_t* counts, int64_t B, int32_t steps, int32_t* quotas) {
  if (B < 0 || steps <= 0) return -1;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t n = std::max<int32_t>(counts[b], 0);
    for (int32_t s = 0; s < steps; ++s)
      quotas[b * steps + s] = static_cast<int32_t>(n / steps + (s < n % steps ? 1 : 0));
  }
  return 0;
}

// block_ranges.  [ARS] function table, "Reference loop" and "Token editing
// (LLaDA2.1)": block boundaries either counted from the end of the prompt or
// aligned on absolute multiples of the block length.  Prompt-relative blocks
// start at P; aligned blocks start at floor(P / bl) * bl.  Every block ends at
// min(start + bl, P + gen_len).
int orc_block_ranges(int64_t P, int64_t gen_len, int64_t block_len, int align,
                     int64_t* ranges, int64_t cap, int64_t* n_out) {
  if (P < 0 || gen_len < 0 || block_len <= 0 || cap < 0 || !n_out) return -1;
  const int64_t first = align ? (P / block_len) * block_len : P;
  const int64_t stop = P + gen_len;
  int64_t n = 0;
  if (gen_len > 0) {
    for (int64_t start = first; start < stop; start += block_len) {
      if (n < cap && ranges) {
        ranges[2 * n] = start;
        ranges[2 * n + 1] = std::min(start + block_len, stop);
      }
      ++n;
    }
  }
  *n_out = n;
  return n > cap ? -2 : 0;
}

// The helpers of uniform-noise decoding.  [ARS] function table
// (linear_temperature, uniform_canvas, renoise, StableConfidentStopping) and
// "Uniform-noise decoding (DiffusionGemma)": the canvas starts as uniformly
// random tokens, the temperature decays linearly with the steps that remain,
// the positions not accepted are re-noised, and a row stops once its argmax
// canvas is stable and confident.

// T = t_min + (t_max - t_min) remaining / num_steps, in double, rounded to fp32.
int orc_linear_temperature(int32_t remaining, int32_t num_steps, float t_min, float t_max, float* T) {
  if (num_steps <= 0 || remaining < 0 || remaining > num_steps || !T) return -1;
  if (!(t_min > 0.0f) || !(t_max >= t_min) || std::isinf(t_max)) return -1;
  const double frac = static_cast<double>(remaining) / static_cast<double>(num_steps);
  *T = static_cast<float>(static_cast<double>(t_min) + (static_cast<double>(t_max) - t_min) * frac);
  return 0;
}

// canvas[b, j] = floor(r V / 2^32), r = Philox4x32-10(counter (j >> 2, b lo,
// b hi, 1), key (lo, hi)), word j & 3: every token of [0, V) is drawn with
// probability within V / 2^32 of 1 / V.
int orc_uniform_canvas(int64_t B, int64_t N, int64_t V, uint64_t key, int32_t* canvas) {
  if (B < 0 || N < 0 || V <= 0 || V > INT32_MAX || (B * N > 0 && !canvas)) return -1;
  const uint32_t k[2] = {static_cast<uint32_t>(key), static_cast<uint32_t>(key >> 32)};
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t j = 0; j < N; ++j) {
      const uint32_t ctr[4] = {static_cast<uint32_t>(j >> 2), static_cast<uint32_t>(b),
                               static_cast<uint32_t>(static_cast<uint64_t>(b) >> 32), 1u};
      uint32_t out[4];
      philox(ctr, k, out);
      const uint64_t r = out[j & 3];
      canvas[b * N + j] = static_cast<int32_t>((r * static_cast<uint64_t>(V)) >> 32);
    }
  }
  return 0;
}

// out[i] = accepted[i] ? sample[i] : noise[i].
int orc_renoise(const int32_t* sample, const uint8_t* accepted, const int32_t* noise, int64_t n, int32_t* out) {
  if (n < 0 || (n > 0 && (!sample || !accepted || !noise || !out))) return -1;
  for (int64_t i = 0; i < n; ++i) out[i] = accepted[i] ? sample[i] : noise[i];
  return 0;
}

// One call of the stopping criterion on the (B, L) argmax canvas and
// entropies.  count[b] < 0 means no previous canvas.  A row is stable when
// its canvas equals the previous one; count[b] counts consecutive stable
// calls; the row is confident when its mean entropy is below
// confidence_threshold, compared exactly in the fixed point of fixed_q:
// sum_l q(H_l) < L q(threshold).  stop[b] = count[b] >= stability_threshold
// and confident.  prev takes the canvas.  L <= 2^16, 0 <= threshold <= 64.
int orc_stable_confident_stop(const int32_t* argmax, const float* entropy, int64_t B, int64_t L,
                              int32_t stability_threshold, float confidence_threshold, int32_t* prev,
                              int32_t* count, uint8_t* stop) {
  if (B < 0 || L <= 0 || L > (static_cast<int64_t>(1) << 16) || stability_threshold < 0) return -1;
  if (!(confidence_threshold >= 0.0f && confidence_threshold <= 64.0f)) return -1;
  if (B > 0 && (!argmax || !entropy || !prev || !count || !stop)) return -1;
  const int64_t thr_q = fixed_q(confidence_threshold);
  for (int64_t b = 0; b < B; ++b) {
    bool same = count[b] >= 0;
    int64_t sum = 0;
    for (int64_t l = 0; l < L; ++l) {
      same = same && argmax[b * L + l] == prev[b * L + l];
      sum += fixed_q(entropy[b * L + l]);
    }
    count[b] = same ? count[b] + 1 : 0;
    for (int64_t l = 0; l < L; ++l) prev[b * L + l] = argmax[b * L + l];
    const bool confident = sum < L * thr_q;
    stop[b] = (count[b] >= stability_threshold && confident) ? 1 : 0;
  }
  return 0;
}

// block_causal_mask.  [ARS] "What mlx-arsenal ships" (attention): the mask
// block-diffusion models are trained with -- bidirectional inside a block,
// causal across blocks, blocks aligned on absolute positions; "Mask
// conventions": additive, 0 where attention is allowed and -inf where it is
// blocked.  Query i sits at absolute position q_offset + i, key j at
// k_offset + j; attend iff block(query) >= block(key), block(p) =
// floor(p / block_len).  out: (Lq, Lk) row-major doubles.
int orc_block_causal_mask(int64_t Lq, int64_t Lk, int64_t q_offset, int64_t k_offset, int64_t block_len,
                          double* out) {
  if (Lq < 0 || Lk < 0 || q_offset < 0 || k_offset < 0 || block_len <= 0 || (Lq * Lk > 0 && !out)) return -1;
  for (int64_t i = 0; i < Lq; ++i) {
    const int64_t bq = (q_offset + i) / block_len;
    for (int64_t j = 0; j < Lk; ++j) {
      const int64_t bk = (k_offset + j) / block_len;
      out[i * Lk + j] = bq >= bk ? 0.0 : -std::numeric_limits<double>::infinity();
    }
  }
  return 0;
}

}  // extern "C"
