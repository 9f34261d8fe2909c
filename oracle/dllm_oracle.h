/*
 * dllm_oracle.h -- plain CPU oracle of the diffusion-LM commit step.
 *
 * TEST INFRASTRUCTURE ONLY.  This header, its implementation and the Python
 * wrapper beside them are the slow, obviously correct reference that the GPU
 * library is checked against.  Only the tests, the smoke check and the
 * bench's CPU-baseline leg may load them; the product path never does.
 *
 * All functions are synchronous host code on host pointers and return 0 on
 * success, a negative value on invalid arguments.
 */
#ifndef DLLM_ORACLE_H
#define DLLM_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): out = philox(ctr, key). */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* The project's fp32 natural logarithm (exponent split + atanh series).
 * Pinned to <= 2.5 ulp of the double logarithm over every u the sampler can
 * draw; its exact bits are this project's own definition, which no value on
 * the pages fixes: parity unpinned beyond that error bound. */
float orc_ln_p(float x);
void orc_ln_p_many(const float* x, int64_t n, float* out);

/* The fp32 Gumbel-perturbed score of vocabulary id v in global row `row`. */
float orc_gumbel_score(float z, float temperature, uint64_t key, int64_t row, int64_t v);

/* Statistics pass: x0, prob and entropy per row, in double.
 * logits: (n_rows, row_stride) row-major; dtype 0 = float32, 1 = bf16 bits.
 * row_ids (nullable): the global row index of each given row (feeds the
 * Gumbel counter); NULL means row i is global row i.
 * n_threads: 0 = every core the process may use. */
int orc_token_stats(const void* logits, int dtype, int64_t n_rows, int64_t V, int64_t row_stride,
                    const int64_t* row_ids, float temperature, uint64_t key,
                    const int32_t* suppress_ids, int32_t n_suppress,
                    int32_t* x0, double* prob, double* entropy, int n_threads);

/* The same pass on scaled logits z' = fp32(z * logit_scale), 0 < logit_scale
 * <= 256 (1 = orc_token_stats).  margin (nullable): prob(x0) minus the
 * probability of the runner-up, the largest z' over the token set without
 * x0.  argmax (nullable): the first id of the largest z' (equal to x0 when
 * temperature == 0). */
int orc_token_stats_ex(const void* logits, int dtype, int64_t n_rows, int64_t V, int64_t row_stride,
                       const int64_t* row_ids, float temperature, uint64_t key, float logit_scale,
                       const int32_t* suppress_ids, int32_t n_suppress,
                       int32_t* x0, double* prob, double* entropy, double* margin, int32_t* argmax,
                       int n_threads);

/* Commit rules over (B, L) row-major confidences and 0/1 candidate masks.
 * entropy_bound sums the ranked entropies exactly in fixed point with 40
 * fractional bits (q as in stable_confident_stop) and compares exactly with
 * gamma; L <= 2^16. */
int orc_threshold_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L,
                           float tau, int strict, uint8_t* commit);
int orc_topk_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L,
                      const int32_t* k, uint8_t* commit);
int orc_factor_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L,
                        float factor, uint8_t* commit);
int orc_entropy_bound_transfer(const float* entropy, const uint8_t* cand, int64_t B, int64_t L,
                               float gamma, uint8_t* commit);
int orc_edit_transfer(const int32_t* x0, const float* prob, const int32_t* tokens,
                      const uint8_t* editable, int64_t n, float tau_edit, uint8_t* edit);

/* Schedules. */
int orc_transfer_schedule(const int32_t* counts, int64_t B, int32_t steps, int32_t* quotas);
int orc_block_ranges(int64_t P, int64_t gen_len, int64_t block_len, int align,
                     int64_t* ranges, int64_t cap, int64_t* n_out);

/* Uniform-noise decoding helpers ("dLLM block decoding", function table and
 * "Uniform-noise decoding (DiffusionGemma)").
 * linear_temperature: T = fp32(t_min + (t_max - t_min) remaining / num_steps).
 * uniform_canvas: (B, N) tokens floor(r V / 2^32), r the Philox4x32-10 word
 *   j & 3 of counter (j >> 2, b lo, b hi, 1) under key.
 * renoise: out = accepted ? sample : noise, elementwise.
 * stable_confident_stop: one call of the stopping criterion; state prev
 *   (B, L) and count (B) (count < 0: no previous canvas); a row is confident
 *   when sum_l q(H_l) < L q(threshold), q(h) = floor(clamp(h, 0, 64) 2^40)
 *   (NaN as 64): the mean entropy against the threshold, exactly.  L <= 2^16. */
int orc_linear_temperature(int32_t remaining, int32_t num_steps, float t_min, float t_max, float* T);
int orc_uniform_canvas(int64_t B, int64_t N, int64_t V, uint64_t key, int32_t* canvas);
int orc_renoise(const int32_t* sample, const uint8_t* accepted, const int32_t* noise, int64_t n, int32_t* out);
int orc_stable_confident_stop(const int32_t* argmax, const float* entropy, int64_t B, int64_t L,
                              int32_t stability_threshold, float confidence_threshold, int32_t* prev,
                              int32_t* count, uint8_t* stop);

/* block_causal_mask ("dLLM block decoding", attention helper and "Mask
 * conventions"): out[i, j] = 0 if floor((q_offset + i) / block_len) >=
 * floor((k_offset + j) / block_len), else -inf.  (Lq, Lk) row-major. */
int orc_block_causal_mask(int64_t Lq, int64_t Lk, int64_t q_offset, int64_t k_offset, int64_t block_len,
                          double* out);

/* Threads orc_token_stats uses when asked for 0. */
int orc_default_threads(void);

#ifdef __cplusplus
}
#endif
#endif /* DLLM_ORACLE_H */
