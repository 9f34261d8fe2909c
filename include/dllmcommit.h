/*
 * dllmcommit.h -- C ABI of libdllmcommit, the commit step of masked
 * (absorbing-state) diffusion-LM block decoding on NVIDIA GB300 (sm_103a).
 *
 * The commit step splits into a statistics pass over the (B, L, V) logits and
 * a commit rule over each batch row's masked candidates, plus the schedules
 * that go with the rules.  Citations name the page and its section:
 *   [ARS]  "dLLM block decoding" research notes (mlx-arsenal): "The pattern",
 *          "What mlx-arsenal ships", "Reference loop", "Token editing
 *          (LLaDA2.1)", "Deviations from the references".
 *   [MOJO] mojo-dllm manual: "The loop LLaDA uses"; "The GPU path",
 *          paragraph "Row statistics on the device".
 *   [MLXC] "Block Diffusion" (mlxcel manual): "Samplers and Reveal Policies".
 *
 * Conventions shared by every entry point:
 *   - The caller owns every buffer.  "device" pointers are CUDA device
 *     memory; "host" pointers are ordinary host memory.  Nothing here
 *     allocates memory.
 *   - Every device-side call is asynchronous on the given stream (0 = the
 *     legacy default stream) and is launched with programmatic dependent
 *     launch, so its prologue may overlap the previous kernel in the stream;
 *     it reads no input before that kernel has finished, except where a
 *     declaration says so (DLLM_FLAG_INPUTS_READY of dllm_commit_step; the
 *     first weight slabs of dllm_lm_head_stats).
 *   - Arguments are validated on the host first; on any error nothing is
 *     launched and the status says why.  A failed launch returns
 *     DLLM_ERR_CUDA (the CUDA error is left for cudaGetLastError).
 *   - Boolean masks are uint8 0/1 (any non-zero byte reads as 1); token ids
 *     are int32; (B, L) arrays are row-major and contiguous; strides are in
 *     elements.
 *   - B == 0 or L == 0 is a valid empty call: nothing is launched.
 *   - Calls on different streams must not share output buffers or a
 *     workspace.
 */
#ifndef DLLMCOMMIT_H
#define DLLMCOMMIT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dllm_stream_t; /* a cudaStream_t */

typedef enum {
  DLLM_OK = 0,
  DLLM_ERR_INVALID_ARGUMENT = 1, /* a shape, pointer, value or alignment is wrong */
  DLLM_ERR_UNSUPPORTED = 2,      /* valid, but outside what this library version handles */
  DLLM_ERR_WORKSPACE = 3,        /* workspace missing or smaller than required */
  DLLM_ERR_CUDA = 4,             /* a CUDA launch or query failed */
  DLLM_ERR_DEVICE = 5            /* reserved: calls are asynchronous, so a kernel's fault is
                                    reported by dllm_workspace_fault, not by the call */
} dllm_status;

typedef enum { DLLM_F32 = 0, DLLM_BF16 = 1 } dllm_dtype;

/* Largest suppress_ids list a statistics call accepts. */
#define DLLM_MAX_SUPPRESS 64
/* Largest L the sorting rules (top-k, factor, entropy bound) accept. */
#define DLLM_MAX_SORT_L 16384

const char* dllm_status_string(dllm_status status);
const char* dllm_version(void);

/* ------------------------------------------------------------------------
 * Statistics pass ([ARS] "What mlx-arsenal ships", token_stats; [MOJO] "Row
 * statistics on the device").
 *
 * For each of the T = B*L logit rows, over the token set A = {0..V-1} minus
 * suppress_ids:
 *   x0      the proposal: the lowest id in A maximising z (temperature == 0),
 *           or maximising the Gumbel score fmaf(t, g_v, z_v) (temperature
 *           t > 0), g_v = -ln_p(-ln_p(u_v)), u_v from Philox4x32-10 with
 *           counter (v >> 2, row lo, row hi, 0), key (key lo, key hi), word
 *           v & 3, u = (2 (r >> 9) + 1) 2^-24; row = b*L + l.
 *   prob    exp(z_x0 - m) / sum_A exp(z - m) of the untempered softmax.
 *   entropy ln Z - S / Z of the same softmax, clamped to [0, ln |A|].
 * bf16 logits widen exactly to fp32.  A NaN carries no mass; every other
 * value is the logit itself: finite logits of any size take the ordinary
 * softmax, +inf entries share all the mass equally, and a row whose every
 * entry carries no mass (NaN or -inf) yields the uniform limit (x0 = min A,
 * prob = 1/|A|, entropy = ln |A|).  Sums are accumulated in fp32.  Rows
 * whose largest logit exceeds about 1.8e8 in magnitude (1.8e8 / s for
 * scaled logits), or that hold no logit above -2^100, are recomputed by a
 * slower exact path inside the same launch (one warp, two or three extra
 * reads of the row); model logits never reach it.
 * temperature   0 (greedy) or a Gumbel temperature in (0, 2^64]; NaN,
 *               negative, infinite or larger values: DLLM_ERR_INVALID_ARGUMENT.
 *
 * logits        device, T rows of row_stride elements (dtype dt); the base
 *               pointer and row_stride * sizeof(element) must be multiples of
 *               16 bytes (else DLLM_ERR_UNSUPPORTED).
 * suppress_ids  HOST array of n_suppress ids in [0, V) (duplicates allowed),
 *               0 <= n_suppress <= DLLM_MAX_SUPPRESS, fewer than |V| distinct.
 * x0, prob, entropy   device outputs, T entries each.
 * workspace     device, >= dllm_token_stats_workspace_size(B, L, V, dt)
 *               bytes, zero-filled before its first use; every call leaves it
 *               zeroed again (the library resets what it uses).  The size
 *               query returns 0 for a negative shape or one beyond 2^56 rows.
 * Errors: DLLM_ERR_INVALID_ARGUMENT also when T * row_stride * 4 does not fit
 * in int64 (no such buffer exists); nothing is launched on any error.
 * ------------------------------------------------------------------------ */
size_t dllm_token_stats_workspace_size(int64_t B, int64_t L, int64_t V, dllm_dtype dt);

dllm_status dllm_token_stats(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V,
                             int64_t row_stride, float temperature, uint64_t key,
                             const int32_t* suppress_ids, int32_t n_suppress,
                             int32_t* x0, float* prob, float* entropy,
                             void* workspace, size_t workspace_bytes, dllm_stream_t stream);

/* ------------------------------------------------------------------------
 * Extended statistics: scaled logits, margin confidence, greedy argmax
 * beside a sample.
 *
 * [MOJO] "Row statistics on the device": besides p = 1/Z, the sampler
 * finishes topk_margin as p minus the runner-up's probability, the runner-up
 * being the largest logit at any other index.  [ARS] "Uniform-noise decoding
 * (DiffusionGemma)": the loop divides the logits by a temperature, measures
 * the entropy of the scaled softmax, keeps the argmax canvas and draws a
 * categorical sample from the same scaled logits.
 *
 * All statistics are those of z' = fp32(z * logit_scale) (one fp32
 * multiplication of the sanitised logit; 1 = unscaled).  x0 is the first
 * argmax of z' (temperature 0) or the Gumbel-max sample of z' (temperature t;
 * t = 1 samples softmax(z')), prob and entropy are those of softmax(z').
 *   margin  prob(x0) - prob(r), r the largest z' over A without x0 (its
 *           probability counts as 0 when A = {x0}).  Negative only when a
 *           sample is not the argmax.
 *   argmax  the first id of the largest z' (equals x0 when temperature == 0).
 * Within tolerance, prob/entropy/margin follow from z * logit_scale rounded
 * once; x0 and argmax are decided on fp32(z * logit_scale) exactly.
 * ------------------------------------------------------------------------ */
typedef struct {
  float logit_scale;        /* 0 < logit_scale <= 256 (else DLLM_ERR_INVALID_ARGUMENT) */
  float* margin;            /* device (B, L) output or NULL */
  int32_t* argmax;          /* device (B, L) output or NULL */
} dllm_stats_ex;

/* dllm_token_stats with the options above (ex == NULL: plain token_stats).
 * Same arguments, workspace and errors otherwise. */
dllm_status dllm_token_stats_ex(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V,
                                int64_t row_stride, float temperature, uint64_t key,
                                const int32_t* suppress_ids, int32_t n_suppress, const dllm_stats_ex* ex,
                                int32_t* x0, float* prob, float* entropy,
                                void* workspace, size_t workspace_bytes, dllm_stream_t stream);

/* ------------------------------------------------------------------------
 * Statistics pass that allocates nothing.  The pages have no counterpart:
 * this entry point is an addition of this library.
 *
 * For callers that may not allocate device memory at all: code whose memory
 * is wholly owned by another allocator (a framework's caching pool, where a
 * cudaMalloc outside the pool can fail or fragment it), inference-server and
 * plugin hosts that hand a kernel only its input and output buffers, and
 * latency-critical loops that forbid allocation after warm-up because
 * cudaMalloc and cudaFree synchronise the device.
 *
 * Arguments, results and errors are those of dllm_token_stats without the
 * workspace.  The scratch memory is one fixed device array inside the
 * library, DLLM_NOALLOC_SCRATCH_BYTES per GPU, held by every GPU that loads
 * the library until the process exits.  A shape whose scratch does not fit
 * (4 bytes per row and 16 per batch row, plus about 40 KB for the partial
 * reductions, so B*L up to roughly 250,000 rows) returns
 * DLLM_ERR_UNSUPPORTED without launching anything.
 *   - The logits and outputs must be on the current CUDA device: the call
 *     takes the array, the device's launch limits and (stream 0) the
 *     default stream from it.
 *   - The first call on each device looks the array's device address up
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.  With CUDA's lazy module loading (the
 *     default), the driver reserves the array on a device only when the
 *     library's kernels are first loaded there, which can be that first
 *     call: make one call of any entry point on each device during warm-up,
 *     before a section that must not allocate.
 *   - Every call first clears the part of the array it uses
 *     (cudaMemsetAsync on the stream), then launches the kernel; nothing is
 *     allocated or freed.
 *   - All calls share the one array and it keeps the last call's contents:
 *     calls that can overlap on the GPU (other streams, other host threads)
 *     race with each other and give wrong results.  Serialise them.
 *   - A kernel fault (a bounded wait that ran out; see dllm_workspace_fault)
 *     is recorded in the array's first word.  dllm_noalloc_fault reads it;
 *     the next dllm_token_stats_noalloc call clears it, so read it after a
 *     call and before the next one.
 * ------------------------------------------------------------------------ */
#define DLLM_NOALLOC_SCRATCH_BYTES (1u << 20)

dllm_status dllm_token_stats_noalloc(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V,
                                     int64_t row_stride, float temperature, uint64_t key,
                                     const int32_t* suppress_ids, int32_t n_suppress,
                                     int32_t* x0, float* prob, float* entropy, dllm_stream_t stream);

/* The fault word of the allocation-free entry's array on the current device,
 * as dllm_workspace_fault reads a workspace's: synchronises `stream`, stores
 * the code in *fault (0: none) and clears the word if it was set.  Errors:
 * DLLM_ERR_INVALID_ARGUMENT for a NULL fault, DLLM_ERR_CUDA if the copy or
 * the synchronisation fails. */
dllm_status dllm_noalloc_fault(dllm_stream_t stream, int32_t* fault);

/* ------------------------------------------------------------------------
 * Commit rules.  One batch row b of L positions; cand (device, (B, L)) marks
 * the masked candidates; commit (device, (B, L)) is written for every
 * position (0 for non-candidates).  Ranking: higher confidence first (NaN
 * ranks as -inf), ties to the lower position; for the entropy bound, lower
 * entropy first (NaN ranks as +inf), ties to the lower position.
 *
 * Optional canvas update, the where(commit, x0, x) of the reference loops:
 * when x0 (device, (B, L)) and canvas (device) are both non-NULL, every
 * committed (b, l) sets canvas[b * canvas_stride + canvas_offset + l] =
 * x0[b * L + l].  Pass NULL for both to skip it.
 * ------------------------------------------------------------------------ */

/* [ARS] threshold_transfer; [MLXC] forced progress: commit cand with
 * conf >= tau (conf > tau when strict != 0); a row with candidates and none
 * passing commits exactly one, the earliest maximal confidence. */
dllm_status dllm_threshold_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L,
                                    float tau, int strict, uint8_t* commit,
                                    const int32_t* x0, int32_t* canvas, int64_t canvas_stride,
                                    int64_t canvas_offset, dllm_stream_t stream);

/* [ARS] topk_transfer; [MOJO] "The loop LLaDA uses": commit the first
 * min(max(k[b], 0), n_cand) candidates of the ranking.  k: device (B,). */
dllm_status dllm_topk_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L,
                               const int32_t* k, uint8_t* commit,
                               const int32_t* x0, int32_t* canvas, int64_t canvas_stride,
                               int64_t canvas_offset, dllm_stream_t stream);

/* [ARS] factor_transfer (without Fast-dLLM's off-by-one): commit the longest
 * prefix of the ranking with (i+1)(1 - c_(i)) <= f, the product evaluated in
 * double; at least one when the row has candidates. */
dllm_status dllm_factor_transfer(const float* conf, const uint8_t* cand, int64_t B, int64_t L,
                                 float factor, uint8_t* commit,
                                 const int32_t* x0, int32_t* canvas, int64_t canvas_stride,
                                 int64_t canvas_offset, dllm_stream_t stream);

/* [ARS] entropy_bound_transfer; [MLXC] at least one accepted: commit the
 * longest prefix of the ascending-entropy ranking whose members have
 * sum_{j<i} H_(j) <= gamma, the sum taken exactly in fixed point with 40
 * fractional bits (each H as floor(clamp(H, 0, 64) 2^40), NaN ranking last)
 * and compared exactly with gamma; at least one when the row has candidates. */
dllm_status dllm_entropy_bound_transfer(const float* entropy, const uint8_t* cand, int64_t B,
                                        int64_t L, float gamma, uint8_t* commit,
                                        const int32_t* x0, int32_t* canvas, int64_t canvas_stride,
                                        int64_t canvas_offset, dllm_stream_t stream);

/* [ARS] edit_transfer and "Token editing (LLaDA2.1)": edit[i] = editable[i]
 * && x0[i] != tokens[i] && prob[i] > tau_edit (NaN prob never edits).  All
 * arrays device, B*L entries. */
dllm_status dllm_edit_transfer(const int32_t* x0, const float* prob, const int32_t* tokens,
                               const uint8_t* editable, int64_t B, int64_t L, float tau_edit,
                               uint8_t* edit, dllm_stream_t stream);

/* [ARS] transfer_schedule; [MOJO] even split over a block's steps:
 * quotas[b, s] = n_b / steps + (s < n_b mod steps), n_b = max(counts[b], 0).
 * counts: device (B,); quotas: device (B, steps).  steps > 0. */
dllm_status dllm_transfer_schedule(const int32_t* counts, int64_t B, int32_t steps,
                                   int32_t* quotas, dllm_stream_t stream);

/* [ARS] block_ranges, "Reference loop", "Token editing": host-only, pure.
 * Blocks start at P (align == 0) or at floor(P / block_len) * block_len
 * (align != 0) and step by block_len; each ends at min(start + block_len,
 * P + gen_len).  gen_len == 0 gives no block.  ranges: HOST (cap, 2) int64
 * (may be NULL when cap == 0); *n_out receives the block count even when it
 * exceeds cap, in which case DLLM_ERR_WORKSPACE is returned and the first
 * cap ranges are written. */
dllm_status dllm_block_ranges(int64_t P, int64_t gen_len, int64_t block_len, int align,
                              int64_t* ranges, int64_t cap, int64_t* n_out);

/* ------------------------------------------------------------------------
 * Uniform-noise decoding helpers ([ARS] function table: linear_temperature,
 * uniform_canvas, renoise, StableConfidentStopping; "Uniform-noise decoding
 * (DiffusionGemma)").  The loop: the canvas starts uniformly random; each
 * step scales the logits by 1 / linear_temperature, takes the argmax,
 * entropy and a categorical sample of the scaled softmax
 * (dllm_token_stats_ex or the fused step with temperature 1), accepts the
 * lowest-entropy positions under the entropy bound over all positions,
 * re-noises the rest, and freezes the rows that meet the stopping criterion.
 * ------------------------------------------------------------------------ */

/* Host-only, pure: *temperature = fp32(t_min + (t_max - t_min) * remaining /
 * num_steps), evaluated in double.  0 <= remaining <= num_steps, num_steps >
 * 0, 0 < t_min <= t_max finite (else DLLM_ERR_INVALID_ARGUMENT). */
dllm_status dllm_linear_temperature(int32_t remaining, int32_t num_steps, float t_min, float t_max,
                                    float* temperature);

/* canvas[b * canvas_stride + j] = floor(r * V / 2^32) for b < B, j < N, with
 * r the word j & 3 of Philox4x32-10(counter (j >> 2, b lo, b hi, 1), key
 * (key lo, key hi)): every id of [0, V) has probability within V / 2^32 of
 * 1/V.  canvas: device int32; canvas_stride >= N; 0 < V <= 2^31 - 1. */
dllm_status dllm_uniform_canvas(int64_t B, int64_t N, int64_t V, uint64_t key, int32_t* canvas,
                                int64_t canvas_stride, dllm_stream_t stream);

/* out[b, j] = accepted[b, j] ? sample[b, j] : noise[b, j] over a (B, N)
 * row-major canvas; accepted == NULL takes sample everywhere (noise may then
 * be NULL).  frozen (device (B) uint8, nullable): rows with frozen[b] != 0
 * keep out as it is (rows that already stopped).  out may alias sample or
 * noise.  All device arrays. */
dllm_status dllm_renoise(const int32_t* sample, const uint8_t* accepted, const int32_t* noise,
                         const uint8_t* frozen, int64_t B, int64_t N, int32_t* out, dllm_stream_t stream);

/* One call of the stable-and-confident stopping criterion on the (B, L)
 * argmax canvas and entropies (device).  State, device, owned by the caller:
 * prev (B, L) int32, the previous canvas; count (B) int32, consecutive
 * stable calls, -1 before the first call (then nothing is stable).  Per row:
 * stable = count >= 0 and argmax == prev everywhere; count = stable ? count
 * + 1 : 0; prev = argmax; confident = the mean entropy is below
 * confidence_threshold, decided exactly in fixed point: sum_l q(H_l) <
 * L q(confidence_threshold), q(h) = floor(clamp(h, 0, 64) 2^40), NaN as 64;
 * stop[b] = count >= stability_threshold and confident.  stop (B) uint8 and
 * done (B) uint8 are nullable outputs; done[b] becomes 1 when stop[b] is
 * (never 0).  L <= 2^16, 0 <= confidence_threshold <= 64, stability >= 0. */
dllm_status dllm_stable_confident_stop(const int32_t* argmax, const float* entropy, int64_t B, int64_t L,
                                       int32_t stability_threshold, float confidence_threshold, int32_t* prev,
                                       int32_t* count, uint8_t* stop, uint8_t* done, dllm_stream_t stream);

/* The rest of one uniform-noise step after the statistics, in one launch,
 * with the same results as these calls in this order (done as the frozen
 * rows of both renoise calls):
 *   dllm_uniform_canvas(B, N, V, noise_key, noise, N);
 *   dllm_renoise(sample, accepted, noise, done, B, N, canvas);
 *   dllm_renoise(step_argmax, NULL, NULL, done, B, N, argmax);
 *   dllm_stable_confident_stop(argmax, entropy, B, N, stability_threshold,
 *                              confidence_threshold, prev, count, NULL, done);
 * All arrays device, (B, N) row-major (count and done (B)).  N <= 2^16. */
dllm_status dllm_uniform_update(const int32_t* sample, const uint8_t* accepted, const int32_t* step_argmax,
                                const float* entropy, int64_t B, int64_t N, int64_t V, uint64_t noise_key,
                                int32_t stability_threshold, float confidence_threshold, int32_t* canvas,
                                int32_t* argmax, int32_t* prev, int32_t* count, uint8_t* done,
                                dllm_stream_t stream);

/* ------------------------------------------------------------------------
 * block_causal_mask ([ARS] "What mlx-arsenal ships": the mask block-diffusion
 * models are trained with -- bidirectional inside a block, causal across
 * blocks, aligned on absolute positions; "Mask conventions": additive, 0
 * attend and -inf blocked; boolean-mask runtimes want the inverse reading).
 *
 * out[i * row_stride + j] for i < Lq (query at absolute position q_offset +
 * i) and j < Lk (key at k_offset + j) is "attend" when floor((q_offset + i)
 * / block_len) >= floor((k_offset + j) / block_len), else "blocked":
 *   DLLM_MASK_F32 / DLLM_MASK_BF16  additive: 0 attend, -inf blocked;
 *   DLLM_MASK_KEEP_U8               1 attend, 0 blocked.
 * block_causal_mask(L, block_len) over a window from position 0 is Lq = Lk =
 * L with zero offsets.  out: device; row_stride (elements) >= Lk.  Rows whose
 * base and stride are 16-byte aligned are written with vector stores.
 * ------------------------------------------------------------------------ */
typedef enum { DLLM_MASK_F32 = 0, DLLM_MASK_BF16 = 1, DLLM_MASK_KEEP_U8 = 2 } dllm_mask_kind;

dllm_status dllm_block_causal_mask(int64_t Lq, int64_t Lk, int64_t q_offset, int64_t k_offset, int64_t block_len,
                                   dllm_mask_kind kind, void* out, int64_t row_stride, dllm_stream_t stream);

/* ------------------------------------------------------------------------
 * LM head fused with the statistics pass (mojo-dllm manual, "The GPU path":
 * the LM head's rows only feed the row statistics; the logits need not reach
 * HBM).  logits[t, v] = sum_k hidden[t, k] weight[v, k] (bf16 inputs, fp32
 * tensor-core accumulation), then x0 / prob / entropy exactly as
 * dllm_token_stats defines them (greedy or Gumbel-max with the same noise:
 * row = t), without the logits ever being stored.
 *
 * hidden  device bf16 (T, d), rows hidden_stride elements apart.
 * weight  device bf16 (V, d), rows weight_stride elements apart (the LM
 *         head's weight in its usual [vocab, hidden] layout).
 * d a multiple of 64; both bases 16-byte aligned and both row strides a
 * multiple of 8 elements (else DLLM_ERR_UNSUPPORTED).
 * logits  optional device fp32 (T, V) output with row stride logits_stride
 *         (NULL: the logits are not written -- the point of the fusion).
 * workspace >= dllm_lm_head_stats_workspace_size(T, V, d) bytes (any
 *         contents; it holds per-CTA partials).  Other arguments as in
 *         dllm_token_stats.
 * Range: the logits this call never stores cannot be read back, so it has
 * no exact path for exotic rows: the products must stay below 1.8e8 in
 * magnitude and must not be NaN (rows beyond that get unspecified
 * statistics; no fault).
 * Ordering: the call is launched as a programmatic dependent of the kernel
 * before it in the stream.  The hidden states (and every output) are touched
 * only after that kernel has completed; the first slabs of the weight are
 * read before, so the weight must not be written by the kernel launched just
 * before this call on the same stream (write it earlier, or on another stream
 * with an event).
 * ------------------------------------------------------------------------ */
size_t dllm_lm_head_stats_workspace_size(int64_t T, int64_t V, int64_t d);

dllm_status dllm_lm_head_stats(const void* hidden, int64_t T, int64_t d, int64_t hidden_stride,
                               const void* weight, int64_t V, int64_t weight_stride, float temperature,
                               uint64_t key, const int32_t* suppress_ids, int32_t n_suppress, int32_t* x0,
                               float* prob, float* entropy, float* logits, int64_t logits_stride,
                               void* workspace, size_t workspace_bytes, dllm_stream_t stream);

/* ------------------------------------------------------------------------
 * Fused commit step: the statistics pass and one commit rule (plus the
 * optional edit rule and canvas update) in one launch.  The rule of batch
 * row b runs as soon as its L rows' statistics are complete, inside the same
 * kernel ([MOJO] spec "possible future fused kernel": softmax, entropy and
 * confidence, top-k, sample, scatter).  Requires L <= 65535, and L <= 1024
 * for the sorting rules (else DLLM_ERR_UNSUPPORTED).
 * ------------------------------------------------------------------------ */
typedef enum {
  DLLM_RULE_NONE = 0,
  DLLM_RULE_THRESHOLD = 1,     /* on prob */
  DLLM_RULE_TOPK = 2,          /* on prob */
  DLLM_RULE_FACTOR = 3,        /* on prob */
  DLLM_RULE_ENTROPY_BOUND = 4  /* on entropy */
} dllm_rule;

typedef struct {
  int32_t rule;             /* a dllm_rule */
  int32_t strict;           /* threshold: > instead of >= */
  float tau;                /* threshold */
  float factor;             /* factor */
  float gamma;              /* entropy bound */
  const int32_t* k;         /* top-k: device (B,) */
  const uint8_t* cand;      /* device (B, L), or NULL: cand = (canvas token == mask_id) */
  int32_t mask_id;          /* used when cand == NULL */
  int32_t edit;             /* non-zero: also run edit_transfer with editable = !cand */
  float tau_edit;
  uint8_t* commit;          /* device (B, L) output, required unless rule == NONE */
  uint8_t* edit_mask;       /* device (B, L) output, required when edit != 0 */
  int32_t* canvas;          /* device; NULL = no canvas update (then cand must be given) */
  int64_t canvas_stride;    /* elements between batch rows of the canvas */
  int64_t canvas_offset;    /* canvas column of position l = 0 */
  int32_t* counts;          /* device (B, 3) or NULL: per batch row [candidates, commits, edits] */
  int32_t flags;            /* 0, or DLLM_FLAG_INPUTS_READY (| DLLM_FLAG_TEST_DROP_COPY in tests) */
  const dllm_stats_ex* ex;  /* NULL, or the extended statistics options (scale, margin, argmax);
                               the rules then decide on the scaled statistics */
} dllm_commit_params;

/* The logits and the candidate mask (when one is given) were complete before
 * the previous kernel in the stream began (they are not that kernel's
 * output): the call may start reading them while that kernel still runs.  It
 * reads the canvas, and writes anything, only after that kernel has finished.
 * Lets back-to-back steps over independent inputs overlap.  Never set it when
 * the previous kernel produces the logits or the mask (an LM-head GEMM, say). */
#define DLLM_FLAG_INPUTS_READY 1

/* Test only, never set in use: the first CTA of the statistics kernel does
 * not issue the bulk copy of its first unit, so that its consumers' bounded
 * wait (about one second) runs out.  The call then takes a second or two,
 * records fault 1 (a consumer gave up waiting for a copy) or 2 (the copy
 * issuer gave up waiting for a free stage) in the workspace, leaves outputs
 * unwritten and workspace counters set.  It exists to exercise the fault path
 * (dllm_workspace_fault, then zeroing the workspace) without a real fault. */
#define DLLM_FLAG_TEST_DROP_COPY 2

dllm_status dllm_commit_step(const void* logits, dllm_dtype dt, int64_t B, int64_t L, int64_t V,
                             int64_t row_stride, float temperature, uint64_t key,
                             const int32_t* suppress_ids, int32_t n_suppress,
                             int32_t* x0, float* prob, float* entropy,
                             const dllm_commit_params* params,
                             void* workspace, size_t workspace_bytes, dllm_stream_t stream);

/* ------------------------------------------------------------------------
 * dllm_commit_step on logits held in host memory, with its results returned
 * to host memory: one call queues, on `stream`, the copy of the (B, L, V)
 * logits (rows contiguous, row stride V) from host_logits into dev_logits,
 * dllm_commit_step on them, and one copy of the per-position results back.
 * Results, in dev_out and then host_out, back to back with T = B L:
 *   x0 int32[T], prob fp32[T], entropy fp32[T], commit uint8[T]
 * (12 T bytes, or 13 T when params->rule != DLLM_RULE_NONE: the commit mask
 * is written to the packed buffer, params->commit is ignored).  The edit
 * mask, the canvas and the counts (when requested) stay on the device.
 * host_logits / host_out: host memory (pinned for the copies to run
 * asynchronously), valid until the stream reaches the copies.
 * dev_logits: device, B L V elements; dev_out: device, 4-byte aligned,
 * >= 13 T bytes.  Other arguments and errors as in dllm_commit_step; the
 * arguments are checked before anything is queued.
 * ------------------------------------------------------------------------ */
dllm_status dllm_commit_step_host(const void* host_logits, void* dev_logits, dllm_dtype dt, int64_t B, int64_t L,
                                  int64_t V, float temperature, uint64_t key, const int32_t* suppress_ids,
                                  int32_t n_suppress, const dllm_commit_params* params, void* dev_out,
                                  void* host_out, void* workspace, size_t workspace_bytes, dllm_stream_t stream);

/* Reads and clears the device fault word of a workspace (synchronises the
 * stream).  *fault = 0 when no kernel reported a fault; otherwise a code
 * naming the wait that gave up (the kernel stopped early; outputs of that
 * call are undefined).  A faulted call can also leave the workspace's
 * per-row and per-batch-row counters non-zero: zero the whole workspace
 * before its next use (only the fault word is cleared here, since the call
 * does not know the workspace's size).  Returns DLLM_ERR_CUDA if the copy
 * fails. */
dllm_status dllm_workspace_fault(void* workspace, dllm_stream_t stream, int32_t* fault);

#ifdef __cplusplus
}
#endif
#endif /* DLLMCOMMIT_H */
