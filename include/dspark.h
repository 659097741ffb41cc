/*
 * dspark.h -- C ABI of the DSpark draft-sampling / verification hot path on one
 * GB300 (sm_103a).
 *
 * Four operations, each one kernel launch on the caller's stream (after a small
 * kernel that clears the workspace header; the scheduler's kernels clear their
 * own status word):
 *
 *   dspark_draft_logits   base logits of the draft LM head (tcgen05 GEMM)
 *   dspark_markov_sample  N-step Markov-biased Gumbel-max sampling (one
 *                         persistent kernel)
 *   dspark_verify         lossless speculative rejection sampling
 *   dspark_schedule       confidence-scheduled admission (survival chain,
 *                         global sort, throughput-optimal K, fill)
 *
 * Conventions shared by every call
 *   - All array arguments are DEVICE pointers on the current CUDA device,
 *     contiguous and row-major, owned by the caller.  The library never
 *     allocates, frees or synchronises inside these calls, so every call can
 *     be captured in a CUDA graph (the caller keeps the buffers at fixed
 *     addresses, as the draft step of "DSpark implementation and evaluation"
 *     §6 does).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).
 *   - Host-side argument errors return DSPARK_ERR_INVALID_ARG or
 *     DSPARK_ERR_UNSUPPORTED synchronously and launch nothing.  A failed
 *     launch returns DSPARK_ERR_CUDA (see dspark_last_error()).
 *   - Errors found on the device (a wait that timed out, non-finite or
 *     out-of-range inputs) set bits in the status word at the start of the
 *     caller's workspace; dspark_read_status() reads it.  Each call clears
 *     the status word of the workspace it is given before launching.
 *   - Random numbers: a counter-based Philox4x32-10 generator keyed by
 *     `seed`; `offset` (< 2^32) selects an independent stream, so the caller
 *     advances it per decode step.  Outputs are a pure function of the inputs
 *     and (seed, offset).
 *   - Workspace: device memory of at least dspark_workspace_size() bytes,
 *     256-byte aligned, used by one call at a time (calls that overlap on the
 *     GPU must use different workspaces).
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DSPARK_API __attribute__((visibility("default")))
#else
#define DSPARK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or workspace  */
    DSPARK_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels handle  */
    DSPARK_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed       */
    DSPARK_ERR_TIMEOUT = 4,       /* a bounded device-side wait ran out         */
    DSPARK_ERR_NUMERIC = 5,       /* non-finite input or a distribution with no mass */
    DSPARK_ERR_INPUT_RANGE = 6    /* a token id, length or probability out of range  */
} dspark_status;

typedef enum { DSPARK_F32 = 0, DSPARK_BF16 = 1 } dspark_dtype;

typedef enum {
    DSPARK_OP_DRAFT_LOGITS = 0,
    DSPARK_OP_MARKOV_SAMPLE = 1,
    DSPARK_OP_VERIFY = 2,
    DSPARK_OP_SCHEDULE = 3,
    DSPARK_OP_VERIFY_GREEDY = 4,
    DSPARK_OP_CONFIDENCE = 5,
    DSPARK_OP_VERIFY_LOGITS = 6,
    DSPARK_OP_VERIFY_GUMBEL = 7
} dspark_op;

/*
 * Device status-word bits (OR-ed by kernels; read with dspark_read_status).
 *   INPUT_RANGE  a value from the caller is out of its range (an anchor or draft
 *                token outside [0, V), a length outside [0, gamma], a mapped
 *                draft-to-target id outside the target vocabulary, a confidence
 *                outside [0, 1], ...); the kernel substitutes a safe value and
 *                never reads memory at the bad index.
 *   INDEX        set only by a library built with -DDSPARK_CHECKED (a debugging
 *                build with no counterpart on the pages, in which every gather
 *                site checks its index): an index at a gather site was out of
 *                range.  Beside INPUT_RANGE it marks a caller's index; alone it
 *                marks an index the library computed itself (a token read back
 *                from a step slot, a sorted candidate, a work-list entry), and
 *                the access was skipped instead of made.
 */
#define DSPARK_STATUS_TIMEOUT      0x1u
#define DSPARK_STATUS_NUMERIC      0x2u
#define DSPARK_STATUS_INPUT_RANGE  0x4u
#define DSPARK_STATUS_INTERNAL     0x8u
#define DSPARK_STATUS_INDEX        0x10u

/*
 * Bytes of workspace an operation needs.  op is a dspark_op; arguments an op
 * does not use are ignored:
 *   DSPARK_OP_DRAFT_LOGITS  256 (the status word)
 *   DSPARK_OP_MARKOV_SAMPLE grows with B*N and B (argmax slots, bounds, lse partials)
 *   DSPARK_OP_VERIFY        grows with B*V/512 (per-512-entry integer masses); N = gamma
 *   DSPARK_OP_SCHEDULE      grows with B*N (radix-sort key buffers)
 *   DSPARK_OP_VERIFY_GREEDY grows with B*(N+1) (row argmax keys); N = gamma
 *   DSPARK_OP_CONFIDENCE    256 (the status word)
 *   DSPARK_OP_VERIFY_LOGITS grows with B*V/2048 (normaliser partials); N = gamma
 *   DSPARK_OP_VERIFY_GUMBEL grows with B*(N+1) (row keys); N = gamma
 * Returns 0 for an unknown op or negative sizes.
 */
DSPARK_API size_t dspark_workspace_size(int op, int B, int N, int V, int r);

/*
 * Base logits of the draft LM head:  logits[m, v] = sum_h hidden[m, h] * lm_head[v, h].
 *
 * "DSpark implementation and evaluation" §2.2 (compute_draft_logits: all N
 * positions of every request through the LM head at once, giving [B, N, V]) and
 * §4 (the draft step).  Here M = B*N rows.
 *
 *   hidden   [M, H]  dtype (bf16 or fp32), device
 *   lm_head  [V, H]  dtype, device
 *   logits   [M, V]  fp32, device (output)
 * bf16 inputs are multiplied exactly and accumulated in fp32 on the tensor
 * cores (tcgen05 kind::f16); fp32 inputs run as tf32 (kind::tf32).
 * Requirements: 1 <= M, 1 <= V < 2^31, 1 <= H, H*sizeof(dtype) a multiple of
 * 16 bytes, hidden/lm_head 16-byte aligned, logits 4-byte aligned.
 * workspace: >= dspark_workspace_size(DSPARK_OP_DRAFT_LOGITS, ...) bytes.
 */
DSPARK_API dspark_status dspark_draft_logits(const void* hidden, const void* lm_head, dspark_dtype dtype,
                                  int M, int H, int V, float* logits,
                                  void* workspace, size_t ws_bytes, void* stream);

/*
 * Sequential Markov-biased Gumbel-max sampling of N draft tokens per request.
 *
 * "DSpark implementation and evaluation" §2.2 (_sample_sequential) and §3
 * (the low-rank Markov head).  For each request b, prev = anchor[b]; for
 * i = 0..N-1:
 *     bias[v] = sum_k w2[v, k] * w1[prev, k]
 *     z[v]    = (base_logits[b, i, v] + bias[v]) / T_b          (T_b > 0)
 *     x       = argmax_v (z[v] + g[v])   ties to the lowest v
 *     draft_tokens[b, i] = x;  prev = x
 * with g a standard Gumbel variate per (b, i, v) from the Philox generator
 * (counter words (c0, c1, c2, c3) = (j, b, (stream << 16) | i, offset), key
 * (lo32 seed, hi32 seed), uniform u = ((w >> 9) + 1/2) * 2^-23), drawn in
 * groups of 16 entries (G = v >> 4, k = v & 15):
 *     W     = word G & 3 of the stream-0 counter j = G >> 2 (the group word)
 *     p     = W & 15, the position of the group's largest variate
 *     E_min = -log(u(W)) / 16, the group's smallest exponential
 *     E_k   = E_min                                 for k == p
 *           = E_min - log(u(w_k))                    otherwise, w_k = word
 *             k & 3 of the stream-3 counter j = (G << 2) | (k >> 2)
 *     g     = -log(E_k)
 * (the 16 E_k are independent Exp(1), so every g is a standard Gumbel, and
 * -log(E_min) bounds the whole group).  T_b = 0 means greedy:
 * x = argmax_v (base + bias), no noise.
 * The [B, V] row of z is never written to device memory.
 *
 *   base_logits  [B, N, V] fp32, device (row (b, i) contiguous over v)
 *   anchor       [B] int32, device, each in [0, V)
 *   w1, w2       [V, r] wdtype (bf16 or fp32), device (markov_w1 embedding and
 *                markov_w2 projection, both stored [V, r])
 *   temperature  [B] fp32, device, each >= 0 and finite
 *   draft_tokens [B, N] int32, device (output)
 *   lse          [B, N] fp32 device output or NULL: log-sum-exp over v of z
 *                (of base + bias when T_b = 0), so that
 *                p_d(x) = exp(z[x] - lse) downstream.
 * Requirements: B, N >= 1, N <= 65535, 2 <= V < 2^31, 1 <= r <= 1024,
 * offset < 2^32.  Device-side: an anchor outside [0, V) sets INPUT_RANGE and
 * is read as 0; a negative or non-finite temperature sets NUMERIC and is read
 * as 0 (greedy); non-finite logits are skipped by the argmax and set NUMERIC.
 * workspace: >= dspark_workspace_size(DSPARK_OP_MARKOV_SAMPLE, B, N, V, r).
 */
DSPARK_API dspark_status dspark_markov_sample(const float* base_logits, const int32_t* anchor,
                                   const void* w1, const void* w2, dspark_dtype wdtype,
                                   const float* temperature, uint64_t seed, uint64_t offset,
                                   int B, int N, int V, int r,
                                   int32_t* draft_tokens, float* lse,
                                   void* workspace, size_t ws_bytes, void* stream);

/*
 * dspark_markov_sample with the calibrated confidence head of every draft token
 * evaluated inside the sampler, step by step.
 *
 * "Speculative decoding: from zero to DSpark" §6: a linear projection of the
 * backbone's hidden state together with the Markov embedding predicts each draft
 * position's conditional acceptance probability, calibrated per position by
 * temperature scaling; the scheduler chains these into survival probabilities:
 *   conf[b, i] = 1 / (1 + exp(-(w_h . hidden[b*N+i] + w_e . w1[prev] + beta) / tau[i]))
 * with prev the token whose embedding step i's Markov bias uses (anchor[b] for
 * i = 0, draft token i-1 after).  The sampler already holds that embedding at
 * step i, so no second pass over the tokens and no separate launch are needed;
 * conf is dspark_schedule's cond_accept.  The result equals dspark_confidence
 * on the tokens this call draws.
 *
 *   hidden  [B*N, H] hdtype (bf16 or fp32), device: the LM head's input rows
 *   w_h [H], w_e [r] fp32, device; beta: host value; tau [N] fp32 > 0, device
 *   conf    [B, N] fp32 output
 * Everything else (arguments, requirements, workspace, device-side status) as
 * dspark_markov_sample; a temperature tau[i] that is not positive and finite
 * gives conf 0 and sets NUMERIC.
 */
DSPARK_API dspark_status dspark_markov_sample_conf(const float* base_logits, const int32_t* anchor,
                                        const void* w1, const void* w2, dspark_dtype wdtype,
                                        const float* temperature, uint64_t seed, uint64_t offset,
                                        int B, int N, int V, int r,
                                        const void* hidden, dspark_dtype hdtype, int H,
                                        const float* w_h, const float* w_e, float beta,
                                        const float* tau, int32_t* draft_tokens, float* conf,
                                        float* lse, void* workspace, size_t ws_bytes, void* stream);

/* Draft-to-target id table conventions of dspark_markov_sample_reduced. */
typedef enum {
    DSPARK_D2T_INDEX = 0,    /* target id = d2t[draft id] (the draft logits scattered into target positions) */
    DSPARK_D2T_OFFSET = 1    /* target id = draft id + d2t[draft id] */
} dspark_d2t_mode;

/*
 * dspark_markov_sample on a reduced draft vocabulary: V is the draft
 * vocabulary (base_logits [B, N, V], w1 and w2 [V, r] and the anchor are in
 * draft ids, and the Markov chain feeds back draft ids); each sampled draft id
 * d is written to draft_tokens as its target-vocabulary id, d2t[d]
 * (DSPARK_D2T_INDEX: "DSpark implementation and evaluation" §5 scatters the
 * draft logits into target positions through an index table) or d + d2t[d]
 * (DSPARK_D2T_OFFSET: "xserv/docs/25-speculative-methods-comparison.md" §3.2,
 * real_id = draft_id + d2t[draft_id]).  Sampling is Gumbel-max over the draft
 * entries with noise indexed by draft id -- the same distribution as over the
 * scattered target-size buffer.
 *
 *   d2t       [V] int32, device
 *   V_target  size of the target vocabulary; a mapped id outside [0, V_target)
 *             is written as -1 and sets INPUT_RANGE
 * Everything else (arguments, requirements, workspace) as dspark_markov_sample;
 * lse, when requested, is over the draft vocabulary.
 */
DSPARK_API dspark_status dspark_markov_sample_reduced(const float* base_logits, const int32_t* anchor,
                                           const void* w1, const void* w2, dspark_dtype wdtype,
                                           const float* temperature, uint64_t seed, uint64_t offset,
                                           int B, int N, int V, int r,
                                           const int32_t* d2t, int d2t_mode, int V_target,
                                           int32_t* draft_tokens, float* lse,
                                           void* workspace, size_t ws_bytes, void* stream);

/*
 * Lossless speculative verification (rejection sampling) of a block of gamma
 * draft tokens per request.
 *
 * "Speculative decoding: from zero to DSpark" §2: draft token x_k is accepted
 * with probability min(1, p_t(x_k) / p_d(x_k)), decided as
 * fl32(u_k * p_d[b,k,x_k]) < p_t[b,k,x_k] with u_k the stream-1 uniform of
 * counter (0, b, k, offset); the first rejected position k* draws a correction
 * from norm(max(0, p_t[k*] - p_d[k*])); if all L_b tested tokens are accepted
 * a bonus token is drawn from p_t[b, L_b].  The draw is an inverse CDF over
 * q_v = floor(w_v * 2^40) with t = floor(R * Q / 2^64), R the stream-2 word
 * pair of counter (0, b, position, offset), Q = sum q_v; the token is the
 * smallest v whose inclusive prefix sum exceeds t.  A residual with no mass
 * falls back to p_t[k*]; a p_t row with no mass gives argmax p_t and sets
 * NUMERIC.
 *
 *   p_target     [B, gamma+1, V] fp32 probabilities, device
 *   p_draft      [B, gamma, V]   fp32 probabilities, device
 *   draft_tokens [B, gamma] int32, device, each in [0, V)
 *   lengths      [B] int32 in [0, gamma], device, or NULL (= gamma): the
 *                scheduler's per-request verify length
 *   out_tokens   [B, gamma+1] int32 output: accepted prefix, then the
 *                correction or bonus token, then -1
 *   num_accepted [B] int32 output
 * Requirements: B >= 1, 1 <= gamma <= 65535, 1 <= V <= 2^24 (keeps Q < 2^64),
 * offset < 2^32; p_target/p_draft 16-byte aligned.
 * Device-side: a token or length out of range sets INPUT_RANGE (the request
 * outputs num_accepted 0 and -1 tokens).
 * Launches one kernel on `stream` (captured by CUDA stream capture).
 * workspace: >= dspark_workspace_size(DSPARK_OP_VERIFY, ...) bytes.
 */
DSPARK_API dspark_status dspark_verify(const float* p_target, const float* p_draft,
                            const int32_t* draft_tokens, const int32_t* lengths,
                            uint64_t seed, uint64_t offset, int B, int gamma, int V,
                            int32_t* out_tokens, int32_t* num_accepted,
                            void* workspace, size_t ws_bytes, void* stream);

/*
 * Greedy (temperature-0) verification of a block of gamma draft tokens per
 * request.
 *
 * "xserv/docs/25-speculative-methods-comparison.md" §2: the longest prefix of
 * draft tokens that each equal the target's argmax at their position is
 * accepted; the target's argmax at the first failing position (position L_b
 * when none fails) is appended.  The output equals the target's own greedy
 * continuation.  Argmax ties go to the lowest token id; NaN entries never win
 * (a row without a non-NaN entry gives token 0 and sets NUMERIC).
 *
 *   target       [B, gamma+1, V] fp32, device: row k scores position k
 *                (logits or probabilities: only the argmax is used)
 *   draft_tokens [B, gamma] int32, device
 *   lengths      [B] int32 in [0, gamma], device, or NULL (= gamma)
 *   out_tokens   [B, gamma+1] int32 output: accepted prefix, the target's
 *                token, then -1
 *   num_accepted [B] int32 output
 * Requirements: B >= 1, 1 <= gamma <= 65535, 1 <= V < 2^31; target 16-byte
 * aligned.  Device-side: a token or length out of range sets INPUT_RANGE
 * (the request outputs num_accepted 0 and -1 tokens).  Only rows k <= L_b
 * are read.
 * workspace: >= dspark_workspace_size(DSPARK_OP_VERIFY_GREEDY, B, gamma, 0, 0).
 */
DSPARK_API dspark_status dspark_verify_greedy(const float* target, const int32_t* draft_tokens,
                                   const int32_t* lengths, int B, int gamma, int V,
                                   int32_t* out_tokens, int32_t* num_accepted,
                                   void* workspace, size_t ws_bytes, void* stream);

/*
 * Verification with the draft's own Gumbel noise ("probabilistic" drafting).
 *
 * "DSpark implementation and evaluation" §5: the draft samples with the
 * Gumbel-max trick and the target verifies with the same Gumbel seed, which
 * keeps the output distribution.  The target draws its own token at each
 * position with the noise the draft drew at that step,
 *   y_k = argmax_v (target_logits[b, k, v] / T[b] + g(b, k, v)),
 * g the draft noise of dspark_markov_sample step k for request b (its seed and
 * offset, the group-of-16 layout of the header of that function); T[b] = 0
 * scores the plain argmax.  Drafted tokens are accepted while x_k = y_k; y at
 * the first mismatch (at L_b when every tested token matches) is appended.
 * The output is the target's own Gumbel-max sample sequence, so its law is the
 * target's whatever the draft; the draft only decides how many of the tokens
 * come from one target pass.  b is the request's row in both calls.  Ties go
 * to the lowest id; NaN entries never win (a row without one gives token 0
 * and sets NUMERIC); a NaN, negative or infinite T is scored greedily and
 * sets NUMERIC.  Scores are fp32 (t * (1/T) + g): a token can differ from an
 * exact evaluation only where the row's top-2 gap is within rounding.
 *
 *   target_logits [B, gamma+1, V] fp32, device: row k scores position k
 *   temperature   [B] fp32, device (the target's; 0 = greedy)
 *   draft_tokens  [B, gamma] int32, device
 *   lengths       [B] int32 in [0, gamma], device, or NULL (= gamma)
 *   seed, offset  the draft sampler's (offset < 2^32)
 *   out_tokens    [B, gamma+1] int32 output: accepted prefix, the target's
 *                 token, then -1
 *   num_accepted  [B] int32 output
 * Requirements: B >= 1, 1 <= gamma <= 65535, 1 <= V < 2^27, B <= 65535;
 * target_logits 16-byte aligned.  Device-side: a token or length out of range
 * sets INPUT_RANGE (the request outputs num_accepted 0 and -1 tokens).  Only
 * rows k <= L_b are read.
 * workspace: >= dspark_workspace_size(DSPARK_OP_VERIFY_GUMBEL, B, gamma, 0, 0).
 */
DSPARK_API dspark_status dspark_verify_gumbel(const float* target_logits, const float* temperature,
                                   const int32_t* draft_tokens, const int32_t* lengths,
                                   uint64_t seed, uint64_t offset, int B, int gamma, int V,
                                   int32_t* out_tokens, int32_t* num_accepted,
                                   void* workspace, size_t ws_bytes, void* stream);

/*
 * Lossless verification from logits, the draft distribution recomputed.
 *
 * "Speculative decoding: from zero to DSpark" §2 (the rule, as dspark_verify)
 * with the distributions of "DSpark implementation and evaluation" §2.2 / §5:
 *   p_t(. | row k) = softmax(target_logits[b, k] / T_t[b])
 *   p_d(. | pos k) = softmax((base_logits[b, k] + w2 . w1[prev_k]) / T_d[b]),
 *                    prev_0 = anchor[b], prev_k = draft_tokens[b, k-1];
 *                    T_d = 0 (a greedy draft): the point mass at draft_tokens[b, k].
 * No [B, gamma, V] draft probabilities are read or written: p_d(x_k) is
 * recomputed at the drafted token from the base logit, one r-long dot product
 * and the sampler's log-sum-exp (draft_lse = dspark_markov_sample's lse
 * output), and at the rejected position only at the entries whose perturbed
 * value can still win the draw (the draw is bounded through p_t, which the
 * residual never exceeds).  The target normalisers are computed here, lazily:
 * row k is read only if every earlier drafted token was accepted, so only the
 * rows k <= k* are streamed.
 * Acceptance: fl32(u_k * p_d(x_k)) < p_t(x_k), u_k the stream-1 uniform as in
 * dspark_verify.  The correction (residual max(0, p_t - p_d) at the first
 * rejection) or bonus (p_t of row L_b) token is drawn by Gumbel-max,
 * argmax_v ln w_v + g_v, g_v the Gumbel variate of Philox stream 4, word v & 3
 * of counter (v >> 2, b, (4 << 16) | position, offset); ties go to the lowest
 * id, a residual with no positive entry falls back to p_t.  Everything is fp32:
 * a decision can differ from an exact evaluation only within rounding of its
 * boundary (relative 1e-5 for an acceptance test, a top-2 gap of ~1e-4 for a
 * draw).
 *
 *   target_logits [B, gamma+1, V] fp32, device
 *   target_temperature [B] fp32, device, > 0
 *   base_logits   [B, gamma, V] fp32, device: the draft's base logits of the
 *                 drafted positions (dspark_draft_logits' output)
 *   anchor        [B] int32, device: the token before the block
 *   w1, w2        [V, r] wdtype (bf16 or fp32), device: markov_w1, markov_w2
 *   draft_temperature [B] fp32, device, >= 0
 *   draft_lse     [B, gamma] fp32, device: the sampler's lse of each drafted
 *                 position (ignored where T_d = 0)
 *   draft_tokens  [B, gamma] int32, device
 *   lengths       [B] int32 in [0, gamma], device, or NULL (= gamma)
 *   out_tokens    [B, gamma+1] int32 output: accepted prefix, the correction
 *                 or bonus token, then -1
 *   num_accepted  [B] int32 output
 * Requirements: B >= 1, 1 <= gamma <= 65535, 2 <= V < 2^31, 1 <= r <= 1024
 * with r * sizeof(wdtype) a multiple of 16 bytes, offset < 2^32;
 * target_logits, base_logits, w1, w2 16-byte aligned.
 * Device-side: a token, anchor or length out of range or a temperature out of
 * its range sets INPUT_RANGE, a non-finite normaliser or draft_lse sets
 * NUMERIC; such a request outputs num_accepted 0 and -1 tokens.
 * Launches two kernels on `stream` (captured by CUDA stream capture), the first
 * a cooperative persistent kernel whose rounds meet at bounded grid barriers
 * (a barrier that gives up sets TIMEOUT).
 * workspace: >= dspark_workspace_size(DSPARK_OP_VERIFY_LOGITS, B, gamma, V, r).
 */
DSPARK_API dspark_status dspark_verify_logits(const float* target_logits, const float* target_temperature,
                                   const float* base_logits, const int32_t* anchor,
                                   const void* w1, const void* w2, dspark_dtype wdtype, int r,
                                   const float* draft_temperature, const float* draft_lse,
                                   const int32_t* draft_tokens, const int32_t* lengths,
                                   uint64_t seed, uint64_t offset, int B, int gamma, int V,
                                   int32_t* out_tokens, int32_t* num_accepted,
                                   void* workspace, size_t ws_bytes, void* stream);

/*
 * Conditional acceptance probability of every draft token from the calibrated
 * confidence head.
 *
 * "Speculative decoding: from zero to DSpark" §6: a linear projection of the
 * backbone's hidden state together with the Markov embedding, calibrated per
 * position by temperature scaling:
 *   conf[b, i] = 1 / (1 + exp(-(w_h . hidden[b*N+i] + w_e . w1[prev] + beta) / tau[i]))
 * with prev = anchor[b] for i = 0 and draft_tokens[b, i-1] after (the
 * embedding the Markov head used at step i).  conf is dspark_schedule's
 * cond_accept.
 *
 *   hidden       [B*N, H] hdtype (bf16 or fp32), device: the LM head's input rows
 *   w1           [V, r] wdtype, device: markov_w1
 *   anchor       [B] int32, draft_tokens [B, N] int32, device
 *   w_h [H], w_e [r] fp32, device: the head's weights; beta: its bias (host value)
 *   tau          [N] fp32 > 0, device: per-position calibration temperatures
 *   conf         [B, N] fp32 output
 * Requirements: B, N, H, r >= 1, V >= 1.  Device-side: a previous token
 * outside [0, V) is read as 0 and sets INPUT_RANGE; a temperature that is not
 * positive and finite gives conf 0 and sets NUMERIC.
 * workspace: >= dspark_workspace_size(DSPARK_OP_CONFIDENCE, ...) bytes.
 */
DSPARK_API dspark_status dspark_confidence(const void* hidden, dspark_dtype hdtype, const void* w1,
                                dspark_dtype wdtype, const int32_t* anchor,
                                const int32_t* draft_tokens, const float* w_h,
                                const float* w_e, float beta, const float* tau,
                                int B, int N, int H, int V, int r, float* conf,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * Confidence-scheduled admission of draft tokens for the next verify batch.
 *
 * "Speculative decoding: from zero to DSpark" §6 and §7:
 *   survival[b, 0] = c[b, 0],  survival[b, k] = fl32(survival[b, k-1] * c[b, k])
 *   candidates (b, k) sorted by survival descending, ties by b*N+k ascending
 *   (a stable device radix sort of all B*N candidates);
 *   if K_in < 0: K = smallest argmax over K in [1, min(B*N, S)] of
 *       f(K) = float64(B * 2^32 + sum_{j<K} floor(s_(j) * 2^32)) * sps[K-1]
 *     (expected tokens of the batch in 32.32 fixed point, times the
 *      steps-per-second table at batch size K; every K is evaluated);
 *   else K = min(K_in, B*N) (capacity fixed ahead of time, §7).
 *   The top K candidates are admitted; lengths[b] counts request b's admitted
 *   candidates, which are always a prefix 0..lengths[b]-1.  The call reads no
 *   token values, so admission of token k never depends on token k's value.
 *
 *   cond_accept [B, N] fp32 in [0, 1], device (values outside are clamped,
 *               NaN read as 0, and INPUT_RANGE is set)
 *   sps         [S] fp64, device, or NULL when K_in >= 0
 *   survival    [B, N] fp32 output
 *   K_out       [1] int32 output
 *   lengths     [B] int32 output
 *   selected    [B*N] int32 output: flat index b*N+k of the admitted
 *               candidates in rank order, then -1
 * Requirements: B, N >= 1, B*N <= 2^20, S >= 1 when K_in < 0.
 * workspace: >= dspark_workspace_size(DSPARK_OP_SCHEDULE, B, N, 0, 0) bytes.
 */
DSPARK_API dspark_status dspark_schedule(const float* cond_accept, const double* sps, int S,
                              int B, int N, int K_in,
                              float* survival, int32_t* K_out, int32_t* lengths,
                              int32_t* selected,
                              void* workspace, size_t ws_bytes, void* stream);

/*
 * Allocation-free variant of dspark_schedule (no counterpart on the pages: it
 * exists for callers, not for the method).  Same arguments, results and
 * requirements as dspark_schedule, without the workspace.
 *
 * For callers that cannot provide device scratch memory: a serving loop that
 * must never block (cudaMalloc/cudaFree can synchronise with work already
 * queued on the device), or a host whose device memory is wholly reserved by
 * another allocator, so that a new allocation would fail.  The scratch lives in
 * one fixed array inside the library (256 bytes: the status header, since pools
 * this size sort in shared memory; held on every GPU that loads the library
 * until the process exits); the call allocates nothing.
 *   - B*N must be at most 16384; larger pools return DSPARK_ERR_INVALID_ARG
 *     (use dspark_schedule with a workspace).
 *   - The first call in each CUDA context looks up the array's device address
 *     (with that context current); make that first call before any stream
 *     capture.  A device reset or another context on the same device gets a
 *     fresh lookup on its first call.
 *   - All calls share the array and each call clears its status header first.
 *     Calls that overlap on the GPU (different streams, or several threads)
 *     race on it and must be serialised by the caller.
 *   - Device-side status bits (clamped confidences) go to the shared array
 *     and are not reported; use dspark_schedule when they are needed.
 */
DSPARK_API dspark_status dspark_schedule_noalloc(const float* cond_accept, const double* sps, int S,
                                                 int B, int N, int K_in,
                                                 float* survival, int32_t* K_out, int32_t* lengths,
                                                 int32_t* selected, void* stream);

/*
 * Synchronises `stream`, reads the status word of `workspace` written by the
 * last call that used it, stores the raw DSPARK_STATUS_* bits in *bits (if
 * bits != NULL) and returns the most severe matching dspark_status
 * (TIMEOUT > NUMERIC > INPUT_RANGE > OK; INTERNAL maps to DSPARK_ERR_CUDA).
 * For tests and debugging: it blocks the host.
 */
DSPARK_API dspark_status dspark_read_status(const void* workspace, uint32_t* bits, void* stream);

/* Static description of a status code. */
DSPARK_API const char* dspark_status_string(dspark_status s);

/* Text of the last host-side error of the calling thread ("" if none). */
DSPARK_API const char* dspark_last_error(void);

/*
 * Self-test of the bounded device-side wait used by every kernel: launches
 * one block that waits on a flag in `workspace` that nothing sets, for at most
 * timeout_ns nanoseconds (1e3 .. 1e10), then records DSPARK_STATUS_TIMEOUT in
 * the workspace status word and returns.  Lets a test show that a wait that
 * runs out ends with an error status and leaves the context usable.
 * workspace: >= 256 bytes.
 */
DSPARK_API dspark_status dspark_selftest_wait_timeout(void* workspace, size_t ws_bytes,
                                           long long timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
