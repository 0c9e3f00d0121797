/*
 * ORACLE - test infrastructure, not product code.
 *
 * A plain, slow, single-threaded CPU statement of the DSpark draft-sampling,
 * exact-verification and acceptance-statistics computations, accumulating in
 * double.  Only the test suite, the smoke check and the benchmark's CPU
 * baseline load it.  It shares no source, header or constant with the CUDA
 * library; the two meet only in the byte layout of their inputs.
 *
 * Sources, cited by page title and section:
 *   [FT] FreeToken PR #69 "[2/3] feat(dsv4): implement exact DSpark speculative
 *        decoding" - sections "End-to-end speculative cycle",
 *        "Checkpoint-faithful DSpark architecture", "Exact decoding semantics".
 *   [MB] NeMo Megatron-Bridge "DSpark Speculative Decoding (Draft Training)
 *        Design" - sections "Semi-autoregressive draft", "Training objective",
 *        "Acceptance and confidence", "Loss return contract".
 *   [PT] pypto "DeepSeek V4 DSpark NPU Serving Dev Notes" - section
 *        "Speculative decoding (K=7)", paragraph "Acceptance".
 *   [SMDS] J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel Random Numbers:
 *        As Easy as 1, 2, 3", SC'11 - the Philox-4x32 generator.
 *
 * Layouts (all row-major, host memory):
 *   logits     dtype 0 = bf16 (uint16 bit patterns), 1 = fp32
 *   backbone   [B, gamma, V]      target [B, gamma+1, V]
 *   U          bf16 [V, r]        W      bf16 [V, r]  (row v holds column v of
 *                                                     the r x V Markov matrix)
 *   E          bf16 [V, H]        h      [B, gamma, H] (dtype h_dtype)
 *   w_conf     fp32 [2H]
 *   policy     four parallel arrays of length B.
 */
#ifndef DSPARK_ORACLE_H
#define DSPARK_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Per-request status values written by the oracle. */
enum {
    ORC_OK = 0,
    ORC_NONFINITE = 1,   /* a NaN or +inf logit in a row the request uses   */
    ORC_EMPTY = 2,       /* a row whose logits are all -inf                  */
    ORC_BAD_POLICY = 4,  /* T <= 0 / NaN, top_k < 0 or top_p NaN (sampled)  */
    ORC_BAD_TOKEN = 5    /* an anchor, proposal or label outside [0, V)      */
};

/* Philox-4x32 with 10 rounds [SMDS]. */
void orc_philox4x32_10(uint32_t key0, uint32_t key1, const uint32_t ctr[4],
                       uint32_t out[4]);

/* The uniform in [0,1) keyed by (seed, request, position, draw):
 * key = (lo32 seed, hi32 seed), counter = (draw, lo32 pos, hi32 pos,
 * lo32 request_id); u = (first output word >> 8) * 2^-24. */
double orc_uniform(uint64_t seed, uint64_t request_id, int64_t pos,
                   uint32_t draw);

/* Sampling policy over one row of logits z (double) [FT Exact decoding ›
 * Probabilistic].  Writes p[V]; returns a status.  *argmax receives the
 * lowest index of the maximum.  *indet is set to 1 when a decision the policy
 * takes lies within the tolerance band; exact_logits says whether z is exact
 * input (verify) or a rounded computation (Markov head). */
int orc_policy_row(const double* z, int V, float temperature, int32_t top_k,
                   float top_p, int32_t greedy, int32_t exact_logits,
                   double* p, int32_t* argmax, int32_t* support_size,
                   int32_t* indet);

/* Inverse-CDF draw in token-index order: the smallest i with
 * sum_{j<=i} w_j > u * sum(w).  *margin receives the distance of u*S to the
 * nearer boundary of the chosen interval, divided by S. */
int32_t orc_sample_index(const double* w, int V, double u, double* margin);

/* (a) Markov-head draft sampling [FT Checkpoint-faithful DSpark architecture;
 * MB Semi-autoregressive draft].  Outputs proposals [B,gamma], q [B,gamma,V]
 * (greedy rows untouched), q_at_x, conf (if h != NULL), status [B], and per
 * (b,k) an indeterminacy flag indet [B,gamma]. */
void orc_markov_sample(const void* backbone, int32_t dtype,
                       const int32_t* anchor, const uint16_t* U,
                       const uint16_t* W, int32_t r, const void* h,
                       int32_t h_dtype, const uint16_t* E, const float* w_conf,
                       int32_t H, const float* temperature,
                       const int32_t* top_k, const float* top_p,
                       const int32_t* greedy, const uint64_t* seed,
                       const uint64_t* request_id, const int64_t* pos0,
                       int32_t B, int32_t gamma, int32_t V, int32_t* proposals,
                       float* q, float* q_at_x, float* conf, int32_t* status,
                       uint8_t* indet);

// RNN-head draft sampling: the Markov sampler with the bias taken from a GRU
// state carried across the block (Wi, Wh bf16 [3r, r] in gate order r, z, n;
// bi, bh fp32 [3r]); states (may be NULL) receives s_k, [B, gamma, r].
void orc_rnn_sample(const void* backbone, int32_t dtype, const int32_t* anchor,
                    const uint16_t* U, const uint16_t* W, int32_t r,
                    const uint16_t* Wi, const uint16_t* Wh, const float* bi,
                    const float* bh, const void* h, int32_t h_dtype,
                    const uint16_t* E, const float* w_conf, int32_t H,
                    const float* temperature, const int32_t* top_k,
                    const float* top_p, const int32_t* greedy,
                    const uint64_t* seed, const uint64_t* request_id,
                    const int64_t* pos0, int32_t B, int32_t gamma, int32_t V,
                    int32_t* proposals, float* q, float* q_at_x, float* conf,
                    int32_t* status, uint8_t* indet, double* states);

/* (b) Exact verify [FT Exact decoding semantics; PT Acceptance].
 * out_tokens [B, gamma+1] (-1 after the emitted tokens), num_accepted [B]
 * (-1 for a failed request), status [B], indet [B].  det_tokens [B] and
 * det_nacc [B] (each may be NULL): the leading out_tokens entries decided
 * before the request's first indeterminate decision, and 1 if num_accepted
 * was decided before it (gamma + 1 and 1 when indet is 0). */
void orc_verify(const void* target, int32_t dtype, const int32_t* proposals,
                const float* q, const float* q_at_x, const float* temperature,
                const int32_t* top_k, const float* top_p, const int32_t* greedy,
                const uint64_t* seed, const uint64_t* request_id,
                const int64_t* pos0, int32_t B, int32_t gamma, int32_t V,
                int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
                uint8_t* indet, int32_t* det_tokens, uint8_t* det_nacc);
/* (b') The same verify over a per-request width: request b checks its first
 * width[b] proposals (0..gamma) against target rows 0..width[b] and draws the
 * bonus from row width[b]; width NULL = gamma for every request.  A width
 * outside [0, gamma] is reported as a bad token. */
void orc_verify_width(const void* target, int32_t dtype, const int32_t* proposals,
                      const float* q, const float* q_at_x, const float* temperature,
                      const int32_t* top_k, const float* top_p, const int32_t* greedy,
                      const uint64_t* seed, const uint64_t* request_id,
                      const int64_t* pos0, int32_t B, int32_t gamma, int32_t V,
                      const int32_t* width, int32_t* out_tokens, int32_t* num_accepted,
                      int32_t* status, uint8_t* indet, int32_t* det_tokens, uint8_t* det_nacc);

/* (c) Analytical acceptance statistics [MB Training objective; Acceptance
 * and confidence; Loss return contract].  draft/target [N,gamma,V] at T=1
 * with no truncation.  l1, accept [N,gamma]; tau [N]; loss_num [4] =
 * (CE, L1, BCE, 0.1 CE + 0.9 L1 + 1.0 BCE) weighted numerators;
 * report [2] = (sum of m*accept, sum of tau); num_tokens = sum of mask;
 * status [N] (may be NULL). */
void orc_accept_stats(const void* draft, const void* target, int32_t dtype,
                      const int32_t* labels, const float* conf_logits,
                      const uint8_t* mask, int32_t N, int32_t gamma, int32_t V,
                      float* l1, float* accept, float* tau, double* loss_num,
                      double* report, int64_t* num_tokens, int32_t* status);

/* (c') Gradient of the loss numerators' total 0.1 CE + 0.9 L1 + 1.0 BCE
 * (weighted, masked) with respect to the draft logits [N,gamma,V] and the
 * confidence logits [N,gamma], the target and the BCE label (accept) held
 * fixed, times scale.  Masked positions: 0; a non-finite logit or a label
 * outside [0, V): NaN. */
void orc_accept_stats_backward(const void* draft, const void* target, int32_t dtype,
                               const int32_t* labels, const float* conf_logits,
                               const uint8_t* mask, int32_t N, int32_t gamma, int32_t V,
                               double scale, float* grad_draft, float* grad_conf);

// Sequential Temperature Scaling: per block position k the inverse
// temperature beta[k] >= 0 minimising the masked BCE of sigmoid(beta z)
// against the accept labels (conf_logits, labels fp32 [N, gamma]); status[k]:
// 0 fitted, 1 no information (beta 1), 2 separated labels (beta 2^20),
// 3 a non-finite logit or a label outside [0, 1] (beta NaN).
void orc_sts_fit(const float* conf_logits, const float* labels, const uint8_t* mask,
                 int32_t N, int32_t gamma, double* beta, int32_t* status);

#ifdef __cplusplus
}
#endif

#endif
