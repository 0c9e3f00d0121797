/*
 * dspark.h - C ABI of the DSpark draft-sampling / exact-verification library
 * for NVIDIA GB300 (sm_103a).
 *
 * Three operations, each a pass over vocabulary-wide logit rows:
 *
 *   dspark_markov_sample  the semi-autoregressive draft's sequential head:
 *                         low-rank Markov logit bias, sampling policy, a
 *                         proposal per position left to right, the full
 *                         proposal distribution q and a confidence per
 *                         position.
 *   dspark_rnn_sample     the same draft with the RNN head: a GRU state
 *                         carried across the block gives the low-rank bias.
 *   dspark_verify         exact verification of a proposal block against the
 *                         target's logits: greedy contiguous-prefix argmax
 *                         acceptance, or accept-with-min(1, p/q), residual
 *                         resampling and a bonus token.
 *   dspark_verify_width   the same over a per-request number of proposals
 *                         to check (0..gamma).
 *   dspark_accept_stats   the analytical training-side statistics: L1
 *                         distance, acceptance rate, tau and the weighted
 *                         CE / L1 / confidence-BCE numerators.
 *   dspark_accept_stats_grad  their loss's gradient with respect to the
 *                         draft logits and the confidence logits.
 *   dspark_sts_fit        Sequential Temperature Scaling: the confidence
 *                         head's per-position inverse temperatures.
 *
 * Sources, by page title and section:
 *   [FT] FreeToken PR #69 "[2/3] feat(dsv4): implement exact DSpark
 *        speculative decoding": "End-to-end speculative cycle",
 *        "Checkpoint-faithful DSpark architecture", "Exact decoding
 *        semantics" (Greedy; Probabilistic), "Scope and limitations" and
 *        the review thread below it.
 *   [MB] NeMo Megatron-Bridge "DSpark Speculative Decoding (Draft Training)
 *        Design": "Semi-autoregressive draft", "Training objective",
 *        "Acceptance and confidence", "Loss return contract", "Memory
 *        contract for the full-vocabulary terms".
 *   [PT] pypto "DeepSeek V4 DSpark NPU Serving Dev Notes": "Speculative
 *        decoding (K=7)" (decode tile, Acceptance).
 *
 * Conventions shared by every entry point
 *   Memory     Every array argument is DEVICE memory owned by the caller.  The
 *              library allocates nothing and keeps no state between calls;
 *              scratch lives in the caller's workspace.
 *   Stream     `stream` is a cudaStream_t (NULL = the legacy default stream).
 *              Work is enqueued asynchronously; nothing synchronises the host.
 *   Layout     Row-major.  Logit rows are contiguous, V elements each.
 *   dtype      DSPARK_BF16 (bfloat16 bit patterns) or DSPARK_F32.
 *   Sizes      1 <= gamma <= DSPARK_MAX_GAMMA; V a multiple of 8 with
 *              8 <= V <= DSPARK_MAX_VOCAB; B (or N) >= 0, and 0 is a no-op.
 *   Alignment  Logit, q and hidden-state arrays start on a 16-byte boundary.
 *   Returns    DSPARK_OK, or a negative dspark_status for an argument error
 *              found on the host before anything is enqueued (nothing is
 *              launched then), or DSPARK_ECUDA if a launch failed.
 *   Status     Problems that depend on data are reported per request in
 *              `status` (dspark_request_status), never by a trap.
 *   Workspace  dspark_workspace_size() gives the bytes an operation needs.
 *              The workspace must be zero-filled once after allocation
 *              (e.g. cudaMemsetAsync(ws, 0, bytes, stream)); every call that
 *              completes returns the words a call reads before writing them
 *              (tickets, records, the error flag) to zero, so it can be
 *              reused by the next call of the same operation on the same
 *              stream without clearing.  The other regions (the Markov
 *              logits, per-CTA partial sums) keep what the call wrote; every
 *              call overwrites them before reading them.  Calls that share one workspace must not overlap in
 *              time, and a workspace serves one operation (clear it before
 *              handing it to another).  The greedy paths keep all their state
 *              on chip and ignore the workspace (it may be NULL): dspark_verify
 *              with policy NULL, and dspark_markov_sample with policy NULL and
 *              r = 0.
 *   Random     Each random decision draws u in [0,1) from Philox-4x32-10
 *              (Salmon et al., SC'11) with key (lo32 seed, hi32 seed) and
 *              counter (draw, lo32 pos, hi32 pos, lo32 request_id):
 *              u = (first output word >> 8) * 2^-24.  pos is the absolute
 *              position of the token being decided; draw 0 = proposal,
 *              1 = accept test, 2 = residual / bonus.  Only the low 32 bits
 *              of request_id enter the counter.
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSPARK_MAX_GAMMA 16
#define DSPARK_MAX_VOCAB (1 << 20)
#define DSPARK_MAX_RANK 256
#define DSPARK_MAX_BATCH 256  /* requests per dspark_markov_sample call */
#define DSPARK_STS_MAX_PASSES 4096  /* largest pass budget of dspark_sts_fit */

/* Sampling policy of one request [FT Exact decoding semantics > Probabilistic:
 * p and q are formed after the request's temperature, top-p and top-k].
 *   greedy != 0   one-hot at the argmax (lowest index on ties); the other
 *                 fields are ignored.
 *   temperature   > 0; logits are scaled by the fp32 value of 1/temperature.
 *   top_k         0 or >= V disables; otherwise exactly top_k tokens are kept,
 *                 taken in (logit descending, index ascending) order.
 *   top_p         >= 1 disables; otherwise the shortest prefix of that order,
 *                 inside the top-k set, whose share of the kept mass is
 *                 >= top_p (at least one token).
 * Temperature is applied first, then top-k, then top-p on the renormalised
 * top-k distribution. */
typedef struct {
    float temperature;
    int32_t top_k;
    float top_p;
    int32_t greedy;
} dspark_policy;

typedef enum {
    DSPARK_OK = 0,
    DSPARK_EINVAL = -1,   /* a size, pointer, alignment or enum is invalid   */
    DSPARK_ENOSPC = -2,   /* workspace smaller than dspark_workspace_size() */
    DSPARK_ECUDA = -3,    /* a CUDA launch or attribute call failed          */
    DSPARK_ENOTSUP = -4   /* valid but unsupported on this device / build    */
} dspark_status;

enum { DSPARK_BF16 = 0, DSPARK_F32 = 1 };

/* Values written to the per-request `status` arrays. */
typedef enum {
    DSPARK_REQ_OK = 0,
    DSPARK_REQ_NONFINITE = 1,  /* a NaN or +inf logit in a row the request uses */
    DSPARK_REQ_EMPTY = 2,      /* a row whose logits are all -inf               */
    DSPARK_REQ_TIMEOUT = 3,    /* a bounded device-side wait gave up            */
    DSPARK_REQ_BAD_POLICY = 4, /* temperature <= 0 or NaN, top_k < 0, top_p NaN */
    DSPARK_REQ_BAD_TOKEN = 5   /* an anchor, proposal or label outside [0, V)   */
} dspark_request_status;

enum {
    DSPARK_OP_MARKOV_SAMPLE = 0,
    DSPARK_OP_VERIFY = 1,
    DSPARK_OP_ACCEPT_STATS = 2,
    DSPARK_OP_STS_FIT = 3,
    DSPARK_OP_RNN_SAMPLE = 4
};

/* Workspace bytes `op` needs for these sizes (r matters only for
 * DSPARK_OP_MARKOV_SAMPLE and DSPARK_OP_RNN_SAMPLE; pass B = N for DSPARK_OP_ACCEPT_STATS and
 * DSPARK_OP_STS_FIT, whose V is not used).  Returns 0 for invalid sizes. */
size_t dspark_workspace_size(int op, int B, int gamma, int V, int r, int H);

/*
 * dspark_markov_sample - the draft's sequential head over one gamma block.
 *
 * [FT Checkpoint-faithful DSpark architecture]: the Markov head runs left to
 * right so proposal k conditions on proposal k-1, the first on the anchor; the
 * full proposal distribution q and the confidences are kept.
 * [MB Semi-autoregressive draft]: the Markov head is a low-rank
 * token-conditioned additive logit bias; the confidence is
 * c_k = sigmoid(w^T [h_k ; embed(x_{k-1})]).
 *
 * For k = 1..gamma, for every request b (x_0 = anchor[b]):
 *   z_k[v]  = backbone[b,k-1,v] + sum_j U[x_{k-1}, j] * W[v, j]   (fp32)
 *   q_k     = policy(z_k)
 *   x_k     = inverse-CDF draw from q_k in token-index order (u: pos0+k,
 *             draw 0); greedy requests take the argmax
 *   c_k     = sigmoid(w_conf[0:H] . h[b,k-1,:] + w_conf[H:2H] . E[x_{k-1},:])
 *
 *   backbone  [B, gamma, V] logits of the parallel backbone, `dtype`.
 *   anchor    int32 [B]: the last committed token of each request.
 *   U         bf16 [V, r]: token embedding of the Markov head (row x).
 *   W         bf16 [V, r]: the r x V output matrix stored transposed, i.e.
 *             row v holds its column v (a Linear(r, V) weight).
 *   r         rank: 0 (no bias; U and W unused) or a multiple of 16 up to
 *             DSPARK_MAX_RANK.
 *   h         [B, gamma, H] draft hidden states (h_dtype), or NULL to skip
 *             the confidence (conf, E, w_conf then unused).
 *   E         bf16 [V, H] draft token embedding;  w_conf  fp32 [2H].
 *   policy    [B] per-request policies, or NULL: every request greedy.
 *   seed, request_id  uint64 [B];  pos0  int64 [B]: position of the anchor.
 *   proposals int32 [B, gamma] out: x_1..x_gamma (-1 after a failure).
 *   q         fp32 [B, gamma, V] out: q_k of sampled requests (0 outside the
 *             support); rows of greedy requests are not written.  May be NULL
 *             only when policy is NULL.
 *   q_at_x    fp32 [B, gamma] out: q_k(x_k); 1 for greedy requests.
 *   conf      fp32 [B, gamma] out (when h != NULL): c_k.
 *   status    int32 [B] out: dspark_request_status.
 *
 * B <= DSPARK_MAX_BATCH.  The gamma steps are sequential.  With a bf16
 * backbone, r a multiple of 64 (64..256), at most 64 requests and a
 * vocabulary the device's SMs hold in eight 128-token tiles each, all steps
 * run in one persistent launch that keeps the biased logits on chip;
 * otherwise each step enqueues at most two kernels (the bias GEMM, then the
 * policy and draw).  dspark_markov_launches() says which.
 */
int dspark_markov_sample(const void* backbone, int dtype, const int32_t* anchor,
                         const uint16_t* U, const uint16_t* W, int r,
                         const void* h, int h_dtype, const uint16_t* E,
                         const float* w_conf, int H, const dspark_policy* policy,
                         const uint64_t* seed, const uint64_t* request_id,
                         const int64_t* pos0, int B, int gamma, int V,
                         int32_t* proposals, float* q, float* q_at_x,
                         float* conf, int32_t* status, void* workspace,
                         size_t workspace_bytes, void* stream);

/* Kernels one dspark_markov_sample call with these sizes enqueues on the
 * current device (the confidence kernel included when with_conf is nonzero),
 * or -1 when the sizes are invalid.  The path depends on the device's SM
 * count, so this asks the CUDA runtime for the current device's properties. */
int dspark_markov_launches(int dtype, int B, int gamma, int V, int r, int with_policy, int with_conf);

/* The same for dspark_rnn_sample (r >= 16). */
int dspark_rnn_launches(int dtype, int B, int gamma, int V, int r, int with_conf);

/*
 * dspark_rnn_sample - the draft's sequential head in its RNN form.
 *
 * [MB Semi-autoregressive draft]: besides the Markov head DSpark offers an
 * RNN head, a GRU-like recurrence carrying prefix state across the block,
 * run serially at inference.  The pages give no equations; the reading: a
 * standard GRU cell (gate order r, z, n) whose input is the rank-r embedding
 * of the previous token, e_k = U[x_{k-1}] (x_0 = the anchor), from the state
 * s_0 = 0 of every block:
 *   r = sigmoid(Wi_r e + bi_r + Wh_r s + bh_r)
 *   z = sigmoid(Wi_z e + bi_z + Wh_z s + bh_z)
 *   n = tanh(Wi_n e + bi_n + r * (Wh_n s + bh_n)),   s_k = (1 - z) n + z s
 * and its state gives a bias of the Markov head's form, added to the backbone
 * logits: z_k[v] = backbone_k[v] + sum_j s_k[j] W[v, j].  Everything else
 * (policy, proposals, q, q_at_x, confidence, statuses, random draws) is
 * dspark_markov_sample's.
 *   U, W       bf16 [V, r], r a multiple of 16 in 16..DSPARK_MAX_RANK.
 *   Wi, Wh     bf16 [3r, r] (rows r, z, n); 16-byte aligned.
 *   bi, bh     fp32 [3r].
 *   Sizes      B <= DSPARK_MAX_BATCH and B <= V.
 *   workspace  dspark_workspace_size(DSPARK_OP_RNN_SAMPLE, B, gamma, V, r, 0).
 * The bias reaches the logits through the tensor cores in bf16: s_k is passed
 * as hi = bf16(s_k) plus lo = bf16(s_k - hi), two products summed in fp32, so
 * the logits carry s_k to about 2^-16 of its size.  Under the same conditions
 * as dspark_markov_sample's one-launch path (bf16 backbone, r a multiple of
 * 64, at most 64 requests) the whole draft, GRU cell included, runs in one
 * persistent launch; otherwise each step enqueues four kernels.
 * dspark_rnn_launches() says which.
 */
int dspark_rnn_sample(const void* backbone, int dtype, const int32_t* anchor,
                      const uint16_t* U, const uint16_t* W, int r,
                      const uint16_t* Wi, const uint16_t* Wh, const float* bi,
                      const float* bh, const void* h, int h_dtype,
                      const uint16_t* E, const float* w_conf, int H,
                      const dspark_policy* policy, const uint64_t* seed,
                      const uint64_t* request_id, const int64_t* pos0, int B,
                      int gamma, int V, int32_t* proposals, float* q,
                      float* q_at_x, float* conf, int32_t* status,
                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * dspark_verify - exact verification of one proposal block per request.
 *
 * [FT Exact decoding semantics > Greedy]: accept the contiguous prefix of
 * proposals equal to the target argmax; at the first disagreement emit the
 * target's own token; a later accidental match is never accepted.
 * [FT > Probabilistic]: accept x_k with probability min(1, p(x_k)/q(x_k)); at
 * the first rejection sample from normalised max(p - q, 0); if every
 * proposal survives, sample a bonus token from the target's next-position
 * distribution.  [PT Acceptance]: 1..gamma+1 tokens per request and step.
 *
 * Target row i (i = 0..gamma) is the target's next-token distribution after
 * (anchor, x_1..x_i): row k-1 scores proposal x_k, row gamma gives the bonus.
 *   target     [B, gamma+1, V] target logits, `dtype`.
 *   proposals  int32 [B, gamma].
 *   q, q_at_x  fp32 [B, gamma, V] and [B, gamma] from dspark_markov_sample;
 *              read only for sampled requests (may be NULL if policy is NULL).
 *   policy     [B], or NULL: every request greedy (the fastest path).
 *   seed, request_id, pos0  as for dspark_markov_sample.  The accept test of
 *              x_k draws at pos0+k (draw 1); the residual at rejection j at
 *              pos0+j (draw 2); the bonus at pos0+gamma+1 (draw 2).
 *   out_tokens int32 [B, gamma+1] out: the emitted tokens, -1 after them.
 *   num_accepted int32 [B] out: accepted proposals n (emitted = n + 1), or -1
 *              for a failed request.
 *   status     int32 [B] out.
 * Sampled accept test: accept iff p(x) > 0 and u < p(x)/q(x) (q(x) = 0 with
 * p(x) > 0 accepts).  A residual with zero mass falls back to p.
 */
int dspark_verify(const void* target, int dtype, const int32_t* proposals,
                  const float* q, const float* q_at_x,
                  const dspark_policy* policy, const uint64_t* seed,
                  const uint64_t* request_id, const int64_t* pos0, int B,
                  int gamma, int V, int32_t* out_tokens, int32_t* num_accepted,
                  int32_t* status, void* workspace, size_t workspace_bytes,
                  void* stream);

/*
 * dspark_verify_width - dspark_verify over a per-request verify width.
 *
 * [FT Scope and limitations, and the review thread]: a serving scheduler
 * may verify fewer than gamma proposals of a request (0..gamma), choosing the
 * width from measured draft and verify costs (the pages give no formula, so
 * the width is an input); [FT Exact decoding semantics] holds at any width.  With width w the request checks x_1..x_w against
 * target rows 0..w-1 exactly as dspark_verify does, and when all w survive
 * the bonus token comes from row w at pos0+w+1 (draw 2).  Rows past w are
 * not read and proposals past x_w are ignored (both may hold anything);
 * emitted tokens are 1..w+1, and out_tokens is -1 after them.
 *   width      int32 [B] device, each in [0, gamma]; NULL = gamma for every
 *              request (exactly dspark_verify).  A width outside [0, gamma]
 *              fails that request with DSPARK_REQ_BAD_TOKEN (num_accepted -1).
 * Every other argument, the layouts (still [B, gamma+1, V] and [B, gamma])
 * and the workspace are those of dspark_verify.  Rows past the width cost a
 * CTA launch each but move no logit bytes.
 */
int dspark_verify_width(const void* target, int dtype, const int32_t* proposals,
                        const float* q, const float* q_at_x,
                        const dspark_policy* policy, const uint64_t* seed,
                        const uint64_t* request_id, const int64_t* pos0,
                        const int32_t* width, int B, int gamma, int V,
                        int32_t* out_tokens, int32_t* num_accepted,
                        int32_t* status, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * dspark_accept_stats - analytical acceptance statistics of a draft against
 * the target, per position, and the weighted loss numerators.
 *
 * [MB Training objective]: weights exp(-k/gamma); L_ce (0.1) against the
 * target's teacher-forced next tokens; L_l1 (0.9) the raw
 * ||p_draft - p_target||_1; L_conf (1.0) BCE of the confidence against the
 * acceptance label.  [MB Acceptance and confidence]: accept_rate =
 * clamp(1 - 0.5 L1, 0, 1); tau = sum_k cumprod(accept_rate)_k + 1.
 * [MB Loss return contract]: numerators and a token count, never ratios.
 *
 *   draft, target  [N, gamma, V] logits (`dtype`); position k = 1..gamma of
 *                  block n; both at temperature 1 with no truncation.
 *   labels         int32 [N, gamma]: the teacher tokens for the CE term.
 *   conf_logits    fp32 [N, gamma]: the confidence head's logits z.
 *   mask           uint8 [N, gamma] (nonzero = counted) or NULL (all).
 *   l1, accept     fp32 [N, gamma] out, for every position.
 *   tau            fp32 [N] out.
 *   loss_num       fp64 [4] out: sum m w_k CE, sum m w_k L1, sum m w_k BCE and
 *                  0.1 CE + 0.9 L1 + 1.0 BCE, with BCE = softplus(z) - a z.
 *   report         fp64 [2] out: sum m accept, sum tau (report numerators;
 *                  their denominators are num_tokens and N).
 *   num_tokens     int64 [1] out: sum m.
 *   status         int32 [N] out, or NULL.
 * Sums are formed in a fixed order: repeated calls give identical bits.
 */
int dspark_accept_stats(const void* draft, const void* target, int dtype,
                        const int32_t* labels, const float* conf_logits,
                        const uint8_t* mask, int N, int gamma, int V,
                        float* l1, float* accept, float* tau, double* loss_num,
                        double* report, int64_t* num_tokens, int32_t* status,
                        void* workspace, size_t workspace_bytes, void* stream);

/*
 * dspark_accept_stats_grad - the backward of dspark_accept_stats' loss: the
 * gradient of J = 0.1 CE + 0.9 L1 + 1.0 BCE (the weighted, masked numerators'
 * total, loss_num[3]) with respect to the draft logits and the confidence
 * logits, times `scale` (e.g. the caller's 1 / num_tokens).  The target is
 * the frozen teacher and the BCE label accept_rate is detached, so
 *   d J / d draft[n,k,v] = scale m w_k (0.1 (p_d,v - [v = label])
 *                                       + 0.9 p_d,v (s_v - sum_u s_u p_d,u)),
 *   s_v = sign(p_d,v - p_t,v) (0 at equality),
 *   d J / d conf_logits[n,k] = scale m w_k (sigmoid(z) - accept_rate).
 * [MB Training objective; Memory contract for the full-vocabulary terms]:
 * the softmax statistics are recomputed per row; nothing full-vocabulary is
 * kept between the passes.
 *
 *   draft, target, labels, conf_logits, mask   as for dspark_accept_stats.
 *   scale          the factor applied to both gradients.
 *   grad_draft     fp32 [N, gamma, V] out (16-byte aligned).
 *   grad_conf      fp32 [N, gamma] out.
 * Masked positions get zeros; a position with a NaN / +inf logit or a label
 * outside [0, V) gets NaN (its whole draft gradient row).  No workspace.
 */
int dspark_accept_stats_grad(const void* draft, const void* target, int dtype,
                             const int32_t* labels, const float* conf_logits,
                             const uint8_t* mask, int N, int gamma, int V,
                             double scale, float* grad_draft, float* grad_conf,
                             void* stream);

/*
 * dspark_verify_greedy_noalloc - the greedy verify of dspark_verify (policy
 * NULL) without workspace arguments, for callers that cannot allocate device
 * memory.  None of the pages has a counterpart; it exists for callers such as
 * a plugin inside a runtime that owns all device memory and offers no
 * allocator, or a latency-critical path that must not call cudaMalloc (which
 * may synchronize the device).
 *
 * Arguments and outputs are those of dspark_verify with every request greedy;
 * the caller provides target, proposals and the three output arrays.  The
 * greedy kernel keeps every intermediate in shared memory (each request's
 * rows are reduced by one thread-block cluster), so the call needs no scratch
 * at all: the library allocates nothing and reserves no device memory for it.
 * Calls on different streams may overlap freely.
 */
int dspark_verify_greedy_noalloc(const void* target, int dtype, const int32_t* proposals, int B,
                                 int gamma, int V, int32_t* out_tokens, int32_t* num_accepted,
                                 int32_t* status, void* stream);

/* A short English description of a dspark_status or request-status code
 * (negative = dspark_status, non-negative = dspark_request_status). */
const char* dspark_status_string(int code);

/* Library version, major * 10000 + minor * 100 + patch. */
int dspark_version(void);

/*
 * dspark_wait_selftest - diagnostic of the library's bounded device waits.
 *
 * The persistent kernels (the fused Markov draft, the temperature-scaling
 * fit) meet at grid barriers whose waits end after about 2 s of global time
 * at most, so that a block that never arrives turns into a status instead of
 * a hung GPU.  This call launches `blocks` thread blocks (1..64, all
 * resident) that meet at one such barrier told to expect blocks + missing
 * arrivals: with missing > 0 the wait can end only by its limit.  Nothing else
 * is in flight meanwhile (no copy, MMA or tensor memory).
 *   limit_us   the wait's limit, 1..2,000,000 microseconds.
 *   status     int32 [blocks] out: DSPARK_REQ_OK when the barrier completed,
 *              DSPARK_REQ_TIMEOUT when the block gave up waiting (a block
 *              that sees another give up stops waiting too).
 *   waited_ns  uint64 [blocks] out: the global time each block waited.
 *   workspace  at least 256 bytes of device memory, 16-byte aligned (the
 *              barrier's count and error word, set by the call).
 * The device stays usable afterwards; any later call may follow on the
 * stream.
 */
int dspark_wait_selftest(int blocks, int missing, int limit_us, int32_t* status, uint64_t* waited_ns,
                         void* workspace, void* stream);

/*
 * dspark_sts_fit - Sequential Temperature Scaling of the confidence head.
 *
 * [MB Acceptance and confidence]: the confidence head regresses to the
 * accept rate, and a post-hoc Sequential Temperature Scaling calibrates it
 * for serving.  The pages give no formula; the reading: temperature scaling
 * with one inverse temperature per block position k, beta_k >= 0, the
 * calibrated confidence being sigmoid(beta_k z); beta_k minimises the masked
 * BCE of sigmoid(beta_k z) against the accept labels over N logged blocks.
 *   conf_logits  fp32 [N, gamma]: the confidence head's logits z.
 *   labels       fp32 [N, gamma]: the accept labels a in [0, 1] (e.g. the
 *                accept rates dspark_accept_stats reports, or observed 0/1
 *                acceptances).
 *   mask         uint8 [N, gamma] (nonzero = counted) or NULL (all).
 *   beta         fp64 [gamma] out.
 *   status       int32 [gamma] out, per position: 0 fitted; 1 no counted
 *                pair with z != 0 (beta = 1); 2 every label agrees with the
 *                sign of its z (a = 1 for z > 0, a = 0 for z < 0), or the
 *                root lies beyond 2^20: no finite fit (beta = 2^20); 3 a
 *                counted pair with a non-finite z or a label outside [0, 1]
 *                (beta = NaN); 4 the pass budget ran out with the search
 *                still open (beta = its last iterate, not the fit); 5 a
 *                wait between the fit's thread blocks ran past its time
 *                limit (about 2 s), so beta is not a fit.  A BCE slope >= 0
 *                at beta = 0 gives beta = 0 (status 0).
 *   passes       int32 [gamma] out, or NULL: the passes over the pairs each
 *                position's search used (every pass reads all positions
 *                until the last one stops).
 *   max_passes   the pass budget, 1..DSPARK_STS_MAX_PASSES, or 0 for 64
 *                (enough for beta to double from 1 to the 2^20 cap and then
 *                halve its bracket below 1e-7; Newton usually ends in ten
 *                or fewer).  The fit stops after the pass in which the last
 *                position stopped.
 *   workspace    dspark_workspace_size(DSPARK_OP_STS_FIT, N, gamma, 0, 0, 0)
 *                bytes; every region is written before it is read.
 * N = 0 is valid (every position reports status 1).  The fit is a root
 * search on the device (Newton steps inside a bracket) in one persistent
 * cooperative launch, with three kernels enqueued in all; beta is accurate
 * to about 1e-6 relative (its sums are fp32 per thread, fp64 across
 * threads) and bit-identical across calls on the same inputs and device
 * (the CTAs' sums are combined in a fixed order).
 */
int dspark_sts_fit(const float* conf_logits, const float* labels,
                   const uint8_t* mask, int N, int gamma, double* beta,
                   int32_t* status, int32_t* passes, int max_passes, void* workspace,
                   size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
