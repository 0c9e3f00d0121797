// Internal launch interface between the C ABI (abi.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

enum { kArgmaxVerify = 0, kArgmaxDraft = 1 };

// Row arg-max and greedy decisions, one cluster per request (argmax.cu).
struct ArgmaxParams {
    const void* logits;       // [groups, rows_per_group, V]
    int dtype;
    int V;
    int rows_per_group;       // rows of one request: gamma+1 (verify) or gamma (draft)
    int gamma;
    int mode;                 // kArgmaxVerify / kArgmaxDraft
    int64_t per;              // elements per CTA of a request (set by the launcher)
    // verify
    const int32_t* proposals;
    int32_t* out_tokens;
    int32_t* num_accepted;
    // draft
    const int32_t* anchor;
    int32_t* props_out;
    float* q_at_x;
    int32_t* status;
};
// Greedy verify over a per-request width: the same block plus the widths, a
// type of its own so that the fixed-width kernel keeps its parameter block.
struct ArgmaxWidthParams : ArgmaxParams {
    const int32_t* width;     // [groups] proposals each request checks (0..gamma)
};
// width null: the fixed-width kernel; otherwise (verify mode) its width variant
cudaError_t launch_argmax_rows(ArgmaxParams p, int groups, cudaStream_t stream,
                               const int32_t* width = nullptr);
int argmax_cluster_size(int dtype, int groups);

// Confidence head c_k = sigmoid(w[:H] . h_k + w[H:] . E[x_{k-1}]) (confidence.cu).
struct ConfParams {
    const void* h;
    int h_dtype;
    const uint16_t* E;
    const float* w;
    int H;
    int B;
    int gamma;
    int V;
    const int32_t* anchor;
    const int32_t* proposals;  // [B, gamma]; x_{k-1} = proposals[k-2] for k >= 2
    int k_first, k_last;       // 1-based positions to compute, inclusive
    float* conf;
};
cudaError_t launch_confidence(const ConfParams& p, cudaStream_t stream);

// Sampled paths on the row engine (policy_kernels.cu).
struct RowRecord {  // the policy of one target row, for the request's decision
    float zmax;
    float inv_t;
    uint32_t tau;     // support = {key > tau} + {key == tau, index <= cut}
    int32_t cut;
    uint64_t mass;    // fixed-point (2^-40) mass of the support
    float p_x;        // p of the proposal this row scores
    int32_t status;
    int32_t argmax;
    int32_t count;    // support size
};
struct VerifyProbParams {
    const void* target;
    int dtype;
    const int32_t* proposals;
    const float* q;
    const float* q_at_x;
    const dspark_policy* policy;
    const uint64_t* seed;
    const uint64_t* request_id;
    const int64_t* pos0;
    int B, gamma, V;
    int slice;                 // elements per CTA of a row's cluster
    int32_t* out_tokens;
    int32_t* num_accepted;
    int32_t* status;
    RowRecord* records;        // [B * (gamma + 1)] workspace
    unsigned int* ticket;      // [B] workspace, zero on entry and exit
};
struct MarkovStepParams {
    const void* backbone;      // [B, gamma, V] (dtype), read when zbuf is null
    int dtype;
    const float* zbuf;         // [B, V] fp32 logits with the Markov bias, or null
    const int32_t* anchor;
    int32_t* proposals;
    float* q;
    float* q_at_x;
    int32_t* status;
    const dspark_policy* policy;   // null: every request greedy
    const uint64_t* seed;
    const uint64_t* request_id;
    const int64_t* pos0;
    int B, gamma, V;
    int slice;
    int k;                     // 1-based step
    const int* error_flag;     // set by the bias kernel when a device wait gave up
};

// Markov bias on the tensor cores (markov_gemm.cu).
struct MarkovGemmParams {
    const void* backbone;      // [B, gamma, V] (dtype)
    int dtype;
    const uint16_t* U;         // bf16 [V, r]
    const uint16_t* W;         // bf16 [V, r]
    const int32_t* anchor;
    const int32_t* proposals;  // [B, gamma]: x_{k-1} = proposals[b, k-2] for k >= 2
    int B, gamma, V, r;
    int k;                     // 1-based step
    float* zbuf;               // [B, V] fp32 out
    int* error_flag;
    // set by prepare_markov_bias
    int mtiles;                // 128-request M tiles (1 or 2)
    int nt;                    // vocabulary rows per tile (MMA N)
    int stages;                // W tiles in flight per CTA
    int rpq;                   // requests per 32-row TMEM lane quadrant of an M tile
    int nbb;                   // backbone blocks in flight per epilogue warp (1 or 2)
    int grid;
};
// Opaque per-call state of the bias GEMM (the W tensor map).
struct MarkovGemmPlan {
    alignas(64) unsigned char tmap[128];
    bool sw128;
};
// Fill the launch shape of `p` and the tensor map of W; false if B or r are
// outside what the kernel supports.
bool prepare_markov_bias(MarkovGemmParams& p, MarkovGemmPlan& plan);
// overlap: a programmatic launch behind the previous step's policy kernel
// (its z buffer must differ from the one that kernel reads).
cudaError_t launch_markov_bias(const MarkovGemmParams& p, const MarkovGemmPlan& plan, bool overlap,
                               cudaStream_t stream);
// The whole draft (every step's bias GEMM, policy and draw) in one persistent
// launch with the biased logits in tensor memory (markov_fused.cu): bf16
// backbone, r a multiple of 64 up to 256, a vocabulary of at most 8 tiles of
// 128 per SM, and one group of at most kFusedMaxBatch requests (the kernel
// runs larger batches as groups one after another, which the per-step path
// beats: 3.1 against 1.2 ms at 256 requests, 129,280 tokens, r = 256).
constexpr int kFusedMaxBatch = 64;
struct MarkovFusedArgs {
    const uint16_t* backbone;  // bf16 [B, gamma, V]
    const uint16_t* U;         // bf16 [V, r]
    const uint16_t* W;         // bf16 [V, r]
    const int32_t* anchor;
    const dspark_policy* policy;
    const uint64_t* seed;
    const uint64_t* request_id;
    const int64_t* pos0;
    int B, gamma, V, r;
    int32_t* proposals;
    float* q;
    float* q_at_x;
    int32_t* status;
    // the RNN head instead of the Markov head (all four set, or all null):
    // the GRU cell's weights; the bias is then W s_k with s_k the GRU state
    const uint16_t* Wi = nullptr;  // bf16 [3r, r], gate order r, z, n
    const uint16_t* Wh = nullptr;  // bf16 [3r, r]
    const float* bi = nullptr;     // [3r]
    const float* bh = nullptr;     // [3r]
};
// rnn: the RNN head's form (one shared-memory operand more, one W stage fewer)
bool markov_fused_supported(int dtype, int B, int V, int r, bool rnn = false);
// Workspace bytes from the start of the Markov workspace (its first 256 bytes
// belong to the per-step path's error word); rnn adds the GRU state buffers.
size_t markov_fused_workspace(int B, int gamma, int V, int r = 0, bool rnn = false);
cudaError_t launch_markov_fused(const MarkovFusedArgs& a, void* ws, size_t ws_bytes, cudaStream_t stream);

// Elements of a row each CTA of the verify / drafting step owns.
int verify_slice(int V);
int step_slice(int V);
int policy_smem_bytes(int V, int store_bf16);
struct VerifyWidthParams : VerifyProbParams {
    const int32_t* width;      // [B] proposals each request checks (0..gamma)
};
// width null: the fixed-width kernel; otherwise its width variant
cudaError_t launch_verify_prob(const VerifyProbParams& p, cudaStream_t stream,
                               const int32_t* width = nullptr);
cudaError_t launch_markov_step(const MarkovStepParams& p, cudaStream_t stream);

// Acceptance statistics (accept_stats.cu).
struct StatsRecord {  // one position's terms, consumed by the fixed-order finaliser
    float ce, l1, bce, acc;
    int32_t code;
    int32_t pad[3];
};
struct StatsParams {
    const void* draft;
    const void* target;
    int dtype;
    const int32_t* labels;
    const float* conf_logits;
    const uint8_t* mask;
    int N, gamma, V;
    int slice;                // elements per CTA slice, a multiple of 8
    float* l1;
    float* accept;
    StatsRecord* rec;         // [N * gamma] workspace
    double* partial;          // [stats_partials(N) * 6] workspace
    float* tau;
    double* loss_num;
    double* report;
    int64_t* num_tokens;
    int32_t* status;
};
int stats_cluster_size();
int stats_partials(int N);
cudaError_t launch_accept_stats(const StatsParams& p, cudaStream_t stream);

// Gradient of the loss numerators' total (accept_stats.cu).
struct StatsGradParams {
    const void* draft;
    const void* target;
    int dtype;
    const int32_t* labels;
    const float* conf_logits;
    const uint8_t* mask;      // or null
    int N, gamma, V;
    int slice;                // elements per CTA slice, a multiple of 8
    double scale;
    float* grad_draft;        // [N, gamma, V]
    float* grad_conf;         // [N, gamma]
};
cudaError_t launch_accept_stats_grad(const StatsGradParams& p, cudaStream_t stream);

// Sequential Temperature Scaling fit (sts.cu): per block position the state
// of its root search, kept in the caller's workspace.
struct StsState {
    double beta;          // the current iterate (the answer once phase == 2)
    double lo, hi;        // bracket of the root (hi = +inf until a slope >= 0 is seen)
    double s1, s2;        // this pass's slope and curvature sums
    unsigned int flags;   // bit 0 a counted z != 0, bit 1 a label against the sign of z, bit 2 an invalid pair
    int phase;            // 0 first pass (beta = 0), 1 searching, 2 done
    int status;           // 0 fitted, 1 no information, 2 no finite root below the cap, 3 invalid input
    int passes;           // passes whose sums the position used
};
struct StsParams {
    const float* conf_logits;  // [N, gamma]
    const float* labels;       // [N, gamma]
    const uint8_t* mask;       // [N, gamma] or null
    int64_t N;
    int gamma;
    double* beta;              // [gamma] out
    int32_t* status;           // [gamma] out
    int32_t* passes;           // [gamma] out, or null
    StsState* state;           // [DSPARK_MAX_GAMMA] workspace
    int* active;               // workspace: positions still searching
    double* partial;           // [kStsMaxGrid][DSPARK_MAX_GAMMA][2] workspace: per-CTA slope and curvature sums
    unsigned* bar;             // workspace: the grid barrier's arrival count
    int* error;                // workspace: set when a barrier wait gave up
    int max_passes;            // the pass budget
};
constexpr int kStsMaxGrid = 1024;   // CTAs of one pass over the pairs, at most
constexpr int kStsDefaultPasses = 64;
cudaError_t launch_sts_fit(const StsParams& p, cudaStream_t stream);

// One step of the RNN head's GRU (rnn.cu): s_k from s_{k-1} and U[x_{k-1}],
// written as fp32 and as the bf16 pair (hi, lo) the bias GEMM reads.
struct GruParams {
    const uint16_t* U;          // bf16 [V, r]
    const uint16_t* Wi;         // bf16 [3r, r], gate order r, z, n
    const uint16_t* Wh;         // bf16 [3r, r]
    const float* bi;            // [3r]
    const float* bh;            // [3r]
    const int32_t* anchor;      // [B]
    const int32_t* proposals;   // [B, gamma]
    int B, gamma, V, r, k;      // k: 1-based step
    const float* state_in;      // [B, r] fp32 workspace: s_{k-1} (unread at k = 1)
    float* state_out;           // [B, r] fp32 workspace: s_k (another buffer than state_in)
    uint16_t* hi;               // [B, r] bf16(s_k)
    uint16_t* lo;               // [B, r] bf16(s_k - hi)
    int32_t* index;             // [B]: b, or -1 when x_{k-1} is not a token (a failed request)
};
cudaError_t launch_gru_step(const GruParams& p, cudaStream_t stream);

// Diagnostic of the bounded grid barrier (selftest.cu): `blocks` blocks wait
// for blocks + missing arrivals, at most limit_ns each.
cudaError_t launch_wait_selftest(int blocks, int missing, uint64_t limit_ns, unsigned* bar, int* error,
                                 int32_t* status, unsigned long long* waited_ns, cudaStream_t stream);

}  // namespace dspark
