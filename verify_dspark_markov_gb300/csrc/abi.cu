// C ABI of the DSpark library: argument validation, workspace layout and
// kernel dispatch.  Everything here runs on the host; every step of the
// computation runs in the kernels it launches on the caller's stream.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "dspark.h"
#include "kernels.h"

namespace dspark {
namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool valid_common(int B, int gamma, int V, int dtype) {
    return B >= 0 && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA && V >= 8 && V <= DSPARK_MAX_VOCAB &&
           V % 8 == 0 && (dtype == DSPARK_BF16 || dtype == DSPARK_F32);
}

// Workspace carve-up.  Regions that must be zero between calls come first.
// The greedy paths keep all their state on chip and use no workspace.
struct VerifyLayout {
    size_t ticket, records, total;
};
VerifyLayout verify_layout(int B, int gamma) {
    VerifyLayout l;
    l.ticket = 0;  // sampled path: one ticket per request (zero between calls)
    l.records = align_up(static_cast<size_t>(B) * sizeof(unsigned int));
    l.total = align_up(l.records + static_cast<size_t>(B) * (gamma + 1) * sizeof(RowRecord));
    return l;
}

// Largest vocabulary the row engine holds in one cluster's shared memory.
bool policy_vocab_ok(int V) { return policy_smem_bytes(V, 0) <= 200 * 1024; }

// The one-launch draft's arguments (the Markov head; the RNN head adds its
// GRU weights) and its launch followed by the confidence kernel.
MarkovFusedArgs fused_args(const void* backbone, const uint16_t* U, const uint16_t* W, const int32_t* anchor,
                           const dspark_policy* policy, const uint64_t* seed, const uint64_t* request_id,
                           const int64_t* pos0, int B, int gamma, int V, int r, int32_t* proposals, float* q,
                           float* q_at_x, int32_t* status) {
    MarkovFusedArgs a{};
    a.backbone = static_cast<const uint16_t*>(backbone);
    a.U = U;
    a.W = W;
    a.anchor = anchor;
    a.policy = policy;
    a.seed = seed;
    a.request_id = request_id;
    a.pos0 = pos0;
    a.B = B;
    a.gamma = gamma;
    a.V = V;
    a.r = r;
    a.proposals = proposals;
    a.q = q;
    a.q_at_x = q_at_x;
    a.status = status;
    return a;
}

int fused_draft(const MarkovFusedArgs& a, const void* h, int h_dtype, const uint16_t* E, const float* w_conf, int H,
                float* conf, void* workspace, size_t workspace_bytes, cudaStream_t s) {
    if (launch_markov_fused(a, workspace, workspace_bytes, s) != cudaSuccess) return DSPARK_ECUDA;
    if (h) {
        ConfParams c{h, h_dtype, E, w_conf, H, a.B, a.gamma, a.V, a.anchor, a.proposals, 1, a.gamma, conf};
        if (launch_confidence(c, s) != cudaSuccess) return DSPARK_ECUDA;
    }
    return DSPARK_OK;
}

struct MarkovLayout {
    size_t error_flag, zbuf, total;
};
// The word that must be zero between calls sits at a fixed offset, so the z
// buffer of one call never overlaps it in a later call of other sizes.
MarkovLayout markov_layout(int B, int gamma, int V, int r) {
    MarkovLayout l;
    (void)gamma;
    l.error_flag = 0;  // zero between calls; set only after a device wait gave up
    l.zbuf = align_up(sizeof(int));
    // two z buffers: step k + 1's bias kernel writes one while step k's
    // policy kernel still reads the other
    const size_t zbytes = r > 0 ? 2 * static_cast<size_t>(B) * V * sizeof(float) : 0;
    l.total = align_up(l.zbuf + zbytes);
    return l;
}

// RNN head: the error flag and two z buffers as for the Markov head (z after
// the hi product, z after the lo product), then the fp32 state, its bf16 hi
// and lo rows and the gather index.
struct RnnLayout {
    size_t error_flag, zbuf, state, hi, lo, index, total;  // state: two [B, r] buffers (steps alternate)
};
RnnLayout rnn_layout(int B, int V, int r) {
    RnnLayout l;
    l.error_flag = 0;
    l.zbuf = align_up(sizeof(int));
    l.state = align_up(l.zbuf + 2 * static_cast<size_t>(B) * V * sizeof(float));
    l.hi = align_up(l.state + 2 * static_cast<size_t>(B) * r * sizeof(float));
    l.lo = align_up(l.hi + static_cast<size_t>(B) * r * sizeof(uint16_t));
    l.index = align_up(l.lo + static_cast<size_t>(B) * r * sizeof(uint16_t));
    l.total = align_up(l.index + static_cast<size_t>(B) * sizeof(int32_t));
    return l;
}

// Statistics: per-position records, then the per-CTA partial sums.
size_t stats_partials_offset(int N, int gamma) {
    return align_up(static_cast<size_t>(N) * gamma * sizeof(StatsRecord));
}
size_t stats_workspace(int N, int gamma) {
    return align_up(stats_partials_offset(N, gamma) + static_cast<size_t>(stats_partials(N)) * 6 * sizeof(double));
}

// Sequential Temperature Scaling: the per-position search states, the count
// of positions still searching, then the per-CTA sums of a pass.
size_t sts_active_offset() { return align_up(static_cast<size_t>(DSPARK_MAX_GAMMA) * sizeof(StsState)); }
// the active count, the barrier count and the error word share one aligned block
size_t sts_partial_offset() { return align_up(sts_active_offset() + 3 * sizeof(int)); }
size_t sts_workspace() {
    return align_up(sts_partial_offset() + static_cast<size_t>(kStsMaxGrid) * DSPARK_MAX_GAMMA * 2 * sizeof(double));
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

}  // namespace
}  // namespace dspark

using namespace dspark;

extern "C" {

int dspark_version(void) { return 100; }

const char* dspark_status_string(int code) {
    switch (code) {
        case DSPARK_OK: return "ok";
        case DSPARK_EINVAL: return "invalid argument";
        case DSPARK_ENOSPC: return "workspace too small";
        case DSPARK_ECUDA: return "CUDA launch failed";
        case DSPARK_ENOTSUP: return "not supported";
        case DSPARK_REQ_NONFINITE: return "request: non-finite logit";
        case DSPARK_REQ_EMPTY: return "request: all logits -inf";
        case DSPARK_REQ_TIMEOUT: return "request: device wait timed out";
        case DSPARK_REQ_BAD_POLICY: return "request: invalid sampling policy";
        case DSPARK_REQ_BAD_TOKEN: return "request: token id outside [0, V)";
        default: return "unknown status";
    }
}

size_t dspark_workspace_size(int op, int B, int gamma, int V, int r, int H) {
    if (op == DSPARK_OP_STS_FIT) return B >= 0 && gamma >= 1 && gamma <= DSPARK_MAX_GAMMA ? sts_workspace() : 0;
    if (!valid_common(B, gamma, V, DSPARK_BF16) || r < 0 || H < 0) return 0;
    switch (op) {
        case DSPARK_OP_MARKOV_SAMPLE:
            // the larger of the two paths' needs (which one runs depends on the device)
            return std::max(markov_layout(B, gamma, V, r).total,
                            r >= 64 && r % 64 == 0 && B <= kFusedMaxBatch ? markov_fused_workspace(B, gamma, V)
                                                                           : size_t(0));
        case DSPARK_OP_VERIFY: return verify_layout(B, gamma).total;
        case DSPARK_OP_ACCEPT_STATS: return stats_workspace(B, gamma);
        case DSPARK_OP_RNN_SAMPLE:
            // the larger of the two paths' needs (which one runs depends on the device)
            return r >= 16 ? std::max(rnn_layout(B, V, r).total,
                                      r >= 64 && r % 64 == 0 && B <= kFusedMaxBatch
                                          ? markov_fused_workspace(B, gamma, V, r, true)
                                          : size_t(0))
                           : 0;
        default: return 0;
    }
}

int dspark_verify_width(const void* target, int dtype, const int32_t* proposals, const float* q,
                        const float* q_at_x, const dspark_policy* policy, const uint64_t* seed,
                        const uint64_t* request_id, const int64_t* pos0, const int32_t* width, int B,
                        int gamma, int V, int32_t* out_tokens, int32_t* num_accepted, int32_t* status,
                        void* workspace, size_t workspace_bytes, void* stream) {
    if (!valid_common(B, gamma, V, dtype)) return DSPARK_EINVAL;
    if (B == 0) return DSPARK_OK;
    if (!target || !proposals || !out_tokens || !num_accepted || !status) return DSPARK_EINVAL;
    if (!aligned16(target)) return DSPARK_EINVAL;
    if (policy && (!q || !q_at_x || !seed || !request_id || !pos0 || !aligned16(q)))
        return DSPARK_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (policy) {  // per-request policies: the row engine
        const VerifyLayout lay = verify_layout(B, gamma);
        if (workspace_bytes < lay.total || !workspace) return DSPARK_ENOSPC;
        if (!policy_vocab_ok(V)) return DSPARK_ENOTSUP;
        VerifyProbParams vp{};
        vp.target = target;
        vp.dtype = dtype;
        vp.proposals = proposals;
        vp.q = q;
        vp.q_at_x = q_at_x;
        vp.policy = policy;
        vp.seed = seed;
        vp.request_id = request_id;
        vp.pos0 = pos0;
        vp.B = B;
        vp.gamma = gamma;
        vp.V = V;
        vp.slice = verify_slice(V);
        vp.out_tokens = out_tokens;
        vp.num_accepted = num_accepted;
        vp.status = status;
        vp.records = at<RowRecord>(workspace, lay.records);
        vp.ticket = at<unsigned int>(workspace, lay.ticket);
        return launch_verify_prob(vp, s, width) == cudaSuccess ? DSPARK_OK : DSPARK_ECUDA;
    }

    ArgmaxParams p{};
    p.logits = target;
    p.dtype = dtype;
    p.V = V;
    p.rows_per_group = gamma + 1;
    p.gamma = gamma;
    p.mode = kArgmaxVerify;
    p.proposals = proposals;
    p.out_tokens = out_tokens;
    p.num_accepted = num_accepted;
    p.status = status;
    return launch_argmax_rows(p, B, s, width) == cudaSuccess ? DSPARK_OK : DSPARK_ECUDA;
}

int dspark_verify(const void* target, int dtype, const int32_t* proposals, const float* q,
                  const float* q_at_x, const dspark_policy* policy, const uint64_t* seed,
                  const uint64_t* request_id, const int64_t* pos0, int B, int gamma, int V,
                  int32_t* out_tokens, int32_t* num_accepted, int32_t* status, void* workspace,
                  size_t workspace_bytes, void* stream) {
    return dspark_verify_width(target, dtype, proposals, q, q_at_x, policy, seed, request_id, pos0, nullptr, B,
                               gamma, V, out_tokens, num_accepted, status, workspace, workspace_bytes, stream);
}

int dspark_markov_sample(const void* backbone, int dtype, const int32_t* anchor, const uint16_t* U,
                         const uint16_t* W, int r, const void* h, int h_dtype, const uint16_t* E,
                         const float* w_conf, int H, const dspark_policy* policy,
                         const uint64_t* seed, const uint64_t* request_id, const int64_t* pos0,
                         int B, int gamma, int V, int32_t* proposals, float* q, float* q_at_x,
                         float* conf, int32_t* status, void* workspace, size_t workspace_bytes,
                         void* stream) {
    if (!valid_common(B, gamma, V, dtype)) return DSPARK_EINVAL;
    if (B > DSPARK_MAX_BATCH) return DSPARK_EINVAL;
    if (r < 0 || r > DSPARK_MAX_RANK || r % 16 != 0) return DSPARK_EINVAL;
    if (B == 0) return DSPARK_OK;
    if (!backbone || !anchor || !proposals || !q_at_x || !status) return DSPARK_EINVAL;
    if (!aligned16(backbone)) return DSPARK_EINVAL;
    if (r > 0 && (!U || !W || !aligned16(U) || !aligned16(W))) return DSPARK_EINVAL;
    if (h && (H <= 0 || !E || !w_conf || !conf || (h_dtype != DSPARK_BF16 && h_dtype != DSPARK_F32)))
        return DSPARK_EINVAL;
    if (policy && (!q || !seed || !request_id || !pos0 || !aligned16(q))) return DSPARK_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (r > 0 && r % 64 == 0 && markov_fused_supported(dtype, B, V, r)) {
        // the whole draft in one persistent launch, z kept in tensor memory
        if (!workspace || workspace_bytes < markov_fused_workspace(B, gamma, V)) return DSPARK_ENOSPC;
        const MarkovFusedArgs a = fused_args(backbone, U, W, anchor, policy, seed, request_id, pos0, B, gamma, V, r,
                                             proposals, q, q_at_x, status);
        return fused_draft(a, h, h_dtype, E, w_conf, H, conf, workspace, workspace_bytes, s);
    }

    if (policy || r > 0) {  // the row engine, one launch per step (after the bias GEMM when r > 0)
        const MarkovLayout lay = markov_layout(B, gamma, V, r);
        if (workspace_bytes < lay.total || !workspace) return DSPARK_ENOSPC;
        if (!policy_vocab_ok(V)) return DSPARK_ENOTSUP;
        int* error_flag = at<int>(workspace, lay.error_flag);
        float* zbuf = r > 0 ? at<float>(workspace, lay.zbuf) : nullptr;
        MarkovGemmParams gp{};
        MarkovGemmPlan plan{};
        if (r > 0) {
            gp.backbone = backbone;
            gp.dtype = dtype;
            gp.U = U;
            gp.W = W;
            gp.anchor = anchor;
            gp.proposals = proposals;
            gp.B = B;
            gp.gamma = gamma;
            gp.V = V;
            gp.r = r;
            gp.zbuf = zbuf;
            gp.error_flag = error_flag;
            if (!prepare_markov_bias(gp, plan)) return DSPARK_ENOTSUP;
        }
        MarkovStepParams mp{};
        mp.backbone = backbone;
        mp.dtype = dtype;
        mp.zbuf = zbuf;
        mp.anchor = anchor;
        mp.proposals = proposals;
        mp.q = q;
        mp.q_at_x = q_at_x;
        mp.status = status;
        mp.policy = policy;
        mp.seed = seed;
        mp.request_id = request_id;
        mp.pos0 = pos0;
        mp.B = B;
        mp.gamma = gamma;
        mp.V = V;
        mp.slice = step_slice(V);
        mp.error_flag = r > 0 ? error_flag : nullptr;
        for (int k = 1; k <= gamma; ++k) {
            if (r > 0) {
                float* zk = zbuf + static_cast<size_t>(k & 1) * B * V;
                gp.k = k;
                gp.zbuf = zk;
                mp.zbuf = zk;
                if (launch_markov_bias(gp, plan, k > 1, s) != cudaSuccess) return DSPARK_ECUDA;
            }
            mp.k = k;
            if (launch_markov_step(mp, s) != cudaSuccess) return DSPARK_ECUDA;
        }
        if (h) {
            ConfParams c{h, h_dtype, E, w_conf, H, B, gamma, V, anchor, proposals, 1, gamma, conf};
            if (launch_confidence(c, s) != cudaSuccess) return DSPARK_ECUDA;
        }
        return DSPARK_OK;
    }

    // Greedy drafting without a Markov bias: x_k = argmax of backbone row k.
    ArgmaxParams p{};
    p.logits = backbone;
    p.dtype = dtype;
    p.V = V;
    p.rows_per_group = gamma;
    p.gamma = gamma;
    p.mode = kArgmaxDraft;
    p.anchor = anchor;
    p.props_out = proposals;
    p.q_at_x = q_at_x;
    p.status = status;
    if (launch_argmax_rows(p, B, s) != cudaSuccess) return DSPARK_ECUDA;
    if (h) {
        ConfParams c{h, h_dtype, E, w_conf, H, B, gamma, V, anchor, proposals, 1, gamma, conf};
        if (launch_confidence(c, s) != cudaSuccess) return DSPARK_ECUDA;
    }
    return DSPARK_OK;
}

int dspark_rnn_launches(int dtype, int B, int gamma, int V, int r, int with_conf) {
    if (!valid_common(B, gamma, V, dtype) || B > DSPARK_MAX_BATCH || B > V) return -1;
    if (r < 16 || r > DSPARK_MAX_RANK || r % 16 != 0) return -1;
    if (B == 0) return 0;
    const int conf = with_conf ? 1 : 0;
    if (r % 64 == 0 && markov_fused_supported(dtype, B, V, r, true)) return 1 + conf;
    return 4 * gamma + conf;  // per step: the GRU cell, the hi and lo products, the policy step
}

int dspark_wait_selftest(int blocks, int missing, int limit_us, int32_t* status, uint64_t* waited_ns,
                         void* workspace, void* stream) {
    if (blocks < 1 || blocks > 64 || missing < 0 || missing > 64 || limit_us < 1 || limit_us > 2000000)
        return DSPARK_EINVAL;
    if (!status || !waited_ns || !workspace || !aligned16(workspace) ||
        (reinterpret_cast<uintptr_t>(status) & 3u) || (reinterpret_cast<uintptr_t>(waited_ns) & 7u))
        return DSPARK_EINVAL;
    unsigned* bar = static_cast<unsigned*>(workspace);
    int* error = reinterpret_cast<int*>(static_cast<char*>(workspace) + 8);
    return launch_wait_selftest(blocks, missing, static_cast<uint64_t>(limit_us) * 1000u, bar, error, status,
                                reinterpret_cast<unsigned long long*>(waited_ns),
                                static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DSPARK_OK
               : DSPARK_ECUDA;
}

int dspark_markov_launches(int dtype, int B, int gamma, int V, int r, int with_policy, int with_conf) {
    if (!valid_common(B, gamma, V, dtype) || B > DSPARK_MAX_BATCH) return -1;
    if (r < 0 || r > DSPARK_MAX_RANK || r % 16 != 0) return -1;
    if (B == 0) return 0;
    const int conf = with_conf ? 1 : 0;
    if (r > 0 && r % 64 == 0 && markov_fused_supported(dtype, B, V, r)) return 1 + conf;
    if (with_policy || r > 0) return gamma * (r > 0 ? 2 : 1) + conf;
    return 1 + conf;
}

int dspark_rnn_sample(const void* backbone, int dtype, const int32_t* anchor, const uint16_t* U,
                      const uint16_t* W, int r, const uint16_t* Wi, const uint16_t* Wh, const float* bi,
                      const float* bh, const void* h, int h_dtype, const uint16_t* E, const float* w_conf,
                      int H, const dspark_policy* policy, const uint64_t* seed, const uint64_t* request_id,
                      const int64_t* pos0, int B, int gamma, int V, int32_t* proposals, float* q,
                      float* q_at_x, float* conf, int32_t* status, void* workspace, size_t workspace_bytes,
                      void* stream) {
    if (!valid_common(B, gamma, V, dtype)) return DSPARK_EINVAL;
    if (B > DSPARK_MAX_BATCH || B > V) return DSPARK_EINVAL;
    if (r < 16 || r > DSPARK_MAX_RANK || r % 16 != 0) return DSPARK_EINVAL;
    if (B == 0) return DSPARK_OK;
    if (!backbone || !anchor || !proposals || !q_at_x || !status) return DSPARK_EINVAL;
    if (!U || !W || !Wi || !Wh || !bi || !bh) return DSPARK_EINVAL;
    if (!aligned16(backbone) || !aligned16(U) || !aligned16(W) || !aligned16(Wi) || !aligned16(Wh))
        return DSPARK_EINVAL;
    if (h && (H <= 0 || !E || !w_conf || !conf || (h_dtype != DSPARK_BF16 && h_dtype != DSPARK_F32)))
        return DSPARK_EINVAL;
    if (policy && (!q || !seed || !request_id || !pos0 || !aligned16(q))) return DSPARK_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    if (r % 64 == 0 && markov_fused_supported(dtype, B, V, r, true)) {
        // the whole draft in one persistent launch: the GRU cell, the bias
        // and the policy of every step, z kept in tensor memory
        if (!workspace || workspace_bytes < markov_fused_workspace(B, gamma, V, r, true)) return DSPARK_ENOSPC;
        MarkovFusedArgs a = fused_args(backbone, U, W, anchor, policy, seed, request_id, pos0, B, gamma, V, r,
                                       proposals, q, q_at_x, status);
        a.Wi = Wi;
        a.Wh = Wh;
        a.bi = bi;
        a.bh = bh;
        return fused_draft(a, h, h_dtype, E, w_conf, H, conf, workspace, workspace_bytes, s);
    }

    const RnnLayout lay = rnn_layout(B, V, r);
    if (workspace_bytes < lay.total || !workspace) return DSPARK_ENOSPC;
    if (!policy_vocab_ok(V)) return DSPARK_ENOTSUP;
    int* error_flag = at<int>(workspace, lay.error_flag);
    float* zA = at<float>(workspace, lay.zbuf);
    float* zB = zA + static_cast<size_t>(B) * V;

    GruParams gru{};
    gru.U = U;
    gru.Wi = Wi;
    gru.Wh = Wh;
    gru.bi = bi;
    gru.bh = bh;
    gru.anchor = anchor;
    gru.proposals = proposals;
    gru.B = B;
    gru.gamma = gamma;
    gru.V = V;
    gru.r = r;
    float* state0 = at<float>(workspace, lay.state);
    float* state1 = state0 + static_cast<size_t>(B) * r;
    gru.hi = at<uint16_t>(workspace, lay.hi);
    gru.lo = at<uint16_t>(workspace, lay.lo);
    gru.index = at<int32_t>(workspace, lay.index);

    // the bias in two products on the tensor cores: zA = backbone_k + hi W^T,
    // then zB = zA + lo W^T; the gather reads row index[b] (= b) of hi / lo
    MarkovGemmParams g1{}, g2{};
    MarkovGemmPlan plan1{}, plan2{};
    g1.backbone = backbone;
    g1.dtype = dtype;
    g1.U = gru.hi;
    g1.W = W;
    g1.anchor = gru.index;
    g1.proposals = proposals;
    g1.B = B;
    g1.gamma = gamma;
    g1.V = V;
    g1.r = r;
    g1.k = 1;
    g1.zbuf = zA;
    g1.error_flag = error_flag;
    g2 = g1;
    g2.backbone = zA;
    g2.dtype = DSPARK_F32;
    g2.U = gru.lo;
    g2.gamma = 1;
    g2.zbuf = zB;
    if (!prepare_markov_bias(g1, plan1) || !prepare_markov_bias(g2, plan2)) return DSPARK_ENOTSUP;

    MarkovStepParams mp{};
    mp.backbone = backbone;
    mp.dtype = dtype;
    mp.zbuf = zB;
    mp.anchor = anchor;
    mp.proposals = proposals;
    mp.q = q;
    mp.q_at_x = q_at_x;
    mp.status = status;
    mp.policy = policy;
    mp.seed = seed;
    mp.request_id = request_id;
    mp.pos0 = pos0;
    mp.B = B;
    mp.gamma = gamma;
    mp.V = V;
    mp.slice = step_slice(V);
    mp.error_flag = error_flag;
    const size_t esz = dtype == DSPARK_BF16 ? 2 : 4;
    for (int k = 1; k <= gamma; ++k) {
        gru.k = k;
        gru.state_in = (k & 1) ? state1 : state0;   // s_{k-1}
        gru.state_out = (k & 1) ? state0 : state1;  // s_k
        if (launch_gru_step(gru, s) != cudaSuccess) return DSPARK_ECUDA;
        // step k's backbone rows, read as the first rows of a [B, gamma, V] array
        g1.backbone = static_cast<const char*>(backbone) + static_cast<size_t>(k - 1) * V * esz;
        if (launch_markov_bias(g1, plan1, false, s) != cudaSuccess) return DSPARK_ECUDA;
        if (launch_markov_bias(g2, plan2, false, s) != cudaSuccess) return DSPARK_ECUDA;
        mp.k = k;
        if (launch_markov_step(mp, s) != cudaSuccess) return DSPARK_ECUDA;
    }
    if (h) {
        ConfParams c{h, h_dtype, E, w_conf, H, B, gamma, V, anchor, proposals, 1, gamma, conf};
        if (launch_confidence(c, s) != cudaSuccess) return DSPARK_ECUDA;
    }
    return DSPARK_OK;
}

int dspark_accept_stats(const void* draft, const void* target, int dtype, const int32_t* labels,
                        const float* conf_logits, const uint8_t* mask, int N, int gamma, int V,
                        float* l1, float* accept, float* tau, double* loss_num, double* report,
                        int64_t* num_tokens, int32_t* status, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (!valid_common(N, gamma, V, dtype)) return DSPARK_EINVAL;
    if (static_cast<int64_t>(N) * gamma * stats_cluster_size() > 0x7FFFFFFFll) return DSPARK_EINVAL;
    if (!loss_num || !report || !num_tokens) return DSPARK_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (N == 0) {  // empty batch: the numerators and the count are zero
        if (cudaMemsetAsync(loss_num, 0, 4 * sizeof(double), s) != cudaSuccess ||
            cudaMemsetAsync(report, 0, 2 * sizeof(double), s) != cudaSuccess ||
            cudaMemsetAsync(num_tokens, 0, sizeof(int64_t), s) != cudaSuccess)
            return DSPARK_ECUDA;
        return DSPARK_OK;
    }
    if (!draft || !target || !labels || !conf_logits || !l1 || !accept || !tau) return DSPARK_EINVAL;
    if (!aligned16(draft) || !aligned16(target)) return DSPARK_EINVAL;
    const size_t need = stats_workspace(N, gamma);
    if (workspace_bytes < need || !workspace) return DSPARK_ENOSPC;
    StatsParams p{};
    p.draft = draft;
    p.target = target;
    p.dtype = dtype;
    p.labels = labels;
    p.conf_logits = conf_logits;
    p.mask = mask;
    p.N = N;
    p.gamma = gamma;
    p.V = V;
    const int C = stats_cluster_size();
    p.slice = ((V + C - 1) / C + 7) / 8 * 8;
    p.l1 = l1;
    p.accept = accept;
    p.rec = at<StatsRecord>(workspace, 0);
    p.partial = at<double>(workspace, stats_partials_offset(N, gamma));
    p.tau = tau;
    p.loss_num = loss_num;
    p.report = report;
    p.num_tokens = num_tokens;
    p.status = status;
    return launch_accept_stats(p, s) == cudaSuccess ? DSPARK_OK : DSPARK_ECUDA;
}

int dspark_accept_stats_grad(const void* draft, const void* target, int dtype, const int32_t* labels,
                             const float* conf_logits, const uint8_t* mask, int N, int gamma, int V,
                             double scale, float* grad_draft, float* grad_conf, void* stream) {
    if (!valid_common(N, gamma, V, dtype)) return DSPARK_EINVAL;
    if (static_cast<int64_t>(N) * gamma * stats_cluster_size() > 0x7FFFFFFFll) return DSPARK_EINVAL;
    if (N == 0) return DSPARK_OK;
    if (!draft || !target || !labels || !conf_logits || !grad_draft || !grad_conf) return DSPARK_EINVAL;
    if (!aligned16(draft) || !aligned16(target) || !aligned16(grad_draft)) return DSPARK_EINVAL;
    if (!(scale == scale)) return DSPARK_EINVAL;
    StatsGradParams p{};
    p.draft = draft;
    p.target = target;
    p.dtype = dtype;
    p.labels = labels;
    p.conf_logits = conf_logits;
    p.mask = mask;
    p.N = N;
    p.gamma = gamma;
    p.V = V;
    const int C = stats_cluster_size();
    p.slice = ((V + C - 1) / C + 7) / 8 * 8;
    p.scale = scale;
    p.grad_draft = grad_draft;
    p.grad_conf = grad_conf;
    return launch_accept_stats_grad(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DSPARK_OK
                                                                                           : DSPARK_ECUDA;
}


int dspark_sts_fit(const float* conf_logits, const float* labels, const uint8_t* mask, int N, int gamma,
                   double* beta, int32_t* status, int32_t* passes, int max_passes, void* workspace,
                   size_t workspace_bytes, void* stream) {
    if (N < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA) return DSPARK_EINVAL;
    if (max_passes < 0 || max_passes > DSPARK_STS_MAX_PASSES) return DSPARK_EINVAL;
    if (!beta || !status) return DSPARK_EINVAL;
    if (N > 0 && (!conf_logits || !labels)) return DSPARK_EINVAL;
    if ((reinterpret_cast<uintptr_t>(conf_logits) & 3u) || (reinterpret_cast<uintptr_t>(labels) & 3u) ||
        (reinterpret_cast<uintptr_t>(beta) & 7u) || (reinterpret_cast<uintptr_t>(status) & 3u) ||
        (reinterpret_cast<uintptr_t>(passes) & 3u))
        return DSPARK_EINVAL;
    if (!workspace || workspace_bytes < sts_workspace()) return DSPARK_ENOSPC;
    StsParams p{};
    p.conf_logits = conf_logits;
    p.labels = labels;
    p.mask = mask;
    p.N = N;
    p.gamma = gamma;
    p.beta = beta;
    p.status = status;
    p.passes = passes;
    p.state = at<StsState>(workspace, 0);
    p.active = at<int>(workspace, sts_active_offset());
    p.bar = at<unsigned>(workspace, sts_active_offset() + sizeof(int));
    p.error = at<int>(workspace, sts_active_offset() + 2 * sizeof(int));
    p.partial = at<double>(workspace, sts_partial_offset());
    p.max_passes = max_passes ? max_passes : kStsDefaultPasses;
    return launch_sts_fit(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DSPARK_OK : DSPARK_ECUDA;
}

}  // extern "C"
