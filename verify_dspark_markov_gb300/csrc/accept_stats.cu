// Analytical acceptance statistics [MB Training objective; Acceptance and
// confidence; Loss return contract].  Per position (n, k):
//   p_d = softmax(draft row), p_t = softmax(target row)   (T = 1, full vocab)
//   L1  = ||p_d - p_t||_1,  accept = clamp(1 - L1/2, 0, 1)
//   CE  = -log p_d[label],  BCE = softplus(z) - accept * z   (z: confidence logit)
// and per block n: tau = 1 + sum_k prod_{j<=k} accept_j; over the batch the
// exp(-k/gamma)-weighted numerators and the token count, never ratios.
//
// Kernel 1 (one cluster of kC CTAs per row pair): each CTA streams a 1/kC
// slice of both rows once from HBM, keeping an online (max, sum of exp) per
// thread; the cluster combines the slices' statistics through distributed
// shared memory; each CTA then re-reads its slice (a ~129 KB working set per
// CTA, so the re-read is served by L2) to form the L1 terms.  The first
// read marks its L2 lines evict_last and the last read evict_first, so that
// the slices of the CTAs in flight (4 per SM) stay in L2 for their re-reads
// while the stream passes through.  NaN / +inf poison the running sums,
// which is how non-finite rows are detected at no cost.
// Kernels 2 and 3: tau and the status per block (one thread each) with the
// weighted sums reduced by fixed binary trees, then the CTA partials in a
// fixed order, so repeated calls give identical bits.
// Kernel 4 (one cluster per row pair, the backward [MB Training objective;
// Memory contract for the full-vocabulary terms: the softmax statistics are
// recomputed, nothing full-vocabulary is kept]): the gradient of the loss
// numerators' total J = sum m w_k (0.1 CE + 0.9 L1 + 1.0 BCE), the target the
// frozen teacher and the BCE label accept held fixed, times a scale:
//   dJ/dd_v = m w_k (0.1 (p_d,v - [v = label]) + 0.9 p_d,v (s_v - S)),
//   s_v = sign(p_d,v - p_t,v), S = sum_v s_v p_d,v,
//   dJ/dz   = m w_k (sigmoid(z) - accept).
// Pass 1 as in kernel 1; pass 2 sums the L1 terms and S; pass 3 re-reads the
// slice (L2, its last read: evict_first) and writes its gradient row with
// streaming stores (kept out of the way of the slices still to be re-read).

#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace dspark {

namespace {

constexpr int kC = 8;          // CTAs per row pair (cluster size)
constexpr int kThreads = 256;
constexpr int kBatch = 5;      // 16-byte vectors per row per thread in flight (64 registers, no spills)
constexpr int kBatchGrad = 4;  // the same in the backward (more would spill at 4 CTAs per SM)
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Online softmax statistics: m = running max (starts at -FLT_MAX so that -inf
// logits contribute exp(-inf) = 0), s = sum of exp(x - m).
struct Online {
    float m, s;
    __device__ __forceinline__ void init() { m = -3.402823466e38f; s = 0.0f; }
    template <int kN>
    __device__ __forceinline__ void add(const float (&x)[kN]) {
        float mx = x[0];
#pragma unroll
        for (int i = 1; i < kN; ++i) mx = fmaxf(mx, x[i]);
        if (mx > m) {
            s *= ex2((m - mx) * kLog2e);
            m = mx;
        }
#pragma unroll
        for (int i = 0; i < kN; ++i) s += ex2((x[i] - m) * kLog2e);
    }
    __device__ __forceinline__ void merge(float m2, float s2) {
        const float mn = fmaxf(m, m2);
        s = s * ex2((m - mn) * kLog2e) + s2 * ex2((m2 - mn) * kLog2e);
        m = mn;
    }
};

template <int kDtype>
__device__ __forceinline__ void unpack(const uint4& v, float (&x)[kDtype == kBF16 ? 8 : 4]) {
    if constexpr (kDtype == kBF16) {
        x[0] = bf16_lo(v.x); x[1] = bf16_hi(v.x); x[2] = bf16_lo(v.y); x[3] = bf16_hi(v.y);
        x[4] = bf16_lo(v.z); x[5] = bf16_hi(v.z); x[6] = bf16_lo(v.w); x[7] = bf16_hi(v.w);
    } else {
        x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
    }
}

template <int kDtype>
__global__ void __cluster_dims__(kC, 1, 1) __launch_bounds__(kThreads, 4)
    stats_pairs_kernel(const StatsParams p) {
    constexpr int kPer = kDtype == kBF16 ? 8 : 4;
    constexpr int64_t kEsize = kDtype == kBF16 ? 2 : 4;
    __shared__ float s_warp[4][kThreads / 32];
    __shared__ float s_stats[4];   // this CTA's (md, sd, mt, st)
    __shared__ double s_l1;        // this CTA's L1 partial

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t pair = blockIdx.x / kC;
    const int64_t lo = static_cast<int64_t>(rank) * p.slice;
    const int64_t hi = min(lo + p.slice, static_cast<int64_t>(p.V));
    const int nvec = hi > lo ? static_cast<int>((hi - lo) / kPer) : 0;
    const char* drow = static_cast<const char*>(p.draft) + (pair * p.V + lo) * kEsize;
    const char* trow = static_cast<const char*>(p.target) + (pair * p.V + lo) * kEsize;

    // ---- pass 1: online max / sum of exp over the slice, both rows
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    Online od, ot;
    od.init();
    ot.init();
    for (int j0 = tid; j0 < nvec; j0 += kBatch * kThreads) {
        uint4 vd[kBatch], vt[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + u * kThreads;
            if (j < nvec) {
                vd[u] = ld_stream_v4(drow + static_cast<int64_t>(j) * 16, keep);
                vt[u] = ld_stream_v4(trow + static_cast<int64_t>(j) * 16, keep);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (j0 + u * kThreads < nvec) {
                float x[kPer];
                unpack<kDtype>(vd[u], x);
                od.add(x);
                unpack<kDtype>(vt[u], x);
                ot.add(x);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        od.merge(__shfl_xor_sync(0xFFFFFFFFu, od.m, o), __shfl_xor_sync(0xFFFFFFFFu, od.s, o));
        ot.merge(__shfl_xor_sync(0xFFFFFFFFu, ot.m, o), __shfl_xor_sync(0xFFFFFFFFu, ot.s, o));
    }
    if (lane == 0) {
        s_warp[0][warp] = od.m; s_warp[1][warp] = od.s;
        s_warp[2][warp] = ot.m; s_warp[3][warp] = ot.s;
    }
    __syncthreads();
    if (tid == 0) {
        Online a, b;
        a.init();
        b.init();
        for (int w = 0; w < kThreads / 32; ++w) {
            a.merge(s_warp[0][w], s_warp[1][w]);
            b.merge(s_warp[2][w], s_warp[3][w]);
        }
        s_stats[0] = a.m; s_stats[1] = a.s; s_stats[2] = b.m; s_stats[3] = b.s;
    }
    cluster.sync();
    // every CTA combines the kC slices in rank order: identical results
    Online gd, gt;
    gd.init();
    gt.init();
    for (int r = 0; r < kC; ++r) {
        const float* st = cluster.map_shared_rank(s_stats, r);
        gd.merge(st[0], st[1]);
        gt.merge(st[2], st[3]);
    }
    const float inv_sd = 1.0f / gd.s, inv_st = 1.0f / gt.s;

    // ---- pass 2: sum of |p_d - p_t| over the slice (re-read, served by L2; its last read)
    float l1 = 0.0f;
    for (int j0 = tid; j0 < nvec; j0 += kBatch * kThreads) {
        uint4 vd[kBatch], vt[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + u * kThreads;
            if (j < nvec) {
                vd[u] = ld_stream_v4(drow + static_cast<int64_t>(j) * 16, drop);
                vt[u] = ld_stream_v4(trow + static_cast<int64_t>(j) * 16, drop);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (j0 + u * kThreads < nvec) {
                float xd[kPer], xt[kPer];
                unpack<kDtype>(vd[u], xd);
                unpack<kDtype>(vt[u], xt);
#pragma unroll
                for (int i = 0; i < kPer; ++i)
                    l1 += fabsf(ex2((xd[i] - gd.m) * kLog2e) * inv_sd - ex2((xt[i] - gt.m) * kLog2e) * inv_st);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
    if (lane == 0) s_warp[0][warp] = l1;
    __syncthreads();
    if (tid == 0) {
        double a = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) a += s_warp[0][w];
        s_l1 = a;
    }
    cluster.sync();
    if (rank == 0 && tid == 0) {
        double dist = 0.0;
        for (int r = 0; r < kC; ++r) dist += *cluster.map_shared_rank(&s_l1, r);
        const float L1 = static_cast<float>(dist);
        const float acc = fminf(1.0f, fmaxf(0.0f, 1.0f - 0.5f * L1));
        int32_t code = (gd.s != gd.s || gt.s != gt.s) ? kReqNonfinite : kReqOk;
        const int32_t y = p.labels[pair];
        float ce;
        if (y < 0 || y >= p.V) {
            code = kReqBadToken;
            ce = __int_as_float(0x7FC00000);
        } else {
            float dy;
            if (kDtype == kBF16)
                dy = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p.draft)[pair * p.V + y]) << 16);
            else
                dy = static_cast<const float*>(p.draft)[pair * p.V + y];
            ce = gd.m + logf(gd.s) - dy;
        }
        const float zc = p.conf_logits[pair];
        const float bce = fmaxf(zc, 0.0f) - acc * zc + log1pf(expf(-fabsf(zc)));
        p.l1[pair] = L1;
        p.accept[pair] = acc;
        StatsRecord rec;
        rec.ce = ce;
        rec.l1 = L1;
        rec.bce = bce;
        rec.acc = acc;
        rec.code = code;
        p.rec[pair] = rec;
    }
    cluster.sync();  // no CTA leaves while rank 0 reads its shared memory
}

// Kernel 4: see the file comment.  Masked positions write zeros; a position
// with a NaN / +inf logit or a label outside [0, V) writes NaN.
template <int kDtype>
__global__ void __cluster_dims__(kC, 1, 1) __launch_bounds__(kThreads, 4)
    stats_grad_kernel(const StatsGradParams p) {
    constexpr int kPer = kDtype == kBF16 ? 8 : 4;
    constexpr int64_t kEsize = kDtype == kBF16 ? 2 : 4;
    __shared__ float s_warp[4][kThreads / 32];
    __shared__ float s_stats[4];   // this CTA's (md, sd, mt, st)
    __shared__ double s_sums[2];   // this CTA's (L1, S) partials

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t pair = blockIdx.x / kC;
    const int k = static_cast<int>(pair % p.gamma) + 1;  // 1-based position in the block
    const int64_t lo = static_cast<int64_t>(rank) * p.slice;
    const int64_t hi = min(lo + p.slice, static_cast<int64_t>(p.V));
    const int nvec = hi > lo ? static_cast<int>((hi - lo) / kPer) : 0;
    const char* drow = static_cast<const char*>(p.draft) + (pair * p.V + lo) * kEsize;
    const char* trow = static_cast<const char*>(p.target) + (pair * p.V + lo) * kEsize;
    float* grow = p.grad_draft + pair * p.V + lo;  // kPer floats per vector, 16-byte aligned

    if (p.mask && p.mask[pair] == 0) {  // the same branch in every CTA of the cluster
        const float4 z4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int j = tid; j < nvec; j += kThreads) {
            float4* g4 = reinterpret_cast<float4*>(grow + static_cast<int64_t>(j) * kPer);
            g4[0] = z4;
            if (kPer == 8) g4[1] = z4;
        }
        if (rank == 0 && tid == 0) p.grad_conf[pair] = 0.0f;
        return;
    }

    // ---- pass 1: online max / sum of exp over the slice, both rows
    const uint64_t keep = l2_policy_evict_last(), drop = l2_policy_evict_first();
    Online od, ot;
    od.init();
    ot.init();
    for (int j0 = tid; j0 < nvec; j0 += kBatchGrad * kThreads) {
        uint4 vd[kBatchGrad], vt[kBatchGrad];
#pragma unroll
        for (int u = 0; u < kBatchGrad; ++u) {
            const int j = j0 + u * kThreads;
            if (j < nvec) {
                vd[u] = ld_stream_v4(drow + static_cast<int64_t>(j) * 16, keep);
                vt[u] = ld_stream_v4(trow + static_cast<int64_t>(j) * 16, keep);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatchGrad; ++u) {
            if (j0 + u * kThreads < nvec) {
                float x[kPer];
                unpack<kDtype>(vd[u], x);
                od.add(x);
                unpack<kDtype>(vt[u], x);
                ot.add(x);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        od.merge(__shfl_xor_sync(0xFFFFFFFFu, od.m, o), __shfl_xor_sync(0xFFFFFFFFu, od.s, o));
        ot.merge(__shfl_xor_sync(0xFFFFFFFFu, ot.m, o), __shfl_xor_sync(0xFFFFFFFFu, ot.s, o));
    }
    if (lane == 0) {
        s_warp[0][warp] = od.m; s_warp[1][warp] = od.s;
        s_warp[2][warp] = ot.m; s_warp[3][warp] = ot.s;
    }
    __syncthreads();
    if (tid == 0) {
        Online a, b;
        a.init();
        b.init();
        for (int w = 0; w < kThreads / 32; ++w) {
            a.merge(s_warp[0][w], s_warp[1][w]);
            b.merge(s_warp[2][w], s_warp[3][w]);
        }
        s_stats[0] = a.m; s_stats[1] = a.s; s_stats[2] = b.m; s_stats[3] = b.s;
    }
    cluster.sync();
    // every CTA combines the kC slices in rank order: identical results
    Online gd, gt;
    gd.init();
    gt.init();
    for (int r = 0; r < kC; ++r) {
        const float* st = cluster.map_shared_rank(s_stats, r);
        gd.merge(st[0], st[1]);
        gt.merge(st[2], st[3]);
    }
    const float inv_sd = 1.0f / gd.s, inv_st = 1.0f / gt.s;
    const int32_t y = p.labels[pair];
    const bool bad = gd.s != gd.s || gt.s != gt.s || y < 0 || y >= p.V;

    // ---- pass 2: the L1 terms and S = sum of sign(p_d - p_t) p_d (re-read, served by L2)
    float l1 = 0.0f, sg = 0.0f;
    for (int j0 = tid; j0 < nvec; j0 += kBatchGrad * kThreads) {
        uint4 vd[kBatchGrad], vt[kBatchGrad];
#pragma unroll
        for (int u = 0; u < kBatchGrad; ++u) {
            const int j = j0 + u * kThreads;
            if (j < nvec) {
                vd[u] = ld_stream_v4(drow + static_cast<int64_t>(j) * 16, keep);
                vt[u] = ld_stream_v4(trow + static_cast<int64_t>(j) * 16, keep);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatchGrad; ++u) {
            if (j0 + u * kThreads < nvec) {
                float xd[kPer], xt[kPer];
                unpack<kDtype>(vd[u], xd);
                unpack<kDtype>(vt[u], xt);
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    // both probabilities rounded before the difference (no
                    // contraction): equal rows give sign 0 exactly
                    const float pd = __fmul_rn(ex2((xd[i] - gd.m) * kLog2e), inv_sd);
                    const float diff = __fsub_rn(pd, __fmul_rn(ex2((xt[i] - gt.m) * kLog2e), inv_st));
                    l1 += fabsf(diff);
                    sg += diff > 0.0f ? pd : (diff < 0.0f ? -pd : 0.0f);
                }
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, o);
        sg += __shfl_xor_sync(0xFFFFFFFFu, sg, o);
    }
    if (lane == 0) {
        s_warp[0][warp] = l1;
        s_warp[1][warp] = sg;
    }
    __syncthreads();
    if (tid == 0) {
        double a = 0.0, b = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) {
            a += s_warp[0][w];
            b += s_warp[1][w];
        }
        s_sums[0] = a;
        s_sums[1] = b;
    }
    cluster.sync();
    double dist = 0.0, S = 0.0;
    for (int r = 0; r < kC; ++r) {
        const double* sr = cluster.map_shared_rank(s_sums, r);
        dist += sr[0];
        S += sr[1];
    }
    const float c = static_cast<float>(p.scale * exp(-static_cast<double>(k) / p.gamma));
    const float Sf = static_cast<float>(S);
    const float nanf = __int_as_float(0x7FC00000);

    // ---- pass 3: the slice's gradient row (re-read, served by L2)
    for (int j0 = tid; j0 < nvec; j0 += kBatchGrad * kThreads) {
        uint4 vd[kBatchGrad], vt[kBatchGrad];
#pragma unroll
        for (int u = 0; u < kBatchGrad; ++u) {
            const int j = j0 + u * kThreads;
            if (j < nvec) {
                vd[u] = ld_stream_v4(drow + static_cast<int64_t>(j) * 16, drop);
                vt[u] = ld_stream_v4(trow + static_cast<int64_t>(j) * 16, drop);
            }
        }
#pragma unroll
        for (int u = 0; u < kBatchGrad; ++u) {
            const int j = j0 + u * kThreads;
            if (j < nvec) {
                float xd[kPer], xt[kPer], g[kPer];
                unpack<kDtype>(vd[u], xd);
                unpack<kDtype>(vt[u], xt);
#pragma unroll
                for (int i = 0; i < kPer; ++i) {
                    const float pd = __fmul_rn(ex2((xd[i] - gd.m) * kLog2e), inv_sd);
                    const float diff = __fsub_rn(pd, __fmul_rn(ex2((xt[i] - gt.m) * kLog2e), inv_st));
                    const float sv = diff > 0.0f ? 1.0f : (diff < 0.0f ? -1.0f : 0.0f);
                    const int64_t v = lo + static_cast<int64_t>(j) * kPer + i;
                    const float gce = pd - (v == y ? 1.0f : 0.0f);
                    g[i] = bad ? nanf : c * (0.1f * gce + 0.9f * pd * (sv - Sf));
                }
                float4* g4 = reinterpret_cast<float4*>(grow + static_cast<int64_t>(j) * kPer);
                __stcs(g4, make_float4(g[0], g[1], g[2], g[3]));
                if constexpr (kPer == 8) __stcs(g4 + 1, make_float4(g[4], g[5], g[6], g[7]));
            }
        }
    }
    if (rank == 0 && tid == 0) {
        const float acc = fminf(1.0f, fmaxf(0.0f, 1.0f - 0.5f * static_cast<float>(dist)));
        const float zc = p.conf_logits[pair];
        p.grad_conf[pair] = bad ? nanf : c * (1.0f / (1.0f + expf(-zc)) - acc);
    }
    cluster.sync();  // no CTA leaves while others read its shared memory
}

constexpr int kFinalThreads = 256;
constexpr int kSums = 6;  // weighted CE, L1, BCE; sum of accept; sum of tau; token count

// Kernel 2 (one thread per block n): tau_n = 1 + sum_k prod_{j<=k} accept_j,
// the block's status, and its share of the sums; each CTA reduces its
// threads' shares by a fixed binary tree and writes one partial per sum.
__global__ void __launch_bounds__(kFinalThreads) stats_blocks_kernel(const StatsParams p) {
    __shared__ double s_w[32];                         // exp(-k / gamma), k = 1..gamma
    __shared__ double s_sum[kSums][kFinalThreads];
    const int tid = threadIdx.x;
    if (tid < p.gamma) s_w[tid] = exp(-static_cast<double>(tid + 1) / p.gamma);
    __syncthreads();
    const int n = blockIdx.x * kFinalThreads + tid;
    double ce = 0.0, l1 = 0.0, bce = 0.0, acc_sum = 0.0, tau = 0.0, cnt = 0.0;
    if (n < p.N) {
        double survive = 1.0;
        tau = 1.0;
        int32_t code = kReqOk;
        for (int k = 1; k <= p.gamma; ++k) {
            const int64_t i = static_cast<int64_t>(n) * p.gamma + (k - 1);
            const StatsRecord r = p.rec[i];
            survive *= r.acc;
            tau += survive;
            code = max(code, r.code);
            if (!p.mask || p.mask[i]) {
                const double w = s_w[k - 1];
                ce += w * r.ce;
                l1 += w * r.l1;
                bce += w * r.bce;
                acc_sum += r.acc;
                cnt += 1.0;
            }
        }
        p.tau[n] = static_cast<float>(tau);
        if (p.status) p.status[n] = code;
    }
    s_sum[0][tid] = ce; s_sum[1][tid] = l1; s_sum[2][tid] = bce;
    s_sum[3][tid] = acc_sum; s_sum[4][tid] = tau; s_sum[5][tid] = cnt;
    __syncthreads();
    for (int h = kFinalThreads / 2; h > 0; h >>= 1) {  // fixed order: identical bits on every call
        if (tid < h)
#pragma unroll
            for (int j = 0; j < kSums; ++j) s_sum[j][tid] += s_sum[j][tid + h];
        __syncthreads();
    }
    if (tid < kSums) p.partial[static_cast<int64_t>(blockIdx.x) * kSums + tid] = s_sum[tid][0];
}

// Kernel 3 (one CTA): the CTA partials in a fixed order.
__global__ void __launch_bounds__(kFinalThreads) stats_total_kernel(const StatsParams p, int nparts) {
    __shared__ double s_sum[kSums][kFinalThreads];
    const int tid = threadIdx.x;
    double t[kSums] = {0, 0, 0, 0, 0, 0};
    for (int c = tid; c < nparts; c += kFinalThreads)  // each thread: a fixed subsequence
#pragma unroll
        for (int j = 0; j < kSums; ++j) t[j] += p.partial[static_cast<int64_t>(c) * kSums + j];
#pragma unroll
    for (int j = 0; j < kSums; ++j) s_sum[j][tid] = t[j];
    __syncthreads();
    for (int h = kFinalThreads / 2; h > 0; h >>= 1) {
        if (tid < h)
#pragma unroll
            for (int j = 0; j < kSums; ++j) s_sum[j][tid] += s_sum[j][tid + h];
        __syncthreads();
    }
    if (tid == 0) {
        p.loss_num[0] = s_sum[0][0];
        p.loss_num[1] = s_sum[1][0];
        p.loss_num[2] = s_sum[2][0];
        p.loss_num[3] = 0.1 * s_sum[0][0] + 0.9 * s_sum[1][0] + 1.0 * s_sum[2][0];
        p.report[0] = s_sum[3][0];
        p.report[1] = s_sum[4][0];
        *p.num_tokens = static_cast<int64_t>(s_sum[5][0]);
    }
}

}  // namespace

int stats_cluster_size() { return kC; }

int stats_partials(int N) { return (N + kFinalThreads - 1) / kFinalThreads; }

cudaError_t launch_accept_stats_grad(const StatsGradParams& p, cudaStream_t stream) {
    const int64_t pairs = static_cast<int64_t>(p.N) * p.gamma;
    const dim3 grid(static_cast<unsigned>(pairs * kC));
    if (p.dtype == kBF16)
        stats_grad_kernel<kBF16><<<grid, kThreads, 0, stream>>>(p);
    else
        stats_grad_kernel<kF32><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_accept_stats(const StatsParams& p, cudaStream_t stream) {
    const int64_t pairs = static_cast<int64_t>(p.N) * p.gamma;
    const dim3 grid(static_cast<unsigned>(pairs * kC));
    if (p.dtype == kBF16)
        stats_pairs_kernel<kBF16><<<grid, kThreads, 0, stream>>>(p);
    else
        stats_pairs_kernel<kF32><<<grid, kThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int nparts = stats_partials(p.N);
    stats_blocks_kernel<<<nparts, kFinalThreads, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    stats_total_kernel<<<1, kFinalThreads, 0, stream>>>(p, nparts);
    return cudaGetLastError();
}

}  // namespace dspark
