// Sequential Temperature Scaling of the confidence head [MB Acceptance and
// confidence]: for each block position k, the inverse temperature
// beta_k >= 0 whose calibrated confidence sigmoid(beta_k z) minimises the
// masked BCE against the accept labels a over logged pairs (z, a).  The BCE
// is convex in beta and its slope sum z (sigmoid(beta z) - a) does not
// decrease, so the fit is the slope's root.
//
// The fit runs on the device in passes; the host only enqueues them:
//  * sts_pass_kernel - one streaming pass over the pairs at the current
//    beta_k of every position: the slope and the curvature
//    sum z^2 sigmoid (1 - sigmoid) per position, and exact flags (a counted
//    z != 0; a label against the sign of its z; an invalid pair).  A thread
//    takes whole rows n (gamma contiguous pairs) with per-position sums in
//    registers; warps reduce by shuffles, CTAs through shared memory, and
//    each CTA writes its per-position sums (fp64) to its own slot.
//  * sts_update_kernel - sums the CTAs' slots per position in a fixed order
//    (a strided sum per thread, then a fixed tree), so beta's bits do not
//    depend on the order the CTAs ran in; then lane k runs sts_search_step
//    (sts_search.cuh) on position k - the degenerate cases on the first pass
//    (taken at beta = 0), then a Newton step kept inside the bracket [lo, hi]
//    of the root, bisection (or doubling while hi is open) when the step
//    leaves it.  A position still searching after the last enqueued pass
//    reports status 4 with its last iterate.
// Once every position has converged the remaining passes return at once.
// HBM-bound: 9 bytes a pair a pass (8 without a mask).

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "sts_search.cuh"

namespace dspark {

namespace {

constexpr int kStsThreads = 256;
constexpr int kStsWarps = kStsThreads / 32;
constexpr int kG = DSPARK_MAX_GAMMA;
constexpr unsigned kInformative = kStsInformative, kViolated = kStsViolated, kInvalid = kStsInvalid;
constexpr int kUpdThreads = 256;
constexpr int32_t kStsNotConverged = 4;

__global__ void sts_init_kernel(StsState* st, int* active, int gamma) {
    const int k = threadIdx.x;
    if (k < kG) {
        StsState s{};
        s.beta = 0.0;
        s.lo = 0.0;
        s.hi = __longlong_as_double(0x7FF0000000000000ll);  // +inf: no upper bound yet
        s.phase = k < gamma ? 0 : 2;
        st[k] = s;
    }
    if (k == 0) *active = gamma;
}

__global__ void __launch_bounds__(kStsThreads) sts_pass_kernel(const float* __restrict__ z,
                                                               const float* __restrict__ a,
                                                               const uint8_t* __restrict__ mask, int64_t N,
                                                               int gamma, StsState* st, const int* active,
                                                               double* partial) {
    if (*active == 0) return;
    __shared__ float s_beta[kG];
    __shared__ float s_red[kStsWarps][kG][2];
    __shared__ unsigned s_flag[3];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < kG) s_beta[tid] = tid < gamma ? static_cast<float>(st[tid].beta) : 0.0f;
    if (tid < 3) s_flag[tid] = 0u;
    __syncthreads();

    float bt[kG], g1[kG], g2[kG];
#pragma unroll
    for (int k = 0; k < kG; ++k) {
        bt[k] = s_beta[k];
        g1[k] = 0.0f;
        g2[k] = 0.0f;
    }
    unsigned inf = 0u, viol = 0u, bad = 0u;  // bit k: position k
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kStsThreads;
    for (int64_t n = static_cast<int64_t>(blockIdx.x) * kStsThreads + tid; n < N; n += stride) {
        const int64_t base = n * gamma;
#pragma unroll
        for (int k = 0; k < kG; ++k) {
            if (k < gamma && (!mask || mask[base + k])) {
                const float zv = z[base + k], av = a[base + k];
                if (!isfinite(zv) || !(av >= 0.0f && av <= 1.0f)) bad |= 1u << k;
                if (zv != 0.0f) inf |= 1u << k;
                if ((zv > 0.0f && av < 1.0f) || (zv < 0.0f && av > 0.0f)) viol |= 1u << k;
                const float sg = 1.0f / (1.0f + expf(-bt[k] * zv));
                g1[k] += zv * (sg - av);
                g2[k] += zv * zv * (sg * (1.0f - sg));
            }
        }
    }

#pragma unroll
    for (int k = 0; k < kG; ++k) {
        if (k < gamma) {
            float x = g1[k], y = g2[k];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
                y += __shfl_xor_sync(0xFFFFFFFFu, y, o);
            }
            if (lane == 0) {
                s_red[warp][k][0] = x;
                s_red[warp][k][1] = y;
            }
        }
    }
    inf = __reduce_or_sync(0xFFFFFFFFu, inf);
    viol = __reduce_or_sync(0xFFFFFFFFu, viol);
    bad = __reduce_or_sync(0xFFFFFFFFu, bad);
    if (lane == 0) {
        if (inf) atomicOr(&s_flag[0], inf);
        if (viol) atomicOr(&s_flag[1], viol);
        if (bad) atomicOr(&s_flag[2], bad);
    }
    __syncthreads();
    if (tid < gamma) {
        double x = 0.0, y = 0.0;
        for (int w = 0; w < kStsWarps; ++w) {
            x += static_cast<double>(s_red[w][tid][0]);
            y += static_cast<double>(s_red[w][tid][1]);
        }
        double* slot = partial + (static_cast<size_t>(blockIdx.x) * kG + tid) * 2;
        slot[0] = x;
        slot[1] = y;
        const unsigned f = (((s_flag[0] >> tid) & 1u) ? kInformative : 0u) |
                           (((s_flag[1] >> tid) & 1u) ? kViolated : 0u) |
                           (((s_flag[2] >> tid) & 1u) ? kInvalid : 0u);
        if (f) atomicOr(&st[tid].flags, f);
    }
}

__global__ void __launch_bounds__(kUpdThreads) sts_update_kernel(StsState* st, int* active, int gamma,
                                                                 const double* partial, int grid, bool last,
                                                                 double* beta_out, int32_t* status_out,
                                                                 int32_t* passes_out) {
    __shared__ double s_sum[kUpdThreads][2];
    const int tid = threadIdx.x;
    if (*active == 0) return;  // the pass kernel wrote no slots (uniform over the CTA)
    // the pass's sums, per position: thread t adds slots t, t + 256, ... in
    // order, then a fixed binary tree over the threads
    for (int k = 0; k < gamma; ++k) {
        double x = 0.0, y = 0.0;
        for (int c = tid; c < grid; c += kUpdThreads) {
            x += partial[(static_cast<size_t>(c) * kG + k) * 2];
            y += partial[(static_cast<size_t>(c) * kG + k) * 2 + 1];
        }
        s_sum[tid][0] = x;
        s_sum[tid][1] = y;
        __syncthreads();
        for (int h = kUpdThreads / 2; h > 0; h >>= 1) {
            if (tid < h) {
                s_sum[tid][0] += s_sum[tid + h][0];
                s_sum[tid][1] += s_sum[tid + h][1];
            }
            __syncthreads();
        }
        if (tid == 0 && st[k].phase != 2) {
            st[k].s1 = s_sum[0][0];
            st[k].s2 = s_sum[0][1];
        }
        __syncthreads();
    }
    if (tid >= 32) return;
    const int k = tid;
    bool finished = false;
    if (k < gamma) {
        StsState s = st[k];
        finished = sts_search_step(s);
        st[k] = s;
        beta_out[k] = s.beta;
        // the budget ran out with the search still open: its last iterate
        status_out[k] = (last && s.phase != 2) ? kStsNotConverged : s.status;
        if (passes_out) passes_out[k] = s.passes;
    }
    const unsigned fin = __ballot_sync(0xFFFFFFFFu, finished);
    if (k == 0 && fin) atomicSub(active, __popc(fin));
}

}  // namespace

cudaError_t launch_sts_fit(const StsParams& p, cudaStream_t stream) {
    if (p.gamma < 1 || p.gamma > kG || p.N < 0 || p.max_passes < 1) return cudaErrorInvalidValue;
    sts_init_kernel<<<1, 32, 0, stream>>>(p.state, p.active, p.gamma);
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t want = (p.N + kStsThreads - 1) / kStsThreads;
    const int grid = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>(std::min<int64_t>(want, static_cast<int64_t>(sms) * 8), kStsMaxGrid)));
    for (int r = 0; r < p.max_passes; ++r) {
        sts_pass_kernel<<<grid, kStsThreads, 0, stream>>>(p.conf_logits, p.labels, p.mask, p.N, p.gamma, p.state,
                                                          p.active, p.partial);
        sts_update_kernel<<<1, kUpdThreads, 0, stream>>>(p.state, p.active, p.gamma, p.partial, grid,
                                                         r == p.max_passes - 1, p.beta, p.status, p.passes);
    }
    return cudaGetLastError();
}

}  // namespace dspark
