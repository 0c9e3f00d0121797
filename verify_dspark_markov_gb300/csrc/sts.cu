// Sequential Temperature Scaling of the confidence head [MB Acceptance and
// confidence]: for each block position k, the inverse temperature
// beta_k >= 0 whose calibrated confidence sigmoid(beta_k z) minimises the
// masked BCE against the accept labels a over logged pairs (z, a).  The BCE
// is convex in beta and its slope sum z (sigmoid(beta z) - a) does not
// decrease, so the fit is the slope's root.
//
// The fit runs on the device in one persistent cooperative launch whose
// CTAs meet at grid barriers (every wait bounded in time):
//  * a pass: one streaming read of the pairs at the current beta_k of every
//    position, giving the slope and the curvature
//    sum z^2 sigmoid (1 - sigmoid) per position, and exact flags (a counted
//    z != 0; a label against the sign of its z; an invalid pair).  A thread
//    takes chunks of four whole rows (4 gamma pairs: gamma 16-byte vectors
//    of z and of a, so the position of every element is fixed at compile
//    time) with per-position sums in registers; warps reduce by shuffles,
//    CTAs through shared memory, and each CTA writes its per-position sums
//    (fp64) to its own slot.  Misaligned inputs and the last N mod 4 rows
//    are read one row at a time.
//  * barrier, then the update, by CTA 0: the CTAs' slots summed per position
//    in a fixed order (a strided sum per lane, then a fixed butterfly), so
//    beta's bits do not depend on the order the CTAs ran in; then lane k
//    runs sts_search_step (sts_search.cuh) on position k - the degenerate
//    cases on the first pass (taken at beta = 0), then a Newton step kept
//    inside the bracket [lo, hi] of the root, bisection (or doubling while
//    hi is open) when the step leaves it.  A position still searching after
//    the last pass of the budget reports status 4 with its last iterate.
//  * barrier; the next pass starts unless every position has stopped.
// A barrier wait that runs past its limit sets an error word and ends the
// CTA; a one-warp kernel after the fit then reports status 5 at every
// position.  HBM-bound: 9 bytes a pair a pass (8 without a mask).

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
constexpr int32_t kStsNotConverged = 4;
constexpr int32_t kStsWaitGaveUp = 5;

__global__ void sts_init_kernel(StsState* st, int* active, unsigned* bar, int* error, int gamma) {
    const int k = threadIdx.x;
    if (k < kG) {
        StsState s{};
        s.beta = 0.0;
        s.lo = 0.0;
        s.hi = __longlong_as_double(0x7FF0000000000000ll);  // +inf: no upper bound yet
        s.phase = k < gamma ? 0 : 2;
        st[k] = s;
    }
    if (k == 0) {
        *active = gamma;
        *bar = 0u;
        *error = 0;
    }
}

// The position state as the other CTAs left it (through L2, not this SM's L1).
__device__ __forceinline__ StsState load_state(const StsState* p) {
    StsState s;
    s.beta = __ldcg(&p->beta);
    s.lo = __ldcg(&p->lo);
    s.hi = __ldcg(&p->hi);
    s.s1 = __ldcg(&p->s1);
    s.s2 = __ldcg(&p->s2);
    s.flags = __ldcg(&p->flags);
    s.phase = __ldcg(&p->phase);
    s.status = __ldcg(&p->status);
    s.passes = __ldcg(&p->passes);
    return s;
}

// One pair's terms at inverse temperature b into the position's sums and flags.
__device__ __forceinline__ void add_pair(float zv, float av, float b, float& g1, float& g2, unsigned& inf,
                                         unsigned& viol, unsigned& bad, unsigned bit) {
    if (!isfinite(zv) || !(av >= 0.0f && av <= 1.0f)) bad |= bit;
    if (zv != 0.0f) inf |= bit;
    if ((zv > 0.0f && av < 1.0f) || (zv < 0.0f && av > 0.0f)) viol |= bit;
    // sigmoid(b z) from the hardware exp2 and a fast reciprocal (each within
    // a few ulp: far below the 1e-7 relative accuracy the fp32 sums allow)
    float e2;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e2) : "f"(-b * zv * 1.4426950408889634f));
    const float sg = __fdividef(1.0f, 1.0f + e2);
    g1 += zv * (sg - av);
    g2 += zv * zv * (sg * (1.0f - sg));
}

template <int G>
__global__ void __launch_bounds__(kStsThreads) sts_fit_kernel(const StsParams p, bool vec) {
    __shared__ float s_beta[kG];
    __shared__ float s_red[kStsWarps][kG][2];
    __shared__ double s_sum[kG][2];
    __shared__ unsigned s_flag[3];
    __shared__ int s_stop, s_ok;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float* __restrict__ z = p.conf_logits;
    const float* __restrict__ a = p.labels;
    const uint8_t* __restrict__ mask = p.mask;
    const int64_t N = p.N;
    const int64_t nthreads = static_cast<int64_t>(gridDim.x) * kStsThreads;
    const int64_t gtid = static_cast<int64_t>(blockIdx.x) * kStsThreads + tid;
    const int64_t chunks = vec ? N / 4 : 0;  // 4-row chunks read as vectors
    unsigned gen = 0;

    for (int pass = 0; pass < p.max_passes; ++pass) {
        if (tid == 0) s_stop = __ldcg(p.active) == 0;
        if (tid < G) s_beta[tid] = static_cast<float>(__ldcg(&p.state[tid].beta));
        if (tid < 3) s_flag[tid] = 0u;
        __syncthreads();
        if (s_stop) break;  // uniform over the grid: every CTA read it after the same barrier

        float bt[G], g1[G], g2[G];
#pragma unroll
        for (int k = 0; k < G; ++k) {
            bt[k] = s_beta[k];
            g1[k] = 0.0f;
            g2[k] = 0.0f;
        }
        unsigned inf = 0u, viol = 0u, bad = 0u;  // bit k: position k
        for (int64_t c = gtid; c < chunks; c += nthreads) {
            const float4* zc = reinterpret_cast<const float4*>(z) + c * G;
            const float4* ac = reinterpret_cast<const float4*>(a) + c * G;
            float4 zv[G], av[G];
            uint32_t mv[G];
#pragma unroll
            for (int i = 0; i < G; ++i) {
                zv[i] = __ldcs(zc + i);
                av[i] = __ldcs(ac + i);
                mv[i] = mask ? __ldcs(reinterpret_cast<const unsigned int*>(mask) + c * G + i) : 0xFFFFFFFFu;
            }
#pragma unroll
            for (int i = 0; i < G; ++i) {
                const float ze[4] = {zv[i].x, zv[i].y, zv[i].z, zv[i].w};
                const float ae[4] = {av[i].x, av[i].y, av[i].z, av[i].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = (4 * i + e) % G;  // compile-time position
                    if ((mv[i] >> (8 * e)) & 0xFFu)
                        add_pair(ze[e], ae[e], bt[k], g1[k], g2[k], inf, viol, bad, 1u << k);
                }
            }
        }
        // rows past the chunks (all rows when the inputs are not aligned)
        for (int64_t n = chunks * 4 + gtid; n < N; n += nthreads) {
            const int64_t base = n * G;
#pragma unroll
            for (int k = 0; k < G; ++k)
                if (!mask || mask[base + k]) add_pair(z[base + k], a[base + k], bt[k], g1[k], g2[k], inf, viol, bad, 1u << k);
        }

#pragma unroll
        for (int k = 0; k < G; ++k) {
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
        inf = __reduce_or_sync(0xFFFFFFFFu, inf);
        viol = __reduce_or_sync(0xFFFFFFFFu, viol);
        bad = __reduce_or_sync(0xFFFFFFFFu, bad);
        if (lane == 0) {
            if (inf) atomicOr(&s_flag[0], inf);
            if (viol) atomicOr(&s_flag[1], viol);
            if (bad) atomicOr(&s_flag[2], bad);
        }
        __syncthreads();
        if (tid < G) {
            double x = 0.0, y = 0.0;
            for (int w = 0; w < kStsWarps; ++w) {
                x += static_cast<double>(s_red[w][tid][0]);
                y += static_cast<double>(s_red[w][tid][1]);
            }
            double* slot = p.partial + (static_cast<size_t>(blockIdx.x) * kG + tid) * 2;
            slot[0] = x;
            slot[1] = y;
            const unsigned f = (((s_flag[0] >> tid) & 1u) ? kInformative : 0u) |
                               (((s_flag[1] >> tid) & 1u) ? kViolated : 0u) |
                               (((s_flag[2] >> tid) & 1u) ? kInvalid : 0u);
            if (f) atomicOr(&p.state[tid].flags, f);
        }
        if (!grid_barrier_bounded(p.bar, p.error, ++gen * gridDim.x, kWaitLimitNs, &s_ok)) return;

        if (blockIdx.x == 0) {
            // the pass's sums per position, in a fixed order: lane l adds
            // slots l, l + 32, ... in turn, then a fixed butterfly
            for (int k = warp; k < G; k += kStsWarps) {
                double x = 0.0, y = 0.0;
                for (int c = lane; c < static_cast<int>(gridDim.x); c += 32) {
                    x += __ldcg(p.partial + (static_cast<size_t>(c) * kG + k) * 2);
                    y += __ldcg(p.partial + (static_cast<size_t>(c) * kG + k) * 2 + 1);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
                    y += __shfl_xor_sync(0xFFFFFFFFu, y, o);
                }
                if (lane == 0) {
                    s_sum[k][0] = x;
                    s_sum[k][1] = y;
                }
            }
            __syncthreads();
            if (warp == 0) {
                const int k = lane;
                bool finished = false;
                if (k < G) {
                    StsState s = load_state(p.state + k);
                    if (s.phase != 2) {
                        s.s1 = s_sum[k][0];
                        s.s2 = s_sum[k][1];
                    }
                    finished = sts_search_step(s);
                    p.state[k] = s;
                    p.beta[k] = s.beta;
                    // the budget ran out with the search still open: its last iterate
                    p.status[k] = (pass == p.max_passes - 1 && s.phase != 2) ? kStsNotConverged : s.status;
                    if (p.passes) p.passes[k] = s.passes;
                }
                const unsigned fin = __ballot_sync(0xFFFFFFFFu, finished);
                if (k == 0 && fin) atomicSub(p.active, __popc(fin));
            }
        }
        if (!grid_barrier_bounded(p.bar, p.error, ++gen * gridDim.x, kWaitLimitNs, &s_ok)) return;
    }
}

// After the fit: a barrier that gave up leaves no fit at any position.
__global__ void sts_finish_kernel(const int* error, int gamma, int32_t* status) {
    if (*error && static_cast<int>(threadIdx.x) < gamma) status[threadIdx.x] = kStsWaitGaveUp;
}

template <int G>
cudaError_t launch_fit(const StsParams& p, int sms, cudaStream_t stream) {
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sts_fit_kernel<G>, kStsThreads, 0);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorLaunchOutOfResources;
    const bool vec = (reinterpret_cast<uintptr_t>(p.conf_logits) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.labels) & 15u) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.mask) & 3u) == 0;
    const int64_t units = vec ? std::max<int64_t>(p.N / 4, p.N % 4) : p.N;
    const int64_t want = (units + kStsThreads - 1) / kStsThreads;
    const int grid = static_cast<int>(std::max<int64_t>(
        1, std::min<int64_t>(std::min<int64_t>(want, static_cast<int64_t>(sms) * per_sm), kStsMaxGrid)));
    StsParams q = p;
    void* args[] = {&q, const_cast<bool*>(&vec)};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(sts_fit_kernel<G>), dim3(grid),
                                       dim3(kStsThreads), args, 0, stream);
}

template <int... Gs>
cudaError_t launch_fit_for(int gamma, const StsParams& p, int sms, cudaStream_t stream,
                           std::integer_sequence<int, Gs...>) {
    cudaError_t e = cudaErrorInvalidValue;
    ((gamma == Gs + 1 ? (e = launch_fit<Gs + 1>(p, sms, stream), true) : false) || ...);
    return e;
}

}  // namespace

cudaError_t launch_sts_fit(const StsParams& p, cudaStream_t stream) {
    if (p.gamma < 1 || p.gamma > kG || p.N < 0 || p.max_passes < 1) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sts_init_kernel<<<1, 32, 0, stream>>>(p.state, p.active, p.bar, p.error, p.gamma);
    e = launch_fit_for(p.gamma, p, sms, stream, std::make_integer_sequence<int, kG>{});
    if (e != cudaSuccess) return e;
    sts_finish_kernel<<<1, 32, 0, stream>>>(p.error, p.gamma, p.status);
    return cudaGetLastError();
}

}  // namespace dspark
