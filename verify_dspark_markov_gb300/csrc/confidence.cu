// Confidence head [MB Semi-autoregressive draft: c_k = sigmoid(w^T [h_k ;
// embed(x_{k-1})])], with embed = the draft token embedding E and no bias.
// One CTA per position; an 8 KB gather per position, negligible next to the
// vocabulary-wide rows, read with 16-byte loads when the rows allow.

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kThreads = 256;

__global__ void __launch_bounds__(kThreads) confidence_kernel(const ConfParams p) {
    const int nk = p.k_last - p.k_first + 1;
    const int b = blockIdx.x / nk;
    const int k = p.k_first + blockIdx.x % nk;  // 1-based position
    const int32_t x_prev = k == 1 ? p.anchor[b] : p.proposals[b * p.gamma + (k - 2)];
    float* out = p.conf + b * p.gamma + (k - 1);
    if (x_prev < 0 || x_prev >= p.V) {  // the request failed before this step
        if (threadIdx.x == 0) *out = 0.0f;
        return;
    }
    const int64_t hrow = (static_cast<int64_t>(b) * p.gamma + (k - 1)) * p.H;
    const uint16_t* e = p.E + static_cast<int64_t>(x_prev) * p.H;
    float acc = 0.0f, acc2 = 0.0f;
    const uintptr_t align = reinterpret_cast<uintptr_t>(p.h) | reinterpret_cast<uintptr_t>(p.E) |
                            reinterpret_cast<uintptr_t>(p.w);
    if (p.H % 8 == 0 && (align & 15) == 0) {
        // 8 elements per 16-byte load of e (and of h in bf16), all of a
        // thread's loads in flight at once: the rows come from HBM
        const uint4* e8 = reinterpret_cast<const uint4*>(e);
        const float4* w4 = reinterpret_cast<const float4*>(p.w);
        const int n8 = p.H / 8;
#pragma unroll 2
        for (int j = threadIdx.x; j < n8; j += kThreads) {
            const uint4 ev = __ldg(e8 + j);
            float hv[8];
            if (p.h_dtype == kBF16) {
                const uint4 hb = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.h) + hrow) + j);
                const uint32_t hw[4] = {hb.x, hb.y, hb.z, hb.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    hv[2 * q] = bf16_lo(hw[q]);
                    hv[2 * q + 1] = bf16_hi(hw[q]);
                }
            } else {
                const float4* h4 = reinterpret_cast<const float4*>(static_cast<const float*>(p.h) + hrow) + 2 * j;
                const float4 a = __ldg(h4), c = __ldg(h4 + 1);
                hv[0] = a.x; hv[1] = a.y; hv[2] = a.z; hv[3] = a.w;
                hv[4] = c.x; hv[5] = c.y; hv[6] = c.z; hv[7] = c.w;
            }
            const float4 wh0 = __ldg(w4 + 2 * j), wh1 = __ldg(w4 + 2 * j + 1);
            const float4 we0 = __ldg(w4 + p.H / 4 + 2 * j), we1 = __ldg(w4 + p.H / 4 + 2 * j + 1);
            const float wh[8] = {wh0.x, wh0.y, wh0.z, wh0.w, wh1.x, wh1.y, wh1.z, wh1.w};
            const float we[8] = {we0.x, we0.y, we0.z, we0.w, we1.x, we1.y, we1.z, we1.w};
            const uint32_t ew[4] = {ev.x, ev.y, ev.z, ev.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc = fmaf(wh[2 * q], hv[2 * q], acc);
                acc2 = fmaf(wh[2 * q + 1], hv[2 * q + 1], acc2);
                acc = fmaf(we[2 * q], bf16_lo(ew[q]), acc);
                acc2 = fmaf(we[2 * q + 1], bf16_hi(ew[q]), acc2);
            }
        }
    } else {
        for (int i = threadIdx.x; i < p.H; i += kThreads) {
            float hv;
            if (p.h_dtype == kBF16)
                hv = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(p.h)[hrow + i]) << 16);
            else
                hv = static_cast<const float*>(p.h)[hrow + i];
            const float ev = __uint_as_float(static_cast<uint32_t>(e[i]) << 16);
            acc = fmaf(p.w[i], hv, acc);
            acc = fmaf(p.w[p.H + i], ev, acc);
        }
    }
    acc += acc2;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
    __shared__ float s[kThreads / 32];
    if ((threadIdx.x & 31) == 0) s[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.0f;
        for (int w = 0; w < kThreads / 32; ++w) a += s[w];
        *out = 1.0f / (1.0f + expf(-a));
    }
}

}  // namespace

cudaError_t launch_confidence(const ConfParams& p, cudaStream_t stream) {
    const int nk = p.k_last - p.k_first + 1;
    if (p.B <= 0 || nk <= 0) return cudaSuccess;
    confidence_kernel<<<p.B * nk, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dspark
