// Confidence head [MB Semi-autoregressive draft: c_k = sigmoid(w^T [h_k ;
// embed(x_{k-1})])], with embed = the draft token embedding E and no bias.
// One CTA per position; an 8 KB gather per position, negligible next to the
// vocabulary-wide rows.

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
    float acc = 0.0f;
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
