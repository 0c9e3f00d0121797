// The RNN head's recurrence [MB Semi-autoregressive draft: a GRU-like
// recurrence carrying prefix state across the block].  The pages give no
// equations; the cell is a standard GRU (gate order r, z, n) on the previous
// token's rank-r embedding e_k = U[x_{k-1}], from s_0 = 0:
//   r = sigma(Wi_r e + bi_r + Wh_r s + bh_r),  z = sigma(Wi_z e + bi_z + Wh_z s + bh_z),
//   n = tanh(Wi_n e + bi_n + r (Wh_n s + bh_n)),  s' = (1 - z) n + z s.
// Its state enters the logits through the Markov head's low-rank bias W s_k,
// computed by the same tcgen05 GEMM: the kernel below writes s_k as two bf16
// rows, hi = bf16(s_k) and lo = bf16(s_k - hi) (s_k to about 2^-16), and an
// index array that lets the GEMM's gather read row b of them.
//
// gru_step_kernel: one CTA per 8 requests, one thread per state unit j.  The
// CTA stages e and s of its requests in shared memory (fp32), then thread j
// streams its six weight rows (Wi and Wh at j, r + j, 2r + j) once, 16 bytes
// at a time, and accumulates the six dot products of all 8 requests.  The
// 2 x 3r x r bf16 weights (768 KB at r = 256) stay in L2 across CTAs.

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kGruReq = 8;  // requests per CTA

__device__ __forceinline__ float sigmoidf_(float a) { return 1.0f / (1.0f + expf(-a)); }

__global__ void __launch_bounds__(256) gru_step_kernel(const GruParams p) {
    __shared__ float s_e[kGruReq][256];
    __shared__ float s_s[kGruReq][256];
    const int r = p.r, j = threadIdx.x;
    const int b0 = blockIdx.x * kGruReq;
    const int nreq = min(kGruReq, p.B - b0);

    // stage e = U[x_{k-1}] and s_{k-1} of the CTA's requests
    for (int m = 0; m < kGruReq; ++m) {
        const int b = b0 + m;
        float e = 0.0f, s = 0.0f;
        if (m < nreq) {
            const int32_t x = p.k == 1 ? p.anchor[b] : p.proposals[static_cast<int64_t>(b) * p.gamma + (p.k - 2)];
            if (x >= 0 && x < p.V) e = __uint_as_float(static_cast<uint32_t>(p.U[static_cast<int64_t>(x) * r + j]) << 16);
            if (p.k > 1) s = p.state[static_cast<int64_t>(b) * r + j];
            if (j == 0) p.index[b] = (x >= 0 && x < p.V) ? b : -1;
        }
        s_e[m][j] = e;
        s_s[m][j] = s;
    }
    __syncthreads();

    // the six dot products of unit j for every request of the CTA
    float acc[6][kGruReq];
#pragma unroll
    for (int g = 0; g < 6; ++g)
#pragma unroll
        for (int m = 0; m < kGruReq; ++m) acc[g][m] = 0.0f;
    const uint16_t* wrow[6] = {p.Wi + static_cast<int64_t>(j) * r, p.Wi + static_cast<int64_t>(r + j) * r,
                               p.Wi + static_cast<int64_t>(2 * r + j) * r, p.Wh + static_cast<int64_t>(j) * r,
                               p.Wh + static_cast<int64_t>(r + j) * r, p.Wh + static_cast<int64_t>(2 * r + j) * r};
    for (int i = 0; i < r; i += 8) {
#pragma unroll
        for (int g = 0; g < 6; ++g) {
            if (g >= 3 && p.k == 1) continue;  // s_0 = 0: the hidden products vanish
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(wrow[g] + i));
            const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
            const float (*v)[256] = g < 3 ? s_e : s_s;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float w0 = bf16_lo(wv[t]), w1 = bf16_hi(wv[t]);
#pragma unroll
                for (int m = 0; m < kGruReq; ++m) {
                    acc[g][m] = fmaf(w0, v[m][i + 2 * t], acc[g][m]);
                    acc[g][m] = fmaf(w1, v[m][i + 2 * t + 1], acc[g][m]);
                }
            }
        }
    }

    for (int m = 0; m < nreq; ++m) {
        const int b = b0 + m;
        const float rg = sigmoidf_((acc[0][m] + p.bi[j]) + (acc[3][m] + p.bh[j]));
        const float zg = sigmoidf_((acc[1][m] + p.bi[r + j]) + (acc[4][m] + p.bh[r + j]));
        const float n = tanhf((acc[2][m] + p.bi[2 * r + j]) + rg * (acc[5][m] + p.bh[2 * r + j]));
        const float s = (1.0f - zg) * n + zg * s_s[m][j];
        const __nv_bfloat16 hi = __float2bfloat16_rn(s);
        const __nv_bfloat16 lo = __float2bfloat16_rn(s - __bfloat162float(hi));
        p.state[static_cast<int64_t>(b) * r + j] = s;
        p.hi[static_cast<int64_t>(b) * r + j] = __bfloat16_as_ushort(hi);
        p.lo[static_cast<int64_t>(b) * r + j] = __bfloat16_as_ushort(lo);
    }
}

}  // namespace

cudaError_t launch_gru_step(const GruParams& p, cudaStream_t stream) {
    if (p.B < 1 || p.r < 16 || p.r > 256 || p.r % 16 != 0) return cudaErrorInvalidValue;
    const int grid = (p.B + kGruReq - 1) / kGruReq;
    gru_step_kernel<<<grid, p.r, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dspark
