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
// gru_step_kernel: one CTA per 8 requests and 8 state units (one per warp).
// The CTA stages e and s_{k-1} of its requests in shared memory (fp32); a
// warp takes one unit, its lanes splitting the K dimension 8 elements each, so that each of the unit's six weight rows (Wi and Wh at j,
// r + j, 2r + j) is one coalesced 512-byte read of the warp; the lanes' partial
// dot products for the 8 requests are summed by a butterfly, and lane m
// applies the gates for request m.  s_{k-1} is read from one state buffer and
// s_k written to the other (the CTAs of a request read all of s_{k-1} while
// others write their units of s_k).  The 2 x 3r x r bf16 weights (768 KB at
// r = 256) stay in L2 across CTAs and steps.

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kGruReq = 8;     // requests per CTA
constexpr int kGruUnits = 8;   // state units per CTA (one per warp: its latency is paid once)
constexpr int kGruThreads = 256;
constexpr int kGruUnitsPerWarp = kGruUnits / (kGruThreads / 32);

__device__ __forceinline__ float sigmoidf_(float a) { return 1.0f / (1.0f + expf(-a)); }

__global__ void __launch_bounds__(kGruThreads) gru_step_kernel(const GruParams p) {
    __shared__ __align__(16) float s_e[kGruReq][256];
    __shared__ __align__(16) float s_s[kGruReq][256];
    __shared__ int32_t s_x[kGruReq];
    const int r = p.r, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b0 = blockIdx.x * kGruReq;
    const int nreq = min(kGruReq, p.B - b0);

    // the CTA's tokens x_{k-1} first, then e = U[x_{k-1}] and s_{k-1} (all r
    // units) of its requests, every thread's loads independent of each other
    if (tid < kGruReq) {
        int32_t x = -1;
        if (tid < nreq) {
            const int b = b0 + tid;
            x = p.k == 1 ? p.anchor[b] : p.proposals[static_cast<int64_t>(b) * p.gamma + (p.k - 2)];
            if (x < 0 || x >= p.V) x = -1;
            if (blockIdx.y == 0) p.index[b] = x >= 0 ? b : -1;
        }
        s_x[tid] = x;
    }
    __syncthreads();
    if (tid < r) {
#pragma unroll
        for (int m = 0; m < kGruReq; ++m) {
            const int32_t x = s_x[m];
            s_e[m][tid] = x >= 0 ? __uint_as_float(static_cast<uint32_t>(p.U[static_cast<int64_t>(x) * r + tid]) << 16)
                                 : 0.0f;
            s_s[m][tid] = (p.k > 1 && m < nreq) ? p.state_in[static_cast<int64_t>(b0 + m) * r + tid] : 0.0f;
        }
    }
    __syncthreads();

    const int k0 = lane * 8;  // this lane's 8 elements of K
    for (int uu = 0; uu < kGruUnitsPerWarp; ++uu) {
        const int j = blockIdx.y * kGruUnits + warp * kGruUnitsPerWarp + uu;  // uniform over the warp
        if (j >= r) break;
        // the unit's six biases, loaded while the dot products run
        const float bir = p.bi[j], biz = p.bi[r + j], bin = p.bi[2 * r + j];
        const float bhr = p.bh[j], bhz = p.bh[r + j], bhn = p.bh[2 * r + j];
        float acc[6][kGruReq];
#pragma unroll
        for (int g = 0; g < 6; ++g)
#pragma unroll
            for (int m = 0; m < kGruReq; ++m) acc[g][m] = 0.0f;
        if (k0 < r) {
#pragma unroll
            for (int g = 0; g < 6; ++g) {
                if (g >= 3 && p.k == 1) continue;  // s_0 = 0: the hidden products vanish
                const uint16_t* row = (g < 3 ? p.Wi : p.Wh) + static_cast<int64_t>((g % 3) * r + j) * r + k0;
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(row));
                const float wf[8] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y),
                                     bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
                const float (*v)[256] = g < 3 ? s_e : s_s;
#pragma unroll
                for (int m = 0; m < kGruReq; ++m) {
                    const float4 a = *reinterpret_cast<const float4*>(&v[m][k0]);
                    const float4 c = *reinterpret_cast<const float4*>(&v[m][k0 + 4]);
                    float t = acc[g][m];
                    t = fmaf(wf[0], a.x, t);
                    t = fmaf(wf[1], a.y, t);
                    t = fmaf(wf[2], a.z, t);
                    t = fmaf(wf[3], a.w, t);
                    t = fmaf(wf[4], c.x, t);
                    t = fmaf(wf[5], c.y, t);
                    t = fmaf(wf[6], c.z, t);
                    t = fmaf(wf[7], c.w, t);
                    acc[g][m] = t;
                }
            }
        }
        // the unit's six dot products for every request, in every lane
#pragma unroll
        for (int g = 0; g < 6; ++g)
#pragma unroll
            for (int m = 0; m < kGruReq; ++m)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[g][m] += __shfl_xor_sync(0xFFFFFFFFu, acc[g][m], o);
#pragma unroll
        for (int m = 0; m < kGruReq; ++m) {
            if (lane != m || m >= nreq) continue;
            const int b = b0 + m;
            const float rg = sigmoidf_((acc[0][m] + bir) + (acc[3][m] + bhr));
            const float zg = sigmoidf_((acc[1][m] + biz) + (acc[4][m] + bhz));
            const float n = tanhf((acc[2][m] + bin) + rg * (acc[5][m] + bhn));
            const float sv = (1.0f - zg) * n + zg * s_s[m][j];
            const __nv_bfloat16 hi = __float2bfloat16_rn(sv);
            const __nv_bfloat16 lo = __float2bfloat16_rn(sv - __bfloat162float(hi));
            p.state_out[static_cast<int64_t>(b) * r + j] = sv;
            p.hi[static_cast<int64_t>(b) * r + j] = __bfloat16_as_ushort(hi);
            p.lo[static_cast<int64_t>(b) * r + j] = __bfloat16_as_ushort(lo);
        }
    }
}

}  // namespace

cudaError_t launch_gru_step(const GruParams& p, cudaStream_t stream) {
    if (p.B < 1 || p.r < 16 || p.r > 256 || p.r % 16 != 0) return cudaErrorInvalidValue;
    const dim3 grid((p.B + kGruReq - 1) / kGruReq, (p.r + kGruUnits - 1) / kGruUnits);
    gru_step_kernel<<<grid, kGruThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dspark
