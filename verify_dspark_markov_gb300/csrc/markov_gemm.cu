// Markov head bias on the tensor cores [MB Semi-autoregressive draft: the
// Markov head is a low-rank, token-conditioned additive logit bias]:
//
//   z[b, v] = backbone[b, k-1, v] + sum_j U[x_{k-1}(b), j] * Wm[j, v]
//
// for one step k, all requests b at once: the gather of B rank-r rows of U
// times the r x V matrix, the one dense contraction on the path.  With W
// stored as [V, r] (row v = column v of Wm) both operands are K-major.
//
// tcgen05 (5th-generation tensor cores), swap-AB so that the long vocabulary
// dimension is M:  D[128 v, N b] = W_tile[128 v, r] x U_x^T[r, N b], bf16
// operands in shared memory (canonical no-swizzle K-major layout: 8-row x
// 16-byte core matrices, K-adjacent core matrices 128 bytes apart), fp32
// accumulator in tensor memory.  One thread issues the MMAs and commits them
// to an mbarrier; four warps read the accumulator back with tcgen05.ld (warp w
// owns TMEM lanes 32w..32w+31 = vocabulary entries), add the backbone and
// write z with coalesced stores.  Persistent CTAs (one per SM) walk the
// vocabulary tiles; the gathered U rows are loaded once per CTA.

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kThreads = 256;  // 8 warps: all stage operands; two per TMEM lane quadrant read back
constexpr int kTileM = 128;

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    // start address >> 4, leading byte offset >> 4 (K direction), stride byte
    // offset >> 4 (M/N direction), descriptor version 1, no swizzle
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
           (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t instr_desc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 16-byte asynchronous copy global -> shared (no register staging), so that
// a thread keeps many copies in flight while staging an operand tile.
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Byte offset of element (row, k) in the canonical no-swizzle K-major layout
// with K columns: 8-row x 8-element core matrices, K-adjacent ones 128 B
// apart, row-group-adjacent ones 16 * K bytes apart.
__device__ __forceinline__ uint32_t canon_off(int row, int kc, int K) {
    return static_cast<uint32_t>((row >> 3) * (16 * K) + kc * 128 + (row & 7) * 16);
}

template <int kDtype>
__global__ void __launch_bounds__(kThreads, 1) markov_bias_kernel(const MarkovGemmParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    __shared__ uint64_t mbar;
    __shared__ uint32_t tmem_base;
    __shared__ int s_timeout;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = p.r, N = p.N;
    const int kchunks = r / 8;  // 16-byte chunks per operand row
    uint8_t* sA = smem;
    uint8_t* sB = smem + kTileM * r * 2;

    if (warp == 0) tmem_alloc(&tmem_base, p.tmem_cols);
    if (tid == 0) {
        mbar_init(&mbar, 1);
        fence_mbar_init();
        s_timeout = 0;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    // B operand: the gathered rows U[x_{k-1}(b)], zero rows past the batch
    for (int c = tid; c < N * kchunks; c += kThreads) {
        const int b = c / kchunks, kc = c % kchunks;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (b < p.B) {
            int32_t x = p.k == 1 ? p.anchor[b] : p.proposals[b * p.gamma + (p.k - 2)];
            if (x < 0 || x >= p.V) x = 0;  // a failed request: its row is ignored downstream
            v = *reinterpret_cast<const uint4*>(p.U + static_cast<int64_t>(x) * r + kc * 8);
        }
        *reinterpret_cast<uint4*>(sB + canon_off(b, kc, r)) = v;
    }

    const uint32_t idesc = instr_desc(kTileM, N);
    const uint32_t aaddr = smem_u32(sA), baddr = smem_u32(sB);
    const int ntiles = (p.V + kTileM - 1) / kTileM;
    uint32_t phase = 0;
    const int64_t bb_stride = static_cast<int64_t>(p.gamma) * p.V;  // backbone [B, gamma, V]
    const char* bb = static_cast<const char*>(p.backbone) + static_cast<int64_t>(p.k - 1) * p.V * (kDtype == kBF16 ? 2 : 4);

    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int v0 = t * kTileM;
        // A operand: W rows v0 .. v0+127, zero past the vocabulary
        for (int c = tid; c < kTileM * kchunks; c += kThreads) {
            const int m = c / kchunks, kc = c % kchunks;
            if (v0 + m < p.V)
                cp_async16(sA + canon_off(m, kc, r), p.W + static_cast<int64_t>(v0 + m) * r + kc * 8);
            else
                *reinterpret_cast<uint4*>(sA + canon_off(m, kc, r)) = make_uint4(0u, 0u, 0u, 0u);
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            for (int ks = 0; ks < r / 16; ++ks) {
                // one K step = two K-adjacent core matrices = 256 bytes further
                const uint64_t ad = smem_desc(aaddr + ks * 256, 128, 16 * r);
                const uint64_t bd = smem_desc(baddr + ks * 256, 128, 16 * r);
                mma_bf16(tmem, ad, bd, idesc, ks > 0 ? 1u : 0u);
            }
            mma_commit(&mbar);
        }
        // backbone values of this thread's entries, read while the MMAs run (all
        // loads issued before any store, so none waits on a store to z)
        const int quad = warp & 3;
        const int v = v0 + quad * 32 + lane;
        const int c_first = (warp >> 2) * 16;
        constexpr int kMaxBatches = 8;  // N <= 256 columns, 16 per batch, two warps per quadrant
        float base[kMaxBatches][16];
#pragma unroll
        for (int bi = 0; bi < kMaxBatches; ++bi) {
            const int c0 = c_first + bi * 32;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int b = c0 + i;
                float x = 0.0f;
                if (c0 < N && b < p.B && v < p.V) {
                    if constexpr (kDtype == kBF16)
                        x = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(
                                                bb + b * bb_stride * 2) + v))
                                            << 16);
                    else
                        x = __ldg(reinterpret_cast<const float*>(bb + b * bb_stride * 4) + v);
                }
                base[bi][i] = x;
            }
        }
        const bool ok = mbar_wait(&mbar, phase, kWaitLimitNs);
        phase ^= 1u;
        if (!ok) s_timeout = 1;
        tc_fence_after();
        // epilogue: warp w reads TMEM lane quadrant w % 4 (vocabulary entries
        // v0 + 32 (w % 4) + lane) and every other 16-column group from w / 4
#pragma unroll
        for (int bi = 0; bi < kMaxBatches; ++bi) {
            const int c0 = c_first + bi * 32;
            if (c0 >= N) break;
            float acc[16];
            tmem_ld16(tmem + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(c0), acc);
            if (v < p.V) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int b = c0 + i;
                    if (b < p.B) p.zbuf[static_cast<int64_t>(b) * p.V + v] = base[bi][i] + acc[i];
                }
            }
        }
        tc_fence_before();
        __syncthreads();  // TMEM and the A tile are free for the next tile
        if (s_timeout) break;
    }
    if (s_timeout) {
        // report, then give MMAs still in flight a bounded chance to land
        // before the tensor memory is released
        if (tid == 0) {
            *p.error_flag = 1;
            mbar_wait(&mbar, phase ^ 1u, kWaitLimitNs);
        }
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, p.tmem_cols);
}

}  // namespace

int markov_gemm_smem(int r, int N) { return (kTileM + N) * r * 2; }

cudaError_t launch_markov_bias(const MarkovGemmParams& p, int grid, cudaStream_t stream) {
    const int smem = markov_gemm_smem(p.r, p.N);
    cudaError_t e;
    if (p.dtype == kBF16) {
        if ((e = cudaFuncSetAttribute(markov_bias_kernel<kBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem)) != cudaSuccess)
            return e;
        markov_bias_kernel<kBF16><<<grid, kThreads, smem, stream>>>(p);
    } else {
        if ((e = cudaFuncSetAttribute(markov_bias_kernel<kF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      smem)) != cudaSuccess)
            return e;
        markov_bias_kernel<kF32><<<grid, kThreads, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace dspark
