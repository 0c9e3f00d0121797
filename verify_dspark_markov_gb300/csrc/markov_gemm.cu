// Markov head bias on the tensor cores [MB Semi-autoregressive draft: the
// Markov head is a low-rank, token-conditioned additive logit bias]:
//
//   z[b, v] = backbone[b, k-1, v] + sum_j U[x_{k-1}(b), j] * Wm[j, v]
//
// for one step k, all requests b at once: the gather of B rank-r rows of U
// times the r x V matrix, the one dense contraction on the path.  With W
// stored as [V, r] (row v = column v of Wm) both operands are K-major.
//
// tcgen05 (5th-generation tensor cores) with the requests on M:
//   D[128 b, NT v] = U_x[128 b, r] x W_tile[NT v, r]^T
// The gathered rows U_x (one or two 128-request M tiles) are written to shared
// memory once per CTA; W streams through a ring of shared-memory stages by TMA
// (128-byte swizzle when r is a multiple of 64, else a no-swizzle 3-D box that
// lands directly in the canonical core-matrix layout), 4 to 6 tiles ahead.
// Warp roles: one thread of warp 0 issues the TMA loads and the MMAs (after
// the MMAs of tile i it refills the stage of tile i - 1), warps 1..8 drain
// the accumulators, one 32 x 32 block of each tile per warp.  Four
// accumulator buffers in tensor memory let the MMAs run up to three tiles
// ahead of the epilogue.  The W stream starts before the gather, which runs as
// asynchronous 16-byte copies.  Requests are spread over the four
// 32-lane TMEM quadrants so that every epilogue warp has rows; each warp
// transposes its 32 x 32 accumulator blocks through a swizzled shared-memory
// tile, so the backbone loads and z stores run along rows (coalesced); its
// backbone blocks arrive two tiles ahead where shared memory allows.
// Persistent CTAs, one per SM, walk the vocabulary tiles.

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_common.cuh"

namespace dspark {

namespace {

using namespace tc;

constexpr int kThreads = 288;  // a control warp (TMA + MMA issue) and 8 epilogue warps
constexpr int kEpiWarps = 8;
constexpr int kMaxStages = 8;
constexpr int kAcc = 4;              // accumulator buffers in tensor memory
constexpr uint32_t kTmemCols = 256;  // kAcc buffers of mtiles * nt = 64 columns
// Per epilogue warp, for its rpq requests (<= 32): an rpq x 32 fp32 transpose
// tile, element (row, col) at row * 32 + (col ^ row) (conflict-free both ways
// without padding), and nbb buffers for the backbone of its block of the next
// tiles (rpq x 32 each, copied asynchronously).
__host__ __device__ constexpr int epi_warp_bytes(int esz, int rpq, int nbb) { return rpq * 32 * (4 + nbb * esz); }
__host__ __device__ constexpr int epi_bytes(int esz, int rpq, int nbb) {
    return kEpiWarps * epi_warp_bytes(esz, rpq, nbb);
}
// Shared memory per CTA (227 KB opt-in) less an allowance for the static part.
constexpr int kSmemMax = 232448 - 1280;

struct GemmSmem {
    uint64_t full[kMaxStages];   // W stage landed (TMA transaction bytes)
    uint64_t empty[kMaxStages];  // W stage consumed (MMA commit)
    uint64_t acc_full[kAcc];     // accumulator ready (MMA commit)
    uint64_t acc_empty[kAcc];    // accumulator drained (one arrival per epilogue warp)
    uint32_t tmem_base;
    int timeout;
    int32_t x[256];  // x_{k-1} of every request (-1: none)
};

__device__ __forceinline__ void set_timeout(GemmSmem& sm, const MarkovGemmParams& p) {
    atomicExch(&sm.timeout, 1);
    *p.error_flag = 1;
}
__device__ __forceinline__ bool timed_out(const GemmSmem& sm) {
    return *reinterpret_cast<const volatile int*>(&sm.timeout) != 0;
}

template <int kDtype, bool kSw128>
__global__ void __launch_bounds__(kThreads, 1)
    markov_bias_kernel(const __grid_constant__ CUtensorMap wmap, const MarkovGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ GemmSmem sm;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = p.r, mt = p.mtiles, NT = p.nt, S = p.stages;
    const int a_rows = 128;
    const uint32_t a_bytes = static_cast<uint32_t>(a_rows * r * 2);  // one M tile
    const uint32_t w_bytes = static_cast<uint32_t>(NT * r * 2);      // one W stage
    uint8_t* sA = smem;
    uint8_t* sW = smem + mt * a_bytes;
    const int ntiles = (p.V + NT - 1) / NT;

    constexpr int kEsz = kDtype == kBF16 ? 2 : 4;
    uint8_t* stage_epi = sW + S * w_bytes;  // epilogue: per warp a transpose tile, then a backbone buffer
    auto issue_w = [&](int t, int s) {
        mbar_arrive_expect_tx(&sm.full[s], w_bytes);
        uint8_t* dst = sW + s * w_bytes;
        if constexpr (kSw128) {
            for (int kb = 0; kb < r / 64; ++kb) tma_load_2d(dst + kb * NT * 128, &wmap, kb * 64, t * NT, &sm.full[s]);
        } else {
            tma_load_3d(dst, &wmap, 0, t * NT, 0, &sm.full[s]);
        }
    };
    int pre = 0;  // W tiles issued before the gather (they do not depend on it)
    if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kMaxStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        for (int a = 0; a < kAcc; ++a) {
            mbar_init(&sm.acc_full[a], 1);
            mbar_init(&sm.acc_empty[a], kEpiWarps);
        }
        sm.timeout = 0;
        fence_mbar_init();
        for (int t = blockIdx.x; t < ntiles && pre < S; t += gridDim.x, ++pre) issue_w(t, pre);
    }
    // With a programmatic launch behind the previous step's policy kernel, the
    // code above (TMEM, barriers, the first W stages) overlapped its tail;
    // x_{k-1} is read only once that kernel has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // A operand: the gathered rows U[x_{k-1}(b)]; row i of lane quadrant q of
    // M tile m holds request m * 128 + q * rpq + i (i < rpq).  Zero rows past
    // the batch and for failed requests (their rows are ignored downstream).
    const int rpq = p.rpq;
    for (int b = threadIdx.x; b < 256; b += kThreads) {
        int32_t x = -1;
        if (b < p.B) {
            x = p.k == 1 ? p.anchor[b] : p.proposals[b * p.gamma + (p.k - 2)];
            if (x < 0 || x >= p.V) x = -1;
        }
        sm.x[b] = x;
    }
    __syncthreads();
    const int kchunks = r / 8;
    for (int c = threadIdx.x; c < mt * 128 * kchunks; c += kThreads) {
        const int row = c / kchunks, kc = c % kchunks;
        const int m = row >> 7, mr = row & 127, i = mr & 31;
        const int b = m * 128 + (mr >> 5) * rpq + i;
        const int32_t x = (i < rpq && b < p.B) ? sm.x[b] : -1;
        uint8_t* d = sA + m * a_bytes + chunk_off<kSw128>(mr, kc, 128);
        if (x >= 0)
            cp_async16(d, p.U + static_cast<int64_t>(x) * r + kc * 8);
        else
            *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
    }
    // The W stream starts once the gather's few latency-bound reads are on
    // their way (issued first, they do not queue behind S stages of W).
    cp_async_wait_all();
    fence_proxy_async_smem();  // generic and async-copy stores -> visible to the tensor cores
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ control: TMA + MMA issue
        if (lane == 0) {
            const uint32_t idesc = instr_desc(128, NT);
            const uint32_t abase = smem_u32(sA), wbase = smem_u32(sW);
            int i = 0, issued = pre;
            for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
                const int s = i % S, a = i % kAcc;
                if (!mbar_wait(&sm.full[s], (i / S) & 1, kWaitLimitNs) ||
                    (i >= kAcc && !mbar_wait(&sm.acc_empty[a], ((i / kAcc) - 1) & 1, kWaitLimitNs))) {
                    set_timeout(sm, p);
                    break;
                }
                tc_fence_after();
                for (int m = 0; m < mt; ++m) {
                    const uint32_t d = tmem + static_cast<uint32_t>(a * mt * NT + m * NT);
                    for (int ks = 0; ks < r / 16; ++ks)
                        mma_bf16(d, op_desc<kSw128>(abase + m * a_bytes, ks, a_rows),
                                 op_desc<kSw128>(wbase + s * w_bytes, ks, NT), idesc, ks > 0 ? 1u : 0u);
                }
                mma_commit(&sm.empty[s]);
                mma_commit(&sm.acc_full[a]);
                // refill the stage of tile i - 1 (its MMAs were issued one step ago)
                if (i >= 1) {
                    const int j = i - 1;
                    const int tj = blockIdx.x + (j + S) * gridDim.x;
                    if (tj < ntiles) {
                        if (!mbar_wait(&sm.empty[j % S], (j / S) & 1, kWaitLimitNs)) {
                            set_timeout(sm, p);
                            break;
                        }
                        issue_w(tj, j % S);
                        ++issued;
                    }
                }
            }
            // Nothing may still be in flight when the tensor memory is released
            // and the CTA exits: the last MMAs, and (after a timeout) copies.
            if (i > 0 && !mbar_wait(&sm.acc_full[(i - 1) % kAcc], ((i - 1) / kAcc) & 1, kWaitLimitNs))
                set_timeout(sm, p);
            if (timed_out(sm))
                for (int k = max(0, issued - S); k < issued; ++k) mbar_wait(&sm.full[k % S], (k / S) & 1, kWaitLimitNs);
        }
    } else {
        // ------------------------------------------------ epilogue
        // Warp e reads TMEM lane quadrant warp % 4 (its requests): the 64
        // flat columns of a tile (mtiles * nt = 64; flat column f is M tile
        // f / nt, column f % nt) split into two 32-column blocks, block e / 4
        // for this warp.  The accumulator block goes to a swizzled shared
        // tile, then each of the block's requests is written along its row
        // (lane = column) with the backbone added.
        const int e = warp - 1;
        const int quad = warp & 3;
        const int f0 = 32 * (e >> 2);
        const int m = f0 / NT, c0 = f0 % NT;
        const int b0 = m * 128 + quad * rpq;             // first request of the block
        const int nrows = max(0, min(rpq, p.B - b0));   // its valid requests
        const int nbb = p.nbb;
        uint8_t* wbase_epi = stage_epi + e * epi_warp_bytes(kEsz, rpq, nbb);
        float* T = reinterpret_cast<float*>(wbase_epi);
        // [nbb][row][32 columns] of the backbone: tile i's block in buffer i % nbb
        uint8_t* bbuf0 = wbase_epi + rpq * 32 * 4;
        const size_t esz = kEsz;
        const char* bb = static_cast<const char*>(p.backbone) + static_cast<size_t>(p.k - 1) * p.V * esz;
        const size_t bb_stride = static_cast<size_t>(p.gamma) * p.V * esz;  // one request
        // Asynchronous copy of the block's backbone of tile t into bbuf, in
        // 16-byte pieces (4 or 8 lanes per row); one commit group per tile.
        auto fetch_bb = [&](int t, uint8_t* bbuf) {
            constexpr int kLanesPerRow = 32 * kEsz / 16;
            constexpr int kRowsPerStep = 32 / kLanesPerRow;
            const int piece = lane % kLanesPerRow;
            const int col = t * NT + c0 + piece * (16 / kEsz);
#pragma unroll
            for (int st = 0; st < 32 / kRowsPerStep; ++st) {
                const int rr = st * kRowsPerStep + lane / kLanesPerRow;
                if (rr < nrows && col < p.V)
                    cp_async16(bbuf + rr * 32 * kEsz + piece * 16,
                               bb + static_cast<size_t>(b0 + rr) * bb_stride + static_cast<size_t>(col) * esz);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        };
        int i = 0;
        if (nrows > 0) {
            for (int q = 0; q < nbb; ++q) {
                const int tq = blockIdx.x + q * static_cast<int>(gridDim.x);
                if (tq < ntiles) fetch_bb(tq, bbuf0 + q * rpq * 32 * kEsz);
                else asm volatile("cp.async.commit_group;" ::: "memory");  // keep one group per tile
            }
        }
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int a = i % kAcc;
            uint8_t* bbuf = bbuf0 + (i % nbb) * rpq * 32 * kEsz;
            if (!mbar_wait(&sm.acc_full[a], (i / kAcc) & 1, kWaitLimitNs)) {
                set_timeout(sm, p);
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                break;
            }
            if (timed_out(sm)) {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
                break;
            }
            tc_fence_after();
            if (nrows > 0) {
                uint32_t acc[32];
                tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) +
                              static_cast<uint32_t>(a * mt * NT + m * NT + c0),
                          acc);
                tmem_wait_ld();
                // this tile's backbone is in bbuf (the next tile's may still be in flight)
                if (nbb == 2) asm volatile("cp.async.wait_group 1;" ::: "memory");
                else asm volatile("cp.async.wait_group 0;" ::: "memory");
                if (lane < rpq) {  // lanes past rpq hold no request
#pragma unroll
                    for (int j = 0; j < 32; ++j) T[lane * 32 + (j ^ lane)] = __uint_as_float(acc[j]);
                }
                __syncwarp();
                const int v = t * NT + c0 + lane;
                float* zrow = p.zbuf + static_cast<size_t>(b0) * p.V + v;
#pragma unroll 4
                for (int rr = 0; rr < nrows; ++rr, zrow += p.V) {
                    if (v < p.V) {
                        float x;
                        if constexpr (kDtype == kBF16)
                            x = __uint_as_float(static_cast<uint32_t>(
                                    reinterpret_cast<const uint16_t*>(bbuf)[rr * 32 + lane]) << 16);
                        else
                            x = reinterpret_cast<const float*>(bbuf)[rr * 32 + lane];
                        *zrow = x + T[rr * 32 + (lane ^ rr)];
                    }
                }
                __syncwarp();
                // the backbone nbb tiles ahead streams in while the accumulators are computed
                const int tn = t + nbb * static_cast<int>(gridDim.x);
                if (tn < ntiles) fetch_bb(tn, bbuf);
                else asm volatile("cp.async.commit_group;" ::: "memory");
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.acc_empty[a]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ host
int smem_bytes(const MarkovGemmParams& p) {
    return p.mtiles * 128 * p.r * 2 + p.stages * p.nt * p.r * 2 +
           epi_bytes(p.dtype == kBF16 ? 2 : 4, p.rpq, p.nbb) + 1024;  // + alignment slack
}

template <int kDtype, bool kSw128>
cudaError_t launch_one(const MarkovGemmParams& p, const CUtensorMap& map, bool overlap, cudaStream_t stream) {
    const int smem = smem_bytes(p);
    cudaError_t e =
        cudaFuncSetAttribute(markov_bias_kernel<kDtype, kSw128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (overlap) {  // may start while the preceding kernel finishes (it waits before reading its outputs)
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    e = cudaLaunchKernelEx(&cfg, markov_bias_kernel<kDtype, kSw128>, map, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

bool prepare_markov_bias(MarkovGemmParams& p, MarkovGemmPlan& plan) {
    if (p.B < 1 || p.B > 256 || p.r < 16 || p.r > 256 || p.r % 16 != 0) return false;
    p.mtiles = (p.B + 127) / 128;
    p.nt = 64 / p.mtiles;
    const int a = p.mtiles * 128 * p.r * 2, w = p.nt * p.r * 2;
    p.rpq = p.mtiles == 1 ? (p.B + 3) / 4 : 32;
    // two backbone buffers per epilogue warp where they leave three W stages, else one
    const int esz = p.dtype == kBF16 ? 2 : 4;
    for (p.nbb = 2; p.nbb >= 1; --p.nbb) {
        const int budget = kSmemMax - epi_bytes(esz, p.rpq, p.nbb) - 1024;  // A + W stages
        p.stages = std::min(kMaxStages, (budget - a) / w);
        if (p.stages >= 3 || (p.nbb == 1 && p.stages >= 2)) break;
    }
    if (p.nbb < 1 || p.stages < 2) return false;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return false;
    const int ntiles = (p.V + p.nt - 1) / p.nt;
    p.grid = std::min(sms, ntiles);

    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return false;
    CUtensorMap* map = reinterpret_cast<CUtensorMap*>(plan.tmap);
    plan.sw128 = p.r % 64 == 0;
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult res;
    if (plan.sw128) {  // [V, r] as 2-D: boxes of 64 columns (128 B) x nt rows, 128-byte swizzle
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.r), static_cast<cuuint64_t>(p.V)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.r) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(p.nt)};
        res = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(p.W), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {  // (8 elements, V rows, r/8 chunks): one box = nt rows in k-chunk-major core-matrix order
        const cuuint64_t dims[3] = {8, static_cast<cuuint64_t>(p.V), static_cast<cuuint64_t>(p.r / 8)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.r) * 2, 16};
        const cuuint32_t box[3] = {8, static_cast<cuuint32_t>(p.nt), static_cast<cuuint32_t>(p.r / 8)};
        res = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(p.W), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return res == CUDA_SUCCESS;
}

cudaError_t launch_markov_bias(const MarkovGemmParams& p, const MarkovGemmPlan& plan, bool overlap,
                               cudaStream_t stream) {
    const CUtensorMap& map = *reinterpret_cast<const CUtensorMap*>(plan.tmap);
    if (p.dtype == kBF16)
        return plan.sw128 ? launch_one<kBF16, true>(p, map, overlap, stream)
                          : launch_one<kBF16, false>(p, map, overlap, stream);
    return plan.sw128 ? launch_one<kF32, true>(p, map, overlap, stream)
                      : launch_one<kF32, false>(p, map, overlap, stream);
}

}  // namespace dspark
