// Greedy paths: the arg-max of every logit row of a request and the
// request's decision, in one launch and one pass over the logits.
//
//  * Greedy verify [FT Exact decoding semantics > Greedy; PT Speculative
//    decoding (K=7) > Acceptance]: a_i = argmax of target row i (lowest index
//    on ties); n = length of the prefix with x_k == a_{k-1}; emit x_1..x_n
//    then a_n.  The width variant (kWidth) checks x_1..x_w of each request
//    (w = its width, 0..gamma): only rows 0..w are streamed and the prefix
//    stops at w.
//  * Greedy drafting without a Markov bias (r = 0): x_k = argmax of backbone
//    row k.
//
// Work split: one thread-block cluster of C CTAs per request (C = 1, 2, 4 or
// 8, the largest that keeps every cluster resident in one wave).  The rows of
// a request are contiguous, so its CTAs take equal contiguous ranges of them.
// In each CTA one producer lane streams the range through a ring of
// shared-memory stages with TMA bulk copies (full / empty mbarriers per
// stage, no CTA-wide barrier in the loop), so the bytes in flight per SM are
// set by the ring, not by registers.  Consumer threads take the packed
// NaN-propagating maximum of the vectors they read from a stage (about one
// instruction per element) and, only when that beats their running best,
// look up the lowest index holding it in the registers they already have.
// Per-thread results are 64-bit keys (ordered value << 32 | ~index) merged
// with atomicMax (max value, then lowest index) into the CTA's row slots;
// each CTA then writes its slots into those of the cluster's first CTA over
// distributed shared memory, a cluster barrier publishes them, and the first
// CTA makes the request's decision with one lane per row.  Nothing goes
// through global memory but the logits and the outputs, so the kernel needs
// no workspace.

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + the producer warp
constexpr int kCtasPerSm = 2;
constexpr int kStages = 3;
constexpr int kStageBytes = 32768;  // two CTAs per SM: 192 KB in flight
constexpr int kVecPerStage = kStageBytes / 16;
constexpr int kVecPerThread = kVecPerStage / kConsumers;
constexpr int kRingBytes = kStages * kStageBytes;
constexpr int kMaxRows = 32;  // rows of one request (gamma + 1 <= 17)
constexpr int kMaxCluster = 8;

struct ArgmaxSmem {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    unsigned long long key[kMaxRows];
    unsigned int bad[kMaxRows];  // bit 0: NaN / +inf seen; bit 1: a device wait gave up
    unsigned int timed_out;
    int32_t x[kMaxRows];  // first CTA: the proposals (verify) or the anchor (drafting)
    // first CTA of the cluster: the row slots of every CTA, written remotely
    unsigned long long rkey[kMaxCluster][kMaxRows];
    unsigned int rbad[kMaxCluster][kMaxRows];
};

__device__ __forceinline__ uint64_t make_key(float v, int64_t idx) {
    return (static_cast<uint64_t>(ordered_key(v)) << 32) |
           static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

// Row status from the merged key and flags, in the oracle's order:
// non-finite first, then empty (every logit -inf).
__device__ __forceinline__ int32_t row_status(uint64_t key, uint32_t flags) {
    if (flags & 2u) return kReqTimeout;
    if (flags & 1u) return kReqNonfinite;
    if (key == 0) return kReqEmpty;
    if (key_to_float(static_cast<uint32_t>(key >> 32)) == -__int_as_float(0x7F800000)) return kReqEmpty;
    return kReqOk;
}
__device__ __forceinline__ int32_t key_index(uint64_t key) {
    return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(key));
}

// ------------------------------------------------ cluster-scope primitives
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}
// The shared::cluster address of `p` in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t map_rank(const void* p, uint32_t rank) {
    uint32_t a;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
    return a;
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, uint64_t v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------- the decision
// All 32 lanes of one warp; lane i < G holds row i's merged key k and flags
// f; for verify lane k < gamma holds the proposal x_{k+1}, for drafting every
// lane holds the anchor.  kWidth: the request checks x_1..x_w (rows 0..w were
// read); a width outside [0, gamma] fails it as a bad token.
template <bool kWidth>
__device__ void decide(const ArgmaxParams& p, int64_t g, int w, uint64_t k, uint32_t f, int32_t x, int lane) {
    const int G = p.rows_per_group;
    const int gamma = p.gamma;
    bool w_ok = true;
    int live = G;  // rows whose status counts
    if constexpr (kWidth) {
        w_ok = w >= 0 && w <= gamma;
        live = w_ok ? w + 1 : 0;
    } else {
        w = gamma;
    }
    const int32_t st = lane < live ? row_status(k, f) : kReqOk;
    const int32_t a = key_index(k);
    const unsigned badrow = __ballot_sync(0xFFFFFFFFu, lane < live && st != kReqOk);

    if (p.mode == kArgmaxVerify) {
        int32_t* out = p.out_tokens + g * (gamma + 1);
        const unsigned badtok = __ballot_sync(0xFFFFFFFFu, lane < w && (x < 0 || x >= p.V));
        int32_t status = kReqOk;
        if (!w_ok || badtok) status = kReqBadToken;
        else if (badrow) status = __shfl_sync(0xFFFFFFFFu, st, __ffs(badrow) - 1);
        if (status != kReqOk) {
            if (lane <= gamma) out[lane] = -1;
            if (lane == 0) {
                p.num_accepted[g] = -1;
                p.status[g] = status;
            }
            return;
        }
        // accepted prefix: the first k with x_k != a_{k-1} ends it
        const unsigned mismatch = __ballot_sync(0xFFFFFFFFu, lane < w && x != a);
        const int n = mismatch ? __ffs(mismatch) - 1 : w;
        const int32_t an = __shfl_sync(0xFFFFFFFFu, a, n);
        if (lane <= gamma) out[lane] = lane < n ? x : (lane == n ? an : -1);
        if (lane == 0) {
            p.num_accepted[g] = n;
            p.status[g] = kReqOk;
        }
    } else {  // greedy drafting, r = 0: group = the gamma backbone rows of request g
        const bool bad_anchor = x < 0 || x >= p.V;
        const int first_bad = bad_anchor ? 0 : (badrow ? __ffs(badrow) - 1 : gamma);
        const int32_t status =
            bad_anchor ? kReqBadToken : (badrow ? __shfl_sync(0xFFFFFFFFu, st, first_bad) : kReqOk);
        if (lane < gamma) {
            const bool ok = lane < first_bad;
            p.props_out[g * gamma + lane] = ok ? a : -1;
            p.q_at_x[g * gamma + lane] = ok ? 1.0f : 0.0f;
        }
        if (lane == 0) p.status[g] = status;
    }
}

// ------------------------------------------------------- streaming arg-max
__device__ __forceinline__ uint32_t bf16x2_max_nan(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Running arg-max of one row segment held by one thread.
struct RowAcc {
    float best;    // largest value seen, -inf if none
    int32_t bidx;  // row-relative index of its first occurrence, -1 if none
    bool bad;      // a NaN or +inf was seen

    __device__ __forceinline__ void reset() {
        best = -__int_as_float(0x7F800000);
        bidx = -1;
        bad = false;
    }
    __device__ __forceinline__ uint64_t key() const { return bidx >= 0 ? make_key(best, bidx) : 0ull; }
};

// Packed maximum of one 16-byte vector (8 bf16 or 4 fp32), NaN-propagating.
template <int kDtype>
__device__ __forceinline__ float vec_max(const uint4& v) {
    if constexpr (kDtype == kBF16) {
        const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(v.x, v.y), bf16x2_max_nan(v.z, v.w));
        return fmax_nan(bf16_lo(m), bf16_hi(m));
    } else {
        return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                        fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
}
template <int kDtype>
__device__ __forceinline__ float vec_elem(const uint4& v, int l) {
    const uint32_t w = l < (kDtype == kBF16 ? 2 : 1) ? v.x : l < (kDtype == kBF16 ? 4 : 2) ? v.y
                     : l < (kDtype == kBF16 ? 6 : 3) ? v.z : v.w;
    if constexpr (kDtype == kBF16) return (l & 1) ? bf16_hi(w) : bf16_lo(w);
    else return __uint_as_float(w);
}

// Fold one 16-byte vector, the `rv`-th vector of its row, into an
// accumulator; vm = its packed maximum.
template <int kDtype>
__device__ __forceinline__ void fold_vector(RowAcc& acc, const uint4& v, float vm, uint32_t rv) {
    constexpr int kPer = kDtype == kBF16 ? 8 : 4;
    if (bad_logit(vm)) {
        acc.bad = true;
    } else if (vm > acc.best) {  // ties keep the earlier (lower-index) occurrence
        acc.best = vm;
        int l0 = kPer - 1;
#pragma unroll
        for (int l = kPer - 1; l >= 0; --l)
            if (vec_elem<kDtype>(v, l) == vm) l0 = l;
        acc.bidx = static_cast<int32_t>(rv * kPer + l0);
    }
}

// NaN-propagating maximum of a thread's vectors of one stage: a packed
// running maximum per 32-bit lane (one max per 4 bytes), reduced at the end.
// Vectors past the stage's end hold -inf.
template <int kDtype>
__device__ __forceinline__ float stage_max(const uint4 (&v)[kVecPerThread]) {
    if constexpr (kDtype == kBF16) {
        uint32_t m0 = v[0].x, m1 = v[0].y, m2 = v[0].z, m3 = v[0].w;
#pragma unroll
        for (int u = 1; u < kVecPerThread; ++u) {
            m0 = bf16x2_max_nan(m0, v[u].x);
            m1 = bf16x2_max_nan(m1, v[u].y);
            m2 = bf16x2_max_nan(m2, v[u].z);
            m3 = bf16x2_max_nan(m3, v[u].w);
        }
        const uint32_t m = bf16x2_max_nan(bf16x2_max_nan(m0, m1), bf16x2_max_nan(m2, m3));
        return fmax_nan(bf16_lo(m), bf16_hi(m));
    } else {
        float m0 = __uint_as_float(v[0].x), m1 = __uint_as_float(v[0].y);
        float m2 = __uint_as_float(v[0].z), m3 = __uint_as_float(v[0].w);
#pragma unroll
        for (int u = 1; u < kVecPerThread; ++u) {
            m0 = fmax_nan(m0, __uint_as_float(v[u].x));
            m1 = fmax_nan(m1, __uint_as_float(v[u].y));
            m2 = fmax_nan(m2, __uint_as_float(v[u].z));
            m3 = fmax_nan(m3, __uint_as_float(v[u].w));
        }
        return fmax_nan(fmax_nan(m0, m1), fmax_nan(m2, m3));
    }
}

// A finite stage maximum cm beat the running best: record its first
// occurrence.  The thread's vectors are rv0, rv0 + kConsumers, ... of the
// row, so the first vector holding cm has the lowest index.
template <int kDtype>
__device__ __forceinline__ void record(RowAcc& acc, const uint4 (&v)[kVecPerThread], float cm, uint32_t rv0) {
    constexpr int kPer = kDtype == kBF16 ? 8 : 4;
    int uf = kVecPerThread - 1;
#pragma unroll
    for (int u = kVecPerThread - 1; u >= 0; --u)
        if (vec_max<kDtype>(v[u]) == cm) uf = u;
    uint4 w = v[0];
#pragma unroll
    for (int u = 1; u < kVecPerThread; ++u)
        if (u == uf) w = v[u];
    int l0 = kPer - 1;
#pragma unroll
    for (int l = kPer - 1; l >= 0; --l)
        if (vec_elem<kDtype>(w, l) == cm) l0 = l;
    acc.best = cm;
    acc.bidx = static_cast<int32_t>((rv0 + static_cast<uint32_t>(uf) * kConsumers) * kPer + l0);
}

// Merge one thread's accumulator of request row `slot` into the CTA's row
// slots (slot < 0: nothing accumulated yet).
__device__ __forceinline__ void flush_row(ArgmaxSmem& sm, const RowAcc& acc, int64_t slot) {
    if (slot < 0) return;
    const uint64_t k = acc.key();
    if (k) atomicMax(&sm.key[slot], static_cast<unsigned long long>(k));
    if (acc.bad) atomicOr(&sm.bad[slot], 1u);
}

// The stages of a CTA's range [v, v_hi) (vector indices), in order.  When a
// row spans at least a whole stage, stages are cut at row ends so that every
// stage lies in one row; shorter rows share stages.  The producer and every
// consumer walk the same sequence.
struct StageWalk {
    int64_t v, v_hi, vpr, rend;
    bool split;
    __device__ __forceinline__ StageWalk(int64_t lo, int64_t hi, int64_t vpr_)
        : v(lo), v_hi(hi), vpr(vpr_), rend((lo / vpr_ + 1) * vpr_), split(vpr_ >= kVecPerStage) {}
    __device__ __forceinline__ bool more() const { return v < v_hi; }
    // Vectors in the stage starting at v.
    __device__ __forceinline__ int count() {
        int64_t n = min(static_cast<int64_t>(kVecPerStage), v_hi - v);
        if (split) {
            if (v >= rend) rend += vpr;
            n = min(n, rend - v);
        }
        return static_cast<int>(n);
    }
};

template <bool kWidth>
using ArgmaxArgs = std::conditional_t<kWidth, ArgmaxWidthParams, ArgmaxParams>;

template <int kDtype, bool kWidth>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) argmax_rows_kernel(const ArgmaxArgs<kWidth> p) {
    extern __shared__ __align__(128) uint8_t ring[];
    __shared__ ArgmaxSmem sm;
    constexpr int kPer = kDtype == kBF16 ? 8 : 4;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t C = cluster_size(), q = cluster_rank();
    const int64_t g = blockIdx.x / C;  // the request
    const int G = p.rows_per_group;
    const int64_t V = p.V;
    const int64_t glen = static_cast<int64_t>(G) * V;
    // elements of the request that are read: every row, or rows 0..w of the
    // width variant (none for an invalid width)
    int w = 0;
    int64_t gread = glen;
    if constexpr (kWidth) {
        w = p.width[g];
        gread = w >= 0 && w <= p.gamma ? static_cast<int64_t>(w + 1) * V : 0;
    }
    const int64_t lo = min(gread, static_cast<int64_t>(q) * p.per);  // request-relative element range
    const int64_t hi = min(gread, lo + p.per);
    const int64_t vpr = V / kPer;    // vectors per row (V is a multiple of 8)
    const int64_t v_lo = lo / kPer;  // request-relative vector index of the range start
    const int64_t v_hi = hi / kPer;
    const char* src = static_cast<const char*>(p.logits) + g * glen * (kDtype == kBF16 ? 2 : 4);

    if (tid < kMaxRows) {
        sm.key[tid] = 0ull;
        sm.bad[tid] = 0u;
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        sm.timed_out = 0u;
        fence_mbar_init();
    }
    __syncthreads();
    // Every CTA's slots and barriers are initialised before any CTA of the
    // cluster touches them remotely (the matching wait is at the end).
    cluster_arrive_release();

    if (warp == kConsumerWarps) {
        // The first CTA's idle producer lanes fetch the proposals (or the
        // anchor) for the decision now, off the critical path.
        if (q == 0 && lane > 0) {
            const int k = lane - 1;
            if (p.mode == kArgmaxVerify) {
                if (k < p.gamma) sm.x[k] = p.proposals[g * p.gamma + k];
            } else if (k == 0) {
                sm.x[0] = p.anchor[g];
            }
        }
        // ------------------------------------------------ producer (one lane)
        if (lane == 0) {
            int issued = 0;
            for (StageWalk w(v_lo, v_hi, vpr); w.more(); ++issued) {
                const int s = issued % kStages;
                if (issued >= kStages &&
                    !mbar_wait(&sm.empty[s], ((issued / kStages) - 1) & 1, kWaitLimitNs)) {
                    atomicOr(&sm.timed_out, 1u);
                    break;
                }
                const int nv = w.count();
                mbar_arrive_expect_tx(&sm.full[s], static_cast<uint32_t>(nv) * 16u);
                bulk_g2s(ring + s * kStageBytes, src + w.v * 16, static_cast<uint32_t>(nv) * 16u, &sm.full[s]);
                w.v += nv;
            }
            // No copy may still be landing when the CTA exits: wait (bounded)
            // for the last copy issued into every stage.
            for (int c = max(0, issued - kStages); c < issued; ++c)
                if (!mbar_wait(&sm.full[c % kStages], (c / kStages) & 1, kWaitLimitNs)) atomicOr(&sm.timed_out, 1u);
        }
    } else {
        // ------------------------------------------------------- consumers
        const uint4 neg = kDtype == kBF16 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                          : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
        RowAcc acc;
        acc.reset();
        int64_t arow = -1, astart = 0, aend = 0;          // this thread's accumulator row and its vectors
        int64_t crow = -1, crow_start = 0, crow_end = 0;  // row holding the current stage's first vector
        StageWalk w(v_lo, v_hi, vpr);
        for (int c = 0; w.more(); ++c) {
            const int s = c % kStages;
            if (!mbar_wait(&sm.full[s], (c / kStages) & 1, kWaitLimitNs)) {
                atomicOr(&sm.timed_out, 1u);
                break;
            }
            const int64_t cv0 = w.v;
            const int nv = w.count();
            w.v += nv;
            const uint8_t* stage = ring + s * kStageBytes;
            uint4 v[kVecPerThread];
#pragma unroll
            for (int u = 0; u < kVecPerThread; ++u) {
                const int j = tid + u * kConsumers;
                v[u] = j < nv ? ld_shared_v4(stage + j * 16) : neg;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);  // the stage's data is in registers now

            if (cv0 >= crow_end) {
                crow = cv0 / vpr;
                crow_start = crow * vpr;
                crow_end = crow_start + vpr;
            }
            if (cv0 + nv <= crow_end) {  // the whole stage lies in one row
                if (arow != crow) {
                    flush_row(sm, acc, arow);
                    acc.reset();
                    arow = crow;
                    astart = crow_start;
                    aend = crow_end;
                }
                // The stage lies in one row for the whole warp, so records are
                // decided warp-wide: only a stage maximum above every lane's
                // best so far (all at lower indices) can be the row's first
                // maximum.  This keeps the divergent record path rare.
                const float cm = stage_max<kDtype>(v);
                const bool bad = bad_logit(cm);
                if (__any_sync(0xFFFFFFFFu, bad)) {  // the row is non-finite: its arg-max is not needed
                    acc.bad |= bad;
                } else {
                    const uint32_t k = ordered_key(cm);
                    const uint32_t wk = __reduce_max_sync(0xFFFFFFFFu, k);
                    if (wk > __reduce_max_sync(0xFFFFFFFFu, ordered_key(acc.best)) && k == wk)
                        record<kDtype>(acc, v, cm, static_cast<uint32_t>(cv0 + tid - astart));
                }
            } else {  // row boundaries inside the stage
#pragma unroll
                for (int u = 0; u < kVecPerThread; ++u) {
                    const int j = tid + u * kConsumers;
                    if (j >= nv) continue;
                    const int64_t vi = cv0 + j;
                    if (vi >= aend) {
                        flush_row(sm, acc, arow);
                        acc.reset();
                        arow = vi / vpr;
                        astart = arow * vpr;
                        aend = astart + vpr;
                    }
                    fold_vector<kDtype>(acc, v[u], vec_max<kDtype>(v[u]), static_cast<uint32_t>(vi - astart));
                }
            }
        }
        flush_row(sm, acc, arow);
    }
    __syncthreads();
    cluster_wait_acquire();

    // Hand this CTA's row slots to the first CTA of the cluster (distributed
    // shared memory), then one cluster barrier: its release orders the remote
    // stores before the first CTA's reads, and no CTA exits while another may
    // still write into its shared memory.  Every wait before the barrier is
    // bounded, so every thread of the cluster reaches it.
    if (warp == 0) {
        const unsigned tflag = sm.timed_out ? 2u : 0u;
        if (lane < G) {
            st_cluster_u64(map_rank(&sm.rkey[q][lane], 0), sm.key[lane]);
            st_cluster_u32(map_rank(&sm.rbad[q][lane], 0), sm.bad[lane] | tflag);
        }
    }
    cluster_arrive_release();
    cluster_wait_acquire();
    if (warp == 0 && q == 0) {
        uint64_t k = 0;
        uint32_t f = 0u;
        if (lane < G) {
            for (uint32_t r = 0; r < C; ++r) {
                const uint64_t kr = sm.rkey[r][lane];
                k = kr > k ? kr : k;
                f |= sm.rbad[r][lane];
            }
        }
        const int32_t x = p.mode == kArgmaxVerify ? (lane < p.gamma ? sm.x[lane] : 0) : sm.x[0];
        decide<kWidth>(p, g, w, k, f, x, lane);
    }
}

template <int kDtype, bool kWidth = false>
const void* kernel_ptr() {
    return reinterpret_cast<const void*>(&argmax_rows_kernel<kDtype, kWidth>);
}

// Opt the kernels into the ring's dynamic shared memory (once per device).
cudaError_t prepare_argmax(int dtype, bool width = false) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // per device, dtype and variant; host threads may race here, so the flags
    // are atomic (setting the attribute twice is harmless)
    static std::atomic<bool> ready[64][2][2] = {};
    if (dev < 64 && ready[dev][dtype][width].load(std::memory_order_acquire)) return cudaSuccess;
    const void* f = width ? (dtype == kBF16 ? kernel_ptr<kBF16, true>() : kernel_ptr<kF32, true>())
                          : (dtype == kBF16 ? kernel_ptr<kBF16>() : kernel_ptr<kF32>());
    e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kRingBytes);
    if (e == cudaSuccess && dev < 64) ready[dev][dtype][width].store(true, std::memory_order_release);
    return e;
}

cudaLaunchConfig_t launch_config(int clusters, int c, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(clusters) * c);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kRingBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Clusters of `c` CTAs that can be resident at once (0 if the query fails).
int resident_clusters(int dtype, int c) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static std::atomic<int> cache[64][2][4] = {};  // 0: not yet queried (atomic: host threads may race)
    const int ci = c == 1 ? 0 : c == 2 ? 1 : c == 4 ? 2 : 3;
    if (dev < 64) {
        const int n = cache[dev][dtype][ci].load(std::memory_order_acquire);
        if (n) return n;
    }
    if (prepare_argmax(dtype) != cudaSuccess) return 0;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(64, c, nullptr, attr);
    int n = 0;
    const void* f = dtype == kBF16 ? kernel_ptr<kBF16>() : kernel_ptr<kF32>();
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) return 0;
    if (dev < 64) cache[dev][dtype][ci].store(n, std::memory_order_release);
    return n;
}

}  // namespace

int argmax_cluster_size(int dtype, int groups) {
    int c = 8;
    while (c > 1) {
        const int n = resident_clusters(dtype, c);
        if (n > 0 && groups <= n) break;
        c /= 2;
    }
    return c;
}

cudaError_t launch_argmax_rows(ArgmaxParams p, int groups, cudaStream_t stream, const int32_t* width) {
    if (groups <= 0) return cudaSuccess;
    if (p.rows_per_group < 1 || p.rows_per_group > kMaxRows || p.gamma < 1 || p.gamma > kMaxRows - 2)
        return cudaErrorInvalidValue;
    if (width && p.mode != kArgmaxVerify) return cudaErrorInvalidValue;
    cudaError_t e = prepare_argmax(p.dtype);
    if (e == cudaSuccess && width) e = prepare_argmax(p.dtype, true);
    if (e != cudaSuccess) return e;
    const int c = argmax_cluster_size(p.dtype, groups);
    const int64_t glen = static_cast<int64_t>(p.rows_per_group) * p.V;
    p.per = ((glen + c - 1) / c + 7) / 8 * 8;  // elements per CTA: ranges start on 16-byte boundaries
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = launch_config(groups, c, stream, attr);
    if (width) {
        ArgmaxWidthParams pw;
        static_cast<ArgmaxParams&>(pw) = p;
        pw.width = width;
        if (p.dtype == kBF16)
            e = cudaLaunchKernelEx(&cfg, argmax_rows_kernel<kBF16, true>, pw);
        else
            e = cudaLaunchKernelEx(&cfg, argmax_rows_kernel<kF32, true>, pw);
    } else if (p.dtype == kBF16) {
        e = cudaLaunchKernelEx(&cfg, argmax_rows_kernel<kBF16, false>, p);
    } else {
        e = cudaLaunchKernelEx(&cfg, argmax_rows_kernel<kF32, false>, p);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark
