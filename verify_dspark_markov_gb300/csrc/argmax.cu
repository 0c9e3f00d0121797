// Greedy paths: a flat-split row argmax over contiguous logit rows, and the
// per-request decisions built on it.
//
//  * Greedy verify [FT Exact decoding semantics > Greedy; PT Speculative
//    decoding (K=7) > Acceptance]: a_i = argmax of target row i (lowest index
//    on ties); n = length of the prefix with x_k == a_{k-1}; emit x_1..x_n
//    then a_n.
//  * Greedy drafting without a Markov bias (r = 0): x_k = argmax of backbone
//    row k.
//
// Work split: the rows of one call are contiguous, so the launch treats them
// as one flat array and gives every CTA an equal contiguous range of it (all
// CTAs resident in one wave).  Each thread streams its share with eight
// 16-byte loads in flight, takes the packed NaN-propagating maximum of each
// batch (about one instruction per element) and, only when a batch beats its
// running best, looks up the lowest index holding it in the registers it
// already has.  At the end of a row segment the CTA reduces to a 64-bit key
// (ordered value << 32 | ~index) and merges it into the row's key with
// atomicMax (max value, then lowest index).  After finishing its part of a
// request the CTA takes a ticket; the CTA that takes the last ticket of a
// request makes that request's decision with one lane per row and returns
// the request's counters to zero.  One launch, one pass over the logits.

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kThreads = 256;
constexpr int kBatch = 8;          // 16-byte loads in flight per thread
constexpr int kMinBlocksPerSM = 4;

__device__ __forceinline__ uint64_t make_key(float v, int64_t idx) {
    return (static_cast<uint64_t>(ordered_key(v)) << 32) |
           static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(idx));
}

// Row status from the merged key and flags, in the oracle's order:
// non-finite first, then empty (every logit -inf).  Flag bit 1 = a device
// wait of this row's CTA timed out.
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

// Called by all 32 lanes of warp 0 once this CTA has merged its share of
// request g: take the request's ticket and, if it is the last one, make the
// request's decision with one lane per row (G <= 17 rows) and return the
// request's counters to zero.
__device__ void ticket_and_finalize(const ArgmaxParams& p, int64_t g, unsigned expected, int lane) {
    unsigned old = 0;
    if (lane == 0) old = atom_add_acq_rel(p.ticket + g, 1u);
    old = __shfl_sync(0xFFFFFFFFu, old, 0);
    if (old != expected - 1) return;
    fence_acq_rel_gpu();

    const int G = p.rows_per_group;
    const int gamma = p.gamma;
    uint64_t k = 0;
    uint32_t f = 0;
    if (lane < G) {
        k = ld_relaxed_u64(p.rowkey + g * G + lane);
        f = ld_relaxed_u32(p.rowbad + g * G + lane);
    }
    const int32_t st = lane < G ? row_status(k, f) : kReqOk;
    const int32_t a = key_index(k);
    if (lane < G) {  // leave the workspace zero-filled for the next call
        p.rowkey[g * G + lane] = 0ull;
        p.rowbad[g * G + lane] = 0u;
    }
    if (lane == 0) p.ticket[g] = 0u;
    const unsigned badrow = __ballot_sync(0xFFFFFFFFu, lane < G && st != kReqOk);

    if (p.mode == kArgmaxVerify) {
        int32_t* out = p.out_tokens + g * (gamma + 1);
        const int32_t x = lane < gamma ? p.proposals[g * gamma + lane] : 0;
        const unsigned badtok = __ballot_sync(0xFFFFFFFFu, lane < gamma && (x < 0 || x >= p.V));
        int32_t status = kReqOk;
        if (badtok) status = kReqBadToken;
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
        const unsigned mismatch = __ballot_sync(0xFFFFFFFFu, lane < gamma && x != a);
        const int n = mismatch ? __ffs(mismatch) - 1 : gamma;
        const int32_t an = __shfl_sync(0xFFFFFFFFu, a, n);
        if (lane <= gamma) out[lane] = lane < n ? x : (lane == n ? an : -1);
        if (lane == 0) {
            p.num_accepted[g] = n;
            p.status[g] = kReqOk;
        }
    } else {  // greedy drafting, r = 0: group = the gamma backbone rows of request g
        const int32_t anchor = p.anchor[g];
        const bool bad_anchor = anchor < 0 || anchor >= p.V;
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

// Fold one 16-byte vector (flat vector index `vi`, whose row starts at flat
// element `row_base`) into an accumulator; vm = its packed maximum.
template <int kDtype>
__device__ __forceinline__ void fold_vector(RowAcc& acc, const uint4& v, float vm, int64_t vi,
                                            int64_t row_base) {
    constexpr int kPer = kDtype == kBF16 ? 8 : 4;
    if (bad_logit(vm)) {
        acc.bad = true;
    } else if (vm > acc.best) {  // ties keep the earlier (lower-index) occurrence
        acc.best = vm;
        int l0 = kPer - 1;
#pragma unroll
        for (int l = kPer - 1; l >= 0; --l)
            if (vec_elem<kDtype>(v, l) == vm) l0 = l;
        acc.bidx = static_cast<int32_t>(vi * kPer + l0 - row_base);
    }
}

constexpr int kSlots = 2;  // rows one CTA folds at a time without a barrier

template <int kDtype>
__global__ void __launch_bounds__(kThreads, kMinBlocksPerSM) argmax_rows_kernel(const ArgmaxParams p) {
    __shared__ uint64_t s_key[kSlots][kThreads / 32];
    __shared__ uint32_t s_bad[kSlots][kThreads / 32];
    constexpr int kPer = kDtype == kBF16 ? 8 : 4;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t lo = static_cast<int64_t>(blockIdx.x) * p.chunk;
    const int64_t hi = min(lo + p.chunk, p.total);
    if (lo >= hi) return;
    const int64_t V = p.V;
    const int64_t gsize = static_cast<int64_t>(p.rows_per_group) * V;
    const char* src = static_cast<const char*>(p.logits);
    const uint4 neg = kDtype == kBF16 ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                      : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);

    // Rows [w0, w0 + kSlots) at a time.  When V exceeds the CTA's range there
    // is a single window, so the stream runs without a barrier to its end.
    for (int64_t w0 = lo / V; w0 <= (hi - 1) / V; w0 += kSlots) {
        const int64_t wl = max(lo, w0 * V), wh = min(hi, (w0 + kSlots) * V);
        const int64_t v_lo = wl / kPer;  // flat vector index of the window start
        const int nvec = static_cast<int>((wh - wl) / kPer);
        RowAcc acc[kSlots];
#pragma unroll
        for (int r = 0; r < kSlots; ++r) acc[r].reset();

        const int64_t vpr = V / kPer;                 // vectors per row (V is a multiple of 8)
        int64_t row = (v_lo + tid) / vpr;             // row of this thread's current vector
        int64_t next_row_vec = (row + 1) * vpr;       // first vector of the following row
        for (int j0 = tid; j0 < nvec; j0 += kBatch * kThreads) {
            uint4 v[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int j = j0 + u * kThreads;
                v[u] = j < nvec ? ld_stream_v4(src + (v_lo + j) * 16) : neg;
            }
            const int64_t vi0 = v_lo + j0;
            while (vi0 >= next_row_vec) { ++row; next_row_vec += vpr; }
            const int u_last = min(kBatch - 1, (nvec - 1 - j0) / kThreads);
            if (vi0 + u_last * kThreads < next_row_vec) {  // the batch lies in one row
                float cm = vec_max<kDtype>(v[0]);
#pragma unroll
                for (int u = 1; u < kBatch; ++u) cm = fmax_nan(cm, vec_max<kDtype>(v[u]));
                const int slot = static_cast<int>(row - w0);
                float best = acc[0].best;
#pragma unroll
                for (int r = 1; r < kSlots; ++r)
                    if (slot == r) best = acc[r].best;
                if (bad_logit(cm) || cm > best) {  // rare: locate it in the registers held
#pragma unroll
                    for (int r = 0; r < kSlots; ++r) {
                        if (r != slot) continue;
#pragma unroll
                        for (int u = 0; u < kBatch; ++u)
                            if (u <= u_last)
                                fold_vector<kDtype>(acc[r], v[u], vec_max<kDtype>(v[u]), vi0 + u * kThreads,
                                                    row * V);
                    }
                }
            } else {  // a row boundary falls inside the batch
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    if (u > u_last) continue;
                    const int64_t vi = vi0 + u * kThreads;
                    const int64_t vrow = vi / vpr;
#pragma unroll
                    for (int r = 0; r < kSlots; ++r)
                        if (r == static_cast<int>(vrow - w0))
                            fold_vector<kDtype>(acc[r], v[u], vec_max<kDtype>(v[u]), vi, vrow * V);
                }
            }
        }

        // merge this CTA's segments of the window's rows
#pragma unroll
        for (int r = 0; r < kSlots; ++r) {
            const uint64_t key = warp_max_u64(acc[r].key());
            const unsigned bad = __ballot_sync(0xFFFFFFFFu, acc[r].bad);
            if (lane == 0) {
                s_key[r][warp] = key;
                s_bad[r][warp] = bad != 0u;
            }
        }
        __syncthreads();
        if (tid == 0) {
            const int nrows = static_cast<int>((wh - 1) / V - w0 + 1);
            for (int r = 0; r < nrows; ++r) {
                uint64_t k = 0;
                uint32_t bad = 0;
                for (int w = 0; w < kThreads / 32; ++w) {
                    k = s_key[r][w] > k ? s_key[r][w] : k;
                    bad |= s_bad[r][w];
                }
                if (k) atomicMax(p.rowkey + w0 + r, static_cast<unsigned long long>(k));
                if (bad) atomicOr(p.rowbad + w0 + r, 1u);
            }
        }
        __syncthreads();
    }

    // Tickets of the requests this CTA touched (thread 0 made the merges, so
    // its acquire-release ticket orders them before the decision).
    if (warp == 0) {
        for (int64_t g = lo / gsize; g <= (hi - 1) / gsize; ++g) {
            const int64_t c0 = (g * gsize) / p.chunk, c1 = ((g + 1) * gsize - 1) / p.chunk;
            ticket_and_finalize(p, g, static_cast<unsigned>(c1 - c0 + 1), lane);
        }
    }
}

}  // namespace

cudaError_t launch_argmax_rows(const ArgmaxParams& p, int grid, cudaStream_t stream) {
    if (p.dtype == kBF16)
        argmax_rows_kernel<kBF16><<<grid, kThreads, 0, stream>>>(p);
    else
        argmax_rows_kernel<kF32><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

// Resident CTAs per SM of the arg-max kernel (the grid is sized to one wave).
int argmax_rows_occupancy(int dtype) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    static int cache[64][2] = {};
    if (dev < 64 && cache[dev][dtype]) return cache[dev][dtype];
    const void* f = dtype == kBF16 ? reinterpret_cast<const void*>(&argmax_rows_kernel<kBF16>)
                                   : reinterpret_cast<const void*>(&argmax_rows_kernel<kF32>);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, f, kThreads, 0) != cudaSuccess) return 0;
    if (dev < 64) cache[dev][dtype] = n;
    return n;
}

int argmax_rows_threads() { return kThreads; }

}  // namespace dspark
