// Row engine: the sampling policy of one vocabulary row, computed by a
// cluster of CTAs (up to kMaxC; the kernel fixes the size) that each own a
// contiguous slice of the row, plus the exact inverse-CDF draw over the
// policy's weights.  The slices stay in global memory: the first pass over a
// row streams it from HBM (or from L2 when the row was just written, like the
// Markov logits), later passes find it in L2.  With no row held in shared
// memory a CTA needs ~37 KB.
//
// The policy [FT Exact decoding semantics > Probabilistic] as this library
// reads it: greedy = one-hot at the lowest-index argmax; otherwise temperature,
// then top-k keeping exactly k tokens in (logit descending, index ascending)
// order, then top-p keeping the shortest prefix of that order (inside the top-k
// set) whose share of the kept mass is >= p; probabilities are the
// renormalised exp((z - zmax) / T) on that support.
//
// Exactness: the support is described by a key threshold and an index cut
// (support = {key > tau} + {key == tau, index <= cut}); masses are fixed-point
// integers w = round(2^40 exp((z - zmax)/T)), so every sum, every top-p
// comparison and every inverse-CDF boundary is an exact, order-independent
// integer decision.  To find the cuts, one pass builds a histogram of
// s = (zmax - z)/T in bins of 1/8 (exact counts, and exact fixed-point masses
// unless the top-k set is small), reduced once over the cluster; its prefix
// sums bound the cuts to a window of bins (usually one), whose elements are
// compacted into rank 0, sorted by (logit descending, index ascending) and cut
// there by exact prefix sums continued from the exact mass above the window.
// A window too large for the buffer (very flat rows) is resolved by radix
// selection on order-preserving 32-bit keys inside its key range.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"

// Barriers of the engine: the CTA's threads and the cluster.  A kernel that
// runs the engine on part of a larger CTA (as a cluster of one) defines both
// as a named barrier of kThreads threads before including this header.
#ifndef RP_SYNC
#define RP_SYNC() __syncthreads()
#endif
#ifndef RP_CL_SYNC
#define RP_CL_SYNC(cl) (cl).sync()
#endif

namespace dspark {
namespace rp {

namespace cg = cooperative_groups;

constexpr int kMaxC = 8;        // CTAs per row, at most (the cluster's size, read at run time)
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 256;      // 8-bit radix digits
constexpr int kWin = 8;         // candidate window widths
constexpr int kCap = 2048;      // candidate buffer of rank 0 (composite keys)
constexpr double kFix = 1099511627776.0;  // 2^40: fixed-point scale of the weights
static_assert(kWarps * kBins <= kCap, "the per-warp histogram masses live in the candidate buffer");
static_assert(kBins == kThreads, "one histogram bin per thread");
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Unnormalised policy weight exp((z - zmax) * invT) and its fixed-point form.
__device__ __forceinline__ float weight_f(float z, float zmax, float inv_t) {
    return ex2(((z - zmax) * inv_t) * kLog2e);
}
__device__ __forceinline__ uint64_t to_fixed(float w) {
    return __float2ull_rn(w * static_cast<float>(kFix));
}

struct Policy {
    float inv_t;
    int32_t top_k;   // 0 = off (already normalised: 0 < top_k < V, else 0)
    float top_p;     // >= 1 = off
    int32_t greedy;
};

// Results of the policy of one row, identical in every CTA of the cluster.
struct RowResult {
    float zmax;
    int32_t argmax;
    int32_t status;
    uint32_t tau;       // support = {key > tau} + {key == tau, index <= cut}
    int32_t cut;
    uint64_t mass;      // sum of fixed-point weights over the support
    int32_t count;      // support size
    int32_t in_buf;     // 1: the support's composite keys are the first `count` of
                        // rank 0's candidate buffer, sorted by (key desc, index asc)
};

// Shared state of one CTA of the engine (static shared memory).
struct Smem {
    // cluster exchange slots, double-buffered so that one cluster barrier per
    // exchange suffices (a slot is rewritten only two exchanges later)
    unsigned long long xu[2][kWin + 2];
    uint32_t hcnt[2][kBins];
    unsigned long long hmass[2][kBins];
    unsigned long long wu[kWarps][kWin + 2];  // per-warp partials
    unsigned long long gat[kMaxC][kWin + 2];  // slots gathered from the cluster's ranks
    unsigned long long tot[kWin + 2];         // their combination, for every thread
    unsigned long long scan_u[kWarps];
    int32_t pick[4];
    int parity;      // which exchange buffer is next
    int hparity;     // which histogram buffer is next
    unsigned int ccount;     // rank 0: candidate slots claimed by the cluster
};
constexpr int kBatch = 4;    // 16-byte vectors per thread in flight in a pass over a slice

// Called by every thread at kernel start, followed by a __syncthreads.
__device__ __forceinline__ void init_smem(Smem& sm) {
    if (threadIdx.x == 0) {
        sm.parity = 0;
        sm.hparity = 0;
        sm.ccount = 0;
    }
    // the candidate histogram (buffer 1 of the radix histograms) starts empty
    for (int b = threadIdx.x; b < kBins; b += kThreads) {
        sm.hcnt[1][b] = 0;
        sm.hmass[1][b] = 0;
    }
}

__device__ __forceinline__ bool in_set(uint32_t key, int32_t idx, uint32_t tau, int32_t cut) {
    return key > tau || (key == tau && idx <= cut);
}
// A value below which no element of the support {key > tau} + {key == tau,
// ...} lies: the value of key tau, or -inf when tau is below the key of -inf
// (tau = 0: the whole row).
__device__ __forceinline__ float support_floor(uint32_t tau) {
    return tau <= ordered_key(-__int_as_float(0x7F800000)) ? -__int_as_float(0x7F800000) : key_to_float(tau);
}

// Block-sum of up to kWin+2 uint64 values per thread, then a cluster-sum; every
// thread of every CTA returns the same totals in out[].
template <int kN>
__device__ __forceinline__ void cluster_sum_u64(Smem& sm, cg::cluster_group& cl, unsigned long long (&v)[kN],
                                                unsigned long long (&out)[kN]) {
    const int nc = static_cast<int>(cl.num_blocks());  // CTAs in the cluster
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < kN; ++i) {
        unsigned long long x = v[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, o);
        if (lane == 0) sm.wu[warp][i] = x;
    }
    RP_SYNC();
    const int buf = sm.parity;
    if (threadIdx.x < kN) {
        unsigned long long t = 0;
        for (int w = 0; w < kWarps; ++w) t += sm.wu[w][threadIdx.x];
        sm.xu[buf][threadIdx.x] = t;
    }
    RP_CL_SYNC(cl);
    // one remote load per (rank, value) pair, then one combination per value
    if (threadIdx.x < nc * kN) {
        const int r = threadIdx.x / kN, i = threadIdx.x % kN;
        sm.gat[r][i] = cl.map_shared_rank(&sm.xu[buf][0], r)[i];
    }
    RP_SYNC();
    if (threadIdx.x < kN) {
        unsigned long long t = 0;
        for (int r = 0; r < nc; ++r) t += sm.gat[r][threadIdx.x];
        sm.tot[threadIdx.x] = t;
    }
    RP_SYNC();
#pragma unroll
    for (int i = 0; i < kN; ++i) out[i] = sm.tot[i];
    RP_SYNC();
    if (threadIdx.x == 0) sm.parity ^= 1;
    RP_SYNC();
}

// Block-max then cluster-max of one uint64 (and OR of a flag word).
__device__ __forceinline__ void cluster_max_u64(Smem& sm, cg::cluster_group& cl, unsigned long long v,
                                                unsigned long long flags, unsigned long long& out_max,
                                                unsigned long long& out_flags) {
    const int nc = static_cast<int>(cl.num_blocks());  // CTAs in the cluster
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = w > v ? w : v;
        flags |= __shfl_xor_sync(0xFFFFFFFFu, flags, o);
    }
    if (lane == 0) {
        sm.wu[warp][0] = v;
        sm.wu[warp][1] = flags;
    }
    RP_SYNC();
    const int buf = sm.parity;
    if (threadIdx.x == 0) {
        unsigned long long m = 0, f = 0;
        for (int w = 0; w < kWarps; ++w) {
            m = sm.wu[w][0] > m ? sm.wu[w][0] : m;
            f |= sm.wu[w][1];
        }
        sm.xu[buf][0] = m;
        sm.xu[buf][1] = f;
    }
    RP_CL_SYNC(cl);
    if (threadIdx.x < 2 * nc) {
        const int r = threadIdx.x >> 1, i = threadIdx.x & 1;
        sm.gat[r][i] = cl.map_shared_rank(&sm.xu[buf][0], r)[i];
    }
    RP_SYNC();
    if (threadIdx.x == 0) {
        unsigned long long m = 0, f = 0;
        for (int r = 0; r < nc; ++r) {
            m = sm.gat[r][0] > m ? sm.gat[r][0] : m;
            f |= sm.gat[r][1];
        }
        sm.tot[0] = m;
        sm.tot[1] = f;
    }
    RP_SYNC();
    out_max = sm.tot[0];
    out_flags = sm.tot[1];
    RP_SYNC();
    if (threadIdx.x == 0) sm.parity ^= 1;
    RP_SYNC();
}

// Gather one uint64 per CTA (thread 0's `mine`) from every CTA of the
// cluster: afterwards sm.gat[r][0] holds rank r's value, for every thread,
// until the next exchange.
__device__ __forceinline__ void cluster_gather_u64(Smem& sm, cg::cluster_group& cl, unsigned long long mine) {
    const int nc = static_cast<int>(cl.num_blocks());  // CTAs in the cluster
    const int buf = sm.parity;
    if (threadIdx.x == 0) sm.xu[buf][0] = mine;
    RP_CL_SYNC(cl);
    if (threadIdx.x < nc) sm.gat[threadIdx.x][0] = cl.map_shared_rank(&sm.xu[buf][0], threadIdx.x)[0];
    RP_SYNC();
    if (threadIdx.x == 0) sm.parity ^= 1;
    RP_SYNC();
}

// Inclusive block scan of one uint64 per thread.
__device__ __forceinline__ unsigned long long block_scan_u64(Smem& sm, unsigned long long x) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.scan_u[warp] = x;
    RP_SYNC();
    unsigned long long base = 0;
    for (int w = 0; w < warp; ++w) base += sm.scan_u[w];
    RP_SYNC();
    return x + base;
}

// The slice [lo, lo + n) of a row owned by this CTA, read in place from
// global memory (z points at element lo; bf16 or fp32; read-only for the
// kernel's lifetime).
struct Slice {
    const void* z;
    int lo, n;
    int per;   // contiguous elements per thread for ordered scans
    int bf16;  // storage format
    int coherent = 0;  // 1: the row was written earlier in the same launch (read through L2, not the read-only path)
    __device__ __forceinline__ float val(int i) const {
        if (coherent) return __ldcg(static_cast<const float*>(z) + i);
        return bf16 ? __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(z) + i)) << 16)
                    : __ldg(static_cast<const float*>(z) + i);
    }
    // 16-byte vectors: 8 (bf16) or 4 (fp32) elements each; n is a multiple of 8
    __device__ __forceinline__ int vper() const { return bf16 ? 8 : 4; }
    __device__ __forceinline__ int nvec() const { return n / vper(); }
    __device__ __forceinline__ uint4 vec(int j) const {
        return coherent ? __ldcg(static_cast<const uint4*>(z) + j) : __ldg(static_cast<const uint4*>(z) + j);
    }
};

__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}
// NaN-propagating maximum of one 16-byte vector of the slice's format.
__device__ __forceinline__ float vec_max(const uint4& v, int bf16) {
    if (bf16) {
        const uint32_t m = bf16x2_max(bf16x2_max(v.x, v.y), bf16x2_max(v.z, v.w));
        return fmax_nan(bf16_lo(m), bf16_hi(m));
    }
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
}
// Element l of a vector of the slice's format.
__device__ __forceinline__ float vec_elem(const uint4& v, int l, int bf16) {
    if (bf16) {
        const uint32_t w = l < 2 ? v.x : l < 4 ? v.y : l < 6 ? v.z : v.w;
        return (l & 1) ? bf16_hi(w) : bf16_lo(w);
    }
    return __uint_as_float(l == 0 ? v.x : l == 1 ? v.y : l == 2 ? v.z : v.w);
}

// The smallest value t (as an ordered key) with pred(t) true, for a predicate
// that is monotone in the value (false below some point, true from there up
// to kmax, and true at kmax): bisection over the ordered keys [1, kmax].
// Every thread computes the same result without communication.
template <typename P>
__device__ __forceinline__ uint32_t lowest_true_key(uint32_t kmax, P pred) {
    uint32_t lo = 1, hi = kmax;  // pred(key_to_float(hi)) holds
    while (lo < hi) {
        const uint32_t mid = lo + (hi - lo) / 2;
        if (pred(key_to_float(mid))) hi = mid;
        else lo = mid + 1;
    }
    return hi;
}

// Every element of the slice, in no particular order: fn(z, index), with
// kBatch 16-byte vectors per thread in flight.
template <typename F>
__device__ __forceinline__ void for_each_elem(const Slice& sl, F fn) {
    const int vp = sl.vper(), nv = sl.nvec();
    for (int j0 = threadIdx.x; j0 < nv; j0 += kThreads * kBatch) {
        uint4 vb[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + u * kThreads;
            vb[u] = j < nv ? sl.vec(j) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + u * kThreads;
            if (j >= nv) break;
#pragma unroll
            for (int l = 0; l < 8; ++l)
                if (l < vp) fn(vec_elem(vb[u], l, sl.bf16), sl.lo + j * vp + l);
        }
    }
}

// This thread's contiguous run of the slice's vectors, [a, e), for scans in
// index order.
__device__ __forceinline__ void thread_run(const Slice& sl, int& a, int& e) {
    const int nv = sl.nvec();
    const int pv = (nv + kThreads - 1) / kThreads;
    a = min(static_cast<int>(threadIdx.x) * pv, nv);
    e = min(a + pv, nv);
}
// fn(z, index) over the vectors [a, e) in index order, kBatch at a time.
template <typename F>
__device__ __forceinline__ void for_run(const Slice& sl, int a, int e, F fn) {
    const int vp = sl.vper();
    for (int j0 = a; j0 < e; j0 += kBatch) {
        uint4 vb[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) vb[u] = j0 + u < e ? sl.vec(j0 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (j0 + u >= e) break;
#pragma unroll
            for (int l = 0; l < 8; ++l)
                if (l < vp) fn(vec_elem(vb[u], l, sl.bf16), sl.lo + (j0 + u) * vp + l);
        }
    }
}

// Radix selection on keys inside the window [klo, khi]: among the elements
// with a key in the window matching `pred`, find the key tau at which the
// descending cumulative measure (count, or fixed-point mass when kMass),
// started at above0 (the measure of everything above the window), reaches
// `target`.  Returns tau, the measure strictly above tau (above0 included)
// and the count / mass of the elements equal to tau (within pred); false when
// the window does not reach target.  Digits of 8 bits below the window's
// common prefix; in bf16 slices the low 16 bits of every key follow from its
// sign bit, so the digits stop at bit 16.  Each warp counts into a private
// copy (wbuf: kWarps x kBins masses, then kWarps x kBins counts), summed per
// CTA and then over the cluster.
template <bool kMass, typename Pred>
__device__ bool radix_select(Smem& sm, cg::cluster_group& cl, const Slice& sl, unsigned long long* wbuf,
                             uint32_t klo, uint32_t khi, unsigned long long above0, unsigned long long target,
                             float zmax, float inv_t, Pred pred, uint32_t& tau, unsigned long long& above,
                             unsigned long long& eq_cnt, unsigned long long& eq_mass) {
    const int nc = static_cast<int>(cl.num_blocks());  // CTAs in the cluster
    const int tid = threadIdx.x;
    const int min_bit = sl.bf16 ? 16 : 0;
    int hi_bit = klo == khi ? 0 : 32 - __clz(static_cast<int>(klo ^ khi));  // bits still open
    if (hi_bit < min_bit) hi_bit = min_bit;
    uint32_t prefix = hi_bit >= 32 ? 0u : (khi >> hi_bit);
    auto full_key = [min_bit](uint32_t pre) -> uint32_t {
        return min_bit ? ((pre << 16) | ((pre & 0x8000u) ? 0u : 0xFFFFu)) : pre;
    };
    above = above0;
    eq_cnt = 0;
    eq_mass = 0;
    if (hi_bit == min_bit) {  // a single key in the window: count it
        const uint32_t k1 = full_key(prefix);
        unsigned long long v[2] = {0, 0};
        if (k1 >= klo && k1 <= khi) {
            for_each_elem(sl, [&](float z, int32_t idx) {
                const uint32_t key = ordered_key(z);
                if (key == k1 && pred(key, idx)) {
                    v[0] += 1;
                    if (kMass) v[1] += to_fixed(weight_f(z, zmax, inv_t));
                }
            });
        }
        unsigned long long o[2];
        cluster_sum_u64<2>(sm, cl, v, o);
        tau = k1;
        eq_cnt = o[0];
        eq_mass = o[1];
        return above0 + (kMass ? o[1] : o[0]) >= target;
    }
    const int warp = tid >> 5;
    uint32_t* wcnt = reinterpret_cast<uint32_t*>(wbuf + kWarps * kBins);
    unsigned long long* wm = wbuf + warp * kBins;
    uint32_t* wc = wcnt + warp * kBins;
    bool found = true;
    while (hi_bit > min_bit) {
        const int nb = min(8, hi_bit - min_bit);
        const int lo_bit = hi_bit - nb;
        const int buf = sm.hparity;
        for (int i = tid; i < kWarps * kBins; i += kThreads) {
            wcnt[i] = 0u;
            if (kMass) wbuf[i] = 0ull;
        }
        RP_SYNC();
        const uint32_t pre = prefix;
        const int hb = hi_bit;
        for_each_elem(sl, [&](float z, int32_t idx) {
            const uint32_t key = ordered_key(z);
            if (key < klo || key > khi || (hb < 32 && (key >> hb) != pre) || !pred(key, idx)) return;
            const int d = static_cast<int>((key >> lo_bit) & ((1u << nb) - 1u));
            atomicAdd(&wc[d], 1u);
            if (kMass) atomicAdd(&wm[d], static_cast<unsigned long long>(to_fixed(weight_f(z, zmax, inv_t))));
        });
        RP_SYNC();
        {  // the CTA's histogram: bin tid over the warps' copies
            uint32_t c = 0;
            unsigned long long m = 0;
            for (int w = 0; w < kWarps; ++w) {
                c += wcnt[w * kBins + tid];
                if (kMass) m += wbuf[w * kBins + tid];
            }
            sm.hcnt[buf][tid] = c;
            if (kMass) sm.hmass[buf][tid] = m;
        }
        RP_CL_SYNC(cl);
        // thread t takes bin (nbins - 1 - t): descending key order
        const int nbins = 1 << nb;
        const int b = nbins - 1 - tid;
        unsigned long long c = 0, m = 0;
        if (b >= 0) {
            for (int r = 0; r < nc; ++r) {
                c += cl.map_shared_rank(&sm.hcnt[buf][0], r)[b];
                if (kMass) m += cl.map_shared_rank(&sm.hmass[buf][0], r)[b];
            }
        }
        const unsigned long long mine = kMass ? m : c;
        if (tid == 0) sm.pick[1] = 0;
        const unsigned long long incl = block_scan_u64(sm, mine);
        if (b >= 0 && above + incl >= target && above + incl - mine < target) {
            sm.pick[0] = b;
            sm.pick[1] = 1;
            reinterpret_cast<unsigned long long*>(&sm.scan_u[0])[0] = incl - mine;  // measure above b
            reinterpret_cast<unsigned long long*>(&sm.wu[0][0])[0] = c;
            reinterpret_cast<unsigned long long*>(&sm.wu[0][1])[0] = m;
        }
        RP_SYNC();
        if (!sm.pick[1]) found = false;
        const int pb = sm.pick[1] ? sm.pick[0] : 0;
        above += sm.pick[1] ? sm.scan_u[0] : 0ull;
        eq_cnt = sm.wu[0][0];
        eq_mass = sm.wu[0][1];
        prefix = (prefix << nb) | static_cast<uint32_t>(pb);
        hi_bit = lo_bit;
        RP_SYNC();
        if (tid == 0) sm.hparity ^= 1;
        RP_SYNC();
    }
    tau = full_key(prefix);
    return found;
}

// Global index of the t-th (1-based) element in index order with key == tau
// and pred; every CTA returns it.
template <typename Pred>
__device__ int32_t tie_index(Smem& sm, cg::cluster_group& cl, const Slice& sl, uint32_t tau,
                             unsigned long long t, Pred pred) {
    const int nc = static_cast<int>(cl.num_blocks());  // CTAs in the cluster
    const int tid = threadIdx.x;
    const int rank = static_cast<int>(cl.block_rank());
    // ordered ownership: each thread a contiguous run of the slice's vectors
    int a, e;
    thread_run(sl, a, e);
    unsigned long long mine = 0;
    for_run(sl, a, e, [&](float z, int32_t idx) {
        const uint32_t key = ordered_key(z);
        if (key == tau && pred(key, idx)) ++mine;
    });
    const unsigned long long incl = block_scan_u64(sm, mine);
    __shared__ unsigned long long s_total;
    if (tid == kThreads - 1) s_total = incl;
    RP_SYNC();
    cluster_gather_u64(sm, cl, s_total);
    const auto totals = [&sm](int r) { return sm.gat[r][0]; };  // per rank
    unsigned long long before = 0;
    int owner = nc - 1;
    for (int r = 0; r < nc; ++r) {
        if (before + totals(r) >= t) { owner = r; break; }
        before += totals(r);
    }
    const int buf = sm.parity;
    if (rank == owner && tid == 0) sm.xu[buf][0] = static_cast<unsigned long long>(sl.lo + max(sl.n - 1, 0));
    RP_SYNC();
    if (rank == owner) {
        const unsigned long long want = t - before;
        if (incl >= want && incl - mine < want) {
            unsigned long long k = incl - mine;
            bool done = false;
            for_run(sl, a, e, [&](float z, int32_t idx) {
                const uint32_t key = ordered_key(z);
                if (!done && key == tau && pred(key, idx) && ++k == want) {
                    sm.xu[buf][0] = static_cast<unsigned long long>(idx);
                    done = true;
                }
            });
        }
    }
    RP_CL_SYNC(cl);
    if (tid == 0) sm.tot[0] = cl.map_shared_rank(&sm.xu[buf][0], owner)[0];
    RP_SYNC();
    const int32_t idx = static_cast<int32_t>(sm.tot[0]);
    RP_SYNC();
    if (tid == 0) sm.parity ^= 1;
    RP_SYNC();
    return idx;
}

// The policy by radix selection over the whole slice (the fallback when the
// candidate set of row_policy would not fit).  z slice already loaded; max
// key, argmax and the bad flag already reduced.
static __device__ void row_policy_radix(Smem& sm, cg::cluster_group& cl, const Slice& sl, int V, const Policy& pol,
                                 RowResult& res, unsigned long long* wbuf) {
    const float zmax = res.zmax;
    const uint32_t kmax = ordered_key(zmax);
    // greedy: the argmax alone
    res.tau = kmax;
    res.cut = res.argmax;
    res.mass = static_cast<unsigned long long>(kFix);
    if (pol.greedy) return;
    const float inv_t = pol.inv_t;

    // ---- top-k: exactly k tokens
    uint32_t tau_k = 0;      // key > 0 holds for every non-NaN value: "all"
    int32_t cut_k = -1;
    const bool use_k = pol.top_k > 0;
    if (use_k) {
        unsigned long long v[kWin + 1], cnt[kWin + 1];
#pragma unroll
        for (int i = 0; i <= kWin; ++i) v[i] = 0;
        for_each_elem(sl, [&](float z, int32_t) {
            const float d = zmax - z;
#pragma unroll
            for (int w = 0; w < kWin; ++w) v[w] += d <= static_cast<float>(1 << w) ? 1ull : 0ull;
        });
        cluster_sum_u64<kWin + 1>(sm, cl, v, cnt);
        // the narrowest width holding k elements, doubled against rounding at its edge
        float zlo = -__int_as_float(0x7F800000);
        for (int w = kWin - 1; w >= 0; --w)
            if (cnt[w] >= static_cast<unsigned long long>(pol.top_k)) zlo = zmax - static_cast<float>(2 << w);
        const uint32_t klo = zlo == -__int_as_float(0x7F800000) ? 0u : ordered_key(zlo);
        unsigned long long above, eqc, eqm;
        auto all = [](uint32_t, int32_t) { return true; };
        if (!radix_select<false>(sm, cl, sl, wbuf, klo, kmax, 0ull, static_cast<unsigned long long>(pol.top_k),
                                 zmax, inv_t, all, tau_k, above, eqc, eqm))
            radix_select<false>(sm, cl, sl, wbuf, 0u, kmax, 0ull, static_cast<unsigned long long>(pol.top_k), zmax,
                                inv_t, all, tau_k, above, eqc, eqm);
        const unsigned long long need = static_cast<unsigned long long>(pol.top_k) - above;
        cut_k = tie_index(sm, cl, sl, tau_k, need, [](uint32_t, int32_t) { return true; });
    }
    auto in_k = [tau_k, cut_k](uint32_t key, int32_t idx) { return in_set(key, idx, tau_k, cut_k); };

    // ---- kept mass, and the mass inside each candidate window (for top-p)
    const bool use_p = pol.top_p < 1.0f;
    unsigned long long v[kWin + 1], ms[kWin + 1];
#pragma unroll
    for (int i = 0; i <= kWin; ++i) v[i] = 0;
    for_each_elem(sl, [&](float z, int32_t idx) {
        const float d = (zmax - z) * inv_t;
        if (d > 41.0f * 0.6931472f + 1.0f) return;  // weight rounds to 0 in 2^-40 units
        const uint32_t key = ordered_key(z);
        if (!in_k(key, idx)) return;
        const unsigned long long w = to_fixed(weight_f(z, zmax, inv_t));
        v[kWin] += w;
#pragma unroll
        for (int wi = 0; wi < kWin; ++wi) v[wi] += d <= static_cast<float>(2 << wi) ? w : 0ull;
    });
    cluster_sum_u64<kWin + 1>(sm, cl, v, ms);
    const unsigned long long kept = ms[kWin];
    res.tau = tau_k;
    res.cut = cut_k;
    res.mass = kept;
    if (!use_p) return;

    // ---- top-p: shortest prefix of the order with mass >= p * kept
    double th = ceil(static_cast<double>(pol.top_p) * static_cast<double>(kept));
    unsigned long long theta = th < 1.0 ? 1ull : static_cast<unsigned long long>(th);
    if (theta > kept) theta = kept;
    float zlo = -__int_as_float(0x7F800000);
    for (int w = kWin - 1; w >= 0; --w)
        if (ms[w] >= theta) zlo = zmax - static_cast<float>(4 << w) / inv_t;  // doubled width
    uint32_t klo = zlo == -__int_as_float(0x7F800000) ? 0u : ordered_key(zlo);
    if (use_k && klo < tau_k) klo = tau_k;  // the cut lies inside the top-k set
    uint32_t tau_p;
    unsigned long long above, eqc, eqm;
    if (!radix_select<true>(sm, cl, sl, wbuf, klo, kmax, 0ull, theta, zmax, inv_t, in_k, tau_p, above, eqc, eqm))
        radix_select<true>(sm, cl, sl, wbuf, 0u, kmax, 0ull, theta, zmax, inv_t, in_k, tau_p, above, eqc, eqm);
    // tied elements share one weight; take just enough of them in index order
    const unsigned long long wt = eqc ? eqm / eqc : 0ull;
    unsigned long long t = wt ? (theta - above + wt - 1) / wt : eqc;
    if (t < 1) t = 1;
    if (t > eqc) t = eqc;
    const int32_t cut_p = tie_index(sm, cl, sl, tau_p, t, in_k);
    res.tau = tau_p;
    res.cut = cut_p;
    res.mass = above + t * wt;
}

// Inverse-CDF draw in token-index order over fixed-point weights w(z, index)
// (index = the token): the smallest index whose inclusive prefix exceeds
// floor(m * total / 2^24), m the 24-bit uniform.  Each thread owns a
// contiguous run of the slice's 16-byte vectors (read kBatch at a time);
// block scan, then the prefix over the cluster's ranks; the owning thread
// re-reads its run to find the token.  Every CTA returns the index.
template <typename Wz>
__device__ int32_t sample_fixed(Smem& sm, cg::cluster_group& cl, const Slice& sl, uint32_t m24, Wz wz,
                                unsigned long long& total_out) {
    const int nc = static_cast<int>(cl.num_blocks());  // CTAs in the cluster
    const int tid = threadIdx.x;
    const int rank = static_cast<int>(cl.block_rank());
    const int vp = sl.vper(), nv = sl.nvec();
    const int pv = (nv + kThreads - 1) / kThreads;  // vectors per thread
    const int a = min(tid * pv, nv), e = min(a + pv, nv);
    auto vec_weight = [&](int j, const uint4& v) {
        unsigned long long w = 0;
#pragma unroll
        for (int l = 0; l < 8; ++l)
            if (l < vp) w += wz(vec_elem(v, l, sl.bf16), sl.lo + j * vp + l);
        return w;
    };
    unsigned long long mine = 0;
    for (int j0 = a; j0 < e; j0 += kBatch) {
        uint4 vb[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) vb[u] = j0 + u < e ? sl.vec(j0 + u) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
            if (j0 + u < e) mine += vec_weight(j0 + u, vb[u]);
    }
    const unsigned long long incl = block_scan_u64(sm, mine);
    __shared__ unsigned long long s_total;
    if (tid == kThreads - 1) s_total = incl;
    RP_SYNC();
    cluster_gather_u64(sm, cl, s_total);
    const auto totals = [&sm](int r) { return sm.gat[r][0]; };  // per rank
    unsigned long long total = 0;
    for (int r = 0; r < nc; ++r) total += totals(r);
    total_out = total;
    if (total == 0) return -1;
    const unsigned long long target =
        static_cast<unsigned long long>((static_cast<unsigned __int128>(m24) * total) >> 24);
    unsigned long long before = 0;
    int owner = nc - 1;
    for (int r = 0; r < nc; ++r) {
        if (before + totals(r) > target) { owner = r; break; }
        before += totals(r);
    }
    const int buf = sm.parity;
    if (rank == owner && tid == 0) sm.xu[buf][0] = static_cast<unsigned long long>(sl.lo + max(sl.n - 1, 0));
    RP_SYNC();
    if (rank == owner) {
        const unsigned long long tl = target - before;  // within this CTA: first prefix > tl
        if (incl > tl && incl - mine <= tl) {
            unsigned long long c = incl - mine;
            bool found = false;
            for (int j = a; j < e && !found; ++j) {
                const uint4 v = sl.vec(j);
                for (int l = 0; l < vp; ++l) {
                    const int32_t idx = sl.lo + j * vp + l;
                    c += wz(vec_elem(v, l, sl.bf16), idx);
                    if (c > tl) {
                        sm.xu[buf][0] = static_cast<unsigned long long>(idx);
                        found = true;
                        break;
                    }
                }
            }
        }
    }
    RP_CL_SYNC(cl);
    if (tid == 0) sm.tot[0] = cl.map_shared_rank(&sm.xu[buf][0], owner)[0];
    RP_SYNC();
    const int32_t idx = static_cast<int32_t>(sm.tot[0]);
    RP_SYNC();
    if (tid == 0) sm.parity ^= 1;
    RP_SYNC();
    return idx;
}

// One pass over this CTA's slice (kBatch 16-byte vectors per thread in
// flight): the row's max key / lowest argmax / non-finite flag, reduced over
// the cluster.  Each thread keeps a packed maximum and looks for the index
// only when a vector beats it.
static __device__ void slice_max(Smem& sm, cg::cluster_group& cl, const Slice& sl, RowResult& res, bool& bad) {
    const int vp = sl.vper(), nv = sl.nvec();
    float nanacc = -__int_as_float(0x7F800000);
    float bval = -__int_as_float(0x7F800000);  // this thread's maximum (vectors in index order)
    int32_t bidx = -1;
    for (int j0 = threadIdx.x; j0 < nv; j0 += kThreads * kBatch) {
        uint4 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + u * kThreads;
            v[u] = j < nv ? sl.vec(j) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + u * kThreads;
            if (j >= nv) break;
            const float vm = vec_max(v[u], sl.bf16);
            nanacc = fmax_nan(nanacc, vm);
            if (vm > bval) {  // rare: a new maximum of this thread; its first occurrence
                int l0 = vp - 1;
#pragma unroll
                for (int l = 7; l >= 0; --l)
                    if (l < vp && vec_elem(v[u], l, sl.bf16) == vm) l0 = l;
                bval = vm;
                bidx = sl.lo + j * vp + l0;
            }
        }
    }
    unsigned long long best = 0;
    if (bidx >= 0 && !bad_logit(bval))
        best = (static_cast<unsigned long long>(ordered_key(bval)) << 32) | (0xFFFFFFFFull - static_cast<uint32_t>(bidx));
    unsigned long long mk, fl;
    cluster_max_u64(sm, cl, best, bad_logit(nanacc) ? 1ull : 0ull, mk, fl);
    bad = fl != 0;
    if (mk == 0) {
        res.zmax = -__int_as_float(0x7F800000);
        res.argmax = -1;
    } else {
        res.zmax = key_to_float(static_cast<uint32_t>(mk >> 32));
        res.argmax = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(mk));
    }
}

// ---------------------------------------------------------------- candidates
// Composite sort key of a logit: larger value first, then lower index.
__device__ __forceinline__ unsigned long long value_order(uint32_t key, int32_t idx) {
    return (static_cast<unsigned long long>(key) << 32) | (0xFFFFFFFFull - static_cast<uint32_t>(idx));
}
// ... and of a token index: lower index first (the key kept in the low word).
__device__ __forceinline__ unsigned long long index_order(uint32_t key, int32_t idx) {
    return (static_cast<unsigned long long>(0xFFFFFFFFu - static_cast<uint32_t>(idx)) << 32) | key;
}
__device__ __forceinline__ uint32_t vo_key(unsigned long long c) { return static_cast<uint32_t>(c >> 32); }
__device__ __forceinline__ int32_t vo_idx(unsigned long long c) {
    return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(c));
}
__device__ __forceinline__ uint32_t io_key(unsigned long long c) { return static_cast<uint32_t>(c); }
__device__ __forceinline__ int32_t io_idx(unsigned long long c) {
    return static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(c >> 32));
}

// Bitonic sort of buf[0, n) in descending order (n <= kCap), padding with 0
// (below every real composite key) up to a power of two.  Each iteration
// handles one compare-exchange pair.  All threads of the CTA.
static __device__ void sort_desc(unsigned long long* buf, int n) {
    int P = 1;
    while (P < n) P <<= 1;
    for (int i = n + threadIdx.x; i < P; i += kThreads) buf[i] = 0ull;
    RP_SYNC();
    const int half = P >> 1;
    for (int k = 2; k <= P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int q = threadIdx.x; q < half; q += kThreads) {
                const int i = ((q & ~(j - 1)) << 1) | (q & (j - 1));
                const int ixj = i + j;
                const unsigned long long a = buf[i], b = buf[ixj];
                if ((i & k) == 0 ? (a < b) : (a > b)) {
                    buf[i] = b;
                    buf[ixj] = a;
                }
            }
            RP_SYNC();
        }
    }
}

// Sort buf[0, n) descending.  Up to kThreads distinct keys: each thread
// places one key at its rank (the number of larger keys), one pass over the
// keys in shared memory; larger sets: the bitonic network.  All threads of
// the CTA.
static __device__ void sort_candidates(unsigned long long* buf, int n) {
    if (n > kThreads) {
        sort_desc(buf, n);
        return;
    }
    const int t = threadIdx.x;
    unsigned long long c = 0;
    int r = 0;
    if (t < n) {
        c = buf[t];
        for (int j = 0; j < n; ++j) r += buf[j] > c ? 1 : 0;
    }
    RP_SYNC();
    if (t < n) buf[r] = c;
    RP_SYNC();
}

// Compact the elements of the slice for which pick(z, index) holds into rank
// 0's candidate buffer as value-order composite keys.  Every picked element
// is >= floor, so whole 16-byte vectors below it are skipped.  Each warp
// claims its slots with one atomic on rank 0's counter (slot order is
// arbitrary; the buffer is sorted afterwards); writes past kCap are dropped.
// Rank 0's counter must be zero and visible to the cluster (a cluster barrier
// after its reset) before the call; ends with a cluster barrier.
template <typename Pick>
__device__ void compact_candidates(Smem& sm, cg::cluster_group& cl, const Slice& sl, unsigned long long* cbuf,
                                   float floor, Pick pick) {
    const int lane = threadIdx.x & 31;
    unsigned int* rcount = cl.map_shared_rank(&sm.ccount, 0);
    unsigned long long* dst = cl.map_shared_rank(cbuf, 0);
    const int vp = sl.vper(), nv = sl.nvec();
    for (int jb = 0; jb < nv; jb += kThreads * kBatch) {  // the same trip count for every thread
      uint4 vb[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
          const int j = jb + u * kThreads + static_cast<int>(threadIdx.x);
          vb[u] = j < nv ? sl.vec(j) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int j = jb + u * kThreads + static_cast<int>(threadIdx.x);
        unsigned mine = 0;  // bit l: element l of vector j is picked
        const uint4 v = vb[u];
        if (j < nv) {
            if (vec_max(v, sl.bf16) >= floor) {
#pragma unroll
                for (int l = 0; l < 8; ++l)
                    if (l < vp && pick(vec_elem(v, l, sl.bf16), sl.lo + j * vp + l)) mine |= 1u << l;
            }
        }
        if (!__any_sync(0xFFFFFFFFu, mine != 0u)) continue;
        const unsigned cnt = static_cast<unsigned>(__popc(mine));
        unsigned incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        unsigned base = 0;
        if (lane == 31) base = atomicAdd(rcount, incl);
        base = __shfl_sync(0xFFFFFFFFu, base, 31) + incl - cnt;
#pragma unroll
        for (int l = 0; l < 8; ++l) {
            if ((mine >> l) & 1u) {
                if (base < static_cast<unsigned>(kCap))
                    dst[base] = value_order(ordered_key(vec_elem(v, l, sl.bf16)), sl.lo + j * vp + l);
                ++base;
            }
        }
      }
    }
    RP_CL_SYNC(cl);
}

// First position i in [0, n) whose inclusive prefix of w(i) satisfies
// prefix >= th (strict = false) or prefix > th (strict = true); n if none.
// Also returns the total.  All threads of one CTA; w is evaluated in
// contiguous per-thread ranges.
template <typename Wf>
__device__ int find_crossing(Smem& sm, int n, unsigned long long th, bool strict, Wf w,
                             unsigned long long& total) {
    const int per = (n + kThreads - 1) / kThreads;
    const int a = min(static_cast<int>(threadIdx.x) * per, n), e = min(a + per, n);
    unsigned long long mine = 0;
    for (int i = a; i < e; ++i) mine += w(i);
    const unsigned long long incl = block_scan_u64(sm, mine);
    __shared__ unsigned long long s_tot;
    __shared__ int s_pos;
    if (threadIdx.x == kThreads - 1) s_tot = incl;
    if (threadIdx.x == 0) s_pos = n;
    RP_SYNC();
    const unsigned long long before = incl - mine;
    const bool here = strict ? (incl > th && before <= th) : (incl >= th && before < th);
    if (here && mine > 0) {
        unsigned long long c = before;
        for (int i = a; i < e; ++i) {
            c += w(i);
            if (strict ? c > th : c >= th) {
                s_pos = i;
                break;
            }
        }
    }
    RP_SYNC();
    total = s_tot;
    const int pos = s_pos;
    RP_SYNC();
    return pos;
}


// One block scan over rank 0's first K candidates (weights wt(i), contiguous
// ranges per thread): total = their weight sum; th = thresh(total); when th
// is nonzero, pos = the first position whose inclusive prefix reaches th
// (K if none) and prefix = the prefix there.  All threads of one CTA.
template <typename Wf, typename Th>
__device__ void cut_scan(Smem& sm, int K, Wf wt, Th thresh, unsigned long long& total, int& pos,
                         unsigned long long& prefix) {
    const int per = (K + kThreads - 1) / kThreads;
    const int a = min(static_cast<int>(threadIdx.x) * per, K), e = min(a + per, K);
    unsigned long long mine = 0;
    for (int i = a; i < e; ++i) mine += wt(i);
    const unsigned long long incl = block_scan_u64(sm, mine);
    __shared__ unsigned long long s_tot, s_pm;
    __shared__ int s_pos;
    if (threadIdx.x == kThreads - 1) s_tot = incl;
    if (threadIdx.x == 0) {
        s_pos = K;
        s_pm = 0ull;
    }
    RP_SYNC();
    total = s_tot;
    const unsigned long long th = thresh(total);
    const unsigned long long before = incl - mine;
    if (th > 0 && mine > 0 && incl >= th && before < th) {
        unsigned long long c = before;
        for (int i = a; i < e; ++i) {
            c += wt(i);
            if (c >= th) {
                s_pos = i;
                s_pm = c;
                break;
            }
        }
    }
    RP_SYNC();
    pos = s_pos;
    prefix = s_pm;
    RP_SYNC();
}

// ceil(p * kept) clamped to [1, kept] (kept = 0 gives 0): the fixed-point
// mass a top-p prefix must reach.
__device__ __forceinline__ unsigned long long p_threshold(float p, unsigned long long kept) {
    const double th = ceil(static_cast<double>(p) * static_cast<double>(kept));
    const unsigned long long t = th < 1.0 ? 1ull : static_cast<unsigned long long>(th);
    return t > kept ? kept : t;
}

// The first bin whose inclusive prefix reaches x (the prefix reaches x at the
// last bin).
template <typename T>
__device__ __forceinline__ int first_at_least(const T* prefix, unsigned long long x) {
    int lo = 0, hi = kBins - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (static_cast<unsigned long long>(prefix[mid]) >= x) hi = mid;
        else lo = mid + 1;
    }
    return lo;
}

// The bin of s = (zmax - z)/T in steps of 1/8 below s = 32 (kBins beyond):
// non-increasing in z.
struct BinOf {
    float zmax, inv_t;
    __device__ __forceinline__ int operator()(float z) const {
        const float sc = (zmax - z) * inv_t;
        return sc < 32.0f ? min(kBins - 1, static_cast<int>(sc * 8.0f)) : kBins;
    }
};

// s = (zmax - z)/T falls in a bin <= b (monotone in z: false below some
// value, true from there up).
struct BinAtMost {
    float zmax, inv_t;
    int b;
    __device__ __forceinline__ bool operator()(float z) const {
        const float sc = (zmax - z) * inv_t;
        return sc < 32.0f && min(kBins - 1, static_cast<int>(sc * 8.0f)) <= b;
    }
};

// One pass over the slice for the histogram of s = (zmax - z)/T in bins of
// 1/8 below s = 32: kMode 0 sums the fixed-point weights alone (returned),
// 1 counts into this warp's bins, 2 counts and adds the weights.  One
// instantiation per mode keeps the weight off the count-only path.
template <int kMode>
__device__ __forceinline__ unsigned long long hist_pass(const Slice& sl, float zmax, float inv_t, uint32_t* whc,
                                                        unsigned long long* whp) {
    unsigned long long tmass = 0;
    const int vp = sl.vper(), nv = sl.nvec();
    for (int j0 = threadIdx.x; j0 < nv; j0 += kThreads * kBatch) {
        uint4 vb[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int j = j0 + u * kThreads;
            vb[u] = j < nv ? sl.vec(j) : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const uint4 v = vb[u];
            if (j0 + u * kThreads >= nv) break;
            if ((zmax - vec_max(v, sl.bf16)) * inv_t >= 32.0f) continue;  // the whole vector is out of range
#pragma unroll
            for (int l = 0; l < 8; ++l) {
                if (l >= vp) break;
                const float z = vec_elem(v, l, sl.bf16);
                const float sc = (zmax - z) * inv_t;
                if (sc < 32.0f) {
                    if (kMode == 0) {
                        tmass += to_fixed(weight_f(z, zmax, inv_t));
                    } else {
                        const int bin = min(kBins - 1, static_cast<int>(sc * 8.0f));
                        if (kMode == 2) atomicAdd(&whp[bin], to_fixed(weight_f(z, zmax, inv_t)));
                        atomicAdd(&whc[bin], 1u);
                    }
                }
            }
        }
    }
    return tmass;
}

// The policy of the row held by the cluster.  One pass builds a histogram of
// s = (zmax - z)/T in bins of 1/8 below s = 32 (beyond, the weight is 0 in
// fixed point), each warp into a private copy, summed per CTA and over the
// cluster: counts alone when top-k keeps at most kThreads tokens (that set is
// compacted whole), otherwise exact counts and exact fixed-point masses.  Its
// prefix sums give the bin where the cumulative count reaches k (top-k),
// bounds on the kept mass, and from them the bins where the cumulative mass
// can reach p of it (top-p): both cuts lie in the window of bins between.
// With top-k and top-p together only the bins where the top-p cut can lie and
// the top-k bin need their tokens; the bins between (the gap) enter as their
// exact count and mass.  The window's elements (but the gap's) are compacted
// into rank 0's buffer, whole vectors below a closed-form floor skipped;
// rank 0 sorts them by (logit descending, index ascending) and takes both cuts
// in one block scan of exact prefix sums continued from the exact mass above
// the window.  A support of at most kThreads tokens is compacted whole, so
// that rank 0 holds it for the draw.  A window too large for the buffer (a
// flat row: thousands of tokens in one bin, bf16 ties) is resolved for top-p
// alone by radix selection inside the window's key range; other such rows
// fall back to row_policy_radix.  cbuf = this CTA's candidate buffer (kCap
// composite keys; only rank 0's receives candidates) followed by
// kWarps x kBins 32-bit counts.
static __device__ void row_policy(Smem& sm, cg::cluster_group& cl, const Slice& sl, int V, const Policy& pol,
                           RowResult& res, unsigned long long* cbuf) {
    const int nc = static_cast<int>(cl.num_blocks());  // CTAs in the cluster
    const float zmax = res.zmax;
    const uint32_t kmax = ordered_key(zmax);
    const int tid = threadIdx.x;
    const int rank = static_cast<int>(cl.block_rank());
    res.tau = kmax;
    res.cut = res.argmax;
    res.mass = static_cast<unsigned long long>(kFix);
    res.count = 1;
    res.in_buf = 0;
    if (pol.greedy) return;
    const float inv_t = pol.inv_t;
    const bool use_k = pol.top_k > 0;
    const bool use_p = pol.top_p < 1.0f;
    const bool trunc = use_k || use_p;
    // Exact masses narrow the window; a top-k set of at most kThreads tokens
    // is compacted whole, so its rows count alone.
    const bool with_mass = !use_k || pol.top_k > kThreads;

    // ---- histogram (rows without truncation need the total mass alone)
    const int warp_id = tid >> 5;
    uint32_t* wcnt = reinterpret_cast<uint32_t*>(cbuf + kWarps * kBins);
    unsigned long long* whp = cbuf + warp_id * kBins;
    uint32_t* whc = wcnt + warp_id * kBins;
    unsigned long long tmass = 0;
    if (trunc) {
        for (int i = tid; i < kWarps * kBins; i += kThreads) {
            if (with_mass) cbuf[i] = 0ull;
            wcnt[i] = 0u;
        }
        RP_SYNC();
    }
    if (!trunc) tmass = hist_pass<0>(sl, zmax, inv_t, whc, whp);
    else if (with_mass) hist_pass<2>(sl, zmax, inv_t, whc, whp);
    else hist_pass<1>(sl, zmax, inv_t, whc, whp);
    RP_SYNC();
    uint32_t* hc = sm.hcnt[1];
    unsigned long long* hp = sm.hmass[1];
    __shared__ unsigned long long s_ctot;  // this CTA's total mass (no truncation)
    if (trunc) {  // the CTA's histogram: bin tid over the warps' copies
        unsigned long long t = 0;
        uint32_t cn = 0;
        for (int w = 0; w < kWarps; ++w) {
            if (with_mass) t += cbuf[w * kBins + tid];
            cn += wcnt[w * kBins + tid];
        }
        hp[tid] = t;
        hc[tid] = cn;
    } else {
        const int lane = tid & 31;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) tmass += __shfl_xor_sync(0xFFFFFFFFu, tmass, o);
        if (lane == 0) sm.wu[warp_id][0] = tmass;
        RP_SYNC();
        if (tid == 0) {
            unsigned long long t = 0;
            for (int w = 0; w < kWarps; ++w) t += sm.wu[w][0];
            s_ctot = t;
        }
    }
    RP_CL_SYNC(cl);
    if (!trunc) {  // the whole vocabulary
        unsigned long long total = 0;
#pragma unroll
        for (int r = 0; r < nc; ++r) total += *cl.map_shared_rank(&s_ctot, r);
        res.tau = 0u;
        res.cut = -1;
        res.mass = total;
        res.count = V;
        return;
    }
    unsigned long long c = 0, m = 0;  // bin tid of the cluster's histogram
#pragma unroll
    for (int r = 0; r < nc; ++r) {
        c += cl.map_shared_rank(hc, r)[tid];
        if (with_mass) m += cl.map_shared_rank(hp, r)[tid];
    }
    __shared__ uint32_t s_cc[kBins];            // inclusive prefix counts
    __shared__ unsigned long long s_cm[kBins];  // inclusive prefix masses
    const unsigned long long cc = block_scan_u64(sm, c);
    const unsigned long long cm = with_mass ? block_scan_u64(sm, m) : 0ull;
    s_cc[tid] = static_cast<uint32_t>(cc);
    s_cm[tid] = cm;
    RP_SYNC();
    const unsigned long long n_in = s_cc[kBins - 1], total_mass = s_cm[kBins - 1];
    // top-k past s = 32 takes every token in range: the others weigh 0
    const unsigned long long k_eff = use_k ? min(static_cast<unsigned long long>(pol.top_k), n_in) : 0ull;

    // ---- the window of bins [wlo, whi] holding the cuts.  With top-k and
    // top-p together the window runs from the top-p crossing down to the top-k
    // bin; only its first bins (those where the top-p crossing can lie, up to
    // phi) and the top-k bin need their tokens: the bins between (the gap)
    // enter the cuts as their exact count and mass.
    __shared__ int s_win[3];
    __shared__ unsigned long long s_pl[6];  // above count / mass, window count, theta (top-p alone), gap count / mass
    if (tid == 0) {
        int whi = use_k ? first_at_least(s_cc, k_eff) : kBins - 1;
        int wlo = 0;
        unsigned long long theta = 0;
        const bool small = s_cc[whi] <= static_cast<uint32_t>(kThreads);
        if (with_mass) {
            // lower bound of the kept mass (exact when top-k is off)
            const unsigned long long mk_lo = use_k ? (whi ? s_cm[whi - 1] : 0ull) : total_mass;
            wlo = whi;
            if (use_p) {
                theta = p_threshold(pol.top_p, mk_lo);
                wlo = first_at_least(s_cm, theta);
                if (!use_k) whi = wlo;
            }
            if (small || s_cc[whi] <= static_cast<uint32_t>(kThreads)) wlo = 0;  // small support: all of it
        }
        int phi = whi;
        if (with_mass && use_k && use_p && !small) {
            // the kept mass is at most the mass through the top-k bin
            const int p_hi = first_at_least(s_cm, p_threshold(pol.top_p, s_cm[whi]));
            if (p_hi + 1 < whi) phi = p_hi;
        }
        const unsigned long long ac = wlo ? s_cc[wlo - 1] : 0ull;
        const unsigned long long gc = phi < whi ? s_cc[whi - 1] - s_cc[phi] : 0ull;
        s_win[0] = wlo;
        s_win[1] = whi;
        s_win[2] = phi;
        s_pl[0] = ac;
        s_pl[1] = wlo ? s_cm[wlo - 1] : 0ull;
        s_pl[2] = s_cc[whi] - ac - gc;
        s_pl[3] = theta;
        s_pl[4] = gc;
        s_pl[5] = phi < whi ? s_cm[whi - 1] - s_cm[phi] : 0ull;
    }
    RP_SYNC();
    const int wlo = s_win[0], whi = s_win[1], phi = s_win[2];
    const unsigned long long above_cnt = s_pl[0], above_mass = s_pl[1], wcount = s_pl[2], theta_p = s_pl[3];
    const unsigned long long gap_cnt = s_pl[4], gap_mass = s_pl[5];
    RP_SYNC();

    if (wcount > static_cast<unsigned long long>(kCap)) {
        const uint32_t klo = lowest_true_key(kmax, BinAtMost{zmax, inv_t, whi});  // the window's lowest key
        if (!use_k) {  // top-p alone: radix selection inside the window
            const uint32_t khi = wlo > 0 ? lowest_true_key(kmax, BinAtMost{zmax, inv_t, wlo - 1}) - 1u : kmax;
            auto all = [](uint32_t, int32_t) { return true; };
            uint32_t tau;
            unsigned long long above, eqc, eqm;
            if (radix_select<true>(sm, cl, sl, cbuf, klo, khi, above_mass, theta_p, zmax, inv_t, all, tau, above,
                                   eqc, eqm) &&
                eqc > 0) {
                // tied elements share one weight; take just enough of them in index order
                const unsigned long long wt = eqm / eqc;
                unsigned long long t = wt ? (theta_p - above + wt - 1) / wt : eqc;
                if (t < 1) t = 1;
                if (t > eqc) t = eqc;
                res.cut = tie_index(sm, cl, sl, tau, t, all);
                res.tau = tau;
                res.mass = above + t * wt;
                res.count = 0x7FFFFFFF;
                return;
            }
        }
        row_policy_radix(sm, cl, sl, V, pol, res, cbuf);
        res.count = 0x7FFFFFFF;
        return;
    }

    // ---- compact the window's elements (but the gap's) into rank 0's buffer.
    // The pick tests the exact bin; the floor only lets whole vectors be
    // skipped, so it is taken below the window's lowest value with margins
    // well past the rounding of s = (zmax - z)/T and of the subtraction.
    {
        const BinOf bin_of{zmax, inv_t};
        float zf = zmax - (static_cast<float>(whi + 1) * 0.125f / inv_t) * 1.0001f;
        zf -= fabsf(zf) * 1e-6f + 1e-30f;
        compact_candidates(sm, cl, sl, cbuf, zf, [=](float z, int32_t) {
            const int b = bin_of(z);
            return b >= wlo && b <= whi && (b <= phi || b == whi);
        });
    }

    // ---- rank 0: sort, take the cuts (prefix sums continue from the mass above the window)
    const int buf = sm.parity;
    if (rank == 0) {
        const int n = static_cast<int>(min(static_cast<unsigned long long>(sm.ccount), wcount));
        sort_candidates(cbuf, n);
        // buffer positions inside the top-k set (the gap's tokens are all in it)
        const int K = use_k ? static_cast<int>(min(k_eff - above_cnt - gap_cnt, static_cast<unsigned long long>(n)))
                            : n;
        auto wt = [&](int i) -> unsigned long long {
            return to_fixed(weight_f(key_to_float(vo_key(cbuf[i])), zmax, inv_t));
        };
        // one scan: the mass of the K kept candidates, then the top-p crossing
        // (theta relative to the mass above the window) and the prefix there
        unsigned long long part, pm;
        int pos;
        cut_scan(sm, K, wt,
                 [&](unsigned long long k_part) -> unsigned long long {
                     if (!use_p) return 0ull;
                     const unsigned long long kept = use_k ? above_mass + gap_mass + k_part : total_mass;
                     return p_threshold(pol.top_p, kept) - above_mass;
                 },
                 part, pos, pm);
        const unsigned long long kept = use_k ? above_mass + gap_mass + part : total_mass;
        int mm = K;
        unsigned long long mass = kept;
        if (use_p) {
            mm = pos < K ? pos + 1 : K;
            mass = above_mass + (pos < K ? pm : part);
        }
        mm = max(mm, 1);
        if (tid == 0) {
            const unsigned long long last = cbuf[mm - 1];
            sm.xu[buf][0] = vo_key(last);
            sm.xu[buf][1] = static_cast<unsigned long long>(static_cast<uint32_t>(vo_idx(last)));
            sm.xu[buf][2] = mass;
            sm.xu[buf][3] = above_cnt + static_cast<unsigned long long>(mm);
        }
    }
    RP_CL_SYNC(cl);
    if (tid < 4) sm.tot[tid] = cl.map_shared_rank(&sm.xu[buf][0], 0)[tid];
    RP_SYNC();
    res.tau = static_cast<uint32_t>(sm.tot[0]);
    res.cut = static_cast<int32_t>(static_cast<uint32_t>(sm.tot[1]));
    res.mass = sm.tot[2];
    res.count = static_cast<int32_t>(min(sm.tot[3], 0x7FFFFFFFull));
    res.in_buf = above_cnt == 0;
    RP_SYNC();
    if (tid == 0) sm.parity ^= 1;
    RP_SYNC();
}

// Inverse-CDF draw over a support held in rank 0's candidate buffer (its
// first n composite keys, in value order), in token-index order: the element
// whose token-order prefix of w(key, index) straddles floor(m * total / 2^24),
// m the 24-bit uniform.  Up to kThreads elements: each thread weighs one
// element once and sums the weights of the lower-indexed ones; larger sets
// are re-keyed by index and sorted.  Returns the token in rank 0 (-1 if the
// total is 0).  Rank 0's threads only; the buffer's upper half is scratch.
template <typename Wf>
__device__ int32_t draw_small_support(Smem& sm, unsigned long long* cbuf, int n, uint32_t m24, Wf w,
                                      unsigned long long& total) {
    if (n <= kThreads) {
        unsigned long long* wbuf = cbuf + kCap / 2;
        int32_t* ibuf = reinterpret_cast<int32_t*>(cbuf + kCap / 2 + kThreads);
        const int t = threadIdx.x;
        unsigned long long wt = 0;
        int32_t idx = 0x7FFFFFFF;
        if (t < n) {
            const unsigned long long c = cbuf[t];
            idx = vo_idx(c);
            wt = w(vo_key(c), idx);
            wbuf[t] = wt;
            ibuf[t] = idx;
        }
        const unsigned long long incl = block_scan_u64(sm, wt);  // also orders the scratch writes
        __shared__ unsigned long long s_tot;
        __shared__ int32_t s_pick;
        if (t == kThreads - 1) s_tot = incl;
        if (t == 0) s_pick = -1;
        RP_SYNC();
        total = s_tot;
        if (total == 0) return -1;
        const unsigned long long target =
            static_cast<unsigned long long>((static_cast<unsigned __int128>(m24) * total) >> 24);
        if (t < n && wt > 0) {
            unsigned long long before = 0;
            for (int j = 0; j < n; ++j) before += ibuf[j] < idx ? wbuf[j] : 0ull;
            if (before <= target && target < before + wt) s_pick = idx;
        }
        RP_SYNC();
        const int32_t pick = s_pick;
        RP_SYNC();
        return pick;
    }
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const unsigned long long c = cbuf[i];
        cbuf[i] = index_order(vo_key(c), vo_idx(c));
    }
    RP_SYNC();
    sort_desc(cbuf, n);
    auto wi = [&](int i) -> unsigned long long { return w(io_key(cbuf[i]), io_idx(cbuf[i])); };
    unsigned long long tot;
    find_crossing(sm, n, 0ull, true, wi, tot);
    total = tot;
    if (tot == 0) return -1;
    const unsigned long long target =
        static_cast<unsigned long long>((static_cast<unsigned __int128>(m24) * tot) >> 24);
    unsigned long long t2;
    const int pos = find_crossing(sm, n, target, true, wi, t2);
    const int32_t pick = pos < n ? io_idx(cbuf[pos]) : io_idx(cbuf[n - 1]);
    RP_SYNC();
    for (int i = threadIdx.x; i < n; i += kThreads) {  // back to value order keys
        const unsigned long long c = cbuf[i];
        cbuf[i] = value_order(io_key(c), io_idx(c));
    }
    RP_SYNC();
    return pick;
}

// Compact the elements of the slice satisfying pred(key, index) into rank 0's
// candidate buffer in value order (as value_order keys); returns their count
// in rank 0 (capped at kCap).  Every element satisfying pred is >= floor.
// Rank 0's counter must have been reset before a preceding cluster barrier.
template <typename Pred>
__device__ int compact_to_rank0(Smem& sm, cg::cluster_group& cl, const Slice& sl, unsigned long long* cbuf,
                                float floor, Pred pred) {
    compact_candidates(sm, cl, sl, cbuf, floor, [&](float z, int32_t idx) { return pred(ordered_key(z), idx); });
    return static_cast<int>(min(sm.ccount, static_cast<unsigned int>(kCap)));
}

// Normalise a request's policy record; returns false for an invalid one.
__device__ __forceinline__ bool make_policy(const dspark_policy& in, int V, Policy& out) {
    out.greedy = in.greedy != 0;
    out.inv_t = 1.0f;
    out.top_k = 0;
    out.top_p = 1.0f;
    if (out.greedy) return true;
    const float T = in.temperature;
    if (!(T > 0.0f) || isinf(T) || in.top_k < 0 || isnan(in.top_p)) return false;
    out.inv_t = 1.0f / T;
    out.top_k = (in.top_k > 0 && in.top_k < V) ? in.top_k : 0;
    out.top_p = in.top_p;
    return true;
}

}  // namespace rp
}  // namespace dspark
