// The draft's sequential head in one persistent launch: every step's Markov
// bias GEMM, sampling policy and draw, with the biased logits z kept in tensor
// memory [MB Semi-autoregressive draft; FT Checkpoint-faithful DSpark
// architecture; FT Exact decoding semantics > Probabilistic].
//
// Per step k (left to right) and request b:
//   z_k[b, v] = backbone[b, k-1, v] + sum_j U[x_{k-1}(b), j] * W[v, j]
//   q_k = policy(z_k) (temperature, top-k, top-p), written in full;
//   x_k = inverse-CDF draw from q_k in token order (greedy: the argmax).
//
// Layout.  Requests go in groups of up to 64 (the MMA's N; the library
// launches the kernel for one group, since groups run one after another and
// the per-step path beats that for larger batches); the vocabulary
// goes to the CTAs in contiguous ranges of 128-row tiles (the MMA's M), so a
// CTA's tokens precede the next CTA's in token order.  Tile j of a CTA lives
// in tensor-memory columns [64 j, 64 j + 64): lane = vocabulary row of the
// tile, column = request.  z never leaves the SM: the GEMM writes it there,
// every later phase of the step reads it there, and only q goes to HBM.
//
// Phases of a step, separated by grid barriers (all CTAs resident: a
// cooperative launch, one CTA per SM):
//   A  gather U[x_{k-1}] (B operand), stream W and backbone tiles by TMA,
//      tcgen05.mma into tensor memory; epilogue warps add the backbone, store
//      z back, and reduce each request's maximum and non-finite flag into
//      global words.                                              | barrier
//   B  greedy rows: the lowest index holding the maximum.  Sampled rows: a
//      16-bin histogram of s = (zmax - z)/T (bins of 2 below s = 32; exact
//      counts and, where top-p or a large top-k needs them, exact fixed-point
//      masses with the row engine's weights), reduced into global words.
//                                                                 | barrier
//   C  (every CTA, for every request) the window of bins holding the top-k
//      and top-p cuts, from the histogram's prefix sums (the row engine's
//      rule).  A one-bin window with more tokens than a candidate list holds
//      is refined once: a 16-bin histogram inside that bin (bins of 1/8),
//      a barrier, the window again over the finer bins.
//   D  compaction of the window's tokens into the request's candidate list
//      in global memory.  A window still too large makes the row "hard":
//      every CTA writes its z there instead.                      | barrier
//   E  the request's owner CTA sorts its candidates and takes the cuts by
//      exact prefix sums; with the whole support in the list it draws x_k at
//      once.  A hard row is done whole by its owner with the row engine
//      (row_policy.cuh) as one CTA.                              | barrier
//   F  every CTA writes its share of q (from tensor memory) and, for rows
//      whose support is not in a list, the support mass of its range.
//                                                      | barrier (if any)
//   G  the CTA whose range holds the draw finds x_k.    | barrier (if any)
// Every sum that decides a token is an integer (fixed-point weights,
// 2^-40), so decisions do not depend on the order of the reductions.
//
// The RNN head (the kernel's second instantiation) differs in two places:
//   A0 before A: the GRU cell s_k = GRU(s_{k-1}, U[x_{k-1}]) for the group's
//      requests, spread over every warp of the grid, into a state buffer in
//      the workspace.                                             | barrier
//   A: the B operand is s_k as two bf16 rows, hi = bf16(s) and lo =
//      bf16(s - hi), and every tile takes two MMAs into one accumulator,
//      z = backbone + hi W^T + lo W^T (s_k to about 2^-16 of its size).
//
// Waits are bounded (kWaitLimitNs); a wait that gives up sets the call's
// error word, every CTA then skips the remaining work, and the requests
// report DSPARK_REQ_TIMEOUT.

#include <cooperative_groups.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
// The row engine (hard rows, the owners' sorts and draws) runs on the first
// 256 threads of this kernel's 512, as a cluster of one CTA: its barriers are
// a named barrier of those threads.
#define RP_SYNC() asm volatile("bar.sync 1, 256;" ::: "memory")
#define RP_CL_SYNC(cl) RP_SYNC()
#include "row_policy.cuh"
#include "tc_common.cuh"

namespace dspark {

namespace {

using namespace tc;
namespace cg = cooperative_groups;

constexpr int kFT = 512;             // threads (16 warps)
constexpr int kEng = rp::kThreads;   // the first kEng threads run the row engine
constexpr int kNG = 64;              // requests per group (MMA N)
constexpr int kMaxLT = 8;            // vocabulary tiles per CTA (8 x 64 columns = all of tensor memory)
constexpr int kTileV = 128;          // vocabulary rows per tile (MMA M)
constexpr int kHB = 16;              // histogram bins: s in [2i, 2i + 2), s < 32; inside one: 16 of 1/8
constexpr int kCand = rp::kCap;      // candidates a list holds (the owner sorts them in shared memory)
constexpr int kWhole = rp::kThreads; // a support this small is compacted whole (drawn by its owner)
constexpr uint32_t kTmemCols = 512;
constexpr int kCountBins = 8;        // counts-only rows count the first 8 coarse bins (s < 16)

// request modes
enum : int { kModeNone = 0, kModeGreedy = 1, kModeWin = 2, kModeAll = 3, kModeHard = 4, kModeRefine = 5 };
// histogram work of a request in phase B: none, greedy argmax, counts, counts and masses
enum : int { kHistNone = 0, kHistGreedy = 1, kHistCount = 2, kHistMass = 3 };
// descriptor flags
enum : uint32_t { kDescDrawn = 1u, kDescPrefix = 2u, kDescDone = 4u };

// Per (group, step) words in the workspace, cleared by the host before the launch.
struct StepWords {
    uint32_t maxkey[kNG];     // ordered key of the row maximum (0: none yet)
    uint32_t bad[kNG];        // a NaN or +inf logit
    uint32_t amax[kNG];       // greedy: 0xFFFFFFFF - (lowest index holding the maximum), max-reduced
    uint32_t ccount[kNG];     // candidates claimed
    uint32_t hcnt[kNG][kHB];
    unsigned long long hmass[kNG][kHB];
    uint32_t hcnt2[kNG][kHB];            // the refinement inside one bin
    unsigned long long hmass2[kNG][kHB];
};
// The owner's result for a request of the current step.
struct Desc {
    uint32_t tau;
    int32_t cut;
    unsigned long long mass;   // fixed-point support mass
    unsigned long long target; // prefix draw: the first token whose inclusive prefix exceeds this
    uint32_t flags;
    int32_t pad;
};
// Window of one request (every CTA computes the same).  lvl 1: bins
// [wlo, whi] but (phi, whi) of the 16 coarse bins; lvl 2: those of the 16
// fine bins that split the coarse bins [rlo, rhi] evenly (fscale fine bins
// per unit of s), and (keep_above) every coarse bin before rlo.
struct Win {
    int mode;
    int lvl, rlo, rhi, keep_above;
    float fscale;
    int wlo, whi, phi;
    unsigned long long above_cnt, above_mass, wcount, gap_cnt, gap_mass, k_eff, total;
};

struct FusedParams {
    const uint16_t* backbone;   // bf16 [B, gamma, V]
    const uint16_t* U;          // bf16 [V, r]
    const int32_t* anchor;
    const dspark_policy* policy;  // null: all greedy
    const uint64_t* seed;
    const uint64_t* request_id;
    const int64_t* pos0;
    int B, gamma, V, r;
    int32_t* proposals;
    float* q;
    float* q_at_x;
    int32_t* status;
    // layout
    int ntiles, tpc, grid, groups, stages, bstages;
    // workspace
    unsigned int* bar;         // barrier arrivals (cleared before the launch)
    int* error;                // set when a wait gave up
    StepWords* words;          // [groups * gamma]
    unsigned long long* cand;  // [kNG][kCand] value-order keys
    Desc* desc;                // [kNG]
    unsigned long long* part;  // [kNG][grid] support mass of each CTA's range
    float* zhard;              // [kNG][V] z of hard rows
    // the RNN head (rnn = 1): the GRU cell's weights and its state s_k,
    // fp32 [2][kNG][r] (step k writes buffer k & 1)
    int rnn;
    const uint16_t* Wi;
    const uint16_t* Wh;
    const float* bi;
    const float* bh;
    float* state;
};

struct FusedSmem {
    uint64_t wfull[4], wempty[4], bfull[4], bempty[4];
    uint64_t accfull[kMaxLT];
    uint32_t tmem_base;
    int abort;
    int barrier_ok;
    int any_prefix;
    int any_refine;
    int32_t x[kNG];
    uint32_t smax[kMaxLT][kNG];  // per tile and request: the largest ordered key of its 128 rows (0: none)
    uint32_t cbad[4][kNG];
    uint32_t floor_key[kNG];     // a pass's threshold: slabs whose maximum is below it hold no work
    // per request of the group, for the policy phases
    float zmax[kNG];
    float inv_t[kNG];
    float inv_s[kNG];    // 1 / support mass (phase F)
    float ba[kNG], bb[kNG];  // bin coefficients (bin_val)
    int mode[kNG];
    int hist[kNG];
    int32_t code[kNG];   // the row's status when it fails at this step
    Win win[kNG];
    Desc d[kNG];
    unsigned long long wpart[4][kNG];   // per quadrant: support mass of the CTA's rows
    unsigned long long qsum[4];         // the draw's scan: per quadrant sums of one tile
    unsigned long long ex;              // the draw's scan: mass of the CTAs before this one
    int32_t pick[4];
};

// ------------------------------------------------------------- helpers
__device__ __forceinline__ uint32_t ld_cg_u32(const uint32_t* p) { return __ldcg(p); }
__device__ __forceinline__ unsigned long long ld_cg_u64(const unsigned long long* p) { return __ldcg(p); }

__device__ __forceinline__ void red_max_u32(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_or_u32(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.or.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add_u32(uint32_t* p, uint32_t v) {
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Grid barrier: arrivals counted on bar[0] for the whole launch (generation
// g waits for g * nctas arrivals); bounded, and a wait that gives up (or an
// error set elsewhere) makes the CTA abort.
// gen: this thread's count of the barriers passed (the same in every thread)
__device__ void grid_sync(const FusedParams& p, FusedSmem& sm, unsigned& gen) {
    if (!grid_barrier_bounded(p.bar, p.error, ++gen * gridDim.x, kWaitLimitNs, &sm.barrier_ok)) sm.abort = 1;
}

// Bins of s = (zmax - z) / T in half units, bf = s / 2, taken as one fma
// -z * ba + bb with ba = inv_t / 2, bb = zmax * ba (monotone in z; every
// phase bins a token the same way): coarse bin floor(bf) below bf = 16 (kHB
// beyond), fine bins splitting the coarse bins [rlo, rhi] in 16 even steps.
__device__ __forceinline__ float bin_val(float z, float ba, float bb) { return fmaf(-z, ba, bb); }
__device__ __forceinline__ int coarse_bin(float bf) { return bf < 16.0f ? min(kHB - 1, static_cast<int>(bf)) : kHB; }
__device__ __forceinline__ int fine_bin(float bf, int rlo, float fscale) {
    return min(kHB - 1, max(0, static_cast<int>((bf - static_cast<float>(rlo)) * fscale)));
}

// An ordered key below which every token has s = (zmax - z) * inv_t >= S
// (margins far past the rounding of s): a slab whose maximum is below it
// has no token with s < S.
__device__ __forceinline__ uint32_t floor_key_s(float zmax, float inv_t, float S) {
    float zf = zmax - (S / inv_t) * 1.0001f;
    zf -= fabsf(zf) * 1e-6f + 1e-30f;
    return ordered_key(zf);
}
// Is any of the 8 slabs (tile j, requests c0..c0+7) at or above its request's floor?
__device__ __forceinline__ bool any_active8(const uint32_t* smax_j, const uint32_t* floor_key, int c0) {
    bool a = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) a |= smax_j[c0 + i] >= floor_key[c0 + i];
    return a;
}

__device__ __forceinline__ float inv_mass(unsigned long long mass) {
    return static_cast<float>(rp::kFix / static_cast<double>(mass));
}

// The window of bins holding a row's cuts from NB bins' inclusive prefix
// sums cc (counts) and cm (masses): the row engine's rule (a support of at
// most kWhole tokens is compacted whole, so that its owner can draw).
template <int NB>
__device__ Win make_window(const rp::Policy& pol, const unsigned long long* cc, const unsigned long long* cm) {
    Win w{};
    const bool use_k = pol.top_k > 0, use_p = pol.top_p < 1.0f;
    w.total = cm[NB - 1];
    w.lvl = 1;
    if (!use_k && !use_p) {
        w.mode = kModeAll;
        return w;
    }
    const bool with_mass = !use_k || pol.top_k > kWhole;
    const unsigned long long n_in = cc[NB - 1];
    w.k_eff = use_k ? min(static_cast<unsigned long long>(pol.top_k), n_in) : 0ull;
    // (unrolled scans and selects: the prefix sums stay in registers)
    auto first_at_least = [](const unsigned long long* pre, unsigned long long x) {
        int i = NB - 1;
#pragma unroll
        for (int b = NB - 2; b >= 0; --b)
            if (pre[b] >= x) i = b;
        return i;
    };
    auto at = [](const unsigned long long* pre, int idx) {
        unsigned long long v = 0;
#pragma unroll
        for (int b = 0; b < NB; ++b)
            if (b == idx) v = pre[b];
        return v;
    };
    int whi = use_k ? first_at_least(cc, w.k_eff) : NB - 1;
    int wlo = 0;
    const bool small = at(cc, whi) <= static_cast<unsigned long long>(kWhole);
    if (with_mass) {
        const unsigned long long mk_lo = use_k ? (whi ? at(cm, whi - 1) : 0ull) : w.total;
        wlo = whi;
        if (use_p) {
            wlo = first_at_least(cm, rp::p_threshold(pol.top_p, mk_lo));
            if (!use_k) whi = wlo;
        }
        if (small || at(cc, whi) <= static_cast<unsigned long long>(kWhole)) wlo = 0;
    }
    int phi = whi;
    if (with_mass && use_k && use_p && !small) {
        const int p_hi = first_at_least(cm, rp::p_threshold(pol.top_p, at(cm, whi)));
        if (p_hi + 1 < whi) phi = p_hi;
    }
    const unsigned long long ac = wlo ? at(cc, wlo - 1) : 0ull;
    const unsigned long long gc = phi < whi ? at(cc, whi - 1) - at(cc, phi) : 0ull;
    w.wlo = wlo;
    w.whi = whi;
    w.phi = phi;
    w.above_cnt = ac;
    w.above_mass = wlo ? at(cm, wlo - 1) : 0ull;
    w.wcount = at(cc, whi) - ac - gc;
    w.gap_cnt = gc;
    w.gap_mass = phi < whi ? at(cm, whi - 1) - at(cm, phi) : 0ull;
    if (NB == kHB && !with_mass && cc[kCountBins - 1] < static_cast<unsigned long long>(pol.top_k)) {
        // counts only: the top-k crossing lies past the counted bins: refine
        // the rest of s < 32, keep the bins before
        w.mode = kModeRefine;
        w.rlo = kCountBins;
        w.rhi = kHB - 1;
        w.fscale = 16.0f / static_cast<float>(w.rhi - w.rlo + 1);
        return w;
    } else if (w.wcount <= static_cast<unsigned long long>(kCand)) {
        w.mode = kModeWin;
    } else {
        // too many tokens: refine the window's coarse bins into 16 finer ones
        // Counts only (top-k <= kWhole): the bins before the top-k bin hold
        // fewer than k tokens; refine the top-k bin and keep them whole.
        w.mode = kModeRefine;
        w.rlo = with_mass ? wlo : whi;
        w.rhi = whi;
        w.fscale = 16.0f / static_cast<float>(w.rhi - w.rlo + 1);
    }
    return w;
}

// Is a token of coarse bin b1 (and fine bin b2, level 2) in the window?
__device__ __forceinline__ bool in_window(const Win& w, int b1, int b2) {
    if (w.lvl == 2) {
        if (b1 < w.rlo) return w.keep_above != 0;
        if (b1 > w.rhi) return false;
        b1 = b2;
    }
    return b1 >= w.wlo && b1 <= w.whi && (b1 <= w.phi || b1 == w.whi);
}

// RNN head, phase A0 of step k: the GRU cell s_k = GRU(s_{k-1}, U[x_{k-1}])
// (gate order r, z, n; s_0 = 0) for the group's nb requests.  Work items
// (state unit u, 4 requests) go to every warp of the grid; a warp's lanes
// split K eight elements each, so each of the unit's six weight rows (Wi and
// Wh at u, r + u, 2r + u) is one coalesced read; the lanes' partial dot
// products are summed by a butterfly and lane m applies the gates for
// request m0 + m.  s_{k-1} is read through L2 (other CTAs wrote it); s_k goes
// to the other state buffer, which the gather reads after a grid barrier.
__device__ __forceinline__ void gru_phase(const FusedParams& p, const int32_t* xsm, int k, int g, int nb, int warp,
                                          int lane) {
    const int r = p.r;
    const float* sprev = p.state + static_cast<size_t>((k - 1) & 1) * kNG * r;
    float* scur = p.state + static_cast<size_t>(k & 1) * kNG * r;
    constexpr int kM = 4;  // requests per work item
    const int items = ((nb + kM - 1) / kM) * r;
    const int k0 = lane * 8;  // this lane's 8 elements of K
    for (int it = blockIdx.x * (kFT / 32) + warp; it < items; it += gridDim.x * (kFT / 32)) {
        const int u = it % r, m0 = (it / r) * kM;
        const float bir = p.bi[u], biz = p.bi[r + u], bin = p.bi[2 * r + u];
        const float bhr = p.bh[u], bhz = p.bh[r + u], bhn = p.bh[2 * r + u];
        // lane m's s_{k-1} at unit u, for the gate update (loaded with the rest)
        const float sp = (k > 1 && lane < kM && m0 + lane < nb) ? __ldcg(sprev + (m0 + lane) * r + u) : 0.0f;
        float acc[6][kM];
#pragma unroll
        for (int q6 = 0; q6 < 6; ++q6)
#pragma unroll
            for (int m = 0; m < kM; ++m) acc[q6][m] = 0.0f;
        if (k0 < r) {
            // every load of the item first (tokens, then embedding and state
            // rows, then weights), so that they overlap
            int32_t xs[kM];  // x_{k-1} of the item's requests (-1: none or invalid)
#pragma unroll
            for (int m = 0; m < kM; ++m) xs[m] = m0 + m < nb ? xsm[m0 + m] : -1;
            uint4 ev[kM];
            float4 s0[kM], s1[kM];
#pragma unroll
            for (int m = 0; m < kM; ++m) {
                const int c = m0 + m;
                ev[m] = xs[m] >= 0 ? __ldg(reinterpret_cast<const uint4*>(p.U + static_cast<int64_t>(xs[m]) * r + k0))
                                   : make_uint4(0u, 0u, 0u, 0u);
                const bool has_s = k > 1 && c < nb;
                s0[m] = has_s ? __ldcg(reinterpret_cast<const float4*>(sprev + c * r + k0)) : make_float4(0.f, 0.f, 0.f, 0.f);
                s1[m] = has_s ? __ldcg(reinterpret_cast<const float4*>(sprev + c * r + k0 + 4))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            uint4 wv[6];
#pragma unroll
            for (int q6 = 0; q6 < 6; ++q6)
                wv[q6] = __ldg(reinterpret_cast<const uint4*>((q6 < 3 ? p.Wi : p.Wh) +
                                                              static_cast<int64_t>((q6 % 3) * r + u) * r + k0));
#pragma unroll
            for (int q6 = 0; q6 < 6; ++q6) {
                const float wf[8] = {bf16_lo(wv[q6].x), bf16_hi(wv[q6].x), bf16_lo(wv[q6].y), bf16_hi(wv[q6].y),
                                     bf16_lo(wv[q6].z), bf16_hi(wv[q6].z), bf16_lo(wv[q6].w), bf16_hi(wv[q6].w)};
#pragma unroll
                for (int m = 0; m < kM; ++m) {
                    float v[8];
                    if (q6 < 3) {
                        v[0] = bf16_lo(ev[m].x); v[1] = bf16_hi(ev[m].x); v[2] = bf16_lo(ev[m].y); v[3] = bf16_hi(ev[m].y);
                        v[4] = bf16_lo(ev[m].z); v[5] = bf16_hi(ev[m].z); v[6] = bf16_lo(ev[m].w); v[7] = bf16_hi(ev[m].w);
                    } else {
                        v[0] = s0[m].x; v[1] = s0[m].y; v[2] = s0[m].z; v[3] = s0[m].w;
                        v[4] = s1[m].x; v[5] = s1[m].y; v[6] = s1[m].z; v[7] = s1[m].w;
                    }
                    float t = acc[q6][m];
#pragma unroll
                    for (int l = 0; l < 8; ++l) t = fmaf(wf[l], v[l], t);
                    acc[q6][m] = t;
                }
            }
        }
#pragma unroll
        for (int q6 = 0; q6 < 6; ++q6)
#pragma unroll
            for (int m = 0; m < kM; ++m)
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[q6][m] += __shfl_xor_sync(0xFFFFFFFFu, acc[q6][m], o);
#pragma unroll
        for (int m = 0; m < kM; ++m) {
            const int c = m0 + m;
            if (lane != m || c >= nb) continue;
            const float rg = 1.0f / (1.0f + expf(-((acc[0][m] + bir) + (acc[3][m] + bhr))));
            const float zg = 1.0f / (1.0f + expf(-((acc[1][m] + biz) + (acc[4][m] + bhz))));
            const float n = tanhf((acc[2][m] + bin) + rg * (acc[5][m] + bhn));
            scur[c * r + u] = (1.0f - zg) * n + zg * sp;
        }
    }
}

// ------------------------------------------------------------------ kernel
// kRnn: the RNN head (p.rnn set), a kernel of its own so that the Markov
// head's registers are not shared with the GRU phase
template <bool kRnn>
__global__ void __launch_bounds__(kFT, 1)
    markov_fused_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap bmap,
                        const FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ FusedSmem sm;
    __shared__ rp::Smem rsm;
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r = p.r, S = p.stages, SB = p.bstages, V = p.V;  // W and backbone stages
    const uint32_t w_bytes = static_cast<uint32_t>(kTileV * r * 2);  // one W stage
    const uint32_t b_bytes = static_cast<uint32_t>(kNG * kTileV * 2);  // one backbone stage
    uint8_t* sW = smem;
    uint8_t* sB = sW + S * w_bytes;
    uint8_t* sU = sB + SB * b_bytes;  // also the owner's candidate buffer (and the row engine's scratch)
    uint8_t* sU2 = sU + kNG * r * 2;  // RNN head: the state's lo rows (sU holds its hi rows)
    unsigned long long* cbuf = reinterpret_cast<unsigned long long*>(sU);
    // the histograms of phases B and C live there too (the step's MMAs have read U by then)
    unsigned long long (*hmass)[kHB] = reinterpret_cast<unsigned long long (*)[kHB]>(sU);
    uint32_t (*hcnt)[kHB] = reinterpret_cast<uint32_t (*)[kHB]>(sU + kNG * kHB * 8);

    const int t0 = blockIdx.x * p.tpc;                        // first tile of this CTA
    const int ntl = max(0, min(p.tpc, p.ntiles - t0));        // its tiles

    if (warp == 0) tmem_alloc(&sm.tmem_base, kTmemCols);
    if (tid == 0) {
        for (int s = 0; s < 4; ++s) {
            mbar_init(&sm.wfull[s], 1);
            mbar_init(&sm.wempty[s], 1);
            mbar_init(&sm.bfull[s], 1);
            mbar_init(&sm.bempty[s], 8);
        }
        for (int j = 0; j < kMaxLT; ++j) mbar_init(&sm.accfull[j], 1);
        sm.abort = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;
    unsigned bar_gen = 0;  // grid barriers passed
    // policy phases: warp w reads TMEM lane quadrant w % 4 and the 16 columns
    // [16 (w / 4), 16 (w / 4) + 16)
    const int q = warp & 3, cq = (warp >> 2) * 16;
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);

    // producers: thread 0 the W tiles and the MMAs, thread 32 the backbone tiles
    int w_issued = 0, b_issued = 0, mma_done = 0;
    const int steps_total = p.groups * p.gamma;
    auto tile_of = [&](int n) { return n % max(ntl, 1); };         // n-th tile of the whole launch
    auto step_of = [&](int n) { return n / max(ntl, 1); };         // its (group, step) index
    // W is read again every step: keep it in L2; the backbone streams through
    const uint64_t pol_keep = l2_policy_evict_last(), pol_stream = l2_policy_evict_first();
    auto issue_w = [&](int n) {
        const int s = n % S;
        mbar_arrive_expect_tx(&sm.wfull[s], w_bytes);
        uint8_t* dst = sW + s * w_bytes;
        const int t = t0 + tile_of(n);
        for (int kb = 0; kb < r / 64; ++kb)
            tma_load_2d_hint(dst + kb * kTileV * 128, &wmap, kb * 64, t * kTileV, &sm.wfull[s], pol_keep);
    };
    auto issue_b = [&](int n) {
        const int s = n % SB;
        const int gs = step_of(n), g = gs / p.gamma, k = gs % p.gamma;  // k 0-based
        mbar_arrive_expect_tx(&sm.bfull[s], b_bytes);
        const int t = t0 + tile_of(n);
        tma_load_3d_hint(sB + s * b_bytes, &bmap, t * kTileV, k, g * kNG, &sm.bfull[s], pol_stream);
    };
    const int total_tiles = steps_total * ntl;
    if (tid == 0)
        for (; w_issued < min(S, total_tiles); ++w_issued) issue_w(w_issued);
    if (tid == 32)
        for (; b_issued < min(SB, total_tiles); ++b_issued) issue_b(b_issued);

    for (int gs = 0; gs < steps_total; ++gs) {
        const int g = gs / p.gamma, k = gs % p.gamma + 1;  // k 1-based
        const int nb = min(kNG, p.B - g * kNG);           // requests of the group
        StepWords& sw = p.words[gs];
        const bool aborted = sm.abort != 0;

        // ------------------------------------------------ A0 (RNN head): the GRU cell
        if constexpr (kRnn) {
            if (tid < kNG) {
                int32_t x = -1;
                if (tid < nb) {
                    const int b = g * kNG + tid;
                    x = k == 1 ? p.anchor[b] : __ldcg(p.proposals + static_cast<int64_t>(b) * p.gamma + (k - 2));
                    if (x < 0 || x >= V) x = -1;
                }
                sm.x[tid] = x;
            }
            __syncthreads();
            if (!sm.abort) gru_phase(p, sm.x, k, g, nb, warp, lane);
            grid_sync(p, sm, bar_gen);  // ---------------------------------- barrier 0
        }

        // ------------------------------------------------ A: gather, GEMM, epilogue
        if (tid < kNG) {
            int32_t x = -1;
            if (tid < nb) {
                const int b = g * kNG + tid;
                x = k == 1 ? p.anchor[b] : __ldcg(p.proposals + static_cast<int64_t>(b) * p.gamma + (k - 2));
                if (x < 0 || x >= V) x = -1;
            }
            sm.x[tid] = x;
        }
        for (int i = tid; i < kMaxLT * kNG; i += kFT) (&sm.smax[0][0])[i] = 0u;
        for (int i = tid; i < 4 * kNG; i += kFT) (&sm.cbad[0][0])[i] = 0u;
        __syncthreads();
        {
            const int kchunks = r / 8;
            if constexpr (!kRnn) {
                for (int c = tid; c < kNG * kchunks; c += kFT) {
                    const int row = c / kchunks, kc = c % kchunks;
                    const int32_t x = sm.x[row];
                    uint8_t* d = sU + chunk_off<true>(row, kc, kNG);
                    if (x >= 0) cp_async16(d, p.U + static_cast<int64_t>(x) * r + kc * 8);
                    else *reinterpret_cast<uint4*>(d) = make_uint4(0u, 0u, 0u, 0u);
                }
                cp_async_wait_all();
            } else {
                // the state s_k as two bf16 operands, hi = bf16(s) and lo =
                // bf16(s - hi) (s to about 2^-16): the bias is hi W^T + lo W^T
                const float* sk = p.state + static_cast<size_t>(k & 1) * kNG * r;
                for (int c = tid; c < kNG * kchunks; c += kFT) {
                    const int row = c / kchunks, kc = c % kchunks;
                    uint4 hv = make_uint4(0u, 0u, 0u, 0u), lv = make_uint4(0u, 0u, 0u, 0u);
                    if (sm.x[row] >= 0) {
                        const float4 a0 = __ldcg(reinterpret_cast<const float4*>(sk + row * r + kc * 8));
                        const float4 a1 = __ldcg(reinterpret_cast<const float4*>(sk + row * r + kc * 8 + 4));
                        const float v[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                        uint32_t hw[4], lw[4];
#pragma unroll
                        for (int l = 0; l < 4; ++l) {
                            const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * l]), h1 = __float2bfloat16_rn(v[2 * l + 1]);
                            const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * l] - __bfloat162float(h0));
                            const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * l + 1] - __bfloat162float(h1));
                            hw[l] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                                    (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
                            lw[l] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
                                    (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
                        }
                        hv = make_uint4(hw[0], hw[1], hw[2], hw[3]);
                        lv = make_uint4(lw[0], lw[1], lw[2], lw[3]);
                    }
                    const uint32_t off = chunk_off<true>(row, kc, kNG);
                    *reinterpret_cast<uint4*>(sU + off) = hv;
                    *reinterpret_cast<uint4*>(sU2 + off) = lv;
                }
            }
            fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t par = static_cast<uint32_t>(gs & 1);  // accumulator barriers complete once per step

        if (warp == 0) {
            if (lane == 0 && !aborted) {
                const uint32_t idesc = instr_desc(128, kNG);
                const uint32_t ubase = smem_u32(sU), ubase2 = smem_u32(sU2), wbase = smem_u32(sW);
                for (int j = 0; j < ntl; ++j) {
                    const int n = gs * ntl + j, s = n % S;
                    if (!mbar_wait(&sm.wfull[s], (n / S) & 1, kWaitLimitNs)) {
                        atomicExch(p.error, 1);
                        sm.abort = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem + static_cast<uint32_t>(j * kNG);
                    for (int ks = 0; ks < r / 16; ++ks)
                        mma_bf16(d, op_desc<true>(wbase + s * w_bytes, ks, kTileV), op_desc<true>(ubase, ks, kNG), idesc,
                                 ks > 0 ? 1u : 0u);
                    if constexpr (kRnn)  // the lo product into the same accumulator
                        for (int ks = 0; ks < r / 16; ++ks)
                            mma_bf16(d, op_desc<true>(wbase + s * w_bytes, ks, kTileV), op_desc<true>(ubase2, ks, kNG),
                                     idesc, 1u);
                    mma_commit(&sm.wempty[s]);
                    mma_commit(&sm.accfull[j]);
                    ++mma_done;
                    // refill this stage S tiles ahead once its MMAs have read it
                    // (a short wait: S tiles stay in flight)
                    if (w_issued < total_tiles && w_issued <= n + S) {
                        if (!mbar_wait(&sm.wempty[s], (n / S) & 1, kWaitLimitNs)) {
                            atomicExch(p.error, 1);
                            sm.abort = 1;
                            break;
                        }
                        issue_w(w_issued++);
                    }
                }
            }
        } else if (warp == 1) {
            // the backbone stream: S tiles ahead of the epilogue, each stage
            // refilled once the epilogue has read it (the epilogue needs only
            // MMAs that thread 0 issues without waiting for this thread)
            if (lane == 0 && !aborted) {
                for (int j = 0; j < ntl; ++j) {
                    const int n = gs * ntl + j;
                    bool ok = true;
                    while (b_issued < total_tiles && b_issued <= n + SB - 1) {
                        const int m = b_issued - SB;
                        if (m >= 0 && !mbar_wait(&sm.bempty[m % SB], (m / SB) & 1, kWaitLimitNs)) {
                            atomicExch(p.error, 1);
                            sm.abort = 1;
                            ok = false;
                            break;
                        }
                        issue_b(b_issued++);
                    }
                    if (!ok) break;
                }
            }
        } else if (warp >= 8) {
            // epilogue: warp w takes TMEM lane quadrant w % 4 of every tile and
            // the 32 columns [32 eh, 32 eh + 32), in chunks of 16
            const int eq = warp & 3, eh = (warp - 8) >> 2;
            const uint32_t te = tmem + (static_cast<uint32_t>(eq * 32) << 16) + static_cast<uint32_t>(eh * 32);
            const float ninf = -__int_as_float(0x7F800000);
            for (int j = 0; j < ntl && !aborted; ++j) {
                const int n = gs * ntl + j, s = n % SB;  // the backbone stage
                if (!mbar_wait(&sm.accfull[j], par, kWaitLimitNs) || !mbar_wait(&sm.bfull[s], (n / SB) & 1, kWaitLimitNs)) {
                    atomicExch(p.error, 1);
                    sm.abort = 1;
                    break;
                }
                tc_fence_after();
                const int vl = eq * 32 + lane;                // row of the tile
                const bool valid = (t0 + j) * kTileV + vl < V;
                const uint16_t* bb = reinterpret_cast<const uint16_t*>(sB + s * b_bytes) + eh * 32 * kTileV + vl;
                float mx[32];  // this row's logit per request, NaN-propagating (rows past V: -inf)
#pragma unroll
                for (int h16 = 0; h16 < 2; ++h16) {
                    uint32_t acc[16];
                    const uint32_t ta = te + static_cast<uint32_t>(j * kNG + h16 * 16);
                    tmem_ld16(ta, acc);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float z = valid ? __uint_as_float(acc[i]) +
                                                    __uint_as_float(static_cast<uint32_t>(bb[(h16 * 16 + i) * kTileV]) << 16)
                                              : ninf;
                        acc[i] = __float_as_uint(z);
                        mx[h16 * 16 + i] = z;
                    }
                    tmem_st16(ta, acc);
                }
                // slab maxima (this tile, 32 requests) over the warp's 32 rows
                // with a NaN-propagating max (a NaN or +inf maximum marks the
                // row non-finite): a transposing butterfly leaves request
                // eh * 32 + lane's in this lane
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const bool upper = (lane & o) != 0;
#pragma unroll
                    for (int i = 0; i < o; ++i) {
                        const float keep = upper ? mx[i + o] : mx[i];
                        const float give = upper ? mx[i] : mx[i + o];
                        mx[i] = fmax_nan(keep, __shfl_xor_sync(0xFFFFFFFFu, give, o));
                    }
                }
                const float m = mx[0];
                if (bad_logit(m)) sm.cbad[eq][eh * 32 + lane] = 1u;
                else if (m != ninf) atomicMax(&sm.smax[j][eh * 32 + lane], ordered_key(m));
                tmem_wait_st();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.bempty[s]);
            }
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid < nb && !sm.abort) {
            uint32_t m = 0u;
            for (int j = 0; j < ntl; ++j) m = max(m, sm.smax[j][tid]);
            const uint32_t bd = sm.cbad[0][tid] | sm.cbad[1][tid] | sm.cbad[2][tid] | sm.cbad[3][tid];
            if (m) red_max_u32(&sw.maxkey[tid], m);
            if (bd) red_or_u32(&sw.bad[tid], 1u);
        }
        grid_sync(p, sm, bar_gen);  // ---------------------------------------- barrier 1

        // ------------------------------------------------ B: greedy argmax, histograms
        if (tid < kNG) {
            int mode = kModeNone, hist = kHistNone;
            int32_t code = kReqOk;
            float zm = 0.0f, it = 1.0f;
            if (tid < nb && sm.x[tid] >= 0 && !sm.abort) {
                const int b = g * kNG + tid;
                const uint32_t mk = ld_cg_u32(&sw.maxkey[tid]);
                const bool bad = ld_cg_u32(&sw.bad[tid]) != 0;
                rp::Policy pol;
                const bool pol_ok = p.policy ? rp::make_policy(p.policy[b], V, pol)
                                             : (pol = rp::Policy{1.0f, 0, 1.0f, 1}, true);
                zm = mk ? key_to_float(mk) : -__int_as_float(0x7F800000);
                const bool empty = mk == 0 || zm == -__int_as_float(0x7F800000);
                it = pol.inv_t;
                // the row engine's order: non-finite, then empty, then an invalid policy
                code = bad ? kReqNonfinite : (empty ? kReqEmpty : (pol_ok ? kReqOk : kReqBadPolicy));
                if (code == kReqOk) {
                    mode = pol.greedy ? kModeGreedy : kModeWin;  // Win refined in C
                    hist = pol.greedy ? kHistGreedy
                                      : ((pol.top_k > 0 && pol.top_k <= kWhole) ? kHistCount : kHistMass);
                }
            }
            sm.mode[tid] = mode;
            sm.hist[tid] = hist;
            sm.code[tid] = code;
            sm.zmax[tid] = zm;
            sm.inv_t[tid] = it;
            sm.ba[tid] = 0.5f * it;
            sm.bb[tid] = zm * (0.5f * it);
            // slabs that can hold work: greedy rows the maximum, counts-only
            // rows s < 16, other sampled rows s < 32
            sm.floor_key[tid] = hist == kHistNone ? 0xFFFFFFFFu
                              : hist == kHistGreedy ? ordered_key(zm)
                              : floor_key_s(zm, it, hist == kHistCount ? 2.0f * kCountBins : 32.0f);
        }
        for (int i = tid; i < kNG * kHB; i += kFT) {
            (&hcnt[0][0])[i] = 0u;
            (&hmass[0][0])[i] = 0ull;
        }
        // next step's first W stages (the W ring is free: this step's MMAs are done)
        if (tid == 0 && !sm.abort) {
            while (w_issued < total_tiles && w_issued < (gs + 1) * ntl + S && w_issued < mma_done + S) {
                const int m = w_issued - S;
                if (m >= 0 && !mbar_wait(&sm.wempty[m % S], (m / S) & 1, kWaitLimitNs)) {
                    atomicExch(p.error, 1);
                    sm.abort = 1;
                    break;
                }
                issue_w(w_issued++);
            }
        }
        __syncthreads();
        if (!sm.abort) {
            for (int c0 = cq; c0 < cq + 16; c0 += 8) {
                // counts-only rows count s < 2 kCountBins only (a top-k
                // crossing past it is refined over the rest in phase C)
                int hmr[8];
                float zmr[8], bar_[8], bbr[8], itr[8];
                uint32_t flr[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    hmr[i] = sm.hist[c0 + i];
                    zmr[i] = sm.zmax[c0 + i];
                    itr[i] = sm.inv_t[c0 + i];
                    bar_[i] = sm.ba[c0 + i];
                    bbr[i] = sm.bb[c0 + i];
                    flr[i] = sm.floor_key[c0 + i];
                }
                for (int j = 0; j < ntl; ++j) {
                    uint32_t act = 0u;
#pragma unroll
                    for (int i = 0; i < 8; ++i) act |= (sm.smax[j][c0 + i] >= flr[i] ? 1u : 0u) << i;
                    if (!act) continue;
                    uint32_t zr[8];
                    tmem_ld8(tq + static_cast<uint32_t>(j * kNG + c0), zr);
                    tmem_wait_ld();
                    const int v = (t0 + j) * kTileV + q * 32 + lane;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int hm = hmr[i];
                        if (hm <= kHistGreedy || !((act >> i) & 1u)) continue;
                        const float z = __uint_as_float(zr[i]);
                        const float bf = v < V ? bin_val(z, bar_[i], bbr[i]) : 16.0f;
                        if (hm == kHistCount) {
                            if (bf < static_cast<float>(kCountBins)) atomicAdd(&hcnt[c0 + i][static_cast<int>(bf)], 1u);
                        } else if (bf < 16.0f) {
                            const int bin = min(kHB - 1, static_cast<int>(bf));
                            atomicAdd(&hcnt[c0 + i][bin], 1u);
                            atomicAdd(&hmass[c0 + i][bin],
                                      static_cast<unsigned long long>(rp::to_fixed(rp::weight_f(z, zmr[i], itr[i]))));
                        }
                    }
                }
                // greedy rows: the lowest index holding the maximum
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (hmr[i] != kHistGreedy) continue;
                    const int c = c0 + i;
                    const uint32_t mk = ordered_key(zmr[i]);
                    for (int j = 0; j < ntl; ++j) {
                        if (sm.smax[j][c] < mk) continue;
                        const uint32_t z = tmem_ld1(tq + static_cast<uint32_t>(j * kNG + c));
                        tmem_wait_ld();
                        const int v = (t0 + j) * kTileV + q * 32 + lane;
                        const bool hit = v < V && ordered_key(__uint_as_float(z)) == mk;
                        const uint32_t best = __reduce_max_sync(0xFFFFFFFFu, hit ? 0xFFFFFFFFu - static_cast<uint32_t>(v) : 0u);
                        if (lane == 0 && best) red_max_u32(&sw.amax[c], best);
                    }
                }
            }
        }
        __syncthreads();
        for (int i = tid; i < kNG * kHB; i += kFT) {
            const int c = i / kHB;
            if (sm.hist[c] < kHistCount) continue;
            const uint32_t cn = (&hcnt[0][0])[i];
            if (cn) {
                red_add_u32(&sw.hcnt[0][0] + i, cn);
                if (sm.hist[c] == kHistMass) red_add_u64(&sw.hmass[0][0] + i, (&hmass[0][0])[i]);
            }
        }
        grid_sync(p, sm, bar_gen);  // ---------------------------------------- barrier 2

        // ------------------------------------------------ C: windows (every CTA)
        for (int i = tid; i < kNG * kHB; i += kFT) {  // the histograms, all loads in flight at once
            const int c = i / kHB;
            if (sm.mode[c] != kModeWin) continue;
            (&hcnt[0][0])[i] = ld_cg_u32(&sw.hcnt[0][0] + i);
            (&hmass[0][0])[i] = sm.hist[c] == kHistMass ? ld_cg_u64(&sw.hmass[0][0] + i) : 0ull;
        }
        __syncthreads();
        if (tid < kNG) {
            const int c = tid;
            if (sm.mode[c] != kModeWin) {
                sm.win[c].mode = sm.mode[c];
            } else {
                unsigned long long cc[kHB], cm[kHB], a = 0, m = 0;
                for (int i = 0; i < kHB; ++i) {
                    a += hcnt[c][i];
                    m += hmass[c][i];
                    cc[i] = a;
                    cm[i] = m;
                }
                rp::Policy pol;
                rp::make_policy(p.policy[g * kNG + c], V, pol);
                sm.win[c] = make_window<kHB>(pol, cc, cm);
            }
        }
        __syncthreads();
        if (tid == 0) {
            int any = 0;
            for (int c = 0; c < nb; ++c) any |= sm.win[c].mode == kModeRefine;
            sm.any_refine = any;
        }
        __syncthreads();
        if (sm.any_refine) {
            // ---- C2: a 16-bin histogram inside each refined row's coarse bins
            for (int i = tid; i < kNG * kHB; i += kFT) {
                (&hcnt[0][0])[i] = 0u;
                (&hmass[0][0])[i] = 0ull;
            }
            if (tid < kNG)
                sm.floor_key[tid] = sm.win[tid].mode == kModeRefine
                                        ? floor_key_s(sm.zmax[tid], sm.inv_t[tid], 2.0f * static_cast<float>(sm.win[tid].rhi + 1))
                                        : 0xFFFFFFFFu;
            __syncthreads();
            if (!sm.abort) {
                for (int c0 = cq; c0 < cq + 16; c0 += 8) {
                    for (int j = 0; j < ntl; ++j) {
                        if (!any_active8(sm.smax[j], sm.floor_key, c0)) continue;
                        uint32_t zr[8];
                        tmem_ld8(tq + static_cast<uint32_t>(j * kNG + c0), zr);
                        tmem_wait_ld();
                        const int v = (t0 + j) * kTileV + q * 32 + lane;
                        if (v >= V) continue;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int c = c0 + i;
                            if (sm.win[c].mode != kModeRefine || sm.smax[j][c] < sm.floor_key[c]) continue;
                            const float z = __uint_as_float(zr[i]);
                            const float zm = sm.zmax[c], it = sm.inv_t[c];
                            const float bf = bin_val(z, sm.ba[c], sm.bb[c]);
                            const int b1 = coarse_bin(bf);
                            if (b1 < sm.win[c].rlo || b1 > sm.win[c].rhi) continue;
                            const int fb = fine_bin(bf, sm.win[c].rlo, sm.win[c].fscale);
                            atomicAdd(&hcnt[c][fb], 1u);
                            atomicAdd(&hmass[c][fb], static_cast<unsigned long long>(rp::to_fixed(rp::weight_f(z, zm, it))));
                        }
                    }
                }
            }
            __syncthreads();
            for (int i = tid; i < kNG * kHB; i += kFT) {
                const int c = i / kHB;
                if (sm.win[c].mode != kModeRefine) continue;
                const uint32_t cn = (&hcnt[0][0])[i];
                if (cn) {
                    red_add_u32(&sw.hcnt2[0][0] + i, cn);
                    red_add_u64(&sw.hmass2[0][0] + i, (&hmass[0][0])[i]);
                }
            }
            grid_sync(p, sm, bar_gen);  // ------------------------------------ barrier 2b
            for (int i = tid; i < kNG * kHB; i += kFT) {
                const int c = i / kHB;
                if (sm.win[c].mode != kModeRefine) continue;
                (&hcnt[0][0])[i] = ld_cg_u32(&sw.hcnt2[0][0] + i);
                (&hmass[0][0])[i] = ld_cg_u64(&sw.hmass2[0][0] + i);
            }
            __syncthreads();
            if (tid < kNG && sm.win[tid].mode == kModeRefine) {
                // bins: everything above the refined range, its 16 fine bins,
                // everything below it (inside s < 32)
                const int c = tid;
                const int rlo = sm.win[c].rlo, rhi = sm.win[c].rhi;
                const float fscale = sm.win[c].fscale;
                unsigned long long cc[kHB + 2], cm[kHB + 2];
                unsigned long long a = 0, m = 0, a1 = 0, m1 = 0, b1 = 0, bm = 0;
#pragma unroll
                for (int i = 0; i < kHB; ++i) {
                    const unsigned long long ci = ld_cg_u32(&sw.hcnt[c][i]), mi = ld_cg_u64(&sw.hmass[c][i]);
                    if (i < rlo) {
                        a1 += ci;
                        m1 += mi;
                    }
                    if (i > rhi) {
                        b1 += ci;
                        bm += mi;
                    }
                }
                cc[0] = a = a1;
                cm[0] = m = m1;
#pragma unroll
                for (int i = 0; i < kHB; ++i) {
                    a += hcnt[c][i];
                    m += hmass[c][i];
                    cc[1 + i] = a;
                    cm[1 + i] = m;
                }
                cc[kHB + 1] = a + b1;
                cm[kHB + 1] = m + bm;
                rp::Policy pol;
                rp::make_policy(p.policy[g * kNG + c], V, pol);
                Win w = make_window<kHB + 2>(pol, cc, cm);
                // the window must end inside the refined bin (fine bins 1..16);
                // starting at bin 0 keeps every coarse bin before it
                if (w.mode == kModeWin && w.whi >= 1 && w.whi <= kHB && w.phi >= 1 && w.phi <= kHB) {
                    w.lvl = 2;
                    w.rlo = rlo;
                    w.rhi = rhi;
                    w.fscale = fscale;
                    w.keep_above = w.wlo == 0;
                    w.wlo = max(w.wlo, 1) - 1;
                    w.whi -= 1;
                    w.phi -= 1;
                } else {
                    w.mode = kModeHard;
                }
                sm.win[c] = w;
            }
            __syncthreads();
        }
        // ------------------------------------------------ D: compaction (and hard rows' z)
        if (tid < kNG) {
            const Win& w = sm.win[tid];
            // picked tokens have bf = s / 2 below the window's last bin's end
            const float bf_end = w.lvl == 1 ? static_cast<float>(w.whi + 1)
                                            : static_cast<float>(w.rlo) + static_cast<float>(w.whi + 1) / w.fscale;
            sm.floor_key[tid] = w.mode == kModeHard ? 0u
                              : w.mode == kModeWin ? floor_key_s(sm.zmax[tid], sm.inv_t[tid], 2.0f * bf_end)
                                                   : 0xFFFFFFFFu;
        }
        __syncthreads();
        if (!sm.abort) {
            for (int c0 = cq; c0 < cq + 16; c0 += 8) {
                for (int j = 0; j < ntl; ++j) {
                    if (!any_active8(sm.smax[j], sm.floor_key, c0)) continue;
                    uint32_t zr[8];
                    tmem_ld8(tq + static_cast<uint32_t>(j * kNG + c0), zr);
                    tmem_wait_ld();
                    const int v = (t0 + j) * kTileV + q * 32 + lane;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int c = c0 + i;
                        const int mode = sm.win[c].mode;
                        if (sm.smax[j][c] < sm.floor_key[c]) continue;
                        const float z = __uint_as_float(zr[i]);
                        if (mode == kModeHard) {
                            if (v < V) p.zhard[static_cast<size_t>(c) * V + v] = z;
                        } else if (mode == kModeWin) {
                            const float bf = bin_val(z, sm.ba[c], sm.bb[c]);
                            const int b1 = v < V ? coarse_bin(bf) : kHB;
                            const Win& w = sm.win[c];
                            const bool pick =
                                b1 < kHB &&
                                in_window(w, b1, (w.lvl == 2 && b1 >= w.rlo && b1 <= w.rhi) ? fine_bin(bf, w.rlo, w.fscale) : 0);
                            const unsigned mask = __ballot_sync(0xFFFFFFFFu, pick);
                            if (mask) {
                                uint32_t base = 0;
                                if (lane == 0) base = atomicAdd(&sw.ccount[c], static_cast<uint32_t>(__popc(mask)));
                                base = __shfl_sync(0xFFFFFFFFu, base, 0) + __popc(mask & ((1u << lane) - 1u));
                                if (pick && base < static_cast<uint32_t>(kCand))
                                    p.cand[static_cast<size_t>(c) * kCand + base] = rp::value_order(ordered_key(z), v);
                            }
                        }
                    }
                }
            }
        }
        grid_sync(p, sm, bar_gen);  // ---------------------------------------- barrier 3

        // ------------------------------------------------ E: owners (cuts, draws, hard rows)
        // on the row engine's threads (the first kEng); the others wait at the barrier
        for (int c = blockIdx.x; c < nb && tid < kEng; c += gridDim.x) {
            if (sm.abort) break;
            const int b = g * kNG + c;
            const int64_t pidx = static_cast<int64_t>(b) * p.gamma + (k - 1);
            const int mode = sm.win[c].mode;
            Desc d{};
            if (mode == kModeNone) {
                if (tid == 0) {
                    // a failed request, or this step's row failed
                    p.proposals[pidx] = -1;
                    p.q_at_x[pidx] = 0.0f;
                    if (sm.x[c] < 0) {
                        if (k == 1) p.status[b] = kReqBadToken;
                    } else {
                        p.status[b] = sm.code[c];
                    }
                    p.desc[c].flags = kDescDone;
                }
                continue;
            }
            if (mode == kModeGreedy) {
                if (tid == 0) {
                    const uint32_t a = ld_cg_u32(&sw.amax[c]);
                    p.proposals[pidx] = static_cast<int32_t>(0xFFFFFFFFu - a);
                    p.q_at_x[pidx] = 1.0f;
                    if (k == 1) p.status[b] = kReqOk;
                    p.desc[c].flags = kDescDone;
                }
                continue;
            }
            rp::Policy pol;
            rp::make_policy(p.policy[b], V, pol);
            const float zmax = sm.zmax[c], inv_t = pol.inv_t;
            const uint32_t m24 = uniform_bits24(p.seed[b], p.request_id[b], p.pos0[b] + k, 0);
            if (mode == kModeAll) {
                if (tid == 0) {
                    d.tau = 0u;
                    d.cut = -1;
                    d.mass = sm.win[c].total;
                    d.target = static_cast<unsigned long long>((static_cast<unsigned __int128>(m24) * d.mass) >> 24);
                    d.flags = kDescPrefix;
                    p.desc[c] = d;
                    p.proposals[pidx] = -1;  // until the CTA holding the draw writes it
                    if (k == 1) p.status[b] = kReqOk;
                }
                continue;
            }
            if (mode == kModeHard) {
                // the row engine on the whole row, this CTA as a cluster of one
                cg::cluster_group cl = cg::this_cluster();
                rp::init_smem(rsm);
                RP_SYNC();
                const float* zrow = p.zhard + static_cast<size_t>(c) * V;
                rp::Slice sl{zrow, 0, V, (V + kEng - 1) / kEng, 0, 1};  // written by this launch: coherent loads
                rp::RowResult res;
                bool bad;
                rp::slice_max(rsm, cl, sl, res, bad);
                res.status = kReqOk;
                res.count = 1;
                res.in_buf = 0;
                rp::row_policy(rsm, cl, sl, V, pol, res, cbuf);
                const float invS = inv_mass(res.mass);
                float* qrow = p.q + pidx * V;
                for (int v = tid; v < V; v += kEng) {
                    const float z = __ldcg(zrow + v);
                    qrow[v] = rp::in_set(ordered_key(z), v, res.tau, res.cut) ? rp::weight_f(z, res.zmax, pol.inv_t) * invS
                                                                              : 0.0f;
                }
                unsigned long long total = 0;
                const int32_t xk = rp::sample_fixed(
                    rsm, cl, sl, m24,
                    [&](float z, int32_t idx) {
                        return rp::in_set(ordered_key(z), idx, res.tau, res.cut)
                                   ? rp::to_fixed(rp::weight_f(z, res.zmax, pol.inv_t))
                                   : 0ull;
                    },
                    total);
                if (tid == 0) {
                    p.proposals[pidx] = xk;
                    p.q_at_x[pidx] = xk >= 0 ? rp::weight_f(__ldcg(zrow + xk), res.zmax, pol.inv_t) * invS : 0.0f;
                    if (k == 1) p.status[b] = kReqOk;
                    d.flags = kDescDone;
                    p.desc[c] = d;
                }
                RP_SYNC();
                continue;
            }
            // kModeWin: the candidates, sorted; the cuts by exact prefix sums
            const Win w = sm.win[c];
            const int n = static_cast<int>(min(static_cast<unsigned long long>(ld_cg_u32(&sw.ccount[c])), w.wcount));
            for (int i = tid; i < n; i += kEng) cbuf[i] = __ldcg(p.cand + static_cast<size_t>(c) * kCand + i);
            RP_SYNC();
            rp::sort_candidates(cbuf, n);
            const bool use_k = pol.top_k > 0, use_p = pol.top_p < 1.0f;
            const int K = use_k ? static_cast<int>(min(w.k_eff - w.above_cnt - w.gap_cnt, static_cast<unsigned long long>(n)))
                                : n;
            auto wt = [&](int i) -> unsigned long long {
                return rp::to_fixed(rp::weight_f(key_to_float(rp::vo_key(cbuf[i])), zmax, inv_t));
            };
            unsigned long long part, pm;
            int pos;
            rp::cut_scan(rsm, K, wt,
                         [&](unsigned long long k_part) -> unsigned long long {
                             if (!use_p) return 0ull;
                             const unsigned long long kept = use_k ? w.above_mass + w.gap_mass + k_part : w.total;
                             return rp::p_threshold(pol.top_p, kept) - w.above_mass;
                         },
                         part, pos, pm);
            const unsigned long long kept = use_k ? w.above_mass + w.gap_mass + part : w.total;
            int mm = K;
            unsigned long long mass = kept;
            if (use_p) {
                mm = pos < K ? pos + 1 : K;
                mass = w.above_mass + (pos < K ? pm : part);
            }
            mm = max(mm, 1);
            const unsigned long long last = cbuf[mm - 1];
            d.tau = rp::vo_key(last);
            d.cut = rp::vo_idx(last);
            d.mass = mass;
            if (w.above_cnt == 0 && mm <= kWhole) {
                // the support is the first mm candidates: draw here
                unsigned long long total = 0;
                const int32_t xk = rp::draw_small_support(
                    rsm, cbuf, mm, m24,
                    [&](uint32_t key, int32_t) { return rp::to_fixed(rp::weight_f(key_to_float(key), zmax, inv_t)); },
                    total);
                if (tid == 0) sm.pick[0] = xk;
                RP_SYNC();
                for (int i = tid; i < mm; i += kEng)
                    if (rp::vo_idx(cbuf[i]) == sm.pick[0])
                        p.q_at_x[pidx] = rp::weight_f(key_to_float(rp::vo_key(cbuf[i])), zmax, inv_t) * inv_mass(mass);
                if (tid == 0) {
                    p.proposals[pidx] = sm.pick[0];
                    d.flags = kDescDrawn;
                }
            } else {
                d.target = static_cast<unsigned long long>((static_cast<unsigned __int128>(m24) * mass) >> 24);
                d.flags = kDescPrefix;
                if (tid == 0) p.proposals[pidx] = -1;  // until the CTA holding the draw writes it
            }
            if (tid == 0) {
                p.desc[c] = d;
                if (k == 1) p.status[b] = kReqOk;
            }
            RP_SYNC();
        }
        grid_sync(p, sm, bar_gen);  // ---------------------------------------- barrier 4

        // ------------------------------------------------ F: q, support mass of this range
        if (tid < kNG) {
            Desc d{};
            float is = 0.0f;
            if (tid < nb && (sm.win[tid].mode == kModeWin || sm.win[tid].mode == kModeAll)) {
                const Desc* gd = p.desc + tid;
                d.tau = __ldcg(&gd->tau);
                d.cut = __ldcg(&gd->cut);
                d.mass = __ldcg(&gd->mass);
                d.target = __ldcg(&gd->target);
                d.flags = __ldcg(&gd->flags);
                is = d.mass ? inv_mass(d.mass) : 0.0f;
            }
            sm.d[tid] = d;
            sm.inv_s[tid] = is;
        }
        __syncthreads();
        if (tid == 0) {
            int any = 0;
            for (int c = 0; c < nb; ++c) any |= (sm.d[c].flags & kDescPrefix) ? 1 : 0;
            sm.any_prefix = any;
        }
        __syncthreads();
        // slabs with a support token (key >= tau) are written from tensor
        // memory; the others of the rows with q get zeros, 16 bytes a lane
        if (tid < kNG) {
            const uint32_t fl = sm.d[tid].flags;
            sm.floor_key[tid] = (fl & (kDescDrawn | kDescPrefix)) ? sm.d[tid].tau : 0xFFFFFFFFu;
        }
        __syncthreads();
        if (!sm.abort) {
            for (int c0 = cq; c0 < cq + 16; c0 += 8) {
                unsigned long long mine[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) mine[i] = 0ull;
                for (int j = 0; j < ntl; ++j) {
                    const int vt = (t0 + j) * kTileV;        // first token of the tile
                    // zeros: lane l takes rows 32q + 4 (l % 8) .. + 3 of requests c0 + l / 8 and c0 + 4 + l / 8
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int c = c0 + half * 4 + (lane >> 3);
                        const int v4 = vt + q * 32 + 4 * (lane & 7);
                        const uint32_t fl = sm.d[c].flags;
                        if ((fl & (kDescDrawn | kDescPrefix)) && sm.smax[j][c] < sm.floor_key[c] && v4 < V)
                            __stcs(reinterpret_cast<float4*>(p.q + (static_cast<int64_t>(g * kNG + c) * p.gamma + (k - 1)) * V + v4),
                                   make_float4(0.0f, 0.0f, 0.0f, 0.0f));
                    }
                    if (!any_active8(sm.smax[j], sm.floor_key, c0)) continue;
                    uint32_t zr[8];
                    tmem_ld8(tq + static_cast<uint32_t>(j * kNG + c0), zr);
                    tmem_wait_ld();
                    const int v = vt + q * 32 + lane;
                    if (v >= V) continue;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int c = c0 + i;
                        if (sm.smax[j][c] < sm.floor_key[c]) continue;
                        const uint32_t fl = sm.d[c].flags;
                        const float z = __uint_as_float(zr[i]);
                        const bool in = rp::in_set(ordered_key(z), v, sm.d[c].tau, sm.d[c].cut);
                        const float wv = in ? rp::weight_f(z, sm.zmax[c], sm.inv_t[c]) : 0.0f;
                        __stcs(p.q + (static_cast<int64_t>(g * kNG + c) * p.gamma + (k - 1)) * V + v, wv * sm.inv_s[c]);
                        if (fl & kDescPrefix) mine[i] += in ? rp::to_fixed(wv) : 0ull;
                    }
                }
                if (sm.any_prefix) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        unsigned long long s = mine[i];
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
                        if (lane == 0) sm.wpart[q][c0 + i] = s;
                    }
                }
            }
        }
        __syncthreads();
        if (sm.any_prefix) {
            if (tid < nb && (sm.d[tid].flags & kDescPrefix))
                p.part[static_cast<size_t>(tid) * gridDim.x + blockIdx.x] =
                    sm.wpart[0][tid] + sm.wpart[1][tid] + sm.wpart[2][tid] + sm.wpart[3][tid];
            grid_sync(p, sm, bar_gen);  // ------------------------------------ barrier 5
            // ------------------------------------------------ G: the CTA holding the draw finds it
            for (int c = 0; c < nb; ++c) {
                if (!(sm.d[c].flags & kDescPrefix) || sm.abort) continue;
                // exclusive prefix of this CTA's range (CTAs in token order)
                if (warp == 0) {
                    unsigned long long ex = 0;
                    for (int o = lane; o < static_cast<int>(blockIdx.x); o += 32)
                        ex += __ldcg(p.part + static_cast<size_t>(c) * gridDim.x + o);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) ex += __shfl_xor_sync(0xFFFFFFFFu, ex, o);
                    if (lane == 0) {
                        const unsigned long long mine = __ldcg(p.part + static_cast<size_t>(c) * gridDim.x + blockIdx.x);
                        const unsigned long long tg = sm.d[c].target;
                        sm.pick[1] = (ex <= tg && tg < ex + mine) ? 1 : 0;
                        sm.ex = ex;
                    }
                }
                __syncthreads();
                if (!sm.pick[1]) continue;
                // scan this range in token order: tiles in order, 128 rows each
                // (warps 0..3 = quadrants 0..3 hold rows 32q..32q+31)
                unsigned long long before = sm.ex;
                const unsigned long long tg = sm.d[c].target;
                const Desc d = sm.d[c];
                int found = -1;
                float fz = 0.0f;
                for (int j = 0; j < ntl && found < 0; ++j) {
                    unsigned long long wq = 0;
                    float z = 0.0f;
                    const int v = (t0 + j) * kTileV + (warp & 3) * 32 + lane;
                    if (warp < 4) {
                        z = __uint_as_float(tmem_ld1(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) +
                                                     static_cast<uint32_t>(j * kNG + c)));
                        tmem_wait_ld();
                        if (v < V && rp::in_set(ordered_key(z), v, d.tau, d.cut))
                            wq = rp::to_fixed(rp::weight_f(z, sm.zmax[c], sm.inv_t[c]));
                    }
                    // inclusive scan over the 128 rows: warp scans, then the quadrant offsets
                    unsigned long long incl = wq;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                        if (lane >= o) incl += y;
                    }
                    if (warp < 4 && lane == 31) sm.qsum[warp] = incl;
                    __syncthreads();
                    unsigned long long off = before;
                    for (int w2 = 0; w2 < (warp & 3) && warp < 4; ++w2) off += sm.qsum[w2];
                    if (warp < 4 && wq > 0 && off + incl > tg && off + incl - wq <= tg) {
                        sm.pick[2] = v;
                        reinterpret_cast<float*>(&sm.pick[3])[0] = z;
                    }
                    const unsigned long long tile_sum = sm.qsum[0] + sm.qsum[1] + sm.qsum[2] + sm.qsum[3];
                    __syncthreads();
                    if (before + tile_sum > tg) {
                        found = sm.pick[2];
                        fz = reinterpret_cast<float*>(&sm.pick[3])[0];
                    }
                    before += tile_sum;
                    __syncthreads();
                }
                if (tid == 0) {
                    const int b = g * kNG + c;
                    const int64_t pidx = static_cast<int64_t>(b) * p.gamma + (k - 1);
                    p.proposals[pidx] = found;
                    p.q_at_x[pidx] = found >= 0 ? rp::weight_f(fz, sm.zmax[c], sm.inv_t[c]) * inv_mass(d.mass) : 0.0f;
                }
                __syncthreads();
            }
            grid_sync(p, sm, bar_gen);  // ------------------------------------ barrier 6
        }
    }

    // ------------------------------------------------ exit
    // On an abort, no copy or MMA may still be landing: wait (bounded) for
    // what was issued.
    if (tid == 0 && sm.abort) {
        for (int n = max(0, w_issued - S); n < w_issued; ++n) mbar_wait(&sm.wfull[n % S], (n / S) & 1, kWaitLimitNs);
        if (mma_done > 0) mbar_wait(&sm.wempty[(mma_done - 1) % S], ((mma_done - 1) / S) & 1, kWaitLimitNs);
    }
    if (tid == 32 && sm.abort)
        for (int n = max(0, b_issued - SB); n < b_issued; ++n) mbar_wait(&sm.bfull[n % SB], (n / SB) & 1, kWaitLimitNs);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kTmemCols);
    // a wait gave up somewhere: no request's outputs can be trusted
    if (blockIdx.x == 0 && *reinterpret_cast<volatile int*>(p.error))
        for (int b = tid; b < p.B; b += kFT) p.status[b] = kReqTimeout;
}

}  // namespace

// ------------------------------------------------------------------ host
namespace {

constexpr int kSmemLimit = 232448;   // opt-in shared memory per CTA
constexpr int kStaticAllowance = 24 * 1024;  // FusedSmem + the row engine's static shared memory
constexpr int kEngineScratch = rp::kCap * 8 + rp::kWarps * rp::kBins * 4;  // the row engine's cbuf

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return n;
}

struct FusedShape {
    int ntiles, tpc, grid, groups, stages, bstages, smem;  // stages: W tiles in flight; bstages: backbone tiles
};

bool fused_shape(int B, int V, int r, bool rnn, FusedShape& f) {
    const int sms = sm_count();
    if (sms <= 0 || B < 1 || r < 64 || r > 256 || r % 64 != 0 || V < kTileV) return false;
    f.ntiles = (V + kTileV - 1) / kTileV;
    f.tpc = (f.ntiles + sms - 1) / sms;
    if (f.tpc > kMaxLT) return false;
    f.grid = (f.ntiles + f.tpc - 1) / f.tpc;
    f.groups = (B + kNG - 1) / kNG;
    // B operands: the gathered U rows, or (RNN head) the state's bf16 hi and lo rows
    const int ops = rnn ? 2 : 1;
    const int w = kTileV * r * 2, b = kNG * kTileV * 2, u = std::max(ops * kNG * r * 2, kEngineScratch);
    const int budget = kSmemLimit - kStaticAllowance - 1024;
    if (!rnn) {
        f.stages = f.bstages = std::min(4, (budget - u) / (w + b));
        if (f.stages < 2) return false;
    } else {
        // the RNN head may take a single W stage (at r = 256 two do not fit
        // beside its second operand; phase A's cadence is set by its epilogue,
        // which overlaps the next tile's W load), keeping two backbone stages
        f.bstages = 2;
        f.stages = std::min(4, (budget - u - f.bstages * b) / w);
        if (f.stages < 1) return false;
    }
    // at least half the SM's shared memory, so that no two CTAs (each taking
    // all of tensor memory) share an SM
    f.smem = std::max(f.stages * w + f.bstages * b + u + 1024, 120 * 1024);
    return true;
}

struct FusedLayout {
    size_t bar, words, clear_end, desc, cand, part, zhard, state, total;
};
// Offsets from `base` (past the slower path's error word, which must stay
// zero between calls); the words up to clear_end are cleared per call.
FusedLayout fused_layout(int B, int gamma, int V, int r_state) {
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    FusedLayout l;
    const int groups = (B + kNG - 1) / kNG, rows = std::min(B, kNG);
    l.bar = 256;
    l.words = up(l.bar + 16);
    l.clear_end = up(l.words + static_cast<size_t>(groups) * gamma * sizeof(StepWords));
    l.desc = l.clear_end;
    l.cand = up(l.desc + kNG * sizeof(Desc));
    l.part = up(l.cand + static_cast<size_t>(kNG) * kCand * 8);
    l.zhard = up(l.part + static_cast<size_t>(kNG) * 1024 * 8);
    l.state = up(l.zhard + static_cast<size_t>(rows) * V * 4);
    l.total = up(l.state + 2 * static_cast<size_t>(kNG) * r_state * 4);  // the GRU state, two buffers
    return l;
}

}  // namespace

bool markov_fused_supported(int dtype, int B, int V, int r, bool rnn) {
    FusedShape f;
    return dtype == kBF16 && B <= kFusedMaxBatch && fused_shape(B, V, r, rnn, f) && f.grid <= 1024;
}

size_t markov_fused_workspace(int B, int gamma, int V, int r, bool rnn) {
    return fused_layout(B, gamma, V, rnn ? r : 0).total;
}

cudaError_t launch_markov_fused(const MarkovFusedArgs& a, void* ws, size_t ws_bytes, cudaStream_t stream) {
    const bool rnn = a.Wi != nullptr;
    if (rnn && (!a.Wh || !a.bi || !a.bh)) return cudaErrorInvalidValue;
    FusedShape f;
    if (!fused_shape(a.B, a.V, a.r, rnn, f)) return cudaErrorInvalidValue;
    if (rnn && f.groups != 1) return cudaErrorInvalidValue;  // the state buffers hold one group
    const FusedLayout lay = fused_layout(a.B, a.gamma, a.V, rnn ? a.r : 0);
    if (ws_bytes < lay.total) return cudaErrorInvalidValue;
    char* base = static_cast<char*>(ws);
    FusedParams p{};
    p.backbone = a.backbone;
    p.U = a.U;
    p.anchor = a.anchor;
    p.policy = a.policy;
    p.seed = a.seed;
    p.request_id = a.request_id;
    p.pos0 = a.pos0;
    p.B = a.B;
    p.gamma = a.gamma;
    p.V = a.V;
    p.r = a.r;
    p.proposals = a.proposals;
    p.q = a.q;
    p.q_at_x = a.q_at_x;
    p.status = a.status;
    p.ntiles = f.ntiles;
    p.tpc = f.tpc;
    p.grid = f.grid;
    p.groups = f.groups;
    p.stages = f.stages;
    p.bstages = f.bstages;
    p.bar = reinterpret_cast<unsigned int*>(base + lay.bar);
    p.error = reinterpret_cast<int*>(base + lay.bar + 8);
    p.words = reinterpret_cast<StepWords*>(base + lay.words);
    p.desc = reinterpret_cast<Desc*>(base + lay.desc);
    p.cand = reinterpret_cast<unsigned long long*>(base + lay.cand);
    p.part = reinterpret_cast<unsigned long long*>(base + lay.part);
    p.zhard = reinterpret_cast<float*>(base + lay.zhard);
    p.rnn = rnn ? 1 : 0;
    p.Wi = a.Wi;
    p.Wh = a.Wh;
    p.bi = a.bi;
    p.bh = a.bh;
    p.state = rnn ? reinterpret_cast<float*>(base + lay.state) : nullptr;

    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    CUtensorMap wmap, bmap;
    const cuuint32_t estr[3] = {1, 1, 1};
    {   // W [V, r]: boxes of 64 columns (128 B) x 128 rows, 128-byte swizzle (the MMA's A operand)
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(a.r), static_cast<cuuint64_t>(a.V)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(a.r) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(kTileV)};
        if (enc(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(a.W), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    {   // backbone [B, gamma, V]: boxes of 128 tokens x 1 step x 64 requests
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(a.V), static_cast<cuuint64_t>(a.gamma),
                                    static_cast<cuuint64_t>(a.B)};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(a.V) * 2, static_cast<cuuint64_t>(a.gamma) * a.V * 2};
        const cuuint32_t box[3] = {static_cast<cuuint32_t>(kTileV), 1, static_cast<cuuint32_t>(kNG)};
        if (enc(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(a.backbone), dims, strides, box,
                estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaMemsetAsync(base + lay.bar, 0, lay.clear_end - lay.bar, stream);
    if (e != cudaSuccess) return e;
    auto kernel = rnn ? markov_fused_kernel<true> : markov_fused_kernel<false>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, f.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(f.grid));
    cfg.blockDim = dim3(kFT);
    cfg.dynamicSmemBytes = static_cast<size_t>(f.smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the grid barriers need it
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, wmap, bmap, p);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace dspark

