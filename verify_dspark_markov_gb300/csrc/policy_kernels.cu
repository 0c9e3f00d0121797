// Sampled paths built on the row engine (row_policy.cuh): one cluster of CTAs
// per vocabulary row, reading the row in place - 4 per target row in the
// verify (384 rows and more fill the GPU), 8 per row in the drafting step,
// whose batch of rows is smaller.
//
//  * verify_rows_kernel - exact verify of a block under per-request policies
//    [FT Exact decoding semantics > Probabilistic]: each cluster forms the
//    policy of one target row and p(x) of the proposal that row scores; the
//    cluster finishing a request's last row (by ticket) takes the accept tests
//    (accept x_k iff p > 0 and u < p(x_k)/q(x_k)), then draws the residual
//    token from normalised max(p - q, 0) at the first rejection, or the bonus
//    token from the last target row, by an exact inverse CDF in token order.
//    Greedy requests in the batch take the contiguous-prefix argmax rule.
//    The width variant (kWidth) checks x_1..x_w of each request (w = its
//    width, 0..gamma): rows past w take their ticket without reading logits,
//    and the bonus comes from row w.
//  * markov_step_kernel - one left-to-right step of the draft's sequential
//    head [FT Checkpoint-faithful DSpark architecture]: q_k = policy(z_k),
//    written in full, and x_k drawn from it (greedy: the argmax).

#include <cooperative_groups.h>

#include <type_traits>

#include "kernels.h"
#include "row_policy.cuh"

namespace dspark {

namespace {

namespace cg = cooperative_groups;
using rp::kThreads;
constexpr int kVerifyC = 4;  // CTAs per target row in the verify
constexpr int kStepC = 8;    // CTAs per row in the drafting step
static_assert(kVerifyC <= rp::kMaxC && kStepC <= rp::kMaxC, "cluster sizes the row engine holds");

__device__ __forceinline__ float inv_mass(uint64_t mass) {
    return static_cast<float>(rp::kFix / static_cast<double>(mass));
}

// Dynamic shared memory: the candidate buffer (used in rank 0) followed by
// the per-warp histogram counts.  The row slices are read in place from
// global memory.

template <bool kWidth>
using VerifyArgs = std::conditional_t<kWidth, VerifyWidthParams, VerifyProbParams>;

// Six CTAs per SM (40 registers, a few spilled): more rows in flight hides
// more of the passes' latency (measured against four and five CTAs per SM).
template <int kDtype, bool kWidth>
__global__ void __cluster_dims__(kVerifyC, 1, 1) __launch_bounds__(rp::kThreads, 6)
    verify_rows_kernel(const VerifyArgs<kWidth> p) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ rp::Smem sm;
    __shared__ float s_px;          // p(x) of this row's proposal, in its owner CTA
    __shared__ int32_t s_last;      // rank 0: this cluster decides the request
    __shared__ int32_t s_plan[4];   // rank 0: (row to draw from, rejected position, token, -)
    __shared__ int32_t s_bcast[4];
    __shared__ int32_t s_w;         // kWidth: the request's width
    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;
    constexpr int kStoreBf16 = kDtype == kBF16;
    unsigned long long* cbuf = reinterpret_cast<unsigned long long*>(dyn);
    rp::init_smem(sm);
    if (tid == 0) {
        s_px = 0.0f;
        s_last = 0;
        s_plan[0] = -1;
        s_plan[1] = 0;
        if constexpr (kWidth) s_w = p.width[blockIdx.x / kVerifyC / (p.gamma + 1)];
    }
    __syncthreads();

    const int rows = p.gamma + 1;
    const int64_t row = blockIdx.x / kVerifyC;
    const int b = static_cast<int>(row / rows), i = static_cast<int>(row % rows);
    // kWidth: rows 0..w-1 score x_1..x_w and row w gives the bonus; a row
    // past w (every row, for an invalid width) gets an empty slice, reads
    // nothing, reports "empty", and the decision never looks at its record
    bool live = true;
    if constexpr (kWidth) live = s_w >= 0 && s_w <= p.gamma && i <= s_w;
    const int lo = rank * p.slice;
    const int n = live ? max(0, min(p.slice, p.V - lo)) : 0;
    const int esize = kDtype == kBF16 ? 2 : 4;
    const char* tgt = static_cast<const char*>(p.target);
    rp::Slice sl{tgt + (row * p.V + lo) * esize, lo, n, (n + kThreads - 1) / kThreads, kStoreBf16};

    rp::Policy pol;
    const bool pol_ok = rp::make_policy(p.policy[b], p.V, pol);
    rp::RowResult res;
    bool bad;
    rp::slice_max(sm, cl, sl, res, bad);
    res.status = bad ? kReqNonfinite : (res.argmax < 0 ? kReqEmpty : (pol_ok ? kReqOk : kReqBadPolicy));
    res.count = 1;
    res.in_buf = 0;
    if (res.status == kReqOk) rp::row_policy(sm, cl, sl, p.V, pol, res, cbuf);

    // p(x) of the proposal scored by this row (rows 0..gamma-1, or 0..w-1), in its owner CTA
    int32_t x = -1;
    if constexpr (kWidth) {
        if (live && i < s_w) x = p.proposals[b * p.gamma + i];
    } else {
        if (i < p.gamma) x = p.proposals[b * p.gamma + i];
    }
    const bool x_ok = x >= 0 && x < p.V;
    const int owner = x_ok ? x / p.slice : 0;
    if (res.status == kReqOk && !pol.greedy && x_ok && rank == owner && tid == 0) {
        const float z = sl.val(x - lo);
        s_px = rp::in_set(ordered_key(z), x, res.tau, res.cut)
                   ? rp::weight_f(z, res.zmax, pol.inv_t) * inv_mass(res.mass)
                   : 0.0f;
    }
    cl.sync();
    if (rank == 0 && tid == 0) {
        RowRecord rec;
        rec.zmax = res.zmax;
        rec.inv_t = pol.inv_t;
        rec.tau = res.tau;
        rec.cut = res.cut;
        rec.mass = res.mass;
        rec.p_x = (x_ok && !pol.greedy) ? *cl.map_shared_rank(&s_px, owner) : 0.0f;
        rec.status = res.status;
        rec.argmax = res.argmax;
        rec.count = res.count;
        p.records[row] = rec;
        const unsigned old = atom_add_acq_rel(p.ticket + b, 1u);
        s_last = old == static_cast<unsigned>(rows - 1);
    }
    cl.sync();
    if (tid == 0) s_bcast[0] = *cl.map_shared_rank(&s_last, 0);
    __syncthreads();
    if (s_bcast[0] == 0) {
        cl.sync();  // keep this CTA's shared memory alive for the cluster's readers
        return;
    }

    // ---- this cluster decides request b
    fence_acq_rel_gpu();
    int32_t* out = p.out_tokens + b * rows;
    if (rank == 0 && tid == 0) {
        p.ticket[b] = 0u;  // leave the workspace zero-filled
        const RowRecord* rec = p.records + static_cast<int64_t>(b) * rows;
        const int32_t* xs = p.proposals + b * p.gamma;
        // proposals checked: gamma, or the width (0 with a failed status
        // when it lies outside [0, gamma])
        int wd = p.gamma;
        bool w_ok = true;
        if constexpr (kWidth) {
            w_ok = s_w >= 0 && s_w <= p.gamma;
            wd = w_ok ? s_w : 0;
        }
        int32_t status = w_ok ? kReqOk : kReqBadToken;
        for (int k = 0; k < wd; ++k)
            if (xs[k] < 0 || xs[k] >= p.V) status = kReqBadToken;
        if (status == kReqOk)
            for (int r = 0; r < wd + 1; ++r)
                if (rec[r].status != kReqOk) { status = rec[r].status; break; }
        if (status != kReqOk) {
            for (int r = 0; r < rows; ++r) out[r] = -1;
            p.num_accepted[b] = -1;
            p.status[b] = status;
        } else if (pol.greedy) {
            int nacc = 0;
            while (nacc < wd && xs[nacc] == rec[nacc].argmax) ++nacc;
            for (int r = 0; r < rows; ++r) out[r] = r < nacc ? xs[r] : (r == nacc ? rec[nacc].argmax : -1);
            p.num_accepted[b] = nacc;
            p.status[b] = kReqOk;
        } else {
            int j = 0;  // first rejected position (1-based), 0 = none
            for (int k = 1; k <= wd; ++k) {
                const float pk = rec[k - 1].p_x;
                const float qk = p.q_at_x[b * p.gamma + (k - 1)];
                const float ratio = qk > 0.0f ? pk / qk : (pk > 0.0f ? __int_as_float(0x7F800000) : 0.0f);
                const float u = uniform01(p.seed[b], p.request_id[b], p.pos0[b] + k, 1);
                if (!(pk > 0.0f && u < ratio)) { j = k; break; }
            }
            for (int r = 0; r < rows; ++r) out[r] = -1;
            for (int r = 0; r < (j ? j - 1 : wd); ++r) out[r] = xs[r];
            s_plan[0] = j ? j - 1 : wd;  // target row to draw from
            s_plan[1] = j;                    // residual against q_j when j > 0
        }
    }
    if (rank == 0 && tid == 0) sm.ccount = 0;  // the draw's candidate slots, published by the barrier below
    cl.sync();
    if (tid < 2) s_bcast[1 + tid] = cl.map_shared_rank(s_plan, 0)[tid];
    __syncthreads();
    const int R = s_bcast[1], j = s_bcast[2];
    if (R >= 0) {
        // draw the residual / bonus token from target row R of request b
        const RowRecord rr = p.records[static_cast<int64_t>(b) * rows + R];
        const int64_t trow = static_cast<int64_t>(b) * rows + R;
        // (the deciding cluster may have had a row past the width: its own
        // slice was empty, row R's is not)
        const int nr = kWidth ? max(0, min(p.slice, p.V - lo)) : n;
        const rp::Slice sr{tgt + (trow * p.V + lo) * esize, lo, nr, (nr + kThreads - 1) / kThreads, kStoreBf16};
        const float invS = inv_mass(rr.mass);
        const float* qrow = j ? p.q + (static_cast<int64_t>(b) * p.gamma + (j - 1)) * p.V : nullptr;
        const int64_t pos = p.pos0[b] + (j ? j : (kWidth ? s_w : p.gamma) + 1);
        const uint32_t m24 = uniform_bits24(p.seed[b], p.request_id[b], pos, 2);
        // p of a support element, its fixed-point weight and residual weight
        auto pw = [&](uint32_t key) { return rp::to_fixed(rp::weight_f(key_to_float(key), rr.zmax, rr.inv_t)); };
        auto resid = [&](uint32_t key, int32_t idx) {
            const float pv = rp::weight_f(key_to_float(key), rr.zmax, rr.inv_t) * invS;
            return rp::to_fixed(fmaxf(pv - qrow[idx], 0.0f));
        };
        int32_t token = -1;
        if (rr.count <= rp::kThreads) {
            // small support: gathered in rank 0, drawn in token order
            const int cnt = rp::compact_to_rank0(sm, cl, sr, cbuf, rp::support_floor(rr.tau), [&](uint32_t key, int32_t idx) {
                return rp::in_set(key, idx, rr.tau, rr.cut);
            });
            if (rank == 0) {
                unsigned long long total = 0;
                if (j) {
                    token = rp::draw_small_support(sm, cbuf, cnt, m24, resid, total);
                    if (total == 0) {  // no residual mass left (round-off): draw from p itself
                        token = rp::draw_small_support(sm, cbuf, cnt, m24,
                                                       [&](uint32_t key, int32_t) { return pw(key); }, total);
                    }
                } else {
                    token = rp::draw_small_support(sm, cbuf, cnt, m24, [&](uint32_t key, int32_t) { return pw(key); },
                                                   total);
                }
            }
        } else {
            // the whole vocabulary: a draw over every CTA's slice
            unsigned long long total = 0;
            if (j) {
                token = rp::sample_fixed(sm, cl, sr, m24,
                                         [&](float z, int32_t idx) {
                                             const uint32_t key = ordered_key(z);
                                             return rp::in_set(key, idx, rr.tau, rr.cut) ? resid(key, idx) : 0ull;
                                         },
                                         total);
            }
            if (!j || total == 0)
                token = rp::sample_fixed(sm, cl, sr, m24,
                                         [&](float z, int32_t idx) {
                                             const uint32_t key = ordered_key(z);
                                             return rp::in_set(key, idx, rr.tau, rr.cut) ? pw(key) : 0ull;
                                         },
                                         total);
        }
        if (rank == 0 && tid == 0) {
            out[R] = token;
            p.num_accepted[b] = R;
            p.status[b] = kReqOk;
        }
    }
    // leave the workspace zero-filled: this request's row records are consumed
    cl.sync();
    if (rank == 0) {
        uint32_t* recw = reinterpret_cast<uint32_t*>(p.records + static_cast<int64_t>(b) * rows);
        for (int e = tid; e < rows * static_cast<int>(sizeof(RowRecord) / 4); e += kThreads) recw[e] = 0u;
    }
    cl.sync();  // keep shared memory alive until every CTA is done reading
}

template <int kDtype>
__global__ void __cluster_dims__(kStepC, 1, 1) __launch_bounds__(rp::kThreads, 4)
    markov_step_kernel(const MarkovStepParams p) {
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ rp::Smem sm;
    __shared__ float s_qx;
    __shared__ int32_t s_x;
    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;
    // the next step's bias kernel may start on SMs this grid leaves free (it
    // waits for this grid's completion before it reads the proposals)
    asm volatile("griddepcontrol.launch_dependents;");
    rp::init_smem(sm);
    if (tid == 0) {
        s_qx = 0.0f;
        s_x = -1;
    }
    __syncthreads();

    const int b = blockIdx.x / kStepC;
    const int k = p.k;  // 1-based position
    const int64_t pidx = static_cast<int64_t>(b) * p.gamma + (k - 1);
    const int32_t x_prev = k == 1 ? p.anchor[b] : p.proposals[pidx - 1];
    // a request that failed at an earlier step (or on its anchor) proposes nothing
    if (x_prev < 0 || x_prev >= p.V) {
        if (rank == 0 && tid == 0) {
            p.proposals[pidx] = -1;
            p.q_at_x[pidx] = 0.0f;
            if (k == 1) p.status[b] = kReqBadToken;
        }
        return;  // uniform over the cluster: no cluster barrier follows
    }
    if (p.error_flag && *p.error_flag) {  // the bias of this step is not trustworthy
        if (rank == 0 && tid == 0) {
            p.proposals[pidx] = -1;
            p.q_at_x[pidx] = 0.0f;
            p.status[b] = kReqTimeout;
        }
        return;
    }
    const bool z_bf16 = !p.zbuf && kDtype == kBF16;
    const int lo = rank * p.slice;
    const int n = max(0, min(p.slice, p.V - lo));
    unsigned long long* cbuf = reinterpret_cast<unsigned long long*>(dyn);
    // the logits with the Markov bias (fp32 [B, V]) or the backbone row
    const void* zrow = p.zbuf ? static_cast<const void*>(p.zbuf + static_cast<int64_t>(b) * p.V + lo)
                              : static_cast<const void*>(static_cast<const char*>(p.backbone) +
                                                         (pidx * p.V + lo) * (kDtype == kBF16 ? 2 : 4));
    rp::Slice sl{zrow, lo, n, (n + kThreads - 1) / kThreads, z_bf16 ? 1 : 0};
    rp::Policy pol;
    const bool pol_ok = p.policy ? rp::make_policy(p.policy[b], p.V, pol)
                                 : (pol = rp::Policy{1.0f, 0, 1.0f, 1}, true);
    rp::RowResult res;
    bool bad;
    rp::slice_max(sm, cl, sl, res, bad);
    res.status = bad ? kReqNonfinite : (res.argmax < 0 ? kReqEmpty : (pol_ok ? kReqOk : kReqBadPolicy));
    if (res.status != kReqOk) {
        if (rank == 0 && tid == 0) {
            p.proposals[pidx] = -1;
            p.q_at_x[pidx] = 0.0f;
            p.status[b] = res.status;
        }
        cl.sync();
        return;
    }
    res.count = 1;
    res.in_buf = 0;
    rp::row_policy(sm, cl, sl, p.V, pol, res, cbuf);
    if (pol.greedy) {
        if (rank == 0 && tid == 0) {
            s_x = res.argmax;
            s_qx = 1.0f;
        }
    } else {
        const float invS = inv_mass(res.mass);
        float* qrow = p.q + pidx * p.V + lo;
        {
            // q over the slice, 16-byte vectors at a time; only support
            // elements (key >= tau) need their weight
            const float zt = rp::support_floor(res.tau);
            const int vp = sl.vper(), nv = sl.nvec();
            for (int j0 = tid; j0 < nv; j0 += kThreads * rp::kBatch) {
              uint4 vb[rp::kBatch];
#pragma unroll
              for (int u = 0; u < rp::kBatch; ++u) {
                  const int jj = j0 + u * kThreads;
                  vb[u] = jj < nv ? sl.vec(jj) : make_uint4(0u, 0u, 0u, 0u);
              }
#pragma unroll
              for (int u = 0; u < rp::kBatch; ++u) {
                const int j = j0 + u * kThreads;
                if (j >= nv) break;
                const uint4 v = vb[u];
                float q8[8];
#pragma unroll
                for (int l = 0; l < 8; ++l) q8[l] = 0.0f;
                if (rp::vec_max(v, sl.bf16) >= zt) {
#pragma unroll
                    for (int l = 0; l < 8; ++l) {
                        if (l >= vp) break;
                        const float z = rp::vec_elem(v, l, sl.bf16);
                        if (rp::in_set(ordered_key(z), lo + j * vp + l, res.tau, res.cut))
                            q8[l] = rp::weight_f(z, res.zmax, pol.inv_t) * invS;
                    }
                }
                float4* d = reinterpret_cast<float4*>(qrow + j * vp);
                d[0] = make_float4(q8[0], q8[1], q8[2], q8[3]);
                if (vp == 8) d[1] = make_float4(q8[4], q8[5], q8[6], q8[7]);
              }
            }
        }
        const uint32_t m24 = uniform_bits24(p.seed[b], p.request_id[b], p.pos0[b] + k, 0);
        if (res.in_buf && res.count <= rp::kThreads) {
            // the support is rank 0's first res.count candidates
            if (rank == 0) {
                unsigned long long total = 0;
                const int32_t xk = rp::draw_small_support(
                    sm, cbuf, res.count, m24,
                    [&](uint32_t key, int32_t) {
                        return rp::to_fixed(rp::weight_f(key_to_float(key), res.zmax, pol.inv_t));
                    },
                    total);
                if (tid == 0) {
                    s_x = xk;
                    s_qx = 0.0f;
                }
                __syncthreads();
                // q(x): the weight of x over the support mass (the buffer is in value order)
                for (int e = tid; e < res.count; e += kThreads)
                    if (rp::vo_idx(cbuf[e]) == xk)
                        s_qx = rp::weight_f(key_to_float(rp::vo_key(cbuf[e])), res.zmax, pol.inv_t) * invS;
            }
        } else {
            unsigned long long total = 0;
            const int32_t xk = rp::sample_fixed(
                sm, cl, sl, m24,
                [&](float z, int32_t idx) {
                    return rp::in_set(ordered_key(z), idx, res.tau, res.cut)
                               ? rp::to_fixed(rp::weight_f(z, res.zmax, pol.inv_t))
                               : 0ull;
                },
                total);
            if (xk >= lo && xk < lo + n && tid == 0) {
                s_x = xk;
                s_qx = rp::weight_f(sl.val(xk - lo), res.zmax, pol.inv_t) * invS;
            }
        }
    }
    cl.sync();
    if (rank == 0 && tid == 0) {
        // the rank holding the draw's results: 0 for greedy / small supports,
        // the owner of x for a draw over every slice
        int src = 0;
        if (!pol.greedy && !(res.in_buf && res.count <= rp::kThreads)) {
            for (int r = 0; r < kStepC; ++r)
                if (*cl.map_shared_rank(&s_x, r) >= 0) { src = r; break; }
        }
        const int32_t xk = *cl.map_shared_rank(&s_x, src);
        p.proposals[pidx] = xk;
        p.q_at_x[pidx] = *cl.map_shared_rank(&s_qx, src);
        if (k == 1) p.status[b] = kReqOk;
    }
    cl.sync();
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

int verify_slice(int V) { return ((V + kVerifyC - 1) / kVerifyC + 7) / 8 * 8; }

int step_slice(int V) { return ((V + kStepC - 1) / kStepC + 7) / 8 * 8; }

int policy_smem_bytes(int V, int store_bf16) {
    (void)V;
    (void)store_bf16;
    return rp::kCap * static_cast<int>(sizeof(unsigned long long)) +
           rp::kWarps * rp::kBins * static_cast<int>(sizeof(uint32_t));
}

template <int kDtype, bool kWidth>
cudaError_t launch_verify_rows(const VerifyArgs<kWidth>& p, int smem, dim3 grid, cudaStream_t stream) {
    const cudaError_t e = set_smem(verify_rows_kernel<kDtype, kWidth>, smem);
    if (e != cudaSuccess) return e;
    verify_rows_kernel<kDtype, kWidth><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_verify_prob(const VerifyProbParams& p, cudaStream_t stream, const int32_t* width) {
    const int smem = policy_smem_bytes(p.V, p.dtype == kBF16);
    const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(p.B) * (p.gamma + 1) * kVerifyC));
    if (width) {
        VerifyWidthParams pw;
        static_cast<VerifyProbParams&>(pw) = p;
        pw.width = width;
        return p.dtype == kBF16 ? launch_verify_rows<kBF16, true>(pw, smem, grid, stream)
                                : launch_verify_rows<kF32, true>(pw, smem, grid, stream);
    }
    return p.dtype == kBF16 ? launch_verify_rows<kBF16, false>(p, smem, grid, stream)
                            : launch_verify_rows<kF32, false>(p, smem, grid, stream);
}

cudaError_t launch_markov_step(const MarkovStepParams& p, cudaStream_t stream) {
    const int smem = policy_smem_bytes(p.V, !p.zbuf && p.dtype == kBF16);
    const dim3 grid(static_cast<unsigned>(p.B * kStepC));
    cudaError_t e;
    if (p.dtype == kBF16) {
        if ((e = set_smem(markov_step_kernel<kBF16>, smem)) != cudaSuccess) return e;
        markov_step_kernel<kBF16><<<grid, kThreads, smem, stream>>>(p);
    } else {
        if ((e = set_smem(markov_step_kernel<kF32>, smem)) != cudaSuccess) return e;
        markov_step_kernel<kF32><<<grid, kThreads, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace dspark
