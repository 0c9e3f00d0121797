// Sampled paths built on the row engine (row_policy.cuh): one cluster of
// rp::kC CTAs per vocabulary row.
//
//  * verify_rows_kernel - exact verify of a block under per-request policies
//    [FT Exact decoding semantics > Probabilistic]: each cluster forms the
//    policy of one target row and p(x) of the proposal that row scores; the
//    cluster finishing a request's last row (by ticket) takes the accept tests
//    (accept x_k iff p > 0 and u < p(x_k)/q(x_k)), then draws the residual
//    token from normalised max(p - q, 0) at the first rejection, or the bonus
//    token from the last target row, by an exact inverse CDF in token order.
//    Greedy requests in the batch take the contiguous-prefix argmax rule.
//  * markov_step_kernel - one left-to-right step of the draft's sequential
//    head [FT Checkpoint-faithful DSpark architecture]: q_k = policy(z_k),
//    written in full, and x_k drawn from it (greedy: the argmax).

#include <cooperative_groups.h>

#include "kernels.h"
#include "row_policy.cuh"

namespace dspark {

namespace {

namespace cg = cooperative_groups;
using rp::kC;
using rp::kThreads;

__device__ __forceinline__ float inv_mass(uint64_t mass) {
    return static_cast<float>(rp::kFix / static_cast<double>(mass));
}

template <int kDtype>
__global__ void __cluster_dims__(rp::kC, 1, 1) __launch_bounds__(rp::kThreads)
    verify_rows_kernel(const VerifyProbParams p) {
    extern __shared__ __align__(16) float zs[];
    __shared__ rp::Smem sm;
    __shared__ float s_px;          // p(x) of this row's proposal, in its owner CTA
    __shared__ int32_t s_last;      // rank 0: this cluster decides the request
    __shared__ int32_t s_plan[4];   // rank 0: (row to sample, residual?, token, status)
    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;
    if (tid == 0) {
        sm.parity = 0;
        sm.hparity = 0;
        s_px = 0.0f;
        s_last = 0;
    }
    __syncthreads();

    const int rows = p.gamma + 1;
    const int64_t row = blockIdx.x / kC;
    const int b = static_cast<int>(row / rows), i = static_cast<int>(row % rows);
    const int lo = rank * p.slice;
    const int n = max(0, min(p.slice, p.V - lo));
    rp::Slice sl{zs, lo, n, (n + kThreads - 1) / kThreads};
    const int esize = kDtype == kBF16 ? 2 : 4;
    const char* tgt = static_cast<const char*>(p.target);

    rp::Policy pol;
    const bool pol_ok = rp::make_policy(p.policy[b], p.V, pol);
    rp::RowResult res;
    bool bad;
    rp::load_slice_and_max<kDtype>(sm, cl, tgt + row * p.V * esize, lo, n, zs, res, bad);
    res.status = bad ? kReqNonfinite : (res.argmax < 0 ? kReqEmpty : (pol_ok ? kReqOk : kReqBadPolicy));
    if (res.status == kReqOk) rp::row_policy(sm, cl, sl, p.V, pol, res);

    // p(x) of the proposal scored by this row (rows 0..gamma-1), in its owner CTA
    int32_t x = -1;
    if (i < p.gamma) x = p.proposals[b * p.gamma + i];
    const bool x_ok = x >= 0 && x < p.V;
    const int owner = x_ok ? x / p.slice : 0;
    if (res.status == kReqOk && !pol.greedy && x_ok && rank == owner && tid == 0) {
        const float z = zs[x - lo];
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
        p.records[row] = rec;
        const unsigned old = atom_add_acq_rel(p.ticket + b, 1u);
        s_last = old == static_cast<unsigned>(rows - 1);
    }
    cl.sync();
    const bool last = *cl.map_shared_rank(&s_last, 0) != 0;
    if (!last) {
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
        int32_t status = kReqOk;
        for (int k = 0; k < p.gamma; ++k)
            if (xs[k] < 0 || xs[k] >= p.V) status = kReqBadToken;
        if (status == kReqOk)
            for (int r = 0; r < rows; ++r)
                if (rec[r].status != kReqOk) { status = rec[r].status; break; }
        s_plan[0] = -1;
        s_plan[3] = status;
        if (status != kReqOk) {
            for (int r = 0; r < rows; ++r) out[r] = -1;
            p.num_accepted[b] = -1;
            p.status[b] = status;
        } else if (pol.greedy) {
            int nacc = 0;
            while (nacc < p.gamma && xs[nacc] == rec[nacc].argmax) ++nacc;
            for (int r = 0; r < rows; ++r) out[r] = r < nacc ? xs[r] : (r == nacc ? rec[nacc].argmax : -1);
            p.num_accepted[b] = nacc;
            p.status[b] = kReqOk;
        } else {
            int j = 0;  // first rejected position (1-based), 0 = none
            for (int k = 1; k <= p.gamma; ++k) {
                const float pk = rec[k - 1].p_x;
                const float qk = p.q_at_x[b * p.gamma + (k - 1)];
                const float ratio = qk > 0.0f ? pk / qk : (pk > 0.0f ? __int_as_float(0x7F800000) : 0.0f);
                const float u = uniform01(p.seed[b], p.request_id[b], p.pos0[b] + k, 1);
                if (!(pk > 0.0f && u < ratio)) { j = k; break; }
            }
            for (int r = 0; r < rows; ++r) out[r] = -1;
            for (int r = 0; r < (j ? j - 1 : p.gamma); ++r) out[r] = xs[r];
            s_plan[0] = j ? j - 1 : p.gamma;  // target row to draw from
            s_plan[1] = j;                    // residual against q_j when j > 0
        }
    }
    cl.sync();
    const int32_t* plan = cl.map_shared_rank(s_plan, 0);
    const int R = plan[0], j = plan[1];
    if (R >= 0) {
        // draw the residual / bonus token from target row R of request b
        const RowRecord rr = p.records[static_cast<int64_t>(b) * rows + R];
        const int64_t trow = static_cast<int64_t>(b) * rows + R;
        rp::RowResult unused;
        bool unused_bad;
        rp::load_slice_and_max<kDtype>(sm, cl, tgt + trow * p.V * esize, lo, n, zs, unused, unused_bad);
        const float invS = inv_mass(rr.mass);
        auto p_of = [&](int li) {
            const float z = zs[li];
            return rp::in_set(ordered_key(z), lo + li, rr.tau, rr.cut) ? rp::weight_f(z, rr.zmax, rr.inv_t) * invS
                                                                       : 0.0f;
        };
        const int64_t pos = p.pos0[b] + (j ? j : p.gamma + 1);
        const uint32_t m24 = uniform_bits24(p.seed[b], p.request_id[b], pos, 2);
        int32_t token = -1;
        unsigned long long total = 0;
        if (j) {
            // residual weights max(p - q_j, 0), formed in a coalesced pass over the
            // slice and kept in place of the logits
            const float* qrow = p.q + (static_cast<int64_t>(b) * p.gamma + (j - 1)) * p.V + lo;
            __syncthreads();
            for (int li = tid; li < n; li += kThreads) {
                const float pv = p_of(li);
                const float qv = qrow[li];
                zs[li] = fmaxf(pv - qv, 0.0f);  // overwrites only this thread's own element
            }
            __syncthreads();
            token = rp::sample_fixed(sm, cl, sl, m24, [&](int li) { return rp::to_fixed(zs[li]); }, total);
            if (total == 0) {  // no residual mass left (round-off): draw from p itself
                rp::load_slice_and_max<kDtype>(sm, cl, tgt + trow * p.V * esize, lo, n, zs, unused, unused_bad);
                token = rp::sample_fixed(
                    sm, cl, sl, m24,
                    [&](int li) {
                        const float z = zs[li];
                        return rp::in_set(ordered_key(z), lo + li, rr.tau, rr.cut)
                                   ? rp::to_fixed(rp::weight_f(z, rr.zmax, rr.inv_t))
                                   : 0ull;
                    },
                    total);
            }
        } else {
            token = rp::sample_fixed(
                sm, cl, sl, m24,
                [&](int li) {
                    const float z = zs[li];
                    return rp::in_set(ordered_key(z), lo + li, rr.tau, rr.cut)
                               ? rp::to_fixed(rp::weight_f(z, rr.zmax, rr.inv_t))
                               : 0ull;
                },
                total);
        }
        if (rank == 0 && tid == 0) {
            out[R] = token;
            p.num_accepted[b] = R;
            p.status[b] = kReqOk;
        }
    }
    cl.sync();  // keep shared memory alive until every CTA is done reading
}

template <int kDtype>
__global__ void __cluster_dims__(rp::kC, 1, 1) __launch_bounds__(rp::kThreads)
    markov_step_kernel(const MarkovStepParams p) {
    extern __shared__ __align__(16) float zs[];
    __shared__ rp::Smem sm;
    __shared__ float s_qx;
    cg::cluster_group cl = cg::this_cluster();
    const int rank = static_cast<int>(cl.block_rank());
    const int tid = threadIdx.x;
    if (tid == 0) {
        sm.parity = 0;
        sm.hparity = 0;
        s_qx = 0.0f;
    }
    __syncthreads();

    const int b = blockIdx.x / kC;
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
    const int lo = rank * p.slice;
    const int n = max(0, min(p.slice, p.V - lo));
    rp::Slice sl{zs, lo, n, (n + kThreads - 1) / kThreads};
    rp::Policy pol;
    const bool pol_ok = p.policy ? rp::make_policy(p.policy[b], p.V, pol)
                                 : (pol = rp::Policy{1.0f, 0, 1.0f, 1}, true);
    const void* zrow;
    int zdtype;
    if (p.zbuf) {  // logits with the Markov bias, fp32 [B, V]
        zrow = p.zbuf + static_cast<int64_t>(b) * p.V;
        zdtype = kF32;
    } else {
        zrow = static_cast<const char*>(p.backbone) + pidx * p.V * (kDtype == kBF16 ? 2 : 4);
        zdtype = kDtype;
    }
    rp::RowResult res;
    bool bad;
    if (zdtype == kF32)
        rp::load_slice_and_max<kF32>(sm, cl, zrow, lo, n, zs, res, bad);
    else
        rp::load_slice_and_max<kBF16>(sm, cl, zrow, lo, n, zs, res, bad);
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
    rp::row_policy(sm, cl, sl, p.V, pol, res);
    int32_t xk;
    if (pol.greedy) {
        xk = res.argmax;
        if (rank == 0 && tid == 0) s_qx = 1.0f;
    } else {
        const float invS = inv_mass(res.mass);
        float* qrow = p.q + pidx * p.V + lo;
        for (int li = tid; li < n; li += kThreads) {
            const float z = zs[li];
            qrow[li] = rp::in_set(ordered_key(z), lo + li, res.tau, res.cut) ? rp::weight_f(z, res.zmax, pol.inv_t) * invS
                                                                               : 0.0f;
        }
        const uint32_t m24 = uniform_bits24(p.seed[b], p.request_id[b], p.pos0[b] + k, 0);
        unsigned long long total = 0;
        xk = rp::sample_fixed(
            sm, cl, sl, m24,
            [&](int li) {
                const float z = zs[li];
                return rp::in_set(ordered_key(z), lo + li, res.tau, res.cut)
                           ? rp::to_fixed(rp::weight_f(z, res.zmax, pol.inv_t))
                           : 0ull;
            },
            total);
        if (xk >= lo && xk < lo + n && tid == 0)
            s_qx = rp::weight_f(zs[xk - lo], res.zmax, pol.inv_t) * invS;
    }
    cl.sync();
    if (rank == 0 && tid == 0) {
        const int owner = pol.greedy ? 0 : xk / p.slice;
        p.proposals[pidx] = xk;
        p.q_at_x[pidx] = *cl.map_shared_rank(&s_qx, owner);
        if (k == 1) p.status[b] = kReqOk;
    }
    cl.sync();
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

int policy_cluster_size() { return kC; }

int policy_slice(int V) { return ((V + kC - 1) / kC + 7) / 8 * 8; }

cudaError_t launch_verify_prob(const VerifyProbParams& p, cudaStream_t stream) {
    const int smem = p.slice * static_cast<int>(sizeof(float));
    const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(p.B) * (p.gamma + 1) * kC));
    cudaError_t e;
    if (p.dtype == kBF16) {
        if ((e = set_smem(verify_rows_kernel<kBF16>, smem)) != cudaSuccess) return e;
        verify_rows_kernel<kBF16><<<grid, kThreads, smem, stream>>>(p);
    } else {
        if ((e = set_smem(verify_rows_kernel<kF32>, smem)) != cudaSuccess) return e;
        verify_rows_kernel<kF32><<<grid, kThreads, smem, stream>>>(p);
    }
    return cudaGetLastError();
}

cudaError_t launch_markov_step(const MarkovStepParams& p, cudaStream_t stream) {
    const int smem = p.slice * static_cast<int>(sizeof(float));
    const dim3 grid(static_cast<unsigned>(p.B * kC));
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
