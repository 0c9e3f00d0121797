// Device-side helpers shared by the DSpark kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

constexpr int kBF16 = DSPARK_BF16;
constexpr int kF32 = DSPARK_F32;

// ---------------------------------------------------------------- floats
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Monotone map from fp32 bit patterns to uint32 (larger value -> larger key);
// -0.0 is folded onto +0.0 so that equal values give equal keys.
__device__ __forceinline__ uint32_t ordered_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_to_float(uint32_t k) {
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// NaN or +inf (a logit the method cannot use; -inf is a legal masked logit).
__device__ __forceinline__ bool bad_logit(float f) {
    return (f != f) || (f == __int_as_float(0x7F800000));
}

// max that propagates NaN (PTX max.NaN).
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// --------------------------------------------------------------- Philox
// Philox-4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds, each
// multiplying counter words 0 and 2 by the round multipliers, folding the
// high product halves into words 1 and 3 with the key, and permuting; the
// key advances by the two Weyl increments after each round.
__device__ __forceinline__ uint32_t philox_first_word(uint32_t k0, uint32_t k1, uint32_t c0,
                                                      uint32_t c1, uint32_t c2, uint32_t c3) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
        const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo2 = 0xCD9E8D57u * c2, hi2 = __umulhi(0xCD9E8D57u, c2);
        const uint32_t n0 = hi2 ^ c1 ^ k0;
        const uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo2; c2 = n2; c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

// The 24-bit integer m of the uniform u = m * 2^-24 for one decision.
__device__ __forceinline__ uint32_t uniform_bits24(uint64_t seed, uint64_t request_id,
                                                   int64_t pos, uint32_t draw) {
    const uint64_t p = static_cast<uint64_t>(pos);
    const uint32_t w = philox_first_word(static_cast<uint32_t>(seed),
                                         static_cast<uint32_t>(seed >> 32), draw,
                                         static_cast<uint32_t>(p), static_cast<uint32_t>(p >> 32),
                                         static_cast<uint32_t>(request_id));
    return w >> 8;
}
__device__ __forceinline__ float uniform01(uint64_t seed, uint64_t request_id, int64_t pos,
                                           uint32_t draw) {
    return static_cast<float>(uniform_bits24(seed, request_id, pos, draw)) * (1.0f / 16777216.0f);
}

// ------------------------------------------------------- memory ordering
__device__ __forceinline__ uint64_t ld_relaxed_u64(const unsigned long long* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const unsigned int* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Ticket increment with acquire-release semantics at GPU scope: orders this
// thread's earlier global writes and atomics before it, and later reads after it.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Streaming 16-byte load that is not kept in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// L2 eviction policies for loads that carry a cache hint: lines to be read
// again soon (evict_last) and lines read for the last time (evict_first).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// ld_stream_v4 with an L2 eviction policy.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(policy));
    return v;
}

// ------------------------------------------------ TMA bulk copies, mbarriers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity to complete; give up after
// limit_ns of global time and return false (the caller reports a timeout).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}
// One-dimensional TMA copy global -> shared, completing `bytes` on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

// Device-side waits give up after this long (the kernels normally wait
// microseconds); the affected requests then report DSPARK_REQ_TIMEOUT.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Grid barrier of a persistent launch whose CTAs are all resident (a
// cooperative launch): thread 0 of each CTA adds one arrival to *bar and
// waits until it reaches `target` (gen * gridDim.x for the gen-th barrier).
// The wait ends after limit_ns of global time, or as soon as another CTA has
// given up (*error set): it then sets *error and returns false in every
// thread of the CTA.  No copy, MMA or other wait of the caller may be in
// flight across the call.
__device__ __forceinline__ bool grid_barrier_bounded(unsigned* bar, int* error, unsigned target, uint64_t limit_ns,
                                                     int* s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        __threadfence();
        atomicAdd(bar, 1u);
        const uint64_t t0 = globaltimer_ns();
        while (ld_relaxed_u32(bar) < target) {
            if (*reinterpret_cast<volatile int*>(error) || globaltimer_ns() - t0 > limit_ns) {
                atomicExch(error, 1);
                ok = 0;
                break;
            }
        }
        __threadfence();
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

// ----------------------------------------------------------- reductions
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint64_t w = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = w > v ? w : v;
    }
    return v;
}

// Host-side status codes of the request-status array.
constexpr int32_t kReqOk = DSPARK_REQ_OK;
constexpr int32_t kReqNonfinite = DSPARK_REQ_NONFINITE;
constexpr int32_t kReqEmpty = DSPARK_REQ_EMPTY;
constexpr int32_t kReqTimeout = DSPARK_REQ_TIMEOUT;
constexpr int32_t kReqBadPolicy = DSPARK_REQ_BAD_POLICY;
constexpr int32_t kReqBadToken = DSPARK_REQ_BAD_TOKEN;

}  // namespace dspark
