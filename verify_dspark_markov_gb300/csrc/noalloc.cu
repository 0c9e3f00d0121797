// dspark_verify_greedy_noalloc: the greedy verify without workspace
// arguments.
//
// Who needs it: a caller that cannot obtain device memory for scratch - for
// example a plugin inside a runtime that owns all device memory and offers its
// plugins no allocator, or a latency-critical path that must not call
// cudaMalloc because cudaMalloc may synchronize the device.  Such a caller
// still passes its own inputs and outputs.
//
// The greedy kernel reduces each request's rows inside one thread-block
// cluster and keeps every intermediate (row keys, flags, the decision's
// inputs) in shared memory, so there is no scratch to provide: this entry
// point allocates nothing, reserves no device memory and holds no state, and
// calls on different streams may overlap.

#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark.h"
#include "kernels.h"

extern "C" int dspark_verify_greedy_noalloc(const void* target, int dtype, const int32_t* proposals,
                                            int B, int gamma, int V, int32_t* out_tokens,
                                            int32_t* num_accepted, int32_t* status, void* stream) {
    using namespace dspark;
    if (B < 0 || gamma < 1 || gamma > DSPARK_MAX_GAMMA || V < 8 || V > DSPARK_MAX_VOCAB || V % 8 != 0 ||
        (dtype != DSPARK_BF16 && dtype != DSPARK_F32))
        return DSPARK_EINVAL;
    if (B == 0) return DSPARK_OK;
    if (!target || !proposals || !out_tokens || !num_accepted || !status) return DSPARK_EINVAL;
    if ((reinterpret_cast<uintptr_t>(target) & 15u) != 0) return DSPARK_EINVAL;

    ArgmaxParams p{};
    p.logits = target;
    p.dtype = dtype;
    p.V = V;
    p.rows_per_group = gamma + 1;
    p.gamma = gamma;
    p.mode = kArgmaxVerify;
    p.proposals = proposals;
    p.out_tokens = out_tokens;
    p.num_accepted = num_accepted;
    p.status = status;
    return launch_argmax_rows(p, B, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DSPARK_OK
                                                                                      : DSPARK_ECUDA;
}
