// Diagnostic of the library's bounded device waits: thread blocks meeting at
// the grid barrier that the persistent kernels use (grid_barrier_bounded),
// told to expect more arrivals than the grid makes, so that the wait can end
// only by its time limit.  Nothing else is in flight while they wait (no
// copy, no MMA, no tensor memory), and every block returns its status.

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

__global__ void wait_selftest_init_kernel(unsigned* bar, int* error) {
    *bar = 0u;
    *error = 0;
}

__global__ void wait_selftest_kernel(unsigned* bar, int* error, unsigned missing, unsigned long long limit_ns,
                                     int32_t* status, unsigned long long* waited_ns) {
    __shared__ int s_ok;
    const uint64_t t0 = globaltimer_ns();
    const bool ok = grid_barrier_bounded(bar, error, gridDim.x + missing, limit_ns, &s_ok);
    if (threadIdx.x == 0) {
        status[blockIdx.x] = ok ? kReqOk : kReqTimeout;
        waited_ns[blockIdx.x] = globaltimer_ns() - t0;
    }
}

}  // namespace

cudaError_t launch_wait_selftest(int blocks, int missing, uint64_t limit_ns, unsigned* bar, int* error,
                                 int32_t* status, unsigned long long* waited_ns, cudaStream_t stream) {
    wait_selftest_init_kernel<<<1, 1, 0, stream>>>(bar, error);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    unsigned m = static_cast<unsigned>(missing);
    unsigned long long lim = limit_ns;
    void* args[] = {&bar, &error, &m, &lim, &status, &waited_ns};
    return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(wait_selftest_kernel), dim3(blocks), dim3(32),
                                       args, 0, stream);
}

}  // namespace dspark
