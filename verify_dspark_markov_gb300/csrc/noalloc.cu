// dspark_verify_greedy_noalloc: the greedy verify with its scratch in a
// statically allocated device array instead of a caller-provided workspace.
//
// Who needs it: a caller that cannot obtain device memory for scratch - for
// example a plugin inside a runtime that owns all device memory and offers its
// plugins no allocator, or a latency-critical path that must not call
// cudaMalloc because cudaMalloc may synchronize the device.  Such a caller
// still passes its own inputs and outputs; only the scratch moves here.
//
// The scratch is one file-scope array of kNoallocScratchBytes bytes.  Every
// GPU that loads this library reserves it until the process exits.  All calls
// on a device share it and it keeps whatever the previous call left, so each
// call clears the bytes it uses before its kernel runs.  Two calls whose work
// overlaps on the same GPU (e.g. on two streams) race on it; callers must
// serialize them.

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "dspark.h"
#include "kernels.h"

namespace {

constexpr int kMaxRequests = DSPARK_NOALLOC_MAX_REQUESTS;
constexpr int kMaxRows = DSPARK_NOALLOC_MAX_ROWS;
constexpr size_t kAlign = 256;
constexpr size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
// per row: a 64-bit arg-max key and a 32-bit flag word; per request: a ticket
constexpr size_t kKeyBytes = align_up(sizeof(unsigned long long) * kMaxRows);
constexpr size_t kFlagBytes = align_up(sizeof(unsigned int) * kMaxRows);
constexpr size_t kTicketBytes = align_up(sizeof(unsigned int) * kMaxRequests);
constexpr size_t kNoallocScratchBytes = kKeyBytes + kFlagBytes + kTicketBytes;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// Device address of g_noalloc_scratch, looked up once per device.  In host
// code the array's name is only a handle for the runtime, not a device
// address, so it must never be passed to a kernel directly.
constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

cudaError_t scratch_address(int device, void** out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[device]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return cudaSuccess;
}

}  // namespace

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
    // sizes beyond what the static scratch holds are refused, never truncated
    if (B > kMaxRequests || static_cast<int64_t>(B) * (gamma + 1) > kMaxRows) return DSPARK_ENOSPC;

    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) return DSPARK_ECUDA;
    void* base = nullptr;
    if (scratch_address(device, &base) != cudaSuccess) return DSPARK_ECUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int rows = B * (gamma + 1);
    unsigned char* scratch = static_cast<unsigned char*>(base);
    ArgmaxParams p{};
    p.logits = target;
    p.dtype = dtype;
    p.V = V;
    p.rows_per_group = gamma + 1;
    p.gamma = gamma;
    p.mode = kArgmaxVerify;
    p.rowkey = reinterpret_cast<unsigned long long*>(scratch);
    p.rowbad = reinterpret_cast<unsigned int*>(scratch + kKeyBytes);
    p.ticket = reinterpret_cast<unsigned int*>(scratch + kKeyBytes + kFlagBytes);
    p.proposals = proposals;
    p.out_tokens = out_tokens;
    p.num_accepted = num_accepted;
    p.status = status;

    // the kernel needs its counters at zero; clear only what this call uses
    if (cudaMemsetAsync(p.rowkey, 0, sizeof(unsigned long long) * rows, s) != cudaSuccess ||
        cudaMemsetAsync(p.rowbad, 0, sizeof(unsigned int) * rows, s) != cudaSuccess ||
        cudaMemsetAsync(p.ticket, 0, sizeof(unsigned int) * B, s) != cudaSuccess)
        return DSPARK_ECUDA;

    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return DSPARK_ECUDA;
    const int occ = argmax_rows_occupancy(dtype);
    if (sms <= 0 || occ <= 0) return DSPARK_ECUDA;
    p.total = static_cast<int64_t>(rows) * V;
    const int64_t slots = static_cast<int64_t>(sms) * occ;
    int64_t chunk = std::max<int64_t>(8192, (p.total + slots - 1) / slots);
    chunk = (chunk + 7) / 8 * 8;
    p.chunk = chunk;
    const int grid = static_cast<int>((p.total + chunk - 1) / chunk);
    return launch_argmax_rows(p, grid, s) == cudaSuccess ? DSPARK_OK : DSPARK_ECUDA;
}
