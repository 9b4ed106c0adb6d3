// dbuf_norm_nonfinite_noalloc: the ragged norm / non-finite check for callers
// that cannot allocate device memory.
//
// Who needs it: a host program that links only this C ABI and has no device
// allocator of its own to hand out scratch (for example a framework that has
// already reserved the device memory in its own pool, where a cudaMalloc would
// fail or fragment that pool), and code on an out-of-memory recovery path that
// still has to check gradients for inf/NaN to decide whether to skip a step.
// Those callers cannot provide the workspace that dbuf_norm_nonfinite takes.
//
// How: the scratch lives in one file-scope device array of kScratchBytes that
// every device loading the library holds until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device (with that device current) asks the runtime for the array's device
// address once and caches it; later calls reuse it.  A cudaDeviceReset after
// that first call is not supported: the cached address would be stale.
// Each call first clears the counters its norm uses in the array (a memset on
// the caller's stream: the per-tensor accumulators, the flag and the ticket,
// which must start at zero), then runs the same two norm launches as
// dbuf_norm_nonfinite with the array as their workspace, so a call never
// depends on what an earlier call left behind, even one that overlapped another
// and raced on the counters.
// All calls share the one array, so calls that overlap on the GPU (different
// streams, or several host threads) race on it and their results are not
// valid; the caller must serialise them.  No cudaMalloc, cudaFree or other
// allocating routine is called.
#include <cuda_runtime.h>

#include <mutex>

#include "dbuf_internal.h"

namespace {

constexpr size_t kScratchBytes = DBUF_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_norm_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).  Returns a cudaError_t value.
int scratch_address(int dev, void **out) {
    if (dev < 0 || dev >= kMaxDevices) return int(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_norm_scratch);
        if (e != cudaSuccess) return int(e);
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return int(cudaSuccess);
}

}  // namespace

extern "C" int dbuf_norm_nonfinite_noalloc(const dbuf_plan_t *p, const void *buf, int32_t dtype,
                                           float *tensor_norms, float *total_norm,
                                           int32_t *nonfinite, void *stream) {
    if (!p) return DBUF_EINVAL;
    if (!p->uploaded) return DBUF_ENOTUPLOADED;
    if (dtype != DBUF_F32 && dtype != DBUF_BF16) return DBUF_EINVAL;
    if (!total_norm || !nonfinite) return DBUF_EINVAL;
    if ((p->n > 0 && !tensor_norms) || (p->total > 0 && !buf)) return DBUF_EINVAL;
    if (dbuf::norm_workspace_bytes(p) > kScratchBytes) return DBUF_ERANGE;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        dbuf::record_cuda_error(int(e));
        return DBUF_ECUDA;
    }
    if (dev != p->dev.device) return DBUF_EDEVICE;
    void *scratch = nullptr;
    int rc = scratch_address(dev, &scratch);
    if (rc != int(cudaSuccess)) {
        dbuf::record_cuda_error(rc);
        return DBUF_ECUDA;
    }
    e = cudaMemsetAsync(static_cast<char *>(scratch) + dbuf::norm_ticket_offset(p), 0,
                        dbuf::norm_ticket_bytes(p), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        dbuf::record_cuda_error(int(e));
        return DBUF_ECUDA;
    }
    rc = dbuf::launch_norm(p, buf, dtype, tensor_norms, total_norm, nonfinite, scratch, stream);
    if (rc != int(cudaSuccess)) {
        dbuf::record_cuda_error(rc);
        return DBUF_ECUDA;
    }
    return DBUF_OK;
}
