// Self-test of the bounded waits: one CTA waits on an mbarrier phase that
// nothing will complete, gives up after the given number of tries, and
// records DBUF_ETIMEOUT in the plan's status word, the same path every
// pipelined kernel takes when a copy does not land.
#include "tma.cuh"

namespace dbuf {
namespace {

__global__ void wait_timeout_kernel(uint32_t tries, int32_t *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
    }
    __syncthreads();
    // nothing arrives on `bar`: its first phase never completes
    const bool got = mbar_wait_limit(&bar, 0u, tries);
    if (__syncthreads_or(!got) && threadIdx.x == 0) atomicExch(status, DBUF_ETIMEOUT);
}

}  // namespace
}  // namespace dbuf

extern "C" int dbuf_selftest_wait_timeout(const dbuf_plan_t *p, uint32_t tries, void *stream) {
    if (!p) return DBUF_EINVAL;
    if (!p->uploaded) return DBUF_ENOTUPLOADED;
    if (tries == 0 || tries > dbuf::kWaitLimit) return DBUF_EINVAL;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev != p->dev.device) return e != cudaSuccess ? DBUF_ECUDA : DBUF_EDEVICE;
    dbuf::wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(tries,
                                                                             p->dev.status);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        dbuf::record_cuda_error(int(e));
        return DBUF_ECUDA;
    }
    return DBUF_OK;
}
