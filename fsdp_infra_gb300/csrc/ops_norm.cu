// Ragged L2 norm with a non-finite flag over the planned flat buffer.
// "veScale 深度技术分析", OpDispatcher: the ragged norm handler computes a vector
// norm when shard boundaries do not match tensor boundaries, and a found_inf
// handler checks for non-finite gradients; "PyTorch FSDP: Experiences on Scaling
// Fully Sharded Data Parallel", sharded gradient scaler and known limitations
// (per-parameter norms need tensor boundaries, not shard boundaries).
//
// Two launches, both deterministic (no floating-point atomics):
//  1. one CTA per chunk: each thread sums squares of its elements in kUnroll
//     independent fp32 accumulators (16 terms each for a full chunk), the CTA
//     combines them in fp64 in a fixed shuffle/shared-memory tree, and writes
//     one fp64 partial and one non-finite flag per chunk to the workspace;
//  2. one CTA: per tensor, a warp adds that tensor's chunk partials in a fixed
//     order; the global sum of squares adds the per-tensor sums in a fixed tree;
//     square roots in fp64, results rounded to fp32.
#include "common.cuh"

namespace dbuf {
namespace {

constexpr int kUnroll = 4;
constexpr int kFinThreads = 1024;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
    norm_partial_kernel(const Chunk *__restrict__ chunks, const TensorDesc *__restrict__ td,
                        const char *__restrict__ buf, double *__restrict__ partial,
                        int32_t *__restrict__ flags) {
    const Chunk c = chunks[blockIdx.x];
    const char *x = buf + (td[c.tensor].buf_off + c.off) * elem_bytes<DT>();
    const int len = c.len;
    float acc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc[u] = 0.0f;
    uint32_t emax = 0;
    const int nv = aligned16(x, x) ? len / kVec : 0;
    for (int base = 0; base < nv; base += kThreads * kUnroll) {
        Raw<DT> r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * kThreads + int(threadIdx.x);
            if (i < nv) r[u] = load_unit<DT>(x, i);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * kThreads + int(threadIdx.x);
            if (i < nv) {
                float v[8];
                to_f32<DT>(r[u], v);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    acc[u] = fmaf(v[k], v[k], acc[u]);
                    emax = max(emax, __float_as_uint(v[k]) & 0x7f800000u);
                }
            }
        }
    }
    for (int i = nv * kVec + int(threadIdx.x); i < len; i += kThreads) {
        const float v = load_scalar<DT>(x, i);
        acc[0] = fmaf(v, v, acc[0]);
        emax = max(emax, __float_as_uint(v) & 0x7f800000u);
    }
    double s = 0.0;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) s += double(acc[u]);
    s = warp_sum(s);
    __shared__ double sh[kThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sh[warp] = s;
    const int bad = __syncthreads_or(emax == 0x7f800000u);
    if (threadIdx.x == 0) {
        double t = 0.0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) t += sh[w];
        partial[blockIdx.x] = t;
        flags[blockIdx.x] = bad ? 1 : 0;
    }
}

__global__ void __launch_bounds__(kFinThreads)
    norm_finalize_kernel(const TensorDesc *__restrict__ td, int n, int nc,
                         const double *__restrict__ partial, const int32_t *__restrict__ flags,
                         double *__restrict__ tsum, float *__restrict__ tensor_norms,
                         float *__restrict__ total_norm, int32_t *__restrict__ nonfinite) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int t = warp; t < n; t += kFinThreads / 32) {
        double s = 0.0;
        for (int i = td[t].chunk_begin + lane; i < td[t].chunk_end; i += 32) s += partial[i];
        s = warp_sum(s);
        if (lane == 0) {
            tsum[t] = s;
            tensor_norms[t] = float(sqrt(s));
        }
    }
    int f = 0;
    for (int i = threadIdx.x; i < nc; i += kFinThreads) f |= flags[i];
    f = __syncthreads_or(f);
    double s = 0.0;
    for (int t = threadIdx.x; t < n; t += kFinThreads) s += tsum[t];
    s = warp_sum(s);
    __shared__ double sh[kFinThreads / 32];
    if (lane == 0) sh[warp] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        double tot = 0.0;
        for (int w = 0; w < kFinThreads / 32; ++w) tot += sh[w];
        *total_norm = float(sqrt(tot));
        *nonfinite = f ? 1 : 0;
    }
}

struct NormWorkspace {
    double *partial;
    int32_t *flags;
    double *tsum;
};

NormWorkspace carve(const dbuf_plan_t *p, void *ws) {
    char *b = static_cast<char *>(ws);
    const size_t nc = p->chunks.size();
    NormWorkspace w;
    w.partial = reinterpret_cast<double *>(b);
    b += align256(sizeof(double) * nc);
    w.flags = reinterpret_cast<int32_t *>(b);
    b += align256(sizeof(int32_t) * nc);
    w.tsum = reinterpret_cast<double *>(b);
    return w;
}

}  // namespace

size_t norm_workspace_bytes(const dbuf_plan_t *p) {
    const size_t nc = p->chunks.size();
    return align256(sizeof(double) * nc) + align256(sizeof(int32_t) * nc) +
           align256(sizeof(double) * size_t(p->n)) + 256;
}

int launch_norm(const dbuf_plan_t *p, const void *buf, int dt, float *tensor_norms,
                float *total_norm, int32_t *nonfinite, void *workspace, void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    NormWorkspace w = carve(p, workspace);
    const unsigned nc = unsigned(p->chunks.size());
    if (nc) {
        if (dt == DBUF_F32)
            norm_partial_kernel<DBUF_F32><<<nc, kThreads, 0, st>>>(
                p->dev.chunks, p->dev.tensors, static_cast<const char *>(buf), w.partial, w.flags);
        else
            norm_partial_kernel<DBUF_BF16><<<nc, kThreads, 0, st>>>(
                p->dev.chunks, p->dev.tensors, static_cast<const char *>(buf), w.partial, w.flags);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    norm_finalize_kernel<<<1, kFinThreads, 0, st>>>(p->dev.tensors, p->n, int(nc), w.partial,
                                                    w.flags, w.tsum, tensor_norms, total_norm,
                                                    nonfinite);
    return cudaGetLastError();
}

}  // namespace dbuf
