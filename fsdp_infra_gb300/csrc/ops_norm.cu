// Ragged L2 norm with a non-finite flag over the planned flat buffer.
// "veScale 深度技术分析", OpDispatcher: the ragged norm handler computes a vector
// norm when shard boundaries do not match tensor boundaries, and a found_inf
// handler checks for non-finite gradients; "PyTorch FSDP: Experiences on Scaling
// Fully Sharded Data Parallel", sharded gradient scaler and known limitations
// (per-parameter norms need tensor boundaries, not shard boundaries).
//
// One launch, deterministic (no floating-point atomics), two-level tree:
//  1. one CTA per chunk: each thread sums squares of its elements in kUnroll
//     independent fp32 accumulators (16 terms each for a full chunk), adds
//     them and the warp adds its 32 lanes in a fixed fp32 shuffle tree (at most
//     about 22 roundings of 2^-24 on any chunk, far inside the 1e-5 tolerance);
//     the 8 warp sums are combined in fp64 in a fixed order, giving one fp64
//     partial and one non-finite flag per chunk in the workspace.  Keeping the
//     lane-level tree in fp32 matters on this GPU, whose fp64 pipe is narrow;
//  2. the last CTA to finish a tensor (an integer ticket per tensor) adds that
//     tensor's chunk partials in a fixed strided order and tree, writes the
//     tensor's norm, and takes a ticket on a global counter; the last tensor
//     finisher adds the per-tensor sums in a fixed order and writes the global
//     norm and flag.  The sums never depend on which CTA finishes last.
// Square roots in fp64, results rounded to fp32.  The tickets start at zero
// (a zero-filled workspace) and each is returned to zero by its last user, so
// every call leaves them as it found them and needs no clearing launch.
#include "common.cuh"

namespace dbuf {
namespace {

constexpr int kUnroll = 4;
constexpr int kWarps = kThreads / 32;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct NormWorkspace {
    double *partial;    // [nc]
    int32_t *flags;     // [nc]
    double *tsum;       // [n]
    int32_t *tflag;     // [n]
    uint32_t *tickets;  // [n + 1]: per-tensor tickets, then the global one
};

NormWorkspace carve(const dbuf_plan_t *p, void *ws) {
    char *b = static_cast<char *>(ws);
    const size_t nc = p->chunks.size(), n = size_t(p->n);
    NormWorkspace w;
    w.partial = reinterpret_cast<double *>(b);
    b += align256(sizeof(double) * nc);
    w.flags = reinterpret_cast<int32_t *>(b);
    b += align256(sizeof(int32_t) * nc);
    w.tsum = reinterpret_cast<double *>(b);
    b += align256(sizeof(double) * n);
    w.tflag = reinterpret_cast<int32_t *>(b);
    b += align256(sizeof(int32_t) * n);
    w.tickets = reinterpret_cast<uint32_t *>(b);
    return w;
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_sum_f32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Chunk sum: lanes in fp32 (fixed xor tree), warps in fp64 in order; every
// thread must call it; the result is valid in thread 0.
__device__ __forceinline__ double chunk_sum(float v, double *sh) {
    v = warp_sum_f32(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) sh[warp] = double(v);
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0)
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += sh[w];
    return t;
}

// Fixed-order CTA sum: lane-xor tree inside each warp, then warps in order.
// Every thread must call it; the result is valid in thread 0.
__device__ __forceinline__ double block_sum(double v, double *sh) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0)
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += sh[w];
    return t;
}

template <int DT>
__global__ void __launch_bounds__(kThreads)
    norm_kernel(const Chunk *__restrict__ chunks, const TensorDesc *__restrict__ td, int n,
                uint32_t n_nonempty, const char *__restrict__ buf, NormWorkspace w,
                float *__restrict__ tensor_norms, float *__restrict__ total_norm,
                int32_t *__restrict__ nonfinite, double *__restrict__ tensor_sumsq) {
    __shared__ double sh[kWarps];
    __shared__ int last;
    pdl_enter();
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
    float sf = 0.0f;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) sf += acc[u];
    const int bad = __syncthreads_or(emax == 0x7f800000u);
    const double s = chunk_sum(sf, sh);

    // ---- level 2a: the last chunk of a tensor to finish sums that tensor
    const int t = c.tensor;
    if (threadIdx.x == 0) {
        w.partial[blockIdx.x] = s;
        w.flags[blockIdx.x] = bad ? 1 : 0;
        __threadfence();
        const uint32_t need = uint32_t(td[t].chunk_end - td[t].chunk_begin);
        last = (atomicAdd(&w.tickets[t], 1u) + 1u == need);
        if (last) w.tickets[t] = 0u;  // no other CTA of this call touches it again
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    const int cb = td[t].chunk_begin, ce = td[t].chunk_end;
    double ts = 0.0;
    int tf = 0;
    for (int i = cb + int(threadIdx.x); i < ce; i += kThreads) {
        ts += __ldcg(&w.partial[i]);
        tf |= __ldcg(&w.flags[i]);
    }
    tf = __syncthreads_or(tf);
    ts = block_sum(ts, sh);
    if (threadIdx.x == 0) {
        w.tsum[t] = ts;
        w.tflag[t] = tf;
        if (tensor_norms) tensor_norms[t] = float(sqrt(ts));
        if (tensor_sumsq) tensor_sumsq[t] = ts;
        __threadfence();
        last = (atomicAdd(&w.tickets[n], 1u) + 1u == n_nonempty);
        if (last) w.tickets[n] = 0u;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();

    // ---- level 2b: the last tensor to finish sums all tensors (fixed order)
    double tot = 0.0;
    int f = 0;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        if (td[i].chunk_end > td[i].chunk_begin) {
            tot += __ldcg(&w.tsum[i]);
            f |= __ldcg(&w.tflag[i]);
        } else {
            if (tensor_norms) tensor_norms[i] = 0.0f;
            if (tensor_sumsq) tensor_sumsq[i] = 0.0;
        }
    }
    f = __syncthreads_or(f);
    tot = block_sum(tot, sh);
    if (threadIdx.x == 0) {
        if (total_norm) *total_norm = float(sqrt(tot));
        *nonfinite = f ? 1 : 0;
    }
}

// Outputs of a group without any element (no chunk to launch a CTA for).
__global__ void norm_empty_kernel(int n, float *tensor_norms, float *total_norm,
                                  int32_t *nonfinite, double *tensor_sumsq) {
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        if (tensor_norms) tensor_norms[i] = 0.0f;
        if (tensor_sumsq) tensor_sumsq[i] = 0.0;
    }
    if (threadIdx.x == 0) {
        if (total_norm) *total_norm = 0.0f;
        *nonfinite = 0;
    }
}

// Norms from per-tensor sums of squares that were added up across shards (the
// AllReduce of the ranks' partials): each tensor's norm, and the global norm
// from the sums in a fixed order (strided per thread, then the CTA tree), in
// fp64, rounded to fp32.  One CTA.
__global__ void __launch_bounds__(kThreads)
    norm_finish_kernel(int n, const double *__restrict__ sumsq, float *__restrict__ tensor_norms,
                       float *__restrict__ total_norm) {
    __shared__ double sh[kWarps];
    double tot = 0.0;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const double v = sumsq[i];
        tensor_norms[i] = float(sqrt(v));
        tot += v;
    }
    tot = block_sum(tot, sh);
    if (threadIdx.x == 0) *total_norm = float(sqrt(tot));
}

}  // namespace

size_t norm_workspace_bytes(const dbuf_plan_t *p) {
    const size_t nc = p->chunks.size(), n = size_t(p->n);
    return align256(sizeof(double) * nc) + align256(sizeof(int32_t) * nc) +
           align256(sizeof(double) * n) + align256(sizeof(int32_t) * n) +
           align256(sizeof(uint32_t) * (n + 1));
}

size_t norm_ticket_offset(const dbuf_plan_t *p) {
    const size_t nc = p->chunks.size(), n = size_t(p->n);
    return align256(sizeof(double) * nc) + align256(sizeof(int32_t) * nc) +
           align256(sizeof(double) * n) + align256(sizeof(int32_t) * n);
}

size_t norm_ticket_bytes(const dbuf_plan_t *p) { return sizeof(uint32_t) * (size_t(p->n) + 1); }

int launch_norm_finish(const dbuf_plan_t *p, const double *sumsq, float *tensor_norms,
                       float *total_norm, void *stream) {
    norm_finish_kernel<<<1, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        p->n, sumsq, tensor_norms, total_norm);
    return cudaGetLastError();
}

int launch_norm(const dbuf_plan_t *p, const void *buf, int dt, float *tensor_norms,
                float *total_norm, int32_t *nonfinite, void *workspace, void *stream,
                double *tensor_sumsq) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const unsigned nc = unsigned(p->chunks.size());
    if (nc == 0) {
        norm_empty_kernel<<<1, 256, 0, st>>>(p->n, tensor_norms, total_norm, nonfinite,
                                             tensor_sumsq);
        return cudaGetLastError();
    }
    NormWorkspace w = carve(p, workspace);
    uint32_t nonempty = 0;
    for (const TensorDesc &d : p->tdesc) nonempty += d.chunk_end > d.chunk_begin ? 1u : 0u;
    const Chunk *chunks = p->dev.chunks;
    const TensorDesc *td = p->dev.tensors;
    const char *b = static_cast<const char *>(buf);
    if (dt == DBUF_F32)
        return launch_pdl(norm_kernel<DBUF_F32>, nc, kThreads, 0, st, chunks, td, p->n, nonempty, b,
                          w, tensor_norms, total_norm, nonfinite, tensor_sumsq);
    return launch_pdl(norm_kernel<DBUF_BF16>, nc, kThreads, 0, st, chunks, td, p->n, nonempty, b, w,
                      tensor_norms, total_norm, nonfinite, tensor_sumsq);
}

}  // namespace dbuf
