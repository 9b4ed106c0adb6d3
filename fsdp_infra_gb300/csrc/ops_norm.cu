// Ragged L2 norm with a non-finite flag over the planned flat buffer.
// "veScale 深度技术分析", OpDispatcher: the ragged norm handler computes a vector
// norm when shard boundaries do not match tensor boundaries, and a found_inf
// handler checks for non-finite gradients; "PyTorch FSDP: Experiences on Scaling
// Fully Sharded Data Parallel", sharded gradient scaler and known limitations
// (per-parameter norms need tensor boundaries, not shard boundaries).
//
// Two launches, deterministic (the same inputs give the same bits, whatever
// order the CTAs run in), no floating-point atomics:
//  1. one CTA per chunk: each thread sums squares of its elements in kUnroll
//     independent fp32 accumulators (16 terms each for a full chunk), the warp
//     adds its 32 lanes in a fixed fp32 shuffle tree (at most about 22 roundings
//     of 2^-24 on any chunk, far inside the 1e-5 tolerance), and the 8 warp sums
//     are combined in fp64 in a fixed order: one fp64 partial per chunk, a fixed
//     function of the chunk's values.  Keeping the lane-level tree in fp32
//     matters on this GPU, whose fp64 pipe is narrow;
//  2. the partial is added to its tensor's exact accumulator: a fixed-point
//     number of kDigits 32-bit digits, digit i of weight 2^(32 i + kDigitBase),
//     each digit held in a 64-bit counter.  The partial's 53-bit significand
//     goes into two or three counters by integer reductions, which are exact
//     and commutative, so a tensor's sum does not depend on the order in which
//     its chunks finish.  A partial is an fp64 sum of eight fp32 values: it lies
//     in [2^-149, 2^131) with its lowest bit at weight >= 2^-201, inside the
//     digits; the top digits take the carries of up to 2^31 partials.  A chunk
//     holding an inf or NaN adds nothing and raises the flag; a partial that
//     overflowed fp32 sets the tensor's infinity mark;
//  3. a second, small launch (a programmatic dependent of the first, so it is
//     resident early and starts as soon as the first completes; one warp for
//     up to 32 tensors, which needs no CTA barrier) finishes: one
//     thread per tensor resolves its carries, rounds the exact sum once to fp64
//     (round to nearest even: tensor_sumsq), takes the square root in fp64 and
//     rounds it to fp32 (tensor_norms), and returns the counters to zero; the
//     global sum adds the per-tensor fp64 sums in a fixed order (strided per
//     thread, then the CTA tree; across CTAs, the last one to take a ticket
//     adds them all), and the flag is read and cleared.  Each call leaves the
//     workspace as it found it.
// The CTAs of the first launch take no ticket and wait for nothing: a chain of
// tickets at the end of a launch cost 6-11 us of a short launch, whatever its
// size, and a ticket per CTA on one counter serialised.
#include "common.cuh"

namespace dbuf {
namespace {

constexpr int kUnroll = 4;
constexpr int kWarps = kThreads / 32;
constexpr int kDigits = 16;        // 32-bit digits of a tensor's exact accumulator
constexpr int kDigitBase = -224;   // weight of digit 0 is 2^kDigitBase

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct NormWorkspace {
    unsigned long long *acc;  // [n][kDigits] digit counters of each tensor's sum of squares
    double *tsum;             // [n] each tensor's sum (a finishing launch of several CTAs)
    uint32_t *ticket;         // [0] finishing CTAs done, [1] non-finite flag
};

NormWorkspace carve(const dbuf_plan_t *p, void *ws) {
    char *b = static_cast<char *>(ws);
    const size_t n = size_t(p->n);
    NormWorkspace w;
    w.acc = reinterpret_cast<unsigned long long *>(b);
    b += align256(sizeof(unsigned long long) * kDigits * n);
    w.tsum = reinterpret_cast<double *>(b);
    b += align256(sizeof(double) * n);
    w.ticket = reinterpret_cast<uint32_t *>(b);
    return w;
}


// Exact addition of a finite partial s in [2^-149, 2^131) to a tensor's digit
// counters: its significand m (53 bits) times 2^(e - 52) sits at bit position
// sh = e - 52 - kDigitBase >= 23 of the fixed-point number.
__device__ __forceinline__ void add_exact(unsigned long long *acc, double s) {
    const unsigned long long bits = static_cast<unsigned long long>(__double_as_longlong(s));
    const int ex = int((bits >> 52) & 0x7ffu);
    const unsigned long long m = (bits & ((1ull << 52) - 1)) | (1ull << 52);
    const int sh = ex - 1075 - kDigitBase;
    const int d = sh >> 5, r = sh & 31;
    const unsigned long long lo = m << r;
    atomicAdd(&acc[d], lo & 0xffffffffull);
    atomicAdd(&acc[d + 1], lo >> 32);
    if (r > 11) atomicAdd(&acc[d + 2], m >> (64 - r));
}

// The exact sum held in a tensor's digit counters, rounded once to fp64 (round
// to nearest, ties to even); +inf when the infinity mark is set.
__device__ __forceinline__ double exact_sum(const unsigned long long (&c)[kDigits]) {
    if (c[kDigits - 1] >> 63) return __longlong_as_double(0x7ff0000000000000ll);
    uint32_t dig[kDigits];
    unsigned long long carry = 0;
#pragma unroll
    for (int i = 0; i < kDigits; ++i) {
        const unsigned long long v = c[i] + carry;
        dig[i] = uint32_t(v);
        carry = v >> 32;
    }
    int top = -1;
#pragma unroll
    for (int i = 0; i < kDigits; ++i)
        if (dig[i]) top = i;
    if (top < 0) return 0.0;
    // 96 bits from the top digit down, then the rest as a sticky bit
    const unsigned long long hi =
        (static_cast<unsigned long long>(dig[top]) << 32) | (top >= 1 ? dig[top - 1] : 0u);
    const uint32_t lo = top >= 2 ? dig[top - 2] : 0u;
    bool rest = false;
#pragma unroll
    for (int i = 0; i < kDigits; ++i)
        if (i < top - 2 && dig[i]) rest = true;
    const int lz = __clzll(static_cast<long long>(hi));  // < 32: the top digit is not zero
    const unsigned long long mm = lz ? (hi << lz) | (static_cast<unsigned long long>(lo) >> (32 - lz)) : hi;
    rest = rest || (lz ? uint32_t(lo << lz) != 0u : lo != 0u);
    unsigned long long keep = mm >> 11;
    const unsigned long long drop = mm & 0x7ffu;
    const bool up = drop > 0x400u || (drop == 0x400u && (rest || (keep & 1u)));
    keep += up ? 1u : 0u;  // 2^53 after a carry out is still exact in fp64
    // weight of mm's bit 0 is 2^(32 (top - 1) + kDigitBase - lz); keep drops 11 bits
    return ldexp(static_cast<double>(keep), 32 * (top - 1) + kDigitBase - lz + 11);
}

// Reads a tensor's digit counters (and returns them to zero): its exact sum of
// squares rounded once to fp64.
__device__ __forceinline__ double take_exact(unsigned long long *acc) {
    unsigned long long cnt[kDigits];
    ulonglong2 *a = reinterpret_cast<ulonglong2 *>(acc);
#pragma unroll
    for (int k = 0; k < kDigits / 2; ++k) {
        const ulonglong2 x = __ldcg(&a[k]);
        cnt[2 * k] = x.x;
        cnt[2 * k + 1] = x.y;
    }
#pragma unroll
    for (int k = 0; k < kDigits / 2; ++k) a[k] = make_ulonglong2(0ull, 0ull);
    return exact_sum(cnt);
}

__device__ __forceinline__ uint32_t ticket_acq_rel(uint32_t *p) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
    return old;
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
__global__ void __launch_bounds__(kThreads, 5)
    norm_kernel(const Chunk *__restrict__ chunks, const TensorDesc *__restrict__ td,
                const char *__restrict__ buf, NormWorkspace w) {
    __shared__ double sh[kWarps];
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

    // ---- the chunk's partial into its tensor's exact accumulator (the
    // finishing launch reads it)
    const int t = c.tensor;
    if (threadIdx.x == 0) {
        if (bad) atomicOr(&w.ticket[1], 1u);
        else if (s < 0x1p131) {
            if (s > 0.0) add_exact(w.acc + size_t(t) * kDigits, s);
        } else atomicOr(&w.acc[size_t(t) * kDigits + kDigits - 1], 1ull << 63);
    }
}

// The finishing launch: CTA b finishes tensors [256 b, 256 b + 256); with more
// than one CTA the last one (a ticket) adds the per-tensor sums in the fixed
// order.  Up to 32 tensors take one warp: its xor tree is the CTA sum's first
// level, and the other warps would only have added zeros.
__global__ void __launch_bounds__(kThreads)
    norm_finish_exact_kernel(int n, NormWorkspace w, float *__restrict__ tensor_norms,
                             float *__restrict__ total_norm, int32_t *__restrict__ nonfinite,
                             double *__restrict__ tensor_sumsq) {
    __shared__ double sh[kWarps];
    __shared__ int last;
    pdl_enter();
    const int i = int(blockIdx.x) * kThreads + int(threadIdx.x);
    double ts = 0.0;
    if (i < n) {
        ts = take_exact(w.acc + size_t(i) * kDigits);
        if (tensor_norms) tensor_norms[i] = float(sqrt(ts));
        if (tensor_sumsq) tensor_sumsq[i] = ts;
        if (gridDim.x > 1) w.tsum[i] = ts;
    }
    if (gridDim.x > 1) {
        __threadfence();  // every thread's per-tensor sum before the CTA's ticket
        __syncthreads();
        if (threadIdx.x == 0) last = ticket_acq_rel(&w.ticket[0]) + 1u == gridDim.x;
        __syncthreads();
        if (!last) return;
        __threadfence();
        ts = 0.0;
        for (int j = threadIdx.x; j < n; j += kThreads) ts += __ldcg(&w.tsum[j]);
    }
    // one warp when the launch has 32 threads (n <= 32): the same xor tree,
    // without the CTA barrier (the other warps would add zeros)
    const double tot = blockDim.x == 32 ? warp_sum(ts) : block_sum(ts, sh);
    if (threadIdx.x == 0) {
        const uint32_t f = __ldcg(&w.ticket[1]);
        if (total_norm) *total_norm = float(sqrt(tot));
        *nonfinite = f ? 1 : 0;
        w.ticket[1] = 0u;
        w.ticket[0] = 0u;
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
    const size_t n = size_t(p->n);
    return align256(sizeof(unsigned long long) * kDigits * n) + align256(sizeof(double) * n) + 256;
}

// Every word of the workspace is a counter that must be zero when a call starts.
size_t norm_ticket_offset(const dbuf_plan_t *) { return 0; }

size_t norm_ticket_bytes(const dbuf_plan_t *p) { return norm_workspace_bytes(p); }

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
    const Chunk *chunks = p->dev.chunks;
    const TensorDesc *td = p->dev.tensors;
    const char *b = static_cast<const char *>(buf);
    cudaError_t e;
    if (dt == DBUF_F32)
        e = launch_pdl(norm_kernel<DBUF_F32>, nc, kThreads, 0, st, chunks, td, b, w);
    else
        e = launch_pdl(norm_kernel<DBUF_BF16>, nc, kThreads, 0, st, chunks, td, b, w);
    if (e != cudaSuccess) return e;
    const unsigned fg = unsigned((p->n + kThreads - 1) / kThreads);
    return launch_pdl(norm_finish_exact_kernel, fg, p->n <= 32 ? 32 : kThreads, 0, st, p->n, w,
                      tensor_norms, total_norm, nonfinite, tensor_sumsq);
}

}  // namespace dbuf
