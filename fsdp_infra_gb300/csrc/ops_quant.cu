// Block-wise absmax quantisation (FP8 E4M3 or INT8) of an fp32 flat buffer.
// "veScale-FSDP: Flexible and High-Performance FSDP at Scale", §4 Block-wise
// RaggedShard: block and shard boundaries coincide, so every shard quantises its
// own blocks without communication; §6.3 8-bit Adam: block-wise INT8
// quantisation of optimizer statistics.
//
// Per block: amax = max |x| (fp32); scale = amax / qmax as one IEEE fp32
// division, 1.0 when not positive; code = enc(x / scale), x / scale rounded to
// nearest even in fp32 (the IEEE quotient).  The quotient is formed from the
// block's correctly rounded reciprocal y = RN(1/scale) with Markstein's
// correction step (P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): q = RN(x*y)
// is within one ulp of x/scale, the remainder r = x - scale*q is exact in one
// fused multiply-add, and RN(q + r*y) is the correctly rounded quotient.  The
// remainder stays exact whenever scale >= 2^-80 (all operands' grids are then
// no finer than the fp32 subnormal spacing wherever the code can be non-zero);
// blocks with a smaller scale use the IEEE division instructions directly.
// The sign is copied from x so that x = -0 gives -0 like the division.  E4M3 encodes with the hardware conversion (round to
// nearest even, saturating to +-448); INT8 rounds half to even and clamps to
// [-127, 127].  Codes share the buffer's layout; scales are tensor by tensor in
// row-major block order.
//
// Two kernels, each one launch over the whole group:
//  - tile kernel (blocks taller than one row, e.g. 128x128): one 512-thread CTA
//    per block; warp w holds rows w, w+16, ... in registers (one float4 per
//    lane per row, a 512-byte coalesced row segment per warp instruction), so
//    the block is read from HBM once; the amax is a shuffle + shared-memory
//    max; codes are written as 4-byte words.
//  - row kernel (1 x qc blocks, e.g. 1x128): one warp per block, 4 blocks per
//    warp and 32 per CTA, loads for all 4 blocks in flight before reducing.
// Shapes outside the vector fast path (odd widths, unaligned rows, blocks
// wider than 128 columns or taller than 128 rows) take a scalar two-pass path
// in the same kernels.
#include "common.cuh"

namespace dbuf {
namespace {

constexpr int kTileThreads = 512;     // one CTA per tile
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kTileRowsPerWarp = 8;   // 16 warps x 8 rows = 128-row tiles
constexpr int kRowBlocksPerWarp = kRowItemBlocks / (kThreads / 32);

template <int Q>
struct QParams;
template <>
struct QParams<DBUF_QUANT_E4M3> {
    static constexpr float qmax = 448.0f;
};
template <>
struct QParams<DBUF_QUANT_INT8> {
    static constexpr float qmax = 127.0f;
};

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ float block_scale(float amax, float qmax) {
    const float s = __fdiv_rn(amax, qmax);
    return (s > 0.0f) ? s : 1.0f;
}

template <int Q>
__device__ __forceinline__ uint32_t encode1(float v);
template <>
__device__ __forceinline__ uint32_t encode1<DBUF_QUANT_E4M3>(float v) {
    return uint32_t(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
template <>
__device__ __forceinline__ uint32_t encode1<DBUF_QUANT_INT8>(float v) {
    int q = __float2int_rn(v);
    q = min(127, max(-127, q));
    return uint32_t(uint8_t(int8_t(q)));
}

// The divisor of one block: scale, its reciprocal, and whether the block takes
// the IEEE division instructions (tiny scales) instead of the reciprocal step.
struct Divisor {
    float s, y;
    bool exact;
};

__device__ __forceinline__ Divisor make_divisor(float scale) {
    Divisor d;
    d.s = scale;
    d.y = __frcp_rn(scale);
    d.exact = !(scale >= 0x1p-80f);
    return d;
}

// x / d.s rounded to nearest even (see the header comment).  EXACT selects the
// IEEE division instructions; callers branch on d.exact once per block so that
// the per-element code holds only one of the two forms.
template <bool EXACT>
__device__ __forceinline__ float quot(float x, const Divisor &d) {
    if (EXACT) return __fdiv_rn(x, d.s);
    const float q = __fmul_rn(x, d.y);
    const float r = __fmaf_rn(-q, d.s, x);
    return copysignf(__fmaf_rn(r, d.y, q), x);
}

template <int Q, bool EXACT>
__device__ __forceinline__ uint32_t encode4(float4 v, const Divisor &d);
template <>
__device__ __forceinline__ uint32_t encode4<DBUF_QUANT_E4M3, false>(float4 v, const Divisor &d) {
    const float2 lo = make_float2(quot<false>(v.x, d), quot<false>(v.y, d));
    const float2 hi = make_float2(quot<false>(v.z, d), quot<false>(v.w, d));
    const uint32_t a = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3);
    const uint32_t b = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3);
    return (a & 0xFFFFu) | (b << 16);
}
template <>
__device__ __forceinline__ uint32_t encode4<DBUF_QUANT_E4M3, true>(float4 v, const Divisor &d) {
    const float2 lo = make_float2(quot<true>(v.x, d), quot<true>(v.y, d));
    const float2 hi = make_float2(quot<true>(v.z, d), quot<true>(v.w, d));
    const uint32_t a = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3);
    const uint32_t b = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3);
    return (a & 0xFFFFu) | (b << 16);
}
template <bool EXACT>
__device__ __forceinline__ uint32_t encode4_int8(float4 v, const Divisor &d) {
    return encode1<DBUF_QUANT_INT8>(quot<EXACT>(v.x, d)) |
           (encode1<DBUF_QUANT_INT8>(quot<EXACT>(v.y, d)) << 8) |
           (encode1<DBUF_QUANT_INT8>(quot<EXACT>(v.z, d)) << 16) |
           (encode1<DBUF_QUANT_INT8>(quot<EXACT>(v.w, d)) << 24);
}
template <>
__device__ __forceinline__ uint32_t encode4<DBUF_QUANT_INT8, false>(float4 v, const Divisor &d) {
    return encode4_int8<false>(v, d);
}
template <>
__device__ __forceinline__ uint32_t encode4<DBUF_QUANT_INT8, true>(float4 v, const Divisor &d) {
    return encode4_int8<true>(v, d);
}

__device__ __forceinline__ float abs_max4(float m, float4 v) {
    return fmaxf(fmaxf(fmaxf(m, fabsf(v.x)), fmaxf(fabsf(v.y), fabsf(v.z))), fabsf(v.w));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float4 ld4(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}

__device__ __forceinline__ bool aligned_mod(const void *p, unsigned a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

// Scalar two-pass quantisation of one h x w block by `nthr` cooperating threads
// (thread index `tid`); the amax is combined through `reduce_max`.
template <int Q, typename ReduceMax>
__device__ __forceinline__ float quant_block_scalar(const float *x, uint8_t *y, int64_t cols, int h,
                                                    int w, int tid, int nthr, ReduceMax reduce_max) {
    float amax = 0.0f;
    const int64_t cnt = int64_t(h) * w;
    for (int64_t i = tid; i < cnt; i += nthr) {
        const int64_t r = i / w, c = i % w;
        amax = fmaxf(amax, fabsf(x[r * cols + c]));
    }
    amax = reduce_max(amax);
    const float scale = block_scale(amax, QParams<Q>::qmax);
    const Divisor d = make_divisor(scale);
    for (int64_t i = tid; i < cnt; i += nthr) {
        const int64_t r = i / w, c = i % w;
        const float v = d.exact ? quot<true>(x[r * cols + c], d) : quot<false>(x[r * cols + c], d);
        y[r * cols + c] = uint8_t(encode1<Q>(v));
    }
    return scale;
}

template <int Q>
__device__ __forceinline__ void tile_body(const QItem &it, const TensorDesc &d,
                                          const float *__restrict__ buf,
                                          uint8_t *__restrict__ codes,
                                          float *__restrict__ scales, float *sh_max) {
    const int64_t bi = it.first / d.nbc, bj = it.first % d.nbc;
    const int64_t r0 = bi * d.qrows, c0 = bj * d.qcols;
    const int h = int(imin64(d.qrows, d.rows - r0));
    const int w = int(imin64(d.qcols, d.cols - c0));
    const int64_t cols = d.cols;
    const float *x = buf + d.buf_off + r0 * cols + c0;
    uint8_t *y = codes + d.buf_off + r0 * cols + c0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool fast = h <= kTileWarps * kTileRowsPerWarp && w <= 128 && (w & 3) == 0 &&
                      (cols & 3) == 0 && aligned_mod(x, 16) && aligned_mod(y, 4);
    float scale;
    if (fast) {
        float4 v[kTileRowsPerWarp];
        float amax = 0.0f;
        const bool col_ok = 4 * lane < w;
#pragma unroll
        for (int k = 0; k < kTileRowsPerWarp; ++k) {
            const int r = warp + k * kTileWarps;
            v[k] = (r < h && col_ok) ? ld4(x + r * cols + 4 * lane) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < kTileRowsPerWarp; ++k) amax = abs_max4(amax, v[k]);
        amax = warp_max(amax);
        if (lane == 0) sh_max[warp] = amax;
        __syncthreads();
        amax = sh_max[0];
#pragma unroll
        for (int i = 1; i < kTileWarps; ++i) amax = fmaxf(amax, sh_max[i]);
        scale = block_scale(amax, QParams<Q>::qmax);
        const Divisor dv = make_divisor(scale);
        if (!dv.exact) {
#pragma unroll
            for (int k = 0; k < kTileRowsPerWarp; ++k) {
                const int r = warp + k * kTileWarps;
                if (r < h && col_ok)
                    __stcs(reinterpret_cast<unsigned int *>(y + r * cols + 4 * lane),
                           encode4<Q, false>(v[k], dv));
            }
        } else {
#pragma unroll
            for (int k = 0; k < kTileRowsPerWarp; ++k) {
                const int r = warp + k * kTileWarps;
                if (r < h && col_ok)
                    __stcs(reinterpret_cast<unsigned int *>(y + r * cols + 4 * lane),
                           encode4<Q, true>(v[k], dv));
            }
        }
    } else {
        scale = quant_block_scalar<Q>(x, y, cols, h, w, threadIdx.x, kTileThreads, [&](float m) {
            m = warp_max(m);
            if (lane == 0) sh_max[warp] = m;
            __syncthreads();
            float r = sh_max[0];
            for (int i = 1; i < kTileWarps; ++i) r = fmaxf(r, sh_max[i]);
            return r;
        });
    }
    if (threadIdx.x == 0) scales[d.scale_off + it.first] = scale;
}

__global__ void __launch_bounds__(kTileThreads, 2)
    quant_tile_kernel(const QItem *__restrict__ items, const TensorDesc *__restrict__ td,
                      const float *__restrict__ buf, uint8_t *__restrict__ codes,
                      float *__restrict__ scales) {
    __shared__ float sh_max[kTileWarps];
    const QItem it = items[blockIdx.x];
    const TensorDesc d = td[it.tensor];
    if (d.quant == DBUF_QUANT_E4M3) tile_body<DBUF_QUANT_E4M3>(it, d, buf, codes, scales, sh_max);
    else tile_body<DBUF_QUANT_INT8>(it, d, buf, codes, scales, sh_max);
}

template <int Q>
__device__ __forceinline__ void row_body(const QItem &it, const TensorDesc &d,
                                         const float *__restrict__ buf,
                                         uint8_t *__restrict__ codes,
                                         float *__restrict__ scales) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t cols = d.cols;
    const float *xt = buf + d.buf_off;
    uint8_t *yt = codes + d.buf_off;
    const bool fast = d.qcols <= 128 && (d.qcols & 3) == 0 && (cols & 3) == 0 &&
                      aligned_mod(xt, 16) && aligned_mod(yt, 4);
    if (fast) {
        float4 v[kRowBlocksPerWarp];
        int64_t boff[kRowBlocksPerWarp];
        int wid[kRowBlocksPerWarp];
#pragma unroll
        for (int j = 0; j < kRowBlocksPerWarp; ++j) {
            const int k = warp + j * (kThreads / 32);
            wid[j] = 0;
            boff[j] = 0;
            v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < it.count) {
                const int64_t b = it.first + k;
                const int64_t bi = b / d.nbc, bj = b % d.nbc;
                const int64_t c0 = bj * d.qcols;
                wid[j] = int(imin64(d.qcols, cols - c0));
                boff[j] = bi * cols + c0;
                if (4 * lane < wid[j]) v[j] = ld4(xt + boff[j] + 4 * lane);
            }
        }
#pragma unroll
        for (int j = 0; j < kRowBlocksPerWarp; ++j) {
            const int k = warp + j * (kThreads / 32);
            if (k >= it.count) continue;  // warp-uniform
            const float amax = warp_max(abs_max4(0.0f, v[j]));
            const float scale = block_scale(amax, QParams<Q>::qmax);
            const Divisor dv = make_divisor(scale);
            unsigned int *dst = reinterpret_cast<unsigned int *>(yt + boff[j] + 4 * lane);
            if (!dv.exact) {
                if (4 * lane < wid[j]) __stcs(dst, encode4<Q, false>(v[j], dv));
            } else {
                if (4 * lane < wid[j]) __stcs(dst, encode4<Q, true>(v[j], dv));
            }
            if (lane == 0) scales[d.scale_off + it.first + k] = scale;
        }
    } else {
        for (int k = warp; k < it.count; k += kThreads / 32) {
            const int64_t b = it.first + k;
            const int64_t bi = b / d.nbc, bj = b % d.nbc;
            const int64_t c0 = bj * d.qcols;
            const int w = int(imin64(d.qcols, cols - c0));
            const float scale = quant_block_scalar<Q>(
                xt + bi * cols + c0, yt + bi * cols + c0, cols, 1, w, lane, 32,
                [](float m) { return warp_max(m); });
            if (lane == 0) scales[d.scale_off + b] = scale;
        }
    }
}

__global__ void __launch_bounds__(kThreads)
    quant_row_kernel(const QItem *__restrict__ items, const TensorDesc *__restrict__ td,
                     const float *__restrict__ buf, uint8_t *__restrict__ codes,
                     float *__restrict__ scales) {
    const QItem it = items[blockIdx.x];
    const TensorDesc d = td[it.tensor];
    if (d.quant == DBUF_QUANT_E4M3) row_body<DBUF_QUANT_E4M3>(it, d, buf, codes, scales);
    else row_body<DBUF_QUANT_INT8>(it, d, buf, codes, scales);
}

}  // namespace

int launch_quant(const dbuf_plan_t *p, const float *buf, uint8_t *codes, float *scales,
                 void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (!p->tile_items.empty()) {
        quant_tile_kernel<<<unsigned(p->tile_items.size()), kTileThreads, 0, st>>>(
            p->dev.tile_items, p->dev.tensors, buf, codes, scales);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (!p->row_items.empty()) {
        quant_row_kernel<<<unsigned(p->row_items.size()), kThreads, 0, st>>>(
            p->dev.row_items, p->dev.tensors, buf, codes, scales);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace dbuf
