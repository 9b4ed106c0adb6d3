// Device helpers shared by the group-operator kernels: 16-byte vector memory
// access and the element conversions.  Every operator streams its tensor ranges
// once through registers (HBM-bound, O(1) flops per byte: no tensor cores).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dbuf_internal.h"

namespace dbuf {

constexpr int kThreads = 256;  // threads per CTA of the chunk kernels
constexpr int kVec = 8;        // elements per vector unit (32 B fp32, 16 B bf16)

template <int DT>
struct Raw;  // the raw bits of one vector unit of 8 elements
template <>
struct Raw<DBUF_F32> {
    uint4 a, b;
};
template <>
struct Raw<DBUF_BF16> {
    uint4 a;
};

template <int DT>
__host__ __device__ constexpr int elem_bytes() {
    return DT == DBUF_F32 ? 4 : 2;
}

// Streaming loads/stores: the data is touched once per operator.
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    return __ldcs(reinterpret_cast<const uint4 *>(p));
}
__device__ __forceinline__ void st_stream(void *p, uint4 v) {
    __stcs(reinterpret_cast<uint4 *>(p), v);
}

template <int DT>
__device__ __forceinline__ Raw<DT> load_unit(const char *base, int i);
template <>
__device__ __forceinline__ Raw<DBUF_F32> load_unit<DBUF_F32>(const char *base, int i) {
    const char *p = base + size_t(i) * 32;
    return Raw<DBUF_F32>{ld_stream(p), ld_stream(p + 16)};
}
template <>
__device__ __forceinline__ Raw<DBUF_BF16> load_unit<DBUF_BF16>(const char *base, int i) {
    return Raw<DBUF_BF16>{ld_stream(base + size_t(i) * 16)};
}

template <int DT>
__device__ __forceinline__ void store_unit(char *base, int i, const Raw<DT> &r);
template <>
__device__ __forceinline__ void store_unit<DBUF_F32>(char *base, int i, const Raw<DBUF_F32> &r) {
    char *p = base + size_t(i) * 32;
    st_stream(p, r.a);
    st_stream(p + 16, r.b);
}
template <>
__device__ __forceinline__ void store_unit<DBUF_BF16>(char *base, int i,
                                                      const Raw<DBUF_BF16> &r) {
    st_stream(base + size_t(i) * 16, r.a);
}

// bf16 -> fp32 is exact: the bf16 bits are the upper half of the fp32 pattern.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> packed bf16x2 (round to nearest even), first value in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// The 8 values of a unit as fp32.
template <int DT>
__device__ __forceinline__ void to_f32(const Raw<DT> &r, float v[8]);
template <>
__device__ __forceinline__ void to_f32<DBUF_F32>(const Raw<DBUF_F32> &r, float v[8]) {
    v[0] = __uint_as_float(r.a.x); v[1] = __uint_as_float(r.a.y);
    v[2] = __uint_as_float(r.a.z); v[3] = __uint_as_float(r.a.w);
    v[4] = __uint_as_float(r.b.x); v[5] = __uint_as_float(r.b.y);
    v[6] = __uint_as_float(r.b.z); v[7] = __uint_as_float(r.b.w);
}
template <>
__device__ __forceinline__ void to_f32<DBUF_BF16>(const Raw<DBUF_BF16> &r, float v[8]) {
    v[0] = bf16_lo(r.a.x); v[1] = bf16_hi(r.a.x);
    v[2] = bf16_lo(r.a.y); v[3] = bf16_hi(r.a.y);
    v[4] = bf16_lo(r.a.z); v[5] = bf16_hi(r.a.z);
    v[6] = bf16_lo(r.a.w); v[7] = bf16_hi(r.a.w);
}

template <int DT>
__device__ __forceinline__ Raw<DT> from_f32(const float v[8]);
template <>
__device__ __forceinline__ Raw<DBUF_F32> from_f32<DBUF_F32>(const float v[8]) {
    Raw<DBUF_F32> r;
    r.a = make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                     __float_as_uint(v[3]));
    r.b = make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]), __float_as_uint(v[6]),
                     __float_as_uint(v[7]));
    return r;
}
template <>
__device__ __forceinline__ Raw<DBUF_BF16> from_f32<DBUF_BF16>(const float v[8]) {
    return Raw<DBUF_BF16>{make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                     pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]))};
}

// Conversion of a whole unit between element types; same-type units keep their
// bits (NaN payloads included).
template <int SRC, int DST>
struct Convert {
    __device__ __forceinline__ static Raw<DST> run(const Raw<SRC> &r) {
        float v[8];
        to_f32<SRC>(r, v);
        return from_f32<DST>(v);
    }
};
template <int DT>
struct Convert<DT, DT> {
    __device__ __forceinline__ static Raw<DT> run(const Raw<DT> &r) { return r; }
};

// Scalar element access (tails and unaligned chunks).
template <int DT>
__device__ __forceinline__ float load_scalar(const char *base, int64_t i) {
    if (DT == DBUF_F32) return reinterpret_cast<const float *>(base)[i];
    return __uint_as_float(uint32_t(reinterpret_cast<const uint16_t *>(base)[i]) << 16);
}
template <int SRC, int DST>
__device__ __forceinline__ void copy_scalar(const char *s, char *d, int64_t i) {
    if (SRC == DST) {
        if (SRC == DBUF_F32)
            reinterpret_cast<uint32_t *>(d)[i] = reinterpret_cast<const uint32_t *>(s)[i];
        else
            reinterpret_cast<uint16_t *>(d)[i] = reinterpret_cast<const uint16_t *>(s)[i];
    } else if (DST == DBUF_F32) {
        reinterpret_cast<float *>(d)[i] = load_scalar<SRC>(s, i);
    } else {
        __nv_bfloat16 h = __float2bfloat16_rn(reinterpret_cast<const float *>(s)[i]);
        reinterpret_cast<uint16_t *>(d)[i] = *reinterpret_cast<uint16_t *>(&h);
    }
}

__device__ __forceinline__ bool aligned16(const void *a, const void *b) {
    return ((reinterpret_cast<uintptr_t>(a) | reinterpret_cast<uintptr_t>(b)) & 15u) == 0;
}

// The elementwise kernels run kChunkSplit CTAs per chunk, each over one part of
// kSubElems elements (a multiple of 8 elements, so a part starts 16-byte
// aligned whenever its chunk does): smaller CTAs shorten the drain of a launch
// without changing the chunk table the norm's partials are kept per.
constexpr int kChunkSplit = 2;
constexpr int kSubElems = int(kChunkElems / kChunkSplit);
static_assert(kSubElems % kVec == 0, "parts keep vector alignment");

// This CTA's part of its chunk (len 0 when the chunk is shorter than the part's start).
__device__ __forceinline__ Chunk sub_chunk(const Chunk *__restrict__ chunks) {
    Chunk c = chunks[blockIdx.x / kChunkSplit];
    const int start = int(blockIdx.x % kChunkSplit) * kSubElems;
    c.off += start;
    c.len = max(0, min(c.len - start, kSubElems));
    return c;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may be
// scheduled while the previous kernel of its stream is still running; it must
// call pdl_enter before its first access to global memory: the wait returns once
// that kernel has completed and its writes are visible (at once for a kernel
// launched the ordinary way), and the trigger then lets the next kernel be
// scheduled in turn.  What overlaps is only launch and CTA scheduling.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace dbuf
