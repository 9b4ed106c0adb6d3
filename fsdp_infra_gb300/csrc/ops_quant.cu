// Block-wise absmax quantisation (FP8 E4M3 or INT8) of an fp32 flat buffer.
// "veScale-FSDP: Flexible and High-Performance FSDP at Scale", §4 Block-wise
// RaggedShard: block and shard boundaries coincide, so every shard quantises its
// own blocks without communication; §6.3 8-bit Adam: block-wise INT8
// quantisation of optimizer statistics.
//
// Per block: amax = max |x| (fp32); scale = amax / qmax as one IEEE fp32
// division, 1.0 when not positive; code = enc(x / scale), x / scale rounded to
// nearest even in fp32 (the IEEE quotient, formed with the reciprocal
// correction step of quant_math.cuh).  The sign is copied from x so that x = -0
// gives -0 like the division.  E4M3 encodes with the hardware conversion (round
// to nearest even, saturating to +-448); INT8 rounds half to even and clamps to
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
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "quant_math.cuh"
#include "tma.cuh"

namespace dbuf {
namespace {

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

constexpr int kTileThreads = 512;     // one CTA per tile
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kTileRowsPerWarp = 8;   // 16 warps x 8 rows = 128-row tiles


// Three-input maximum (sm_100+); the inputs here are never NaN.
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float abs_max4(float m, float4 v) {
    return max3f(max3f(m, fabsf(v.x), fabsf(v.y)), fabsf(v.z), fabsf(v.w));
}

// Maximum over the warp of non-negative, NaN-free values (block maxima of |x|
// taken with NaN-ignoring max): their bit patterns order like the values, so
// one integer max reduction does it.
__device__ __forceinline__ float warp_max(float v) {
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

__device__ __forceinline__ float4 ld4(const float *p) {
    return __ldcs(reinterpret_cast<const float4 *>(p));
}

__host__ __device__ __forceinline__ bool aligned_mod(const void *p, unsigned a) {
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
        amax = sh_max[lane % kTileWarps];
#pragma unroll
        for (int o = kTileWarps / 2; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
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
    pdl_enter();
    const QItem it = items[blockIdx.x];
    const TensorDesc d = td[it.tensor];
    if (d.quant == DBUF_QUANT_E4M3) tile_body<DBUF_QUANT_E4M3>(it, d, buf, codes, scales, sh_max);
    else tile_body<DBUF_QUANT_INT8>(it, d, buf, codes, scales, sh_max);
}

// The register-tile kernel over the pipelined list, for buffers that are not
// 16-byte aligned (the rows then cannot be bulk-copied).
__global__ void __launch_bounds__(kTileThreads, 2)
    quant_tile_pipe_list_kernel(const TileItem *__restrict__ items,
                                const TensorDesc *__restrict__ td, const float *__restrict__ buf,
                                uint8_t *__restrict__ codes, float *__restrict__ scales) {
    __shared__ float sh_max[kTileWarps];
    pdl_enter();
    const TileItem ti = items[blockIdx.x];
    const TensorDesc d = td[ti.tensor];
    const QItem it{int64_t(ti.bi) * d.nbc + ti.bj, ti.tensor, 1};
    if (d.quant == DBUF_QUANT_E4M3) tile_body<DBUF_QUANT_E4M3>(it, d, buf, codes, scales, sh_max);
    else tile_body<DBUF_QUANT_INT8>(it, d, buf, codes, scales, sh_max);
}

// Row blocks: 8 lanes per 1 x qc block (qc <= 128), each lane holding up to 4
// float4 (16 elements) of it, so a warp covers 4 blocks and a CTA 32 blocks per
// round; a thread keeps both rounds of its item in flight before reducing.
// The block amax is a 3-level xor shuffle inside the 8-lane group.
constexpr int kRowLanes = 8;
constexpr int kRowGroups = kThreads / kRowLanes;
constexpr int kRowRounds = kRowItemBlocks / kRowGroups;
constexpr int kRowVecs = 128 / 4 / kRowLanes;  // float4 per lane per block

template <int Q>
__device__ __forceinline__ void row_body(const RowItem &it, const TensorDesc &d,
                                         const float *__restrict__ buf,
                                         uint8_t *__restrict__ codes,
                                         float *__restrict__ scales) {
    const int64_t cols = d.cols;
    const float *xt = buf + d.buf_off;
    uint8_t *yt = codes + d.buf_off;
    const uint32_t nbc = uint32_t(d.nbc);
    const bool fast = d.qcols <= 128 && (d.qcols & 3) == 0 && (cols & 3) == 0 &&
                      aligned_mod(xt, 16) && aligned_mod(yt, 4);
    if (fast) {
        const int grp = threadIdx.x / kRowLanes, gl = threadIdx.x % kRowLanes;
        float4 v[kRowRounds][kRowVecs];
        int64_t off[kRowRounds], sidx[kRowRounds];
        int wid[kRowRounds];
#pragma unroll
        for (int j = 0; j < kRowRounds; ++j) {
            const int k = grp + j * kRowGroups;
            wid[j] = 0;
            off[j] = 0;
            sidx[j] = 0;
            if (k < it.count) {
                const uint32_t t = uint32_t(it.bj0) + uint32_t(k);
                const int64_t bi = int64_t(it.bi0) + t / nbc, bj = t % nbc;
                const int64_t c0 = bj * d.qcols;
                wid[j] = int(imin64(d.qcols, cols - c0));
                off[j] = bi * cols + c0;
                sidx[j] = d.scale_off + bi * d.nbc + bj;
            }
#pragma unroll
            for (int u = 0; u < kRowVecs; ++u) {
                const int f = 4 * (gl + u * kRowLanes);
                v[j][u] = f < wid[j] ? ld4(xt + off[j] + f) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int j = 0; j < kRowRounds; ++j) {
            float amax = 0.0f;
#pragma unroll
            for (int u = 0; u < kRowVecs; ++u) amax = abs_max4(amax, v[j][u]);
            // all lanes take part: groups past the item's end reduce zeros
#pragma unroll
            for (int o = kRowLanes / 2; o > 0; o >>= 1)
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            if (wid[j] == 0) continue;
            const float scale = block_scale(amax, QParams<Q>::qmax);
            const Divisor dv = make_divisor(scale);
            if (!dv.exact) {
#pragma unroll
                for (int u = 0; u < kRowVecs; ++u) {
                    const int f = 4 * (gl + u * kRowLanes);
                    if (f < wid[j])
                        __stcs(reinterpret_cast<unsigned int *>(yt + off[j] + f),
                               encode4<Q, false>(v[j][u], dv));
                }
            } else {
#pragma unroll
                for (int u = 0; u < kRowVecs; ++u) {
                    const int f = 4 * (gl + u * kRowLanes);
                    if (f < wid[j])
                        __stcs(reinterpret_cast<unsigned int *>(yt + off[j] + f),
                               encode4<Q, true>(v[j][u], dv));
                }
            }
            if (gl == 0) scales[sidx[j]] = scale;
        }
    } else {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int k = warp; k < it.count; k += kThreads / 32) {
            const uint32_t t = uint32_t(it.bj0) + uint32_t(k);
            const int64_t bi = int64_t(it.bi0) + t / nbc, bj = t % nbc;
            const int64_t c0 = bj * d.qcols;
            const int w = int(imin64(d.qcols, cols - c0));
            const float scale = quant_block_scalar<Q>(
                xt + bi * cols + c0, yt + bi * cols + c0, cols, 1, w, lane, 32,
                [](float m) { return warp_max(m); });
            if (lane == 0) scales[d.scale_off + bi * d.nbc + bj] = scale;
        }
    }
}

__global__ void __launch_bounds__(kThreads)
    quant_row_kernel(const RowItem *__restrict__ items, const TensorDesc *__restrict__ td,
                     const float *__restrict__ buf, uint8_t *__restrict__ codes,
                     float *__restrict__ scales) {
    pdl_enter();
    const RowItem it = items[blockIdx.x];
    const TensorDesc d = td[it.tensor];
    if (d.quant == DBUF_QUANT_E4M3) row_body<DBUF_QUANT_E4M3>(it, d, buf, codes, scales);
    else row_body<DBUF_QUANT_INT8>(it, d, buf, codes, scales);
}

// ---------------------------------------------------------------------------
// Pipelined tile kernel.  One 512-thread CTA per SM walks its tiles (item
// blockIdx.x, blockIdx.x + gridDim.x, ...) in two groups of 8 warps that take
// alternate tiles, so that one group's per-tile chain (wait, maxima, group
// barrier, scale, encode) overlaps the other's.  Each group owns one tile
// buffer: its phases are consumed by that group alone and strictly in order,
// which a parity wait needs (with buffers shared round-robin between groups,
// one group could run two phases ahead on a buffer and take a stale phase for
// its own).  One thread fetches a whole tile with a single 2-D
// tensor-memory-access copy (cp.async.bulk.tensor, tensor map of that tensor,
// zero fill past the tensor's edge) completing on the buffer's mbarrier; the
// group's warps pull the tile into registers (warp w of the group holds rows
// w, w+8, ...), meet the maximum at the group's named barrier, and the
// group's first thread refills the buffer with the group's next tile while
// the codes are encoded and stored.  Every mbarrier
// wait is bounded: a group decides a failed wait together at its barrier,
// records DBUF_ETIMEOUT in the plan's status word and stops; after a CTA-wide
// barrier thread 0 waits (bounded again) for copies still in flight.
// ---------------------------------------------------------------------------
constexpr int kPipeThreads = 512;
constexpr int kPipeWarps = kPipeThreads / 32;
constexpr int kPipeGroupWarps = kPipeWarps / 2;     // warps per ping-pong group
// Each group owns a ring of three half-tile buffers: a tile's two halves (rows
// [0, hr) and [hr, 2 hr), hr = ceil(qrows / 2)) are the group's halves 2t and
// 2t + 1, half h lands in the group's buffer h % 3, so that while the group
// works on tile t the first half of tile t + 1 is in flight and the rest
// follows as soon as tile t is in registers (1.5 tiles in flight per group).
constexpr int kPipeHalves = 3;
constexpr int kPipeBuffers = 2 * kPipeHalves;
constexpr int kPipeHalfBytes = (kPipeMaxRows / 2) * kPipeMaxCols * 4;
constexpr int kPipeRowsPerWarp = kPipeMaxRows / kPipeGroupWarps;
constexpr size_t kPipeSmemBytes = size_t(kPipeBuffers) * kPipeHalfBytes + 1024 + 256;

struct TmaMaps {
    CUtensorMap map[kPipeMaxTensors];
};

struct PipeTile {
    uint8_t *y;
    int64_t cols;
    int64_t scale_idx;
    int h, w, quant, qrows, qcols, slot, x0, y0, hr;
};

__device__ __forceinline__ PipeTile pipe_tile(const TileItem &it, const TensorDesc *__restrict__ td,
                                              uint8_t *codes) {
    const TensorDesc &d = td[it.tensor];
    PipeTile g;
    const int64_t r0 = int64_t(it.bi) * d.qrows, c0 = int64_t(it.bj) * d.qcols;
    g.cols = d.cols;
    g.h = int(imin64(d.qrows, d.rows - r0));
    g.w = int(imin64(d.qcols, d.cols - c0));
    g.y = codes + d.buf_off + r0 * d.cols + c0;
    g.scale_idx = d.scale_off + int64_t(it.bi) * d.nbc + it.bj;
    g.quant = d.quant;
    g.qrows = d.qrows;
    g.qcols = d.qcols;
    g.slot = it.slot;
    g.x0 = int(c0);
    g.y0 = int(r0);
    g.hr = (d.qrows + 1) / 2;
    return g;
}

// One thread: expect half e of the tile's box (hr rows; edges are zero-filled)
// and fetch it.
__device__ __forceinline__ void pipe_issue(const PipeTile &g, const TmaMaps &maps, int e,
                                           char *stage, uint64_t *bar) {
    mbar_arrive_expect_tx(bar, uint32_t(g.hr) * uint32_t(g.qcols) * 4u);
    tma_load_2d(stage, &maps.map[g.slot], g.x0, g.y0 + e * g.hr, bar);
}

template <int Q>
__device__ __forceinline__ void pipe_encode_store(const PipeTile &g, const float4 (&v)[kPipeRowsPerWarp],
                                                  const Divisor &dv, int warp, int lane) {
    const bool col_ok = 4 * lane < g.w;
    if (!dv.exact) {
#pragma unroll
        for (int k = 0; k < kPipeRowsPerWarp; ++k) {
            const int r = warp + k * kPipeGroupWarps;
            if (r < g.h && col_ok)
                __stcs(reinterpret_cast<unsigned int *>(g.y + r * g.cols + 4 * lane),
                       encode4<Q, false>(v[k], dv));
        }
    } else {
#pragma unroll
        for (int k = 0; k < kPipeRowsPerWarp; ++k) {
            const int r = warp + k * kPipeGroupWarps;
            if (r < g.h && col_ok)
                __stcs(reinterpret_cast<unsigned int *>(g.y + r * g.cols + 4 * lane),
                       encode4<Q, true>(v[k], dv));
        }
    }
}

__global__ void __launch_bounds__(kPipeThreads, 1)
    quant_pipe_kernel(const __grid_constant__ TmaMaps maps, const TileItem *__restrict__ items,
                      int nitems, const TensorDesc *__restrict__ td, uint8_t *__restrict__ codes,
                      float *__restrict__ scales, int32_t *__restrict__ status) {
    extern __shared__ unsigned char smem_raw[];
    // tensor copies land at 1024-byte-aligned buffers
    char *stages = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(stages + size_t(kPipeBuffers) * kPipeHalfBytes);
    float *sh_max = reinterpret_cast<float *>(bars + kPipeBuffers);  // [2 groups][2][kPipeGroupWarps]
    int *last = reinterpret_cast<int *>(sh_max + 4 * kPipeGroupWarps);  // last half issued per buffer
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = warp / kPipeGroupWarps, gw = warp % kPipeGroupWarps;
    const int gtid = tid - grp * kPipeGroupWarps * 32;   // thread index in the group
    const int gbar = 1 + grp;                            // the group's named barrier
    const int G = gridDim.x;
    const float iq448 = __frcp_rn(448.0f), iq127 = __frcp_rn(127.0f);  // RN(1 / qmax)

    if (tid == 0) {
        for (int b = 0; b < kPipeBuffers; ++b) {
            mbar_init(&bars[b], 1);
            last[b] = -1;
        }
        mbar_fence_init();
    }

    // Group grp takes this CTA's tiles k = grp, grp + 2, ...: its t-th tile is
    // k = 2t + grp, whose halves are the group's halves 2t and 2t + 1.
    const int mine = int(blockIdx.x) < nitems ? (nitems - 1 - int(blockIdx.x)) / G + 1 : 0;
    const int ntiles = (mine - grp + 1) / 2;
    auto issue_half_of = [&](int h, const PipeTile &g) {  // half h into buffer h % 3
        const int b = grp * kPipeHalves + h % kPipeHalves;
        last[b] = h;  // before the copy, whose arrive releases it to the group
        pipe_issue(g, maps, h & 1, stages + size_t(b) * kPipeHalfBytes, &bars[b]);
    };
    auto issue_half = [&](int h) {  // the group's first thread
        const int t = h >> 1;
        if (t >= ntiles) return;
        issue_half_of(h, pipe_tile(items[int(blockIdx.x) + (2 * t + grp) * G], td, codes));
    };
    // The work items and tensor descriptors are written once, at upload, so the
    // first tiles' descriptors are read before the wait for the previous kernel;
    // only the copies of the buffer it may have written wait.
    PipeTile first0, first1;
    if (gtid == 0) {
        if (ntiles > 0) first0 = pipe_tile(items[int(blockIdx.x) + grp * G], td, codes);
        if (ntiles > 1) first1 = pipe_tile(items[int(blockIdx.x) + (2 + grp) * G], td, codes);
    }
    __syncthreads();
    pdl_enter();
    if (gtid == 0) {
        if (ntiles > 0) {
            issue_half_of(0, first0);
            issue_half_of(1, first0);
        }
        if (ntiles > 1) issue_half_of(2, first1);
    }

    for (int t = 0; t < ntiles; ++t) {
        const int i = int(blockIdx.x) + (2 * t + grp) * G;
        const PipeTile g = pipe_tile(items[i], td, codes);
        const int h0 = 2 * t, h1 = 2 * t + 1;
        const int b0 = grp * kPipeHalves + h0 % kPipeHalves;
        const int b1 = grp * kPipeHalves + h1 % kPipeHalves;
        const bool got0 = mbar_wait_bounded(&bars[b0], uint32_t(h0 / kPipeHalves) & 1u);
        const bool got = got0 && mbar_wait_bounded(&bars[b1], uint32_t(h1 / kPipeHalves) & 1u);

        const float *st0 = reinterpret_cast<const float *>(stages + size_t(b0) * kPipeHalfBytes);
        const float *st1 = reinterpret_cast<const float *>(stages + size_t(b1) * kPipeHalfBytes);
        const bool col_ok = 4 * lane < g.w;
        float4 v[kPipeRowsPerWarp];
        float amax = 0.0f;
#pragma unroll
        for (int r8 = 0; r8 < kPipeRowsPerWarp; ++r8) {
            const int r = gw + r8 * kPipeGroupWarps;
            const bool second = r >= g.hr;
            const float *st = second ? st1 : st0;
            const int lr = second ? r - g.hr : r;
            v[r8] = (r < g.h && col_ok)
                        ? *reinterpret_cast<const float4 *>(st + lr * g.qcols + 4 * lane)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
            amax = abs_max4(amax, v[r8]);
        }
        amax = warp_max(amax);
        float *slot = sh_max + (grp * 2 + (t & 1)) * kPipeGroupWarps;
        if (lane == 0) slot[gw] = amax;
        // Every thread of the group has its rows in registers: both halves may be
        // refilled.  The barrier also settles the group's verdict on the waits.
        if (group_any(!got, gbar, kPipeGroupWarps * 32)) {
            if (gtid == 0) atomicExch(status, DBUF_ETIMEOUT);
            break;
        }
        if (gtid == 0) {
            issue_half(h0 + kPipeHalves);  // the second half of tile t + 1, into b0
            issue_half(h1 + kPipeHalves);  // the first half of tile t + 2, into b1
        }
        amax = warp_max(slot[lane % kPipeGroupWarps]);
        if (g.quant == DBUF_QUANT_E4M3) {
            const float scale = block_scale_cr(amax, QParams<DBUF_QUANT_E4M3>::qmax, iq448);
            pipe_encode_store<DBUF_QUANT_E4M3>(g, v, make_divisor(scale), gw, lane);
            if (gtid == 0) scales[g.scale_idx] = scale;
        } else {
            const float scale = block_scale_cr(amax, QParams<DBUF_QUANT_INT8>::qmax, iq127);
            pipe_encode_store<DBUF_QUANT_INT8>(g, v, make_divisor(scale), gw, lane);
            if (gtid == 0) scales[g.scale_idx] = scale;
        }
    }
    // A copy issued for a tile that a failed group no longer takes may still be
    // in flight into this CTA's shared memory: wait (bounded) for the last copy
    // issued into each buffer before the CTA exits.
    __syncthreads();
    if (tid == 0)
        for (int b = 0; b < kPipeBuffers; ++b)
            if (last[b] >= 0) (void)mbar_wait_bounded(&bars[b], uint32_t(last[b] / kPipeHalves) & 1u);
}

// Host: the tensor-map encoder, looked up once from the driver.
std::mutex g_encode_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

}  // namespace

bool encode_map_2d(CUtensorMap *map, bool f32, void *base, int64_t cols, int64_t rows,
                   int box_cols, int box_rows) {
    if (!g_encode) return false;
    const int es = f32 ? 4 : 1;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * cuuint64_t(es)};
    const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                                2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int prepare_quant_kernels() {
    cudaError_t e = cudaFuncSetAttribute(quant_pipe_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kPipeSmemBytes));
    if (e != cudaSuccess) return int(e);
    std::lock_guard<std::mutex> lock(g_encode_mutex);
    if (!g_encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q);
        if (e != cudaSuccess) return int(e);
        if (q != cudaDriverEntryPointSuccess || !fn) return int(cudaErrorNotSupported);
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    return int(cudaSuccess);
}

namespace {

// Tensor maps of the pipelined tensors of `p` over the buffer `buf` (one 2-D
// map per tensor: columns x rows, row pitch cols*4 bytes, box qcols x qrows).
// The maps of the plan's pipelined tensors b0 .. b0 + count - 1 (one launch).
bool encode_maps(const dbuf_plan_t *p, const float *buf, TmaMaps *maps, size_t b0, size_t count) {
    for (size_t slot = 0; slot < count; ++slot) {
        const TensorDesc &d = p->tdesc[p->pipe_tensors[b0 + slot]];
        if (!encode_map_2d(&maps->map[slot], true, const_cast<float *>(buf + d.buf_off), d.cols,
                           d.rows, d.qcols, (d.qrows + 1) / 2))
            return false;
    }
    return true;
}

}  // namespace

// Persistent grid of the pipelined tile kernel for n tiles on `sms` SMs.  CTA b
// takes tiles b, b + G, ... and its two groups alternate, so a launch lasts as
// many tile rounds as its busiest group has tiles: ceil(ceil(n / G) / 2).  With
// G = sms that is the fewest rounds; from two rounds per group on, the grid is
// then cut to the fewest CTAs that still finish in those rounds (at least 90%
// of the SMs): the same bytes in the same rounds on fewer, fuller groups.
static int pipe_grid(int n, int sms) {
    if (n < 4 * sms) return n < sms ? n : sms;
    const int rounds = ((n + sms - 1) / sms + 1) / 2;
    const int per_cta = 2 * rounds;
    const int g = (n + per_cta - 1) / per_cta;
    const int lo = (9 * sms + 9) / 10;
    return g < lo ? lo : g;
}

int launch_quant(const dbuf_plan_t *p, const float *buf, uint8_t *codes, float *scales,
                 void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Pipelined tiles need 16-byte aligned rows: a 16-byte-aligned fp32 buffer
    // and 4-byte-aligned codes (the plan checked the offsets and widths).
    bool pipe_ok = !p->pipe_items.empty() && aligned_mod(buf, 16) && aligned_mod(codes, 4);
    // one launch per kPipeMaxTensors tensors; every map is encoded before the
    // first launch, so that a map the encoder rejects sends all tiles to the
    // register-tile kernel
    const size_t nslot = p->pipe_tensors.size();
    std::vector<TmaMaps> batches;
    for (size_t b0 = 0; pipe_ok && b0 < nslot; b0 += kPipeMaxTensors) {
        batches.emplace_back();
        pipe_ok = encode_maps(p, buf, &batches.back(), b0,
                              std::min<size_t>(kPipeMaxTensors, nslot - b0));
    }
    if (pipe_ok) {
        for (size_t b = 0; b < batches.size(); ++b) {
            const size_t b0 = b * kPipeMaxTensors;
            const size_t i0 = p->pipe_item_start[b0];
            const size_t i1 = p->pipe_item_start[std::min(nslot, b0 + kPipeMaxTensors)];
            const int n = int(i1 - i0);
            if (n == 0) continue;
            const int grid = pipe_grid(n, p->dev.num_sms);
            const cudaError_t e = launch_pdl(
                quant_pipe_kernel, grid, kPipeThreads, kPipeSmemBytes, st, batches[b],
                static_cast<const TileItem *>(p->dev.pipe_items + i0), n,
                static_cast<const TensorDesc *>(p->dev.tensors), codes, scales, p->dev.status);
            if (e != cudaSuccess) return e;
        }
    } else if (!p->pipe_items.empty()) {
        const cudaError_t e = launch_pdl(
            quant_tile_pipe_list_kernel, unsigned(p->pipe_items.size()), kTileThreads, 0, st,
            static_cast<const TileItem *>(p->dev.pipe_items),
            static_cast<const TensorDesc *>(p->dev.tensors), buf, codes, scales);
        if (e != cudaSuccess) return e;
    }
    if (!p->tile_items.empty()) {
        const cudaError_t e = launch_pdl(
            quant_tile_kernel, unsigned(p->tile_items.size()), kTileThreads, 0, st,
            static_cast<const QItem *>(p->dev.tile_items),
            static_cast<const TensorDesc *>(p->dev.tensors), buf, codes, scales);
        if (e != cudaSuccess) return e;
    }
    if (!p->row_items.empty()) {
        const cudaError_t e = launch_pdl(
            quant_row_kernel, unsigned(p->row_items.size()), kThreads, 0, st,
            static_cast<const RowItem *>(p->dev.row_items),
            static_cast<const TensorDesc *>(p->dev.tensors), buf, codes, scales);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace dbuf
