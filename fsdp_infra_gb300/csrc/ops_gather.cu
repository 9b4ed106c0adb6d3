// Whole-matrix gather and scatter between the m shard buffers and full 2-D
// matrices, for Muon-style updates that need each matrix whole.
// "veScale-FSDP: Flexible and High-Performance FSDP at Scale", §6.3 Distributed
// Muon: each matrix is redistributed to a root as the full matrix, updated
// there, and the update redistributed back (Algorithm 2).  With every shard in
// this GPU's memory the redistribution is a copy: one launch over the plan's
// pieces (tensor chunks cut at shard bounds), each CTA moving one piece with
// 16-byte streaming loads and stores when both ends are aligned.  A NULL
// matrix pointer skips that tensor.  Bytes move unchanged (no conversion).
#include "common.cuh"

namespace dbuf {
namespace {

constexpr int kCopyUnroll = 4;

__device__ __forceinline__ void copy_bytes(char *__restrict__ dst, const char *__restrict__ src,
                                           int64_t bytes, int es) {
    const int tid = int(threadIdx.x);
    int64_t done = 0;
    if (((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15) == 0) {
        const int64_t nv = bytes / 16;
        const uint4 *s = reinterpret_cast<const uint4 *>(src);
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        for (int64_t b0 = 0; b0 < nv; b0 += int64_t(kThreads) * kCopyUnroll) {
            uint4 r[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const int64_t i = b0 + int64_t(u) * kThreads + tid;
                if (i < nv) r[u] = __ldcs(s + i);
            }
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const int64_t i = b0 + int64_t(u) * kThreads + tid;
                if (i < nv) __stcs(d + i, r[u]);
            }
        }
        done = nv * 16;
    }
    // the rest, one element at a time
    if (es == 4) {
        const float *s = reinterpret_cast<const float *>(src + done);
        float *d = reinterpret_cast<float *>(dst + done);
        for (int64_t i = tid; i < (bytes - done) / 4; i += kThreads) d[i] = s[i];
    } else {
        const uint16_t *s = reinterpret_cast<const uint16_t *>(src + done);
        uint16_t *d = reinterpret_cast<uint16_t *>(dst + done);
        for (int64_t i = tid; i < (bytes - done) / 2; i += kThreads) d[i] = s[i];
    }
}

template <bool GATHER>
__global__ void __launch_bounds__(kThreads)
    piece_copy_kernel(const Piece *__restrict__ pieces, void *const *__restrict__ shards,
                      void *const *__restrict__ tensors, int es) {
    // kChunkSplit CTAs per piece, as the elementwise kernels split their chunks
    Piece pc = pieces[blockIdx.x / kChunkSplit];
    const int start = int(blockIdx.x % kChunkSplit) * kSubElems;
    pc.off += start;
    pc.shard_off += start;
    pc.len = max(0, min(pc.len - start, kSubElems));
    char *tp = static_cast<char *>(tensors[pc.tensor]);
    if (!tp) return;
    char *sp = static_cast<char *>(shards[pc.shard]);
    char *t = tp + pc.off * es;
    char *sh = sp + pc.shard_off * es;
    if (GATHER)
        copy_bytes(t, sh, int64_t(pc.len) * es, es);
    else
        copy_bytes(sh, t, int64_t(pc.len) * es, es);
}

}  // namespace

int launch_gather(const dbuf_plan_t *p, void *const *shards, int dt, void *const *dst,
                  void *stream) {
    if (p->pieces.empty()) return cudaSuccess;
    piece_copy_kernel<true><<<unsigned(p->pieces.size()) * kChunkSplit, kThreads, 0,
                              static_cast<cudaStream_t>(stream)>>>(
        p->dev.pieces, shards, dst, dt == DBUF_F32 ? 4 : 2);
    return cudaGetLastError();
}

int launch_scatter(const dbuf_plan_t *p, const void *const *src, int dt, void *const *shards,
                   void *stream) {
    if (p->pieces.empty()) return cudaSuccess;
    piece_copy_kernel<false><<<unsigned(p->pieces.size()) * kChunkSplit, kThreads, 0,
                               static_cast<cudaStream_t>(stream)>>>(
        p->dev.pieces, shards, const_cast<void *const *>(src), dt == DBUF_F32 ? 4 : 2);
    return cudaGetLastError();
}

}  // namespace dbuf
