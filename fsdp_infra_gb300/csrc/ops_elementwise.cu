// Elementwise group operators over the planned flat buffer, one launch each:
//   pack (copy-in, fused fp32->bf16 cast), unpack (copy-out), and gradient
//   scale/accumulate/zero.
// "veScale-FSDP: Flexible and High-Performance FSDP at Scale", §5 DBuffer:
// group-level operators replace one add/scale/zero/copy kernel per tensor with
// one kernel over the tensor group; Figure 2 is the copy-in/copy-out these
// operators perform between user tensors and the buffer.
// "PyTorch FSDP: Experiences on Scaling Fully Sharded Data Parallel": native
// mixed precision (one cast per flat parameter), gradient accumulation.
//
// Work split: the plan's chunk table cuts every tensor into chunks of at most
// kChunkElems elements; kChunkSplit CTAs share a chunk, each handling its part
// with 16-byte vector loads and stores (8 elements per thread per unit, kUnroll
// units in flight per thread), and a scalar tail.  Padding between tensors is never touched.
// In a slice plan a tensor is its piece inside one shard: the user tensor is read
// or written from the piece's first element (src_off) on.
#include "common.cuh"

namespace dbuf {
namespace {

constexpr int kUnroll = 4;

template <int SRC, int DST>
__device__ __forceinline__ void copy_cast_range(const char *__restrict__ s, char *__restrict__ d,
                                                int len) {
    const int nv = aligned16(s, d) ? len / kVec : 0;
    for (int base = 0; base < nv; base += kThreads * kUnroll) {
        Raw<SRC> r[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * kThreads + int(threadIdx.x);
            if (i < nv) r[u] = load_unit<SRC>(s, i);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = base + u * kThreads + int(threadIdx.x);
            if (i < nv) store_unit<DST>(d, i, Convert<SRC, DST>::run(r[u]));
        }
    }
    for (int i = nv * kVec + int(threadIdx.x); i < len; i += kThreads) copy_scalar<SRC, DST>(s, d, i);
}

template <int SRC, int DST>
__global__ void __launch_bounds__(kThreads)
    pack_kernel(const Chunk *__restrict__ chunks, const TensorDesc *__restrict__ td,
                const void *const *__restrict__ src, char *__restrict__ buf) {
    pdl_enter();
    const Chunk c = sub_chunk(chunks);
    const TensorDesc &t = td[c.tensor];
    const char *s = static_cast<const char *>(src[c.tensor]) + (t.src_off + c.off) * elem_bytes<SRC>();
    char *d = buf + (t.buf_off + c.off) * elem_bytes<DST>();
    copy_cast_range<SRC, DST>(s, d, c.len);
}

template <int SRC, int DST>
__global__ void __launch_bounds__(kThreads)
    unpack_kernel(const Chunk *__restrict__ chunks, const TensorDesc *__restrict__ td,
                  const char *__restrict__ buf, void *const *__restrict__ dst) {
    pdl_enter();
    const Chunk c = sub_chunk(chunks);
    const TensorDesc &t = td[c.tensor];
    const char *s = buf + (t.buf_off + c.off) * elem_bytes<SRC>();
    char *d = static_cast<char *>(dst[c.tensor]) + (t.src_off + c.off) * elem_bytes<DST>();
    copy_cast_range<SRC, DST>(s, d, c.len);
}

// acc = acc + g*scale (product and sum each rounded to fp32: no FMA), g = +0.
template <int GDT>
__global__ void __launch_bounds__(kThreads)
    sac_kernel(const Chunk *__restrict__ chunks, const TensorDesc *__restrict__ td,
               char *__restrict__ grad, float *__restrict__ acc, float scale) {
    pdl_enter();
    const Chunk c = sub_chunk(chunks);
    const int64_t base = td[c.tensor].buf_off + c.off;
    char *g = grad + base * elem_bytes<GDT>();
    char *a = reinterpret_cast<char *>(acc + base);
    const int len = c.len;
    const int nv = aligned16(g, a) ? len / kVec : 0;
    for (int b0 = 0; b0 < nv; b0 += kThreads * kUnroll) {
        Raw<GDT> gr[kUnroll];
        Raw<DBUF_F32> ar[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = b0 + u * kThreads + int(threadIdx.x);
            if (i < nv) {
                gr[u] = load_unit<GDT>(g, i);
                ar[u] = load_unit<DBUF_F32>(a, i);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = b0 + u * kThreads + int(threadIdx.x);
            if (i < nv) {
                float gv[8], av[8];
                to_f32<GDT>(gr[u], gv);
                to_f32<DBUF_F32>(ar[u], av);
#pragma unroll
                for (int k = 0; k < 8; ++k) av[k] = __fadd_rn(av[k], __fmul_rn(gv[k], scale));
                store_unit<DBUF_F32>(a, i, from_f32<DBUF_F32>(av));
                Raw<GDT> z;
                if constexpr (GDT == DBUF_F32) {
                    z.a = make_uint4(0, 0, 0, 0);
                    z.b = make_uint4(0, 0, 0, 0);
                } else {
                    z.a = make_uint4(0, 0, 0, 0);
                }
                store_unit<GDT>(g, i, z);
            }
        }
    }
    float *af = reinterpret_cast<float *>(a);
    for (int i = nv * kVec + int(threadIdx.x); i < len; i += kThreads) {
        const float gv = load_scalar<GDT>(g, i);
        af[i] = __fadd_rn(af[i], __fmul_rn(gv, scale));
        if (GDT == DBUF_F32) reinterpret_cast<float *>(g)[i] = 0.0f;
        else reinterpret_cast<uint16_t *>(g)[i] = 0;
    }
}

template <int SRC, int DST>
cudaError_t run_pack(const dbuf_plan_t *p, const void *const *src, void *buf, cudaStream_t st) {
    const unsigned grid = unsigned(p->chunks.size()) * kChunkSplit;
    return launch_pdl(pack_kernel<SRC, DST>, grid, kThreads, 0, st,
                      static_cast<const Chunk *>(p->dev.chunks),
                      static_cast<const TensorDesc *>(p->dev.tensors), src, static_cast<char *>(buf));
}

template <int SRC, int DST>
cudaError_t run_unpack(const dbuf_plan_t *p, const void *buf, void *const *dst, cudaStream_t st) {
    const unsigned grid = unsigned(p->chunks.size()) * kChunkSplit;
    return launch_pdl(unpack_kernel<SRC, DST>, grid, kThreads, 0, st,
                      static_cast<const Chunk *>(p->dev.chunks),
                      static_cast<const TensorDesc *>(p->dev.tensors),
                      static_cast<const char *>(buf), dst);
}

}  // namespace

int launch_pack(const dbuf_plan_t *p, const void *const *src, int sdt, void *buf, int bdt,
                void *stream) {
    if (p->chunks.empty()) return cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (sdt == DBUF_F32 && bdt == DBUF_F32) return run_pack<DBUF_F32, DBUF_F32>(p, src, buf, st);
    if (sdt == DBUF_F32 && bdt == DBUF_BF16) return run_pack<DBUF_F32, DBUF_BF16>(p, src, buf, st);
    if (sdt == DBUF_BF16 && bdt == DBUF_BF16) return run_pack<DBUF_BF16, DBUF_BF16>(p, src, buf, st);
    return run_pack<DBUF_BF16, DBUF_F32>(p, src, buf, st);
}

int launch_unpack(const dbuf_plan_t *p, const void *buf, int bdt, void *const *dst, int ddt,
                  void *stream) {
    if (p->chunks.empty()) return cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (bdt == DBUF_F32 && ddt == DBUF_F32) return run_unpack<DBUF_F32, DBUF_F32>(p, buf, dst, st);
    if (bdt == DBUF_F32 && ddt == DBUF_BF16) return run_unpack<DBUF_F32, DBUF_BF16>(p, buf, dst, st);
    if (bdt == DBUF_BF16 && ddt == DBUF_BF16) return run_unpack<DBUF_BF16, DBUF_BF16>(p, buf, dst, st);
    return run_unpack<DBUF_BF16, DBUF_F32>(p, buf, dst, st);
}

int launch_sac(const dbuf_plan_t *p, void *grad, int gdt, float *acc, float scale, void *stream) {
    if (p->chunks.empty()) return cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const unsigned grid = unsigned(p->chunks.size()) * kChunkSplit;
    const Chunk *chunks = p->dev.chunks;
    const TensorDesc *td = p->dev.tensors;
    if (gdt == DBUF_F32)
        return launch_pdl(sac_kernel<DBUF_F32>, grid, kThreads, 0, st, chunks, td,
                          static_cast<char *>(grad), acc, scale);
    return launch_pdl(sac_kernel<DBUF_BF16>, grid, kThreads, 0, st, chunks, td,
                      static_cast<char *>(grad), acc, scale);
}

}  // namespace dbuf
