// Fused group optimizer step: AdamW over the planned flat buffer, one launch.
// "veScale 深度技术分析", OpDispatcher: the fused AdamW/SGD handler runs the
// fused optimizer on the local shard; "veScale-FSDP: Flexible and
// High-Performance FSDP at Scale", §5 DBuffer: one kernel over the tensor group
// instead of per-tensor kernels.  The pages name the fused optimizer but not its
// formula: this is the standard decoupled-weight-decay AdamW update, written as
// a fixed sequence of IEEE fp32 operations (no contraction):
//   g = grad * coef;  p = p * (1 - lr*wd)
//   m = beta1*m + (1-beta1)*g;  v = beta2*v + ((1-beta2)*g)*g
//   p = p - (lr/bc1) * (m / (sqrt(v / bc2) + eps))
// coef = min(1, max_norm / (total_norm + 1e-6)) is read from the device norm
// of the same step (gradient-norm clipping, no host round trip); a set
// non-finite flag skips the whole step, as a gradient scaler skips a step with
// inf/NaN gradients.  Tensor ranges only; 28 bytes per element (read p, g, m,
// v; write p, m, v).
#include "common.cuh"

namespace dbuf {
namespace {

constexpr int kUnroll = 2;

struct AdamScalars {
    float coef, decay, step, beta1, beta2, omb1, omb2, bc2, eps;
};

__device__ __forceinline__ AdamScalars adam_scalars(const dbuf_adamw_hparams &hp,
                                                    const float *total_norm) {
    AdamScalars s;
    s.coef = 1.0f;
    if (hp.max_norm > 0.0f && total_norm) {
        const float c = __fdiv_rn(hp.max_norm, __fadd_rn(*total_norm, 1e-6f));
        s.coef = c < 1.0f ? c : 1.0f;
    }
    s.decay = __fsub_rn(1.0f, __fmul_rn(hp.lr, hp.weight_decay));
    s.step = __fdiv_rn(hp.lr, hp.bias_correction1);
    s.beta1 = hp.beta1;
    s.beta2 = hp.beta2;
    s.omb1 = __fsub_rn(1.0f, hp.beta1);
    s.omb2 = __fsub_rn(1.0f, hp.beta2);
    s.bc2 = hp.bias_correction2;
    s.eps = hp.eps;
    return s;
}

__device__ __forceinline__ void adam_elem(const AdamScalars &s, float &p, float g, float &m,
                                          float &v) {
    g = __fmul_rn(g, s.coef);
    const float pd = __fmul_rn(p, s.decay);
    m = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.omb1, g));
    v = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(__fmul_rn(s.omb2, g), g));
    const float denom = __fadd_rn(__fsqrt_rn(__fdiv_rn(v, s.bc2)), s.eps);
    p = __fsub_rn(pd, __fmul_rn(s.step, __fdiv_rn(m, denom)));
}

__global__ void __launch_bounds__(kThreads)
    adamw_kernel(const Chunk *__restrict__ chunks, const TensorDesc *__restrict__ td,
                 float *__restrict__ params, const float *__restrict__ grads,
                 float *__restrict__ exp_avg, float *__restrict__ exp_avg_sq,
                 const dbuf_adamw_hparams hp, const float *__restrict__ total_norm,
                 const int32_t *__restrict__ nonfinite) {
    if (nonfinite && *nonfinite) return;  // skipped step: nothing is written
    const AdamScalars s = adam_scalars(hp, total_norm);
    const Chunk c = chunks[blockIdx.x];
    const int64_t base = td[c.tensor].buf_off + c.off;
    char *p = reinterpret_cast<char *>(params + base);
    const char *g = reinterpret_cast<const char *>(grads + base);
    char *m = reinterpret_cast<char *>(exp_avg + base);
    char *v = reinterpret_cast<char *>(exp_avg_sq + base);
    const int len = c.len;
    const bool vec = aligned16(p, g) && aligned16(m, v);
    const int nv = vec ? len / kVec : 0;
    for (int b0 = 0; b0 < nv; b0 += kThreads * kUnroll) {
        Raw<DBUF_F32> rp[kUnroll], rg[kUnroll], rm[kUnroll], rv[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = b0 + u * kThreads + int(threadIdx.x);
            if (i < nv) {
                rp[u] = load_unit<DBUF_F32>(p, i);
                rg[u] = load_unit<DBUF_F32>(g, i);
                rm[u] = load_unit<DBUF_F32>(m, i);
                rv[u] = load_unit<DBUF_F32>(v, i);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int i = b0 + u * kThreads + int(threadIdx.x);
            if (i < nv) {
                float pv[8], gv[8], mv[8], vv[8];
                to_f32<DBUF_F32>(rp[u], pv);
                to_f32<DBUF_F32>(rg[u], gv);
                to_f32<DBUF_F32>(rm[u], mv);
                to_f32<DBUF_F32>(rv[u], vv);
#pragma unroll
                for (int k = 0; k < 8; ++k) adam_elem(s, pv[k], gv[k], mv[k], vv[k]);
                store_unit<DBUF_F32>(p, i, from_f32<DBUF_F32>(pv));
                store_unit<DBUF_F32>(m, i, from_f32<DBUF_F32>(mv));
                store_unit<DBUF_F32>(v, i, from_f32<DBUF_F32>(vv));
            }
        }
    }
    float *pf = reinterpret_cast<float *>(p);
    const float *gf = reinterpret_cast<const float *>(g);
    float *mf = reinterpret_cast<float *>(m);
    float *vf = reinterpret_cast<float *>(v);
    for (int i = nv * kVec + int(threadIdx.x); i < len; i += kThreads) {
        float pe = pf[i], me = mf[i], ve = vf[i];
        adam_elem(s, pe, gf[i], me, ve);
        pf[i] = pe;
        mf[i] = me;
        vf[i] = ve;
    }
}

}  // namespace

int launch_adamw(const dbuf_plan_t *p, float *params, const float *grads, float *exp_avg,
                 float *exp_avg_sq, const dbuf_adamw_hparams &hp, const float *total_norm,
                 const int32_t *nonfinite, void *stream) {
    if (p->chunks.empty()) return cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    adamw_kernel<<<unsigned(p->chunks.size()), kThreads, 0, st>>>(
        p->dev.chunks, p->dev.tensors, params, grads, exp_avg, exp_avg_sq, hp, total_norm,
        nonfinite);
    return cudaGetLastError();
}

}  // namespace dbuf
