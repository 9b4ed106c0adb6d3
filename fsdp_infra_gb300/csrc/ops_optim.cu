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
//
// 8-bit AdamW (§6.3 8-bit Adam: block-wise INT8 quantisation of the gradient
// statistics, blocks inside shards) runs the same step on block-quantised
// moments: per quantisation block of a tensor, m = code * scale (signed INT8,
// scale = amax / 127) and v = (code + 1) * scale (unsigned 8-bit without a zero
// level, scale = amax / 256); the fp32 step; new block scales from the new
// moments' amax; re-encoding with the correctly rounded quotient of
// quant_math.cuh.  A group of 4..32 lanes owns one block: pass 1 loads the
// gradients and codes, keeps the new moments in registers and reduces the block
// maxima with shuffles; pass 2 loads the parameters, updates them and writes
// the codes (blocks with more than lanes * kOptUnitsPerLane units recompute the
// moments in pass 2 instead).  Unquantised tensors keep compact fp32 moments and
// take the fp32 path in the same launch.  16 bytes per element (read p, g and
// two codes; write p and two codes) plus 16 bytes per block.
#include <algorithm>

#include "quant_math.cuh"
#include "tma.cuh"

namespace dbuf {
namespace {

constexpr int kUnroll = 2;

struct AdamScalars {
    float coef, decay, step, beta1, beta2, omb1, omb2, bc2, eps;
    float ibc2;  // RN(1 / bc2), for the 8-bit step's quotient
    float i127;  // RN(1 / 127), for the 8-bit step's block scale
    bool fast;   // bc2 and eps inside the range of the correctly rounded forms
};

// The clipping coefficient min(1, max_norm / (total_norm + 1e-6)), 1 without clipping.
__device__ __forceinline__ float clip_coef(const AdamParams &hp, const float *total_norm) {
    if (hp.max_norm > 0.0f && total_norm) {
        const float c = __fdiv_rn(hp.max_norm, __fadd_rn(*total_norm, 1e-6f));
        return c < 1.0f ? c : 1.0f;
    }
    return 1.0f;
}

__device__ __forceinline__ AdamScalars adam_scalars(const AdamParams &hp,
                                                    const float *total_norm) {
    AdamScalars s;
    s.coef = clip_coef(hp, total_norm);
    s.decay = __fsub_rn(1.0f, __fmul_rn(hp.lr, hp.weight_decay));
    s.step = __fdiv_rn(hp.lr, hp.bias_correction1);
    s.beta1 = hp.beta1;
    s.beta2 = hp.beta2;
    s.omb1 = __fsub_rn(1.0f, hp.beta1);
    s.omb2 = __fsub_rn(1.0f, hp.beta2);
    s.bc2 = hp.bias_correction2;
    s.eps = hp.eps;
    s.ibc2 = __frcp_rn(s.bc2);
    s.i127 = __frcp_rn(127.0f);
    s.fast = s.bc2 >= 0x1p-40f && s.bc2 <= 1.0f && s.eps >= 0.0f && s.eps <= 0x1p40f;
    return s;
}

// The same scalars but coef, computed on the host for a kernel that takes them
// as parameters (operands from the constant bank instead of registers).  Each
// operation is one IEEE single-precision operation rounded to nearest, as on
// the device; a volatile result keeps every product and quotient rounded on
// its own (no contraction into a fused multiply-add).
AdamScalars host_scalars(const AdamParams &hp) {
    AdamScalars s;
    volatile float t;
    s.coef = 1.0f;
    t = hp.lr * hp.weight_decay;
    s.decay = 1.0f - t;
    t = hp.lr / hp.bias_correction1;
    s.step = t;
    s.beta1 = hp.beta1;
    s.beta2 = hp.beta2;
    t = 1.0f - hp.beta1;
    s.omb1 = t;
    t = 1.0f - hp.beta2;
    s.omb2 = t;
    s.bc2 = hp.bias_correction2;
    s.eps = hp.eps;
    t = 1.0f / s.bc2;
    s.ibc2 = t;
    t = 1.0f / 127.0f;
    s.i127 = t;
    s.fast = s.bc2 >= 0x1p-40f && s.bc2 <= 1.0f && s.eps >= 0.0f && s.eps <= 0x1p40f;
    return s;
}

// The moments' update (m, v in and out).
__device__ __forceinline__ void adam_moments(const AdamScalars &s, float g, float &m, float &v) {
    g = __fmul_rn(g, s.coef);
    m = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.omb1, g));
    v = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(__fmul_rn(s.omb2, g), g));
}

// The parameter's update from the new moments.
__device__ __forceinline__ float adam_param(const AdamScalars &s, float p, float m, float v) {
    const float pd = __fmul_rn(p, s.decay);
    const float denom = __fadd_rn(__fsqrt_rn(__fdiv_rn(v, s.bc2)), s.eps);
    return __fsub_rn(pd, __fmul_rn(s.step, __fdiv_rn(m, denom)));
}

// adam_param with the correctly rounded forms; equal to it whenever |m| and v
// lie in [2^-60, 2^60] and s.fast holds: v/bc2 is then in [2^-60, 2^100], its
// square root plus eps in [2^-30, 2^51], and m over that in the normal range.
__device__ __forceinline__ float adam_param_cr(const AdamScalars &s, float p, float m, float v) {
    const float pd = __fmul_rn(p, s.decay);
    const float denom = __fadd_rn(sqrt_cr(div_cr(v, s.bc2, s.ibc2)), s.eps);
    return __fsub_rn(pd, __fmul_rn(s.step, div_cr(m, denom, rcp_cr(denom))));
}

// Three-input maximum (a NaN input is ignored, as by fmaxf) and minimum (a NaN
// input gives NaN) of sm_100+.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float fmin3_nan(float a, float b, float c) {
    float r;
    asm("min.NaN.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// adam_moments on a pair: the products packed, each sum scalar (a packed
// product may only feed a scalar, correctly rounded sum, never a packed one).
__device__ __forceinline__ void adam_moments2(const AdamScalars &s, float g0, float g1, float &m0,
                                              float &m1, float &v0, float &v1) {
    const float2 g = __fmul2_rn(make_float2(g0, g1), make_float2(s.coef, s.coef));
    const float2 a = __fmul2_rn(make_float2(s.beta1, s.beta1), make_float2(m0, m1));
    const float2 b = __fmul2_rn(make_float2(s.omb1, s.omb1), g);
    m0 = __fadd_rn(a.x, b.x);
    m1 = __fadd_rn(a.y, b.y);
    const float2 c = __fmul2_rn(make_float2(s.beta2, s.beta2), make_float2(v0, v1));
    const float2 d = __fmul2_rn(__fmul2_rn(make_float2(s.omb2, s.omb2), g), g);
    v0 = __fadd_rn(c.x, d.x);
    v1 = __fadd_rn(c.y, d.y);
}

// adam_param_cr on a pair with the packed fp32x2 multiply, fused multiply-add
// and add: per element the same IEEE operations in the same order.  No packed
// multiply feeds a packed add here (each feeds a fused multiply-add), so the
// compiler has nothing to contract; p * decay - step * q, the one place where
// a product meets a sum, stays scalar.
__device__ __forceinline__ float2 neg2(float2 a) { return make_float2(-a.x, -a.y); }

__device__ __forceinline__ void adam_param_cr2(const AdamScalars &s, float &p0, float &p1, float m0,
                                               float m1, float v0, float v1) {
    const float2 v = make_float2(v0, v1), m = make_float2(m0, m1);
    // v / bc2
    const float2 ib = make_float2(s.ibc2, s.ibc2);
    const float2 q1 = __fmul2_rn(v, ib);
    const float2 a = __ffma2_rn(__ffma2_rn(q1, make_float2(-s.bc2, -s.bc2), v), ib, q1);
    // its square root, plus eps
    const float2 r = make_float2(rsqrt_approx(a.x), rsqrt_approx(a.y));
    const float2 sq = __fmul2_rn(a, r);
    const float2 h = __fmul2_rn(make_float2(0.5f, 0.5f), r);
    const float2 root = __ffma2_rn(__ffma2_rn(neg2(sq), sq, a), h, sq);
    const float2 den = __fadd2_rn(root, make_float2(s.eps, s.eps));
    // its reciprocal, then m / den
    const float2 nden = neg2(den), one = make_float2(1.0f, 1.0f);
    float2 y = make_float2(rcp_approx(den.x), rcp_approx(den.y));
    y = __ffma2_rn(__ffma2_rn(nden, y, one), y, y);
    y = __ffma2_rn(__ffma2_rn(nden, y, one), y, y);
    const float2 q2 = __fmul2_rn(m, y);
    const float2 t = __ffma2_rn(__ffma2_rn(q2, nden, m), y, q2);
    p0 = __fsub_rn(__fmul_rn(p0, s.decay), __fmul_rn(s.step, t.x));
    p1 = __fsub_rn(__fmul_rn(p1, s.decay), __fmul_rn(s.step, t.y));
}

__device__ __forceinline__ void adam_elem(const AdamScalars &s, float &p, float g, float &m,
                                          float &v) {
    adam_moments(s, g, m, v);
    p = adam_param(s, p, m, v);
}

// AdamW over `len` elements of fp32 parameters, gradients and moments.
__device__ __forceinline__ void adamw_range(const AdamScalars &s, float *params,
                                            const float *grads, float *exp_avg,
                                            float *exp_avg_sq, int len) {
    char *p = reinterpret_cast<char *>(params);
    const char *g = reinterpret_cast<const char *>(grads);
    char *m = reinterpret_cast<char *>(exp_avg);
    char *v = reinterpret_cast<char *>(exp_avg_sq);
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

__global__ void __launch_bounds__(kThreads)
    adamw_kernel(const Chunk *__restrict__ chunks, const TensorDesc *__restrict__ td,
                 float *__restrict__ params, const float *__restrict__ grads,
                 float *__restrict__ exp_avg, float *__restrict__ exp_avg_sq,
                 const AdamParams hp, const float *__restrict__ total_norm,
                 const int32_t *__restrict__ nonfinite) {
    if (nonfinite && *nonfinite) return;  // skipped step: nothing is written
    const AdamScalars s = adam_scalars(hp, total_norm);
    const Chunk c = sub_chunk(chunks);
    const int64_t base = td[c.tensor].buf_off + c.off;
    adamw_range(s, params + base, grads + base, exp_avg + base, exp_avg_sq + base, c.len);
}

// ---------------------------------------------------------------------------
// 8-bit AdamW
// ---------------------------------------------------------------------------

// AdamW over `len` fp32 elements, one float4 per thread per iteration: the
// unquantised tensors of the 8-bit step (norm weights, biases) are small, and
// this body keeps the launch's register count at the block path's.
__device__ __forceinline__ void adamw_range_lean(const AdamScalars &s, float *p, const float *g,
                                                 float *m, float *v, int len) {
    const bool vec = aligned16(p, g) && aligned16(m, v);
    const int nv = vec ? len / 4 : 0;
    for (int i = int(threadIdx.x); i < nv; i += kThreads) {
        float4 pp = __ldcs(reinterpret_cast<const float4 *>(p) + i);
        const float4 gg = __ldcs(reinterpret_cast<const float4 *>(g) + i);
        float4 mm = __ldcs(reinterpret_cast<const float4 *>(m) + i);
        float4 vv = __ldcs(reinterpret_cast<const float4 *>(v) + i);
        adam_elem(s, pp.x, gg.x, mm.x, vv.x);
        adam_elem(s, pp.y, gg.y, mm.y, vv.y);
        adam_elem(s, pp.z, gg.z, mm.z, vv.z);
        adam_elem(s, pp.w, gg.w, mm.w, vv.w);
        __stcs(reinterpret_cast<float4 *>(p) + i, pp);
        __stcs(reinterpret_cast<float4 *>(m) + i, mm);
        __stcs(reinterpret_cast<float4 *>(v) + i, vv);
    }
    for (int i = nv * 4 + int(threadIdx.x); i < len; i += kThreads) {
        float pe = p[i], me = m[i], ve = v[i];
        adam_elem(s, pe, g[i], me, ve);
        p[i] = pe;
        m[i] = me;
        v[i] = ve;
    }
}

// Exact conversions through the fp32 significand.  A byte u placed under the
// exponent of 2^23 (bits 0x4B0000uu) is the float 2^23 + u.  For |q| < 2^22,
// RN(q + 1.5*2^23) is 1.5*2^23 + rint(q) with ties to even (fp32 spacing is 1
// in [2^23, 2^24)), and its bits are 0x4B400000 + rint(q), so the low byte is
// rint(q) mod 256.
constexpr float kMagicRound = 12582912.0f;     // 1.5 * 2^23
constexpr uint32_t kMagicByte = 0x4B000000u;   // 2^23

__device__ __forceinline__ float2 splat(float a) { return make_float2(a, a); }

// Packed fp32x2 operations are used only where no packed multiply feeds a
// packed add: the compiler fuses such a pair into one fp32x2 multiply-add (a
// single rounding) even when both carry an explicit round-to-nearest modifier,
// which the scalar __fmul_rn / __fadd_rn never are.  Dequantisation (add, then
// multiply) and encoding (multiply-add, then add) are safe; the moment and
// parameter updates use the scalar forms.

__device__ __forceinline__ float byte_float(uint32_t w, int k) {
    return __uint_as_float(__byte_perm(w, kMagicByte, 0x7650u | unsigned(k)));
}

// The low bytes of four floats' bits, packed into one word.
__device__ __forceinline__ uint32_t low_bytes(float a, float b, float c, float d) {
    const uint32_t ab = __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x0040u);
    const uint32_t cd = __byte_perm(__float_as_uint(c), __float_as_uint(d), 0x0040u);
    return __byte_perm(ab, cd, 0x5410u);
}

// Whether pass 1 also loads the parameters of an in-register block (one memory
// latency per round, more registers) or pass 2 does.
constexpr bool kLoadParamsEarly = true;

// Whether dequantisation and encoding use packed fp32x2 operations (half the
// floating-point instructions, but operands in aligned register pairs) or
// scalar ones.
constexpr bool kPackedCodes = true;

// x / d.s for a scale inside the reciprocal step's range, without the sign
// fix-up (a zero quotient's sign does not change an 8-bit code).
__device__ __forceinline__ float quot_nosign(float x, const Divisor &d) {
    const float q = __fmul_rn(x, d.y);
    return __fmaf_rn(__fmaf_rn(-q, d.s, x), d.y, q);
}

// A lane's unit is W consecutive elements of one block row (W = 4 on the
// vector path).  STREAM marks loads of data read once (evict-first).
template <int W, bool STREAM>
__device__ __forceinline__ void load_f(const float *p, int64_t e, float (&x)[W]) {
    if constexpr (W == 4) {
        const float4 *a = reinterpret_cast<const float4 *>(p + e);
        const float4 t = STREAM ? __ldcs(a) : *a;
        x[0] = t.x; x[1] = t.y; x[2] = t.z; x[3] = t.w;
    } else {
        x[0] = STREAM ? __ldcs(p + e) : p[e];
    }
}

template <int W>
__device__ __forceinline__ void store_f(float *p, int64_t e, const float (&x)[W]) {
    if constexpr (W == 4)
        __stcs(reinterpret_cast<float4 *>(p + e), make_float4(x[0], x[1], x[2], x[3]));
    else
        __stcs(p + e, x[0]);
}

template <int W, bool STREAM>
__device__ __forceinline__ uint32_t load_c(const uint8_t *c, int64_t e) {
    if constexpr (W == 4) {
        const unsigned int *a = reinterpret_cast<const unsigned int *>(c + e);
        return STREAM ? __ldcs(a) : *a;
    } else {
        return c[e];
    }
}

template <int W>
__device__ __forceinline__ void store_c(uint8_t *c, int64_t e, uint32_t x) {
    if constexpr (W == 4)
        __stcs(reinterpret_cast<unsigned int *>(c + e), x);
    else
        c[e] = uint8_t(x);
}

// Dequantise a unit's codes (m = code * scale, v = (code + 1) * scale) and
// step its moments; updates the block maxima.
template <int W, bool STREAM>
__device__ __forceinline__ void unit_moments(const AdamScalars &s, const float *grads,
                                             const uint8_t *mc, const uint8_t *vc, int64_t e,
                                             float ms_old, float vs_old, float (&m)[W],
                                             float (&v)[W], float &mamax, float &vamax) {
    float g[W];
    load_f<W, STREAM>(grads, e, g);
    const uint32_t cm = load_c<W, STREAM>(mc, e), cv = load_c<W, STREAM>(vc, e);
    if constexpr (W == 4 && !kPackedCodes) {
        const uint32_t xm = cm ^ 0x80808080u;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            m[w] = __fmul_rn(__fadd_rn(byte_float(xm, w), -8388736.0f), ms_old);
            v[w] = __fmul_rn(__fadd_rn(byte_float(cv, w), -8388607.0f), vs_old);
            adam_moments(s, g[w], m[w], v[w]);
            mamax = fmaxf(mamax, fabsf(m[w]));
            vamax = fmaxf(vamax, v[w]);
        }
    } else if constexpr (W == 4) {
        // int8 c: the byte c ^ 0x80 = c + 128, so c = (2^23 + c + 128) - (2^23 + 128)
        const uint32_t xm = cm ^ 0x80808080u;
        const float2 om = splat(-8388736.0f), ov = splat(-8388607.0f);
        const float2 sm = splat(ms_old), sv = splat(vs_old);
        float2 m01 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(xm, 0), byte_float(xm, 1)), om), sm);
        float2 m23 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(xm, 2), byte_float(xm, 3)), om), sm);
        float2 v01 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(cv, 0), byte_float(cv, 1)), ov), sv);
        float2 v23 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(cv, 2), byte_float(cv, 3)), ov), sv);
        m[0] = m01.x; m[1] = m01.y; m[2] = m23.x; m[3] = m23.y;
        v[0] = v01.x; v[1] = v01.y; v[2] = v23.x; v[3] = v23.y;
#pragma unroll
        for (int w = 0; w < 4; ++w) adam_moments(s, g[w], m[w], v[w]);
        mamax = fmaxf(fmaxf(mamax, fabsf(m[0])), fmaxf(fabsf(m[1]), fabsf(m[2])));
        mamax = fmaxf(mamax, fabsf(m[3]));
        vamax = fmaxf(fmaxf(vamax, v[0]), fmaxf(v[1], v[2]));
        vamax = fmaxf(vamax, v[3]);
    } else {
        m[0] = __fmul_rn(__int2float_rn(int(int8_t(uint8_t(cm)))), ms_old);
        v[0] = __fmul_rn(__int2float_rn(int(cv & 0xFFu) + 1), vs_old);
        adam_moments(s, g[0], m[0], v[0]);
        mamax = fmaxf(mamax, fabsf(m[0]));
        vamax = fmaxf(vamax, v[0]);
    }
}

// The second moment's code: nearest level (c + 1) * scale, c in [0, 255].
template <bool EXACT>
__device__ __forceinline__ uint32_t v_code(float v, const Divisor &d) {
    const int c = __float2int_rn(quot<EXACT>(v, d));
    return uint32_t(min(256, max(1, c)) - 1);
}

// Pass 2 of one unit: parameters from the new moments, then both codes.  The
// reciprocal-step path (!EXACT: both scales in [2^-80, 2^100]) rounds through
// the magic constant: |m / scale_m| <= 127 (1 + 2^-24) and 0 <= v / scale_v <=
// 256 there, so no clamp can bind beyond max(q, 1) for v.
template <int W, bool EXACT>
__device__ __forceinline__ void unit_update(const AdamScalars &s, float *params, uint8_t *mc,
                                            uint8_t *vc, int64_t e, const float (&pin)[W],
                                            const float (&m)[W], const float (&v)[W],
                                            const Divisor &dm, const Divisor &dv, bool vzero,
                                            bool fast) {
    float p[W];
    uint32_t cm = 0, cv = 0;
    if constexpr (W == 4) {
        bool cr = fast;
#pragma unroll
        for (int w = 0; w < 4; ++w) cr = cr && v[w] >= 0x1p-60f && fabsf(m[w]) >= 0x1p-60f;
        if (cr) {
#pragma unroll
            for (int w = 0; w < 4; ++w) p[w] = adam_param_cr(s, pin[w], m[w], v[w]);
        } else {
#pragma unroll
            for (int w = 0; w < 4; ++w) p[w] = adam_param(s, pin[w], m[w], v[w]);
        }
        if (!EXACT && !kPackedCodes) {
            float qm[4], qv[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                qm[w] = __fadd_rn(quot_nosign(m[w], dm), kMagicRound);
                qv[w] = __fadd_rn(__fadd_rn(fmaxf(quot_nosign(v[w], dv), 1.0f), kMagicRound),
                                  -1.0f);
            }
            cm = low_bytes(qm[0], qm[1], qm[2], qm[3]);
            cv = low_bytes(qv[0], qv[1], qv[2], qv[3]);
        } else if (!EXACT) {
            const float2 mg = splat(kMagicRound);
            const float2 qm01 = __fadd2_rn(quot2(make_float2(m[0], m[1]), dm), mg);
            const float2 qm23 = __fadd2_rn(quot2(make_float2(m[2], m[3]), dm), mg);
            cm = low_bytes(qm01.x, qm01.y, qm23.x, qm23.y);
            float2 qv01 = quot2(make_float2(v[0], v[1]), dv);
            float2 qv23 = quot2(make_float2(v[2], v[3]), dv);
            qv01 = make_float2(fmaxf(qv01.x, 1.0f), fmaxf(qv01.y, 1.0f));
            qv23 = make_float2(fmaxf(qv23.x, 1.0f), fmaxf(qv23.y, 1.0f));
            qv01 = __fadd2_rn(__fadd2_rn(qv01, mg), splat(-1.0f));
            qv23 = __fadd2_rn(__fadd2_rn(qv23, mg), splat(-1.0f));
            cv = low_bytes(qv01.x, qv01.y, qv23.x, qv23.y);
        } else {
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                cm |= encode1<DBUF_QUANT_INT8>(quot<true>(m[w], dm)) << (8 * w);
                cv |= (vzero ? 0u : v_code<true>(v[w], dv)) << (8 * w);
            }
        }
    } else {
        p[0] = adam_param(s, pin[0], m[0], v[0]);
        cm = encode1<DBUF_QUANT_INT8>(quot<EXACT>(m[0], dm));
        cv = vzero ? 0u : v_code<EXACT>(v[0], dv);
    }
    store_f<W>(params, e, p);
    store_c<W>(mc, e, cm);
    store_c<W>(vc, e, cv);
}

// The codes of a unit of 4 from its new moments by the reciprocal-step
// quotient (both scales in [2^-80, 2^100]), as in unit_update<4, false>.
__device__ __forceinline__ void unit_codes_fast(const float (&m)[4], const float (&v)[4],
                                                const Divisor &dm, const Divisor &dv, uint32_t &cm,
                                                uint32_t &cv) {
    const float2 mg = splat(kMagicRound);
    const float2 qm01 = __fadd2_rn(quot2(make_float2(m[0], m[1]), dm), mg);
    const float2 qm23 = __fadd2_rn(quot2(make_float2(m[2], m[3]), dm), mg);
    cm = low_bytes(qm01.x, qm01.y, qm23.x, qm23.y);
    float2 qv01 = quot2(make_float2(v[0], v[1]), dv);
    float2 qv23 = quot2(make_float2(v[2], v[3]), dv);
    qv01 = make_float2(fmaxf(qv01.x, 1.0f), fmaxf(qv01.y, 1.0f));
    qv23 = make_float2(fmaxf(qv23.x, 1.0f), fmaxf(qv23.y, 1.0f));
    qv01 = __fadd2_rn(__fadd2_rn(qv01, mg), splat(-1.0f));
    qv23 = __fadd2_rn(__fadd2_rn(qv23, mg), splat(-1.0f));
    cv = low_bytes(qv01.x, qv01.y, qv23.x, qv23.y);
}

// Walk of one lane over its units u = j, j + lanes, ... of a block with `upr`
// units per row: (row, cu) advances by (dr, dc) with one carry.
struct UnitWalk {
    int row, cu, dr, dc, upr;
    __device__ __forceinline__ UnitWalk(int j, int lanes, int upr_) : upr(upr_) {
        row = j / upr;
        cu = j - row * upr;
        dr = lanes / upr;
        dc = lanes - dr * upr;
    }
    __device__ __forceinline__ void next() {
        cu += dc;
        row += dr;
        if (cu >= upr) {
            cu -= upr;
            ++row;
        }
    }
};

// The same walk as a 32-bit element offset from the block's first element:
// each step adds dr rows and dc units, and a wrap moves to the next row.  Used
// for blocks whose offsets stay below 2^31 (qrows * cols < 2^31).
template <int W>
struct Walk32 {
    int cu, dc, upr;
    unsigned off, step, wrap;  // unsigned: steps past the block's last unit wrap harmlessly
    __device__ __forceinline__ Walk32(int j, int lanes, int upr_, int cols) : upr(upr_) {
        const int row = j / upr;
        cu = j - row * upr;
        off = unsigned(row) * unsigned(cols) + unsigned(cu * W);
        const int dr = lanes / upr;
        dc = lanes - dr * upr;
        step = unsigned(dr) * unsigned(cols) + unsigned(dc * W);
        wrap = unsigned(cols) - unsigned(upr * W);
    }
    __device__ __forceinline__ void next() {
        cu += dc;
        off += step;
        if (cu >= upr) {
            cu -= upr;
            off += wrap;
        }
    }
};

template <int W, bool EXACT>
__device__ __forceinline__ void pass2(const AdamScalars &s, float *params, const float *grads,
                                      uint8_t *mc, uint8_t *vc, int64_t base, int64_t cols,
                                      int j, int lanes, UnitWalk wk, Walk32<W> w32, int nu,
                                      bool inreg, float ms_old, float vs_old,
                                      const float (&pr)[kOptUnitsPerLane][W],
                                      const float (&mr)[kOptUnitsPerLane][W],
                                      const float (&vr)[kOptUnitsPerLane][W], const Divisor &dm,
                                      const Divisor &dv, bool vzero, bool fast) {
    if (inreg) {
        float *pb = params + base;
        uint8_t *mb = mc + base;
        uint8_t *vb = vc + base;
        float pl[kOptUnitsPerLane][W];
        if (!kLoadParamsEarly) {
            Walk32<W> w0 = w32;
#pragma unroll
            for (int i = 0; i < kOptUnitsPerLane; ++i) {
                if (j + i * lanes < nu) load_f<W, true>(pb, w0.off, pl[i]);
                w0.next();
            }
        }
#pragma unroll
        for (int i = 0; i < kOptUnitsPerLane; ++i) {
            if (j + i * lanes < nu) {
                if constexpr (kLoadParamsEarly)
                    unit_update<W, EXACT>(s, pb, mb, vb, w32.off, pr[i], mr[i], vr[i], dm, dv,
                                          vzero, fast);
                else
                    unit_update<W, EXACT>(s, pb, mb, vb, w32.off, pl[i], mr[i], vr[i], dm, dv,
                                          vzero, fast);
            }
            w32.next();
        }
    } else {
        for (int u = j; u < nu; u += lanes) {
            const int64_t e = base + int64_t(wk.row) * cols + wk.cu * W;
            float p[W], m[W], v[W], ma = 0.0f, va = 0.0f;
            load_f<W, true>(params, e, p);
            unit_moments<W, false>(s, grads, mc, vc, e, ms_old, vs_old, m, v, ma, va);
            unit_update<W, EXACT>(s, params, mc, vc, e, p, m, v, dm, dv, vzero, fast);
            wk.next();
        }
    }
}

// One work item: groups of `lanes` threads take its blocks in rounds.  Pass 1
// loads every unit of the block (parameters too, when the block fits in
// registers), pass 2 computes and stores; the block maxima meet by shuffles
// within a warp and through shared memory across warps (lanes > 32), with the
// slots alternating between rounds so that one barrier per round suffices.
template <int W>
__device__ __forceinline__ void opt_item(const AdamScalars &s, const OptItem &it,
                                         const TensorDesc &d, float *params, const float *grads,
                                         uint8_t *mc, uint8_t *vc, float *ms, float *vs,
                                         float2 (*red)[kThreads / 32]) {
    constexpr int U = kOptUnitsPerLane;
    const int lanes = it.lanes;
    const int sh = __ffs(lanes) - 1;
    const int groups = kThreads >> sh;
    const int tid = int(threadIdx.x);
    const int grp = tid >> sh, j = tid & (lanes - 1);
    const int nbc = d.nbc;
    // the lanes of this thread's group within its warp (the whole warp when the
    // group spans warps)
    const unsigned gmask = lanes >= 32 ? 0xFFFFFFFFu
                                       : ((1u << lanes) - 1u) << ((tid & 31) & ~(lanes - 1));
    // the walk over a full-width block, shared by all but the right-edge blocks
    const UnitWalk wfull(j, lanes, d.qcols / W);
    // 32-bit offsets inside a block when its rows span less than 2^31 elements
    const bool small = int64_t(d.qrows) * d.cols < (int64_t(1) << 31);
    const Walk32<W> w32full(j, lanes, d.qcols / W, small ? int(d.cols) : 0);
    int par = 0;
    for (int k0 = 0; k0 < it.count; k0 += groups, par ^= 1) {
        const int k = k0 + grp;
        const bool active = k < it.count;
        int64_t base = 0, si = 0;
        int upr = 1, nu = 0;
        float ms_old = 0.0f, vs_old = 0.0f;
        UnitWalk wk = wfull;
        Walk32<W> w32 = w32full;
        if (active) {
            int bi = it.bi0, bj = it.bj0 + k;
            if (bj >= nbc) {
                const int q = bj / nbc;
                bi += q;
                bj -= q * nbc;
            }
            const int64_t r0 = int64_t(bi) * d.qrows;
            const int c0 = bj * d.qcols;
            const int br = int(min(int64_t(d.qrows), d.rows - r0));
            const int bc = int(min(int64_t(d.qcols), d.cols - c0));
            base = d.buf_off + r0 * d.cols + c0;
            upr = bc / W;
            nu = br * upr;
            if (bc != d.qcols) {
                wk = UnitWalk(j, lanes, upr);
                w32 = Walk32<W>(j, lanes, upr, small ? int(d.cols) : 0);
            }
            si = d.scale_off + int64_t(bi) * nbc + bj;
            ms_old = ms[si];
            vs_old = vs[si];
        }
        const bool inreg = small && nu <= lanes * U;
        float pr[U][W], mr[U][W], vr[U][W];
        float mamax = 0.0f, vamax = 0.0f;
        {
            UnitWalk w1 = wk;
            if (inreg) {
                const float *pb = params + base;
                const float *gb = grads + base;
                const uint8_t *mb = mc + base;
                const uint8_t *vb = vc + base;
                Walk32<W> w2 = w32;
#pragma unroll
                for (int i = 0; i < U; ++i) {
                    if (j + i * lanes < nu) {
                        if (kLoadParamsEarly) load_f<W, true>(pb, w2.off, pr[i]);
                        unit_moments<W, true>(s, gb, mb, vb, w2.off, ms_old, vs_old, mr[i], vr[i],
                                              mamax, vamax);
                    }
                    w2.next();
                }
            } else {
                for (int u = j; u < nu; u += lanes) {
                    float m[W], v[W];
                    unit_moments<W, false>(s, grads, mc, vc,
                                           base + int64_t(w1.row) * d.cols + w1.cu * W, ms_old,
                                           vs_old, m, v, mamax, vamax);
                    w1.next();
                }
            }
        }
        // both maxima are non-negative and NaN-free (fmaxf drops NaN), so their
        // bit patterns order like their values: one integer max per warp group
        mamax = __uint_as_float(__reduce_max_sync(gmask, __float_as_uint(mamax)));
        vamax = __uint_as_float(__reduce_max_sync(gmask, __float_as_uint(vamax)));
        if (lanes > 32) {
            if ((tid & 31) == 0) red[par][tid >> 5] = make_float2(mamax, vamax);
            __syncthreads();
            const int w0 = (grp << sh) >> 5;
            for (int q = 0; q < (lanes >> 5); ++q) {
                const float2 r = red[par][w0 + q];
                mamax = fmaxf(mamax, r.x);
                vamax = fmaxf(vamax, r.y);
            }
        }
        if (!active) continue;
        const float ms_new = block_scale_cr(mamax, 127.0f, s.i127);
        const float vs_new = __fmul_rn(vamax, 0x1p-8f);  // = RN(vamax / 256), underflow included
        const Divisor dm = make_divisor(ms_new), dv = make_divisor(vs_new);
        const bool vzero = !(vs_new > 0.0f);
        // the correctly rounded update needs every |m| and v <= 2^60 (lower
        // bounds are checked per unit)
        const bool fast = s.fast && mamax <= 0x1p60f && vamax <= 0x1p60f;
        if (dm.exact || dv.exact)
            pass2<W, true>(s, params, grads, mc, vc, base, d.cols, j, lanes, wk, w32, nu, inreg,
                           ms_old, vs_old, pr, mr, vr, dm, dv, vzero, fast);
        else
            pass2<W, false>(s, params, grads, mc, vc, base, d.cols, j, lanes, wk, w32, nu, inreg,
                            ms_old, vs_old, pr, mr, vr, dm, dv, vzero, fast);
        if (j == 0) {
            ms[si] = ms_new;
            vs[si] = vs_new;
        }
    }
}

// Four CTAs per SM (64 registers): the step is bound by memory latency as much
// as by instruction issue, and 32 warps per SM beat fewer, spill-free warps.
__global__ void __launch_bounds__(kThreads, 4)
    adamw8_kernel(const Chunk *__restrict__ chunks, const int32_t *__restrict__ plain,
                  int32_t n_plain, const OptItem *__restrict__ items,
                  const TensorDesc *__restrict__ td, float *__restrict__ params,
                  const float *__restrict__ grads, uint8_t *__restrict__ mc,
                  uint8_t *__restrict__ vc, float *__restrict__ ms, float *__restrict__ vs,
                  float *__restrict__ m32, float *__restrict__ v32, const AdamParams hp,
                  const float *__restrict__ total_norm, const int32_t *__restrict__ nonfinite) {
    __shared__ float2 red[2][kThreads / 32];
    if (nonfinite && *nonfinite) return;  // skipped step: nothing is written
    const AdamScalars s = adam_scalars(hp, total_norm);
    if (int(blockIdx.x) < n_plain) {
        const Chunk c = chunks[plain[blockIdx.x]];
        const int64_t base = td[c.tensor].buf_off + c.off;
        const int64_t sb = td[c.tensor].state_off + c.off;
        adamw_range_lean(s, params + base, grads + base, m32 + sb, v32 + sb, c.len);
        return;
    }
    const OptItem it = items[blockIdx.x - n_plain];
    const TensorDesc &d = td[it.tensor];
    const bool vec = d.qcols % 4 == 0 && d.cols % 4 == 0 && d.buf_off % 4 == 0 &&
                     aligned16(params, grads) &&
                     ((reinterpret_cast<uintptr_t>(mc) | reinterpret_cast<uintptr_t>(vc)) & 3) == 0;
    if (vec)
        opt_item<4>(s, it, d, params, grads, mc, vc, ms, vs, red);
    else
        opt_item<1>(s, it, d, params, grads, mc, vc, ms, vs, red);
}

// ---------------------------------------------------------------------------
// Pipelined 8-bit AdamW.  One CTA of 16 warps per SM.  Each stage is a box of
// whole quantisation blocks of one tensor holding kP8StageElems elements,
// fetched with four 2-D tensor-map copies (p, g, m codes, v codes) into one of
// two shared-memory buffers and completing on the buffer's "full" mbarrier.
// The warp that releases the buffer of stage k last (a shared-memory count,
// one acquire-release increment per warp once the warp has its data in
// registers) issues the copies of stage k+2 into it, so that no warp waits
// for the others to release.  Every thread takes 16
// elements (four units of 4) of one block: it steps the moments, the block's
// threads meet their maxima (integer max within a warp; across warps through
// shared memory and a named barrier whose id range belongs to one group size),
// and it updates the parameters and stores them and the codes to HBM.  A
// thread whose 16 |m| and v all lie in the exact forms' range (the common
// case) takes one branch for all of them, so that their update chains
// interleave, on packed fp32x2 instructions.  Per-tensor geometry sits in a
// shared-memory table; stage items are loaded two iterations ahead and old
// scales one.  A launch takes the tensors of at most kP8MaxTensors tensor-map
// slots.  Every wait is bounded: a block group decides a failed wait
// together before its next barrier, records DBUF_ETIMEOUT and stops (a stage
// that a stopped warp never releases is never refilled, so the others stop at
// their next wait); thread 0 waits (bounded) for copies still in flight
// before the CTA exits.
// ---------------------------------------------------------------------------
constexpr int kP8Warps = kP8ComputeWarps;
constexpr int kP8Threads = kP8Warps * 32;
constexpr int kP8U = kP8UnitsPerThread;
constexpr int kP8StageBytes = kP8StageElems * 10;    // p, g (fp32) + m, v codes
constexpr int kP8Stages = 2;

__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
                 : "=r"(old)
                 : "r"(smem_u32(p)), "r"(v)
                 : "memory");
    return old;
}

// The tensor maps of one launch: the plan's p8 tensors b * kP8MaxTensors ..
// b * kP8MaxTensors + nslots - 1 for launch b, whose items carry their slot
// within the launch.
struct P8Maps {
    CUtensorMap map[kP8MaxTensors][4];  // p, g, m codes, v codes
    int32_t tensor[kP8MaxTensors];      // slot -> tensor
    int32_t nslots;
};

// Geometry of one tensor's stages: blocks per stage nblk = Rb x K, box width bw.
struct P8Slot {
    int64_t buf_off, rows, cols, scale_off;
    int qrows, qcols, nbc, lanes, lg_lanes, K, lg_K, bw, ucols, lg_ucols, id_base, pad;
};

constexpr size_t kP8SmemBytes = size_t(kP8Stages) * kP8StageBytes + 1024 +
                                2 * kP8Stages * 8 + 16 * kP8Warps * 8 +
                                kP8MaxTensors * sizeof(P8Slot);

// The block of stage item `it` that thread `tid` works on, and its scale index.
struct P8Place {
    int bl, j, rb, kb, bi, bj;
    bool block;
    int64_t si;
};

__device__ __forceinline__ P8Place p8_place(const P8Slot &g, const P8Item &it, int tid) {
    P8Place q;
    q.bl = tid >> g.lg_lanes;
    q.j = tid & (g.lanes - 1);
    q.rb = q.bl >> g.lg_K;
    q.kb = q.bl & (g.K - 1);
    q.bi = it.bi0 + q.rb;
    q.bj = it.bj0 + q.kb;
    q.block = int64_t(q.bi) * g.qrows < g.rows && q.bj < g.nbc;
    q.si = g.scale_off + int64_t(q.bi) * g.nbc + q.bj;
    return q;
}

__device__ __forceinline__ void p8_issue(const P8Maps &maps, const P8Slot *slots, const P8Item &it,
                                         char *buf, uint64_t *full) {
    const P8Slot &g = slots[it.slot];
    const int x = it.bj0 * g.qcols, y = it.bi0 * g.qrows;
    mbar_arrive_expect_tx(full, uint32_t(kP8StageBytes));
    tma_load_2d(buf, &maps.map[it.slot][0], x, y, full);
    tma_load_2d(buf + kP8StageElems * 4, &maps.map[it.slot][1], x, y, full);
    tma_load_2d(buf + kP8StageElems * 8, &maps.map[it.slot][2], x, y, full);
    tma_load_2d(buf + kP8StageElems * 9, &maps.map[it.slot][3], x, y, full);
}

__global__ void __launch_bounds__(kP8Threads, 1)
    adamw8_pipe_kernel(const __grid_constant__ P8Maps maps, const P8Item *__restrict__ items,
                       int nitems, const TensorDesc *__restrict__ td, float *__restrict__ params,
                       uint8_t *__restrict__ mc, uint8_t *__restrict__ vc, float *__restrict__ ms,
                       float *__restrict__ vs, const AdamParams hp,
                       const AdamScalars hs, const float *__restrict__ total_norm,
                       const int32_t *__restrict__ nonfinite, int32_t *__restrict__ status) {
    extern __shared__ unsigned char smem_raw[];
    char *stages = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + size_t(kP8Stages) * kP8StageBytes);
    // per buffer: warps that have released it; then the number of stages issued
    uint32_t *rel = reinterpret_cast<uint32_t *>(full + kP8Stages);
    int *nissued = reinterpret_cast<int *>(rel + kP8Stages);
    // block maxima across warps: one row of slots per named barrier, so that a
    // slot is only ever shared by the warps of one group
    float2 *red = reinterpret_cast<float2 *>(full + 2 * kP8Stages);  // [16][kP8Warps]
    P8Slot *slots = reinterpret_cast<P8Slot *>(red + 16 * kP8Warps);
    const int tid = int(threadIdx.x), warp = tid >> 5, lane = tid & 31;
    const int G = int(gridDim.x);
    if (nonfinite && *nonfinite) return;  // skipped step: nothing is written
    if (tid < maps.nslots) {
        const TensorDesc &d = td[maps.tensor[tid]];
        P8Slot g;
        g.buf_off = d.buf_off;
        g.rows = d.rows;
        g.cols = d.cols;
        g.scale_off = d.scale_off;
        g.qrows = d.qrows;
        g.qcols = d.qcols;
        g.nbc = d.nbc;
        const int qe = d.qrows * d.qcols;
        g.lanes = qe / (4 * kP8U);
        g.lg_lanes = __ffs(g.lanes) - 1;
        const int nblk = kP8StageElems / qe;
        g.K = min(256 / d.qcols, nblk);
        g.lg_K = __ffs(g.K) - 1;
        g.bw = g.K * d.qcols;
        g.ucols = d.qcols >> 2;
        g.lg_ucols = __ffs(g.ucols) - 1;
        g.id_base = g.lanes == 64 ? 1 : g.lanes == 128 ? 9 : g.lanes == 256 ? 13 : 15;
        g.pad = 0;
        slots[tid] = g;
    }
    if (tid == 0) {
        for (int st = 0; st < kP8Stages; ++st) {
            mbar_init(&full[st], 1);
            rel[st] = 0;
        }
        mbar_fence_init();
    }
    __syncthreads();
    AdamScalars s = hs;
    s.coef = clip_coef(hp, total_norm);
    const int mine = int(blockIdx.x) < nitems ? (nitems - 1 - int(blockIdx.x)) / G + 1 : 0;
    if (mine == 0) return;
    if (tid == 0) {
        int issued = 0;
        for (; issued < kP8Stages && issued < mine; ++issued)
            p8_issue(maps, slots, items[int(blockIdx.x) + issued * G],
                     stages + size_t(issued) * kP8StageBytes, &full[issued]);
        *nissued = issued;
    }

    P8Item cur = items[blockIdx.x];
    P8Item nxt = mine > 1 ? items[int(blockIdx.x) + G] : cur;  // loaded a stage ahead
    float ms_cur = 0.0f, vs_cur = 0.0f;
    {
        const P8Place q = p8_place(slots[cur.slot], cur, tid);
        if (q.block) {
            ms_cur = ms[q.si];
            vs_cur = vs[q.si];
        }
    }
    for (int k = 0; k < mine; ++k) {
        const int st = k % kP8Stages;
        // the item after next (its load has a stage to land), and the next
        // item's old scales, one iteration ahead
        P8Item nxt2 = nxt;
        if (k + 2 < mine) nxt2 = items[int(blockIdx.x) + (k + 2) * G];
        float ms_nxt = 0.0f, vs_nxt = 0.0f;
        if (k + 1 < mine) {
            const P8Place qn = p8_place(slots[nxt.slot], nxt, tid);
            if (qn.block) {
                ms_nxt = ms[qn.si];
                vs_nxt = vs[qn.si];
            }
        }

        const P8Slot &g = slots[cur.slot];
        const P8Place q = p8_place(g, cur, tid);
        const bool got = mbar_wait_bounded(&full[st], uint32_t(k / kP8Stages) & 1u);

        const char *buf = stages + size_t(st) * kP8StageBytes;
        float p[kP8U][4], m[kP8U][4], v[kP8U][4];
        int64_t e[kP8U];
        bool valid[kP8U];
        float mamax = 0.0f, vamax = 0.0f;
        float mmin = __int_as_float(0x7F800000), vmin = __int_as_float(0x7F800000);
        uint32_t cmw[kP8U], cvw[kP8U];
        float gw[kP8U][4];
#pragma unroll
        for (int u2 = 0; u2 < kP8U; ++u2) {
            const int u = q.j + u2 * g.lanes;
            const int row = u >> g.lg_ucols, cq = u & (g.ucols - 1);
            const int so = (q.rb * g.qrows + row) * g.bw + q.kb * g.qcols + 4 * cq;
            const int64_t r = int64_t(q.bi) * g.qrows + row;
            const int c = q.bj * g.qcols + 4 * cq;
            valid[u2] = q.block && r < g.rows && c < g.cols;
            e[u2] = g.buf_off + r * g.cols + c;
            const float4 pp = *reinterpret_cast<const float4 *>(buf + size_t(so) * 4);
            const float4 gg =
                *reinterpret_cast<const float4 *>(buf + kP8StageElems * 4 + size_t(so) * 4);
            p[u2][0] = pp.x; p[u2][1] = pp.y; p[u2][2] = pp.z; p[u2][3] = pp.w;
            gw[u2][0] = gg.x; gw[u2][1] = gg.y; gw[u2][2] = gg.z; gw[u2][3] = gg.w;
            cmw[u2] = *reinterpret_cast<const uint32_t *>(buf + kP8StageElems * 8 + so);
            cvw[u2] = *reinterpret_cast<const uint32_t *>(buf + kP8StageElems * 9 + so);
        }
        // the buffer may be refilled once every warp has its data in registers:
        // the last warp to release it issues stage k + kP8Stages into it (the
        // count is next used with that stage, whose copies follow the reset)
        __syncwarp();
        if (lane == 0 && atom_add_acq_rel(&rel[st], 1u) == kP8Warps - 1) {
            rel[st] = 0;
            const int j = k + kP8Stages;
            if (j < mine) {
                p8_issue(maps, slots, items[int(blockIdx.x) + j * G],
                         stages + size_t(st) * kP8StageBytes, &full[st]);
                *nissued = j + 1;
            }
        }

#pragma unroll
        for (int u2 = 0; u2 < kP8U; ++u2) {
            const uint32_t xm = cmw[u2] ^ 0x80808080u;
            const float2 om = splat(-8388736.0f), ov = splat(-8388607.0f);
            const float2 sm = splat(ms_cur), sv = splat(vs_cur);
            const float2 m01 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(xm, 0), byte_float(xm, 1)), om), sm);
            const float2 m23 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(xm, 2), byte_float(xm, 3)), om), sm);
            const float2 v01 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(cvw[u2], 0), byte_float(cvw[u2], 1)), ov), sv);
            const float2 v23 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(cvw[u2], 2), byte_float(cvw[u2], 3)), ov), sv);
            m[u2][0] = m01.x; m[u2][1] = m01.y; m[u2][2] = m23.x; m[u2][3] = m23.y;
            v[u2][0] = v01.x; v[u2][1] = v01.y; v[u2][2] = v23.x; v[u2][3] = v23.y;
#pragma unroll
            for (int w = 0; w < 4; w += 2)
                adam_moments2(s, gw[u2][w], gw[u2][w + 1], m[u2][w], m[u2][w + 1], v[u2][w],
                              v[u2][w + 1]);
            if (valid[u2]) {
                const float a0 = fabsf(m[u2][0]), a1 = fabsf(m[u2][1]);
                const float a2 = fabsf(m[u2][2]), a3 = fabsf(m[u2][3]);
                mamax = fmax3(fmax3(mamax, a0, a1), a2, a3);
                vamax = fmax3(fmax3(vamax, v[u2][0], v[u2][1]), v[u2][2], v[u2][3]);
                mmin = fmin3_nan(fmin3_nan(mmin, a0, a1), a2, a3);
                vmin = fmin3_nan(fmin3_nan(vmin, v[u2][0], v[u2][1]), v[u2][2], v[u2][3]);
            }
        }
        // every |m| and v of the thread's units inside the range of the exact forms
        // (false for a NaN)
        const bool inrange = mmin >= 0x1p-60f && vmin >= 0x1p-60f;

        // block maxima and the group's verdict on the wait
        bool failed;
        if (g.lanes <= 32) {
            const unsigned gmask = g.lanes == 32
                                       ? 0xFFFFFFFFu
                                       : ((1u << g.lanes) - 1u) << (lane & ~(g.lanes - 1));
            failed = __any_sync(gmask, !got);
            mamax = __uint_as_float(__reduce_max_sync(gmask, __float_as_uint(mamax)));
            vamax = __uint_as_float(__reduce_max_sync(gmask, __float_as_uint(vamax)));
        } else {
            const int gid = g.id_base + q.bl;
            failed = group_any(!got, gid, g.lanes);
            mamax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mamax)));
            vamax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(vamax)));
            const int w0 = (q.bl << g.lg_lanes) >> 5;
            if (lane == 0) red[gid * kP8Warps + (warp - w0)] = make_float2(mamax, vamax);
            group_sync(gid, g.lanes);
            for (int w = 0; w < (g.lanes >> 5); ++w) {
                const float2 r = red[gid * kP8Warps + w];
                mamax = fmaxf(mamax, r.x);
                vamax = fmaxf(vamax, r.y);
            }
        }
        if (failed) {
            if (q.j == 0) atomicExch(status, DBUF_ETIMEOUT);
            break;
        }
        if (q.block) {
            const float ms_new = block_scale_cr(mamax, 127.0f, s.i127);
            const float vs_new = __fmul_rn(vamax, 0x1p-8f);
            const Divisor dm = make_divisor(ms_new), dv = make_divisor(vs_new);
            const bool vzero = !(vs_new > 0.0f);
            const bool fast = s.fast && mamax <= 0x1p60f && vamax <= 0x1p60f;
            const bool exact = dm.exact || dv.exact;
            // the common case decided once for the thread's 16 elements, so that
            // their update chains share one basic block and interleave
            if (fast && !exact && inrange) {
#pragma unroll
                for (int u2 = 0; u2 < kP8U; ++u2)
#pragma unroll
                    for (int w = 0; w < 4; w += 2)
                        adam_param_cr2(s, p[u2][w], p[u2][w + 1], m[u2][w], m[u2][w + 1],
                                       v[u2][w], v[u2][w + 1]);
                uint32_t cm[kP8U], cv[kP8U];
#pragma unroll
                for (int u2 = 0; u2 < kP8U; ++u2)
                    unit_codes_fast(m[u2], v[u2], dm, dv, cm[u2], cv[u2]);
#pragma unroll
                for (int u2 = 0; u2 < kP8U; ++u2) {
                    if (!valid[u2]) continue;
                    store_f<4>(params, e[u2], p[u2]);
                    store_c<4>(mc, e[u2], cm[u2]);
                    store_c<4>(vc, e[u2], cv[u2]);
                }
            } else {
                // per unit: IEEE forms where a value leaves the range, exact quotients
                // for scales outside [2^-80, 2^100]
#pragma unroll
                for (int u2 = 0; u2 < kP8U; ++u2) {
                    if (!valid[u2]) continue;
                    if (exact)
                        unit_update<4, true>(s, params, mc, vc, e[u2], p[u2], m[u2], v[u2], dm,
                                             dv, vzero, fast);
                    else
                        unit_update<4, false>(s, params, mc, vc, e[u2], p[u2], m[u2], v[u2], dm,
                                              dv, vzero, fast);
                }
            }
            if (q.j == 0) {
                ms[q.si] = ms_new;
                vs[q.si] = vs_new;
            }
        }
        cur = nxt;
        nxt = nxt2;
        ms_cur = ms_nxt;
        vs_cur = vs_nxt;
    }
    __syncthreads();  // every warp has left the loop: the count of stages issued is final
    if (tid == 0) {
        // copies of the last stages issued may still be in flight: wait for them
        // (bounded) before the CTA exits (stages are issued in order)
        const int issued = *nissued;
        for (int j = (issued > kP8Stages ? issued - kP8Stages : 0); j < issued; ++j)
            (void)mbar_wait_bounded(&full[j % kP8Stages], uint32_t(j / kP8Stages) & 1u);
    }
}

// ---------------------------------------------------------------------------
// Pipelined 8-bit AdamW for blocks of kBigBlockElems (16384) elements, twice a
// stage of the kernel above (128 x 128, 64 x 256 or 256 x 64 blocks).  One CTA
// of 16 warps per SM takes one block at a time.  The block's gradients and both
// code arrays (6 bytes per element, 96 KB) come in by three 2-D tensor-map
// copies into one of two shared-memory buffers; the parameters are read
// straight into registers, issued before the wait on the buffer, from L2, where
// a tensor-map prefetch issued with the block's copies has brought them.  The
// boxes of the block after are prefetched into L2 at the same time, so that its
// copies, issued one block later, land from L2.
// Pass 1: every thread (8 units of 4 consecutive elements of one block row; a
// warp covers 128 consecutive columns) dequantises, steps the moments, keeps
// them in registers, updates its parameters and stores them (the correctly
// rounded forms when every |m| and v of the thread lies in [2^-60, 2^60] and
// the step's scalars allow; IEEE forms otherwise: equal results).  The block
// maxima meet across the CTA (integer max within a warp, shared memory across
// warps, one barrier, which also settles the CTA's verdict on the wait and
// frees the buffer: thread 0 then issues the block after next into it).  Pass
// 2 encodes the codes from the moments in registers and stores them.  Sixteen
// bytes per element move, as in the kernel above; the register kernel reads
// the gradients and codes of these blocks twice.
// ---------------------------------------------------------------------------
constexpr int kBigThreads = 512;
constexpr int kBigWarps = kBigThreads / 32;
constexpr int kBigU = int(kBigBlockElems) / 4 / kBigThreads;  // units of 4 per thread
constexpr int kBigStageBytes = int(kBigBlockElems) * 6;       // g (fp32) + m, v codes
constexpr int kBigStages = 2;

struct BigMaps {
    CUtensorMap map[kP8MaxTensors][4];  // g, m codes, v codes; p (prefetched into L2)
    int32_t tensor[kP8MaxTensors];      // slot -> tensor
    int32_t nslots;
};

struct BigSlot {
    int64_t buf_off, rows, cols, scale_off;
    int qrows, qcols, nbc, lg_upr;
};

constexpr size_t kBigSmemBytes = size_t(kBigStages) * kBigStageBytes + 1024 + kBigStages * 8 +
                                 2 * kBigWarps * 8 + kP8MaxTensors * sizeof(BigSlot);

__device__ __forceinline__ void big_issue(const BigMaps &maps, const BigSlot *slots,
                                          const P8Item &it, char *buf, uint64_t *full) {
    const BigSlot &g = slots[it.slot];
    const int x = it.bj0 * g.qcols, y = it.bi0 * g.qrows;
    mbar_arrive_expect_tx(full, uint32_t(kBigStageBytes));
    tma_load_2d(buf, &maps.map[it.slot][0], x, y, full);
    tma_load_2d(buf + kBigBlockElems * 4, &maps.map[it.slot][1], x, y, full);
    tma_load_2d(buf + kBigBlockElems * 5, &maps.map[it.slot][2], x, y, full);
    // the block's parameters are read directly from global memory when its turn
    // comes; bringing them into L2 now takes DRAM latency off that first read
    tma_prefetch_l2_2d(&maps.map[it.slot][3], x, y);
}

// The boxes of the block issued after `it` into L2 (its copies come one block
// later and find them there).
__device__ __forceinline__ void big_prefetch(const BigMaps &maps, const BigSlot *slots,
                                             const P8Item &it) {
    const BigSlot &g = slots[it.slot];
    const int x = it.bj0 * g.qcols, y = it.bi0 * g.qrows;
#pragma unroll
    for (int a = 0; a < 3; ++a) tma_prefetch_l2_2d(&maps.map[it.slot][a], x, y);
}

__global__ void __launch_bounds__(kBigThreads, 1)
    adamw8_big_kernel(const __grid_constant__ BigMaps maps, const P8Item *__restrict__ items,
                      int nitems, const TensorDesc *__restrict__ td, float *__restrict__ params,
                      uint8_t *__restrict__ mc, uint8_t *__restrict__ vc, float *__restrict__ ms,
                      float *__restrict__ vs, const AdamParams hp, const AdamScalars hs,
                      const float *__restrict__ total_norm, const int32_t *__restrict__ nonfinite,
                      int32_t *__restrict__ status) {
    extern __shared__ unsigned char smem_raw[];
    char *stages = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + size_t(kBigStages) * kBigStageBytes);
    float2 *red = reinterpret_cast<float2 *>(full + kBigStages);  // [2][kBigWarps]
    BigSlot *slots = reinterpret_cast<BigSlot *>(red + 2 * kBigWarps);
    const int tid = int(threadIdx.x), warp = tid >> 5, lane = tid & 31;
    const int G = int(gridDim.x);
    if (nonfinite && *nonfinite) return;  // skipped step: nothing is written
    if (tid < maps.nslots) {
        const TensorDesc &d = td[maps.tensor[tid]];
        BigSlot g;
        g.buf_off = d.buf_off;
        g.rows = d.rows;
        g.cols = d.cols;
        g.scale_off = d.scale_off;
        g.qrows = d.qrows;
        g.qcols = d.qcols;
        g.nbc = d.nbc;
        g.lg_upr = __ffs(d.qcols >> 2) - 1;
        slots[tid] = g;
    }
    if (tid == 0) {
        for (int st = 0; st < kBigStages; ++st) mbar_init(&full[st], 1);
        mbar_fence_init();
    }
    __syncthreads();
    AdamScalars s = hs;
    s.coef = clip_coef(hp, total_norm);
    const int mine = int(blockIdx.x) < nitems ? (nitems - 1 - int(blockIdx.x)) / G + 1 : 0;
    if (mine == 0) return;
    int issued = 0;
    if (tid == 0)
        for (; issued < kBigStages && issued < mine; ++issued)
            big_issue(maps, slots, items[int(blockIdx.x) + issued * G],
                      stages + size_t(issued) * kBigStageBytes, &full[issued]);
    if (tid == 0 && issued < mine) big_prefetch(maps, slots, items[int(blockIdx.x) + issued * G]);

    for (int k = 0; k < mine; ++k) {
        const int st = k % kBigStages;
        const P8Item it = items[int(blockIdx.x) + k * G];
        const BigSlot &g = slots[it.slot];
        const int64_t si = g.scale_off + int64_t(it.bi0) * g.nbc + it.bj0;
        const float ms_old = ms[si], vs_old = vs[si];
        const int upr = g.qcols >> 2;
        const int64_t r0 = int64_t(it.bi0) * g.qrows;
        const int c0 = it.bj0 * g.qcols;
        // the thread's units u = tid + kBigThreads * i share one column and lie dr
        // rows apart: unit i is row row0 + i * dr of the block
        const int row0 = tid >> g.lg_upr, cu = tid & (upr - 1);
        const int dr = kBigThreads >> g.lg_upr;
        const int c = c0 + 4 * cu;
        const int so0 = row0 * g.qcols + 4 * cu, dso = dr * g.qcols;
        const int64_t e0 = g.buf_off + (r0 + row0) * g.cols + c, de = int64_t(dr) * g.cols;
        const int64_t rleft = g.rows - (r0 + row0);  // unit i is inside the tensor if i * dr < rleft
        const bool col_ok = c < g.cols;
        float p[kBigU][4], m[kBigU][4], v[kBigU][4];
        uint32_t valid = 0;  // bit i: unit i lies inside the tensor
#pragma unroll
        for (int i = 0; i < kBigU; ++i) {
            if (col_ok && int64_t(i) * dr < rleft) {
                valid |= 1u << i;
                load_f<4, true>(params, e0 + i * de, p[i]);
            } else {
                p[i][0] = p[i][1] = p[i][2] = p[i][3] = 0.0f;
            }
        }
        const bool got = mbar_wait_bounded(&full[st], uint32_t(k / kBigStages) & 1u);

        // pass 1: the new moments (kept), the block maxima, the parameters (updated
        // and stored unit by unit, so that a unit's parameters die as its moments
        // are born)
        const char *buf = stages + size_t(st) * kBigStageBytes;
        float mamax = 0.0f, vamax = 0.0f;
#pragma unroll
        for (int i = 0; i < kBigU; ++i) {
            const int so = so0 + i * dso;
            const float4 gg = *reinterpret_cast<const float4 *>(buf + size_t(so) * 4);
            const uint32_t cmw = *reinterpret_cast<const uint32_t *>(buf + kBigBlockElems * 4 + so);
            const uint32_t cvw = *reinterpret_cast<const uint32_t *>(buf + kBigBlockElems * 5 + so);
            const uint32_t xm = cmw ^ 0x80808080u;
            const float2 om = splat(-8388736.0f), ov = splat(-8388607.0f);
            const float2 sm = splat(ms_old), sv = splat(vs_old);
            const float2 m01 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(xm, 0), byte_float(xm, 1)), om), sm);
            const float2 m23 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(xm, 2), byte_float(xm, 3)), om), sm);
            const float2 v01 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(cvw, 0), byte_float(cvw, 1)), ov), sv);
            const float2 v23 = __fmul2_rn(__fadd2_rn(make_float2(byte_float(cvw, 2), byte_float(cvw, 3)), ov), sv);
            m[i][0] = m01.x; m[i][1] = m01.y; m[i][2] = m23.x; m[i][3] = m23.y;
            v[i][0] = v01.x; v[i][1] = v01.y; v[i][2] = v23.x; v[i][3] = v23.y;
            adam_moments2(s, gg.x, gg.y, m[i][0], m[i][1], v[i][0], v[i][1]);
            adam_moments2(s, gg.z, gg.w, m[i][2], m[i][3], v[i][2], v[i][3]);
            if ((valid >> i) & 1u) {
                const float a0 = fabsf(m[i][0]), a1 = fabsf(m[i][1]);
                const float a2 = fabsf(m[i][2]), a3 = fabsf(m[i][3]);
                const float ma = fmax3(fmax3(0.0f, a0, a1), a2, a3);
                const float va = fmax3(fmax3(0.0f, v[i][0], v[i][1]), v[i][2], v[i][3]);
                mamax = fmaxf(mamax, ma);
                vamax = fmaxf(vamax, va);
                float lo = fmin3_nan(fmin3_nan(a0, a1, a2), a3, v[i][0]);
                lo = fmin3_nan(fmin3_nan(lo, v[i][1], v[i][2]), v[i][3], lo);
                // every |m| and v of the unit inside the correctly rounded forms'
                // range (false for a NaN)
                if (s.fast && lo >= 0x1p-60f && fmaxf(ma, va) <= 0x1p60f) {
                    adam_param_cr2(s, p[i][0], p[i][1], m[i][0], m[i][1], v[i][0], v[i][1]);
                    adam_param_cr2(s, p[i][2], p[i][3], m[i][2], m[i][3], v[i][2], v[i][3]);
                } else {
#pragma unroll
                    for (int w = 0; w < 4; ++w) p[i][w] = adam_param(s, p[i][w], m[i][w], v[i][w]);
                }
                store_f<4>(params, e0 + i * de, p[i]);
            }
        }

        // the block maxima (non-negative, NaN-free: their bits order like their
        // values) across the CTA; the barrier also frees the buffer
        mamax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mamax)));
        vamax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(vamax)));
        float2 *rk = red + (k & 1) * kBigWarps;
        if (lane == 0) rk[warp] = make_float2(mamax, vamax);
        if (__syncthreads_or(!got)) {
            if (tid == 0) atomicExch(status, DBUF_ETIMEOUT);
            break;
        }
        if (tid == 0 && k + kBigStages < mine) {
            big_issue(maps, slots, items[int(blockIdx.x) + (k + kBigStages) * G],
                      stages + size_t(st) * kBigStageBytes, &full[st]);
            if (k + kBigStages + 1 < mine)
                big_prefetch(maps, slots, items[int(blockIdx.x) + (k + kBigStages + 1) * G]);
            issued = k + kBigStages + 1;
        }
#pragma unroll
        for (int w = 0; w < kBigWarps; ++w) {
            const float2 r = rk[w];
            mamax = fmaxf(mamax, r.x);
            vamax = fmaxf(vamax, r.y);
        }

        // pass 2: new scales and the codes
        const float ms_new = block_scale_cr(mamax, 127.0f, s.i127);
        const float vs_new = __fmul_rn(vamax, 0x1p-8f);
        const Divisor dm = make_divisor(ms_new), dv = make_divisor(vs_new);
        const bool vzero = !(vs_new > 0.0f);
        if (!(dm.exact || dv.exact)) {
#pragma unroll
            for (int i = 0; i < kBigU; ++i) {
                uint32_t cm, cv;
                unit_codes_fast(m[i], v[i], dm, dv, cm, cv);
                if ((valid >> i) & 1u) {
                    store_c<4>(mc, e0 + i * de, cm);
                    store_c<4>(vc, e0 + i * de, cv);
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < kBigU; ++i) {
                if (!((valid >> i) & 1u)) continue;
                uint32_t cm = 0, cv = 0;
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    cm |= encode1<DBUF_QUANT_INT8>(quot<true>(m[i][w], dm)) << (8 * w);
                    cv |= (vzero ? 0u : v_code<true>(v[i][w], dv)) << (8 * w);
                }
                store_c<4>(mc, e0 + i * de, cm);
                store_c<4>(vc, e0 + i * de, cv);
            }
        }
        if (tid == 0) {
            ms[si] = ms_new;
            vs[si] = vs_new;
        }
    }
    __syncthreads();
    if (tid == 0) {
        // copies of the last blocks issued may still be in flight: wait for them
        // (bounded) before the CTA exits (blocks are issued in order)
        for (int j = (issued > kBigStages ? issued - kBigStages : 0); j < issued; ++j)
            (void)mbar_wait_bounded(&full[j % kBigStages], uint32_t(j / kBigStages) & 1u);
    }
}

}  // namespace

int launch_adamw(const dbuf_plan_t *p, float *params, const float *grads, float *exp_avg,
                 float *exp_avg_sq, const AdamParams &hp, const float *total_norm,
                 const int32_t *nonfinite, void *stream) {
    if (p->chunks.empty()) return cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    adamw_kernel<<<unsigned(p->chunks.size()) * kChunkSplit, kThreads, 0, st>>>(
        p->dev.chunks, p->dev.tensors, params, grads, exp_avg, exp_avg_sq, hp, total_norm,
        nonfinite);
    return cudaGetLastError();
}

int prepare_optim_kernels() {
    cudaError_t e = cudaFuncSetAttribute(adamw8_pipe_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(kP8SmemBytes));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(adamw8_big_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kBigSmemBytes));
    return int(e);
}

int launch_adamw8(const dbuf_plan_t *p, float *params, const float *grads, uint8_t *m_codes,
                  uint8_t *v_codes, float *m_scales, float *v_scales, float *m32, float *v32,
                  const AdamParams &hp, const float *total_norm, const int32_t *nonfinite,
                  void *stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The pipelined kernel takes the tensors with tensor maps when every buffer
    // is 16-byte aligned and the maps encode; the register kernel takes the rest
    // (all quantised tensors otherwise).
    const uintptr_t bits = reinterpret_cast<uintptr_t>(params) | reinterpret_cast<uintptr_t>(grads) |
                           reinterpret_cast<uintptr_t>(m_codes) | reinterpret_cast<uintptr_t>(v_codes);
    bool pipe = (!p->p8_items.empty() || !p->big_items.empty()) && (bits & 15) == 0;
    // one launch per kP8MaxTensors tensors; every map is encoded before the first
    // launch, so that a tensor the encoder rejects sends all of them to the
    // register kernel
    const size_t nslot = p->p8_tensors.size();
    std::vector<P8Maps> batches;
    for (size_t b0 = 0; pipe && b0 < nslot; b0 += kP8MaxTensors) {
        P8Maps maps;
        maps.nslots = int32_t(std::min<size_t>(kP8MaxTensors, nslot - b0));
        for (int slot = 0; pipe && slot < maps.nslots; ++slot) {
            const int32_t t = p->p8_tensors[b0 + slot];
            maps.tensor[slot] = t;
            const TensorDesc &d = p->tdesc[t];
            const int qe = d.qrows * d.qcols, nblk = kP8StageElems / qe;
            const int K = std::min(256 / d.qcols, nblk), bw = K * d.qcols, bh = (nblk / K) * d.qrows;
            pipe = encode_map_2d(&maps.map[slot][0], true, params + d.buf_off, d.cols, d.rows, bw,
                                 bh) &&
                   encode_map_2d(&maps.map[slot][1], true, const_cast<float *>(grads) + d.buf_off,
                                 d.cols, d.rows, bw, bh) &&
                   encode_map_2d(&maps.map[slot][2], false, m_codes + d.buf_off, d.cols, d.rows,
                                 bw, bh) &&
                   encode_map_2d(&maps.map[slot][3], false, v_codes + d.buf_off, d.cols, d.rows,
                                 bw, bh);
        }
        batches.push_back(maps);
    }
    // the big-block tensors: gradients and both codes by tensor maps, one block a
    // box, and the parameters' map for the L2 prefetch
    const size_t nbig = p->big_tensors.size();
    std::vector<BigMaps> big_batches;
    for (size_t b0 = 0; pipe && b0 < nbig; b0 += kP8MaxTensors) {
        BigMaps maps;
        maps.nslots = int32_t(std::min<size_t>(kP8MaxTensors, nbig - b0));
        for (int slot = 0; pipe && slot < maps.nslots; ++slot) {
            const int32_t t = p->big_tensors[b0 + slot];
            maps.tensor[slot] = t;
            const TensorDesc &d = p->tdesc[t];
            pipe = encode_map_2d(&maps.map[slot][0], true, const_cast<float *>(grads) + d.buf_off,
                                 d.cols, d.rows, d.qcols, d.qrows) &&
                   encode_map_2d(&maps.map[slot][1], false, m_codes + d.buf_off, d.cols, d.rows,
                                 d.qcols, d.qrows) &&
                   encode_map_2d(&maps.map[slot][2], false, v_codes + d.buf_off, d.cols, d.rows,
                                 d.qcols, d.qrows) &&
                   encode_map_2d(&maps.map[slot][3], true, params + d.buf_off, d.cols, d.rows,
                                 d.qcols, d.qrows);
        }
        big_batches.push_back(maps);
    }
    const size_t n_items = pipe ? p->n_opt_rest : p->opt_items.size();
    const size_t grid = p->opt_plain.size() + n_items;
    for (size_t b = 0; pipe && b < batches.size(); ++b) {
        const size_t b0 = b * kP8MaxTensors;
        const size_t i0 = p->p8_item_start[b0], i1 = p->p8_item_start[b0 + batches[b].nslots];
        const int n = int(i1 - i0);
        if (n == 0) continue;
        const int g = n < p->dev.num_sms ? n : p->dev.num_sms;
        adamw8_pipe_kernel<<<g, kP8Threads, kP8SmemBytes, st>>>(
            batches[b], p->dev.p8_items + i0, n, p->dev.tensors, params, m_codes, v_codes,
            m_scales, v_scales, hp, host_scalars(hp), total_norm, nonfinite, p->dev.status);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    for (size_t b = 0; pipe && b < big_batches.size(); ++b) {
        const size_t b0 = b * kP8MaxTensors;
        const size_t i0 = p->big_item_start[b0], i1 = p->big_item_start[b0 + big_batches[b].nslots];
        const int n = int(i1 - i0);
        if (n == 0) continue;
        const int g = n < p->dev.num_sms ? n : p->dev.num_sms;
        adamw8_big_kernel<<<g, kBigThreads, kBigSmemBytes, st>>>(
            big_batches[b], p->dev.big_items + i0, n, p->dev.tensors, params, m_codes, v_codes,
            m_scales, v_scales, hp, host_scalars(hp), total_norm, nonfinite, p->dev.status);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (grid == 0) return cudaSuccess;
    adamw8_kernel<<<unsigned(grid), kThreads, 0, st>>>(
        p->dev.chunks, p->dev.opt_plain, int32_t(p->opt_plain.size()), p->dev.opt_items,
        p->dev.tensors, params, grads, m_codes, v_codes, m_scales, v_scales, m32, v32, hp,
        total_norm, nonfinite);
    return cudaGetLastError();
}

}  // namespace dbuf
