/*
 * dbuf_oracle.c -- plain, slow, single-threaded CPU oracle for the DBuffer
 * group-operator path.  TEST INFRASTRUCTURE ONLY: it is called by the tests, by
 * the smoke check and by the benchmark's CPU-baseline leg, never by the product
 * path.  It shares no source with the CUDA library.
 *
 * Build: gcc -std=c11 -O2 -fno-fast-math -ffp-contract=off -shared -fPIC
 * (no FMA contraction, no fast-math, IEEE fp32 arithmetic, default rounding).
 *
 * Sources (page title, section):
 *  [FSDP-1] "veScale-FSDP: Flexible and High-Performance FSDP at Scale",
 *           §4 RaggedShard format; §5 Planning algorithm (problem formulation,
 *           default tensor order, 3-case analysis); §5 DBuffer (group-level
 *           operators, zero-copy access); §6.3 8-bit Adam (block-wise quantisation
 *           of the local shard without communication); §6.3 Distributed Muon
 *           (whole-matrix redistribution to a root and back, Algorithm 2).
 *  [FSDP-2] "PyTorch FSDP: Experiences on Scaling Fully Sharded Data Parallel",
 *           FlatParameter; native mixed precision; gradient accumulation;
 *           sharded gradient scaler; known limitations.
 *  [veScale-3] "veScale 深度技术分析", RaggedShard Placement (placement_types.py:
 *           flattened storage, local_units); OpDispatcher (ragged norm handler,
 *           found_inf handler, fused AdamW/SGD handler).
 *
 * Readings where the pages leave a step open are stated at each function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

#define ORC_QNONE 0
#define ORC_QE4M3 1
#define ORC_QINT8 2

/* ------------------------------------------------------------------------ */
/* Layout                                                                    */
/* ------------------------------------------------------------------------ */

/* Sharding granularity g_t in elements.  RaggedShard works on flattened
 * storage: the sharded prefix dimension is the row, the rest is the tail
 * [veScale-3, RaggedShard Placement].  A unit of gran_rows rows of a row-major
 * [rows, cols] tensor therefore covers gran_rows*cols consecutive elements.
 * gran_rows <= 0, or a unit at least as tall as the tensor, makes the whole
 * tensor one unit (it may never be cut). */
static int64_t unit_elems(int64_t rows, int64_t cols, int64_t gran_rows)
{
    int64_t n = rows * cols;
    if (gran_rows <= 0 || gran_rows >= rows) return n;
    return gran_rows * cols;
}

static int64_t round_up(int64_t x, int64_t a) { return ((x + a - 1) / a) * a; }

static int64_t gcd64(int64_t a, int64_t b)
{
    while (b) { int64_t t = a % b; a = b; b = t; }
    return a;
}

/* Constraint (iii) of [FSDP-1, §5 formulation], checked literally: every shard
 * boundary B_k that falls strictly inside [p, p+n) must be a whole number of
 * units g from the tensor's start, so no block is split between two shards. */
static int cuts_ok(int64_t p, int64_t n, int64_t g, const int64_t *B, int m)
{
    for (int k = 1; k < m; ++k) {
        if (B[k] <= p) continue;
        if (B[k] >= p + n) break;
        if ((B[k] - p) % g != 0) return 0;
    }
    return 1;
}

/* Smallest aligned start >= p that satisfies (iii) for a tensor of n elements
 * and unit g, given shard boundaries B[0..m].  Returns a start with
 * start + n > B[m] when the tensor no longer fits (constraint (iv) fails).
 *
 * Shard by shard: a start p in shard j = [B_j, B_{j+1}) either keeps the tensor
 * inside the shard (the first case of the pages' 3-case analysis), or the
 * tensor runs past B_{j+1}; then B_{j+1} is inside it, so B_{j+1} - p must be a
 * multiple of g (and p a multiple of the alignment a): p = B_{j+1} - q*lcm(a,g).
 * The smallest such p >= the current candidate is tried; if a later boundary is
 * still violated (the tensor contains a whole shard whose size is not a multiple
 * of g), every larger start in this shard contains that boundary too at the same
 * residue, so the search moves to the next shard's start. */
static int64_t first_start(int64_t p, int64_t n, int64_t g, int64_t a,
                           const int64_t *B, int m)
{
    if (n == 0) return p;
    for (;;) {
        if (p + n > B[m]) return p;
        if (cuts_ok(p, n, g, B, m)) return p;
        int j = 0;
        while (j + 1 < m && B[j + 1] <= p) ++j;
        int64_t end = B[j + 1];
        if (g < n) {
            int64_t L = a / gcd64(a, g) * g;
            int64_t q = end - ((end - p) / L) * L;
            if (q > p && q < end && cuts_ok(q, n, g, B, m)) return q;
        }
        p = end;
    }
}

/* Greedy-leftmost placement of the tensors, in the given (default) order, at a
 * fixed shard unit size U.  Shard k spans [U*c_k, U*c_{k+1}) with c_k the prefix
 * sums of the per-shard units (all 1 for even shards).  Constraints of
 * [FSDP-1, §5 formulation]: (i) order kept, tensors do not overlap, padding only
 * between tensors; (ii) every start a multiple of a; (iii) as cuts_ok; (iv) the
 * last tensor ends within the buffer.  Returns 1 if all tensors fit. */
static int place_all(int32_t n, const int64_t *numel, const int64_t *unit,
                     int64_t a, const int64_t *B, int m, int64_t *offsets)
{
    int64_t pos = 0;
    for (int32_t t = 0; t < n; ++t) {
        int64_t p = first_start(round_up(pos, a), numel[t], unit[t], a, B, m);
        if (p + numel[t] > B[m]) return 0;
        offsets[t] = p;
        pos = p + numel[t];
    }
    return 1;
}

/* The minimum per-shard size S* of [FSDP-1, §5 formulation] for the default
 * tensor order (the order the pages adopt), found by scanning every multiple
 * of a upward from a lower bound; the canonical layout is the greedy-leftmost
 * one at S*.  With local_units u_k (RaggedShard's per-device shares,
 * [veScale-3, RaggedShard Placement]) shard k holds u_k*U elements and U is
 * minimised instead; even shards are u_k = 1.
 *
 * Lower bound: the buffer must hold all E elements, and some shard must hold
 * the largest unit whole: U >= max(ceil(E / sum u), ceil(max unit / max u)).
 *
 * Outputs S (= U), offsets[n], bounds[m+1].  Returns 0, or -1 on bad input. */
int orc_plan(int32_t n, const int64_t *rows, const int64_t *cols,
             const int64_t *gran_rows, int32_t m, const int32_t *units,
             int64_t align, int64_t *S_out, int64_t *offsets, int64_t *bounds)
{
    if (n < 0 || m < 1 || align < 1) return -1;
    int64_t *numel = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    int64_t *unit = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    int64_t *c = (int64_t *)malloc(sizeof(int64_t) * (size_t)(m + 1));
    if (!numel || !unit || !c) { free(numel); free(unit); free(c); return -1; }

    int64_t E = 0, big = 0;
    for (int32_t t = 0; t < n; ++t) {
        if (rows[t] < 0 || cols[t] < 0) { free(numel); free(unit); free(c); return -1; }
        numel[t] = rows[t] * cols[t];
        unit[t] = unit_elems(rows[t], cols[t], gran_rows[t]);
        if (unit[t] < 1) unit[t] = 1;
        E += numel[t];
        int64_t need = unit[t] < numel[t] ? unit[t] : numel[t];
        if (need > big) big = need;
    }
    int64_t umax = 0;
    c[0] = 0;
    for (int32_t k = 0; k < m; ++k) {
        int64_t u = units ? units[k] : 1;
        if (u < 1) { free(numel); free(unit); free(c); return -1; }
        c[k + 1] = c[k] + u;
        if (u > umax) umax = u;
    }
    int64_t lb = (E + c[m] - 1) / c[m];
    int64_t lb2 = (big + umax - 1) / umax;
    if (lb2 > lb) lb = lb2;
    lb = round_up(lb, align);

    int64_t *B = bounds;
    for (int64_t S = lb;; S += align) {
        for (int32_t k = 0; k <= m; ++k) B[k] = S * c[k];
        if (place_all(n, numel, unit, align, B, m, offsets)) {
            *S_out = S;
            break;
        }
    }
    free(numel); free(unit); free(c);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static float bits_f32(uint32_t u) { float x; memcpy(&x, &u, 4); return x; }

/* bfloat16 is the upper half of an IEEE binary32 pattern.  Round to nearest,
 * ties to even: the discarded low 16 bits are compared with half an ulp
 * (0x8000); above it rounds away from zero, below it truncates, at exactly half
 * it picks the candidate whose last kept bit is 0.  A carry out of the
 * mantissa correctly moves to the next binade (or to infinity past the largest
 * finite value).  NaN stays NaN (quiet bit set, sign kept). */
uint16_t orc_f32_to_bf16(float x)
{
    uint32_t u = f32_bits(x);
    if (isnan(x)) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t upper = u >> 16, lower = u & 0xFFFFu;
    if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
    return (uint16_t)upper;
}

float orc_bf16_to_f32(uint16_t h) { return bits_f32((uint32_t)h << 16); }

/* Magnitude of a non-negative OCP FP8 E4M3 code 0..126: 4 exponent bits with
 * bias 7 and 3 mantissa bits; exponent field 0 holds subnormals m/8 * 2^-6.
 * 0x7F is NaN and there is no infinity; the largest finite value is 448. */
double orc_e4m3_value(uint8_t code)
{
    int e = (code >> 3) & 15, mt = code & 7;
    double v = (e == 0) ? ldexp(mt / 8.0, -6) : ldexp(1.0 + mt / 8.0, e - 7);
    if ((code & 0x7F) == 0x7F) v = NAN;
    return (code & 0x80) ? -v : v;
}

/* fp32 -> E4M3, round to nearest with ties to the even code, saturating to
 * +-448 (values at or beyond 448 in magnitude, infinities included).  The
 * nearest code is found among the 127 finite magnitudes by bisection; the
 * distances are exact in double. */
uint8_t orc_f32_to_e4m3(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sign | 0x7F);
    double ax = fabs((double)x);
    if (ax >= 448.0) return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 126;           /* value(lo) <= ax < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (orc_e4m3_value((uint8_t)mid) <= ax) lo = mid; else hi = mid;
    }
    double dlo = ax - orc_e4m3_value((uint8_t)lo);
    double dhi = orc_e4m3_value((uint8_t)hi) - ax;
    int code;
    if (dlo < dhi) code = lo;
    else if (dhi < dlo) code = hi;
    else code = (lo & 1) ? hi : lo;   /* the code's last bit is the mantissa's */
    return (uint8_t)(sign | code);
}

/* fp32 -> INT8: round half to even (rintf under the default rounding mode),
 * then clamp to the symmetric range [-127, 127]. */
int8_t orc_f32_to_int8(float v)
{
    if (isnan(v)) return 0;
    float r = rintf(v);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    return (int8_t)r;
}

void orc_f32_to_bf16_array(const float *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_bf16(x[i]);
}

void orc_f32_to_e4m3_array(const float *x, uint8_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_e4m3(x[i]);
}

void orc_f32_to_int8_array(const float *x, int8_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = orc_f32_to_int8(x[i]);
}

/* ------------------------------------------------------------------------ */
/* Group operators on the planned flat buffer                                */
/* ------------------------------------------------------------------------ */

static float load_elem(const void *p, int32_t dtype, int64_t i)
{
    if (dtype == ORC_BF16) return orc_bf16_to_f32(((const uint16_t *)p)[i]);
    return ((const float *)p)[i];
}

static void store_elem(void *p, int32_t dtype, int64_t i, float v)
{
    if (dtype == ORC_BF16) ((uint16_t *)p)[i] = orc_f32_to_bf16(v);
    else ((float *)p)[i] = v;
}

/* One element from src[i] to dst[j]: a copy of its bytes when both sides have
 * the same type (a copy-in or copy-out is a copy, so every bit pattern, NaN
 * payloads included, arrives unchanged), else the cast through fp32. */
static void move_elem(const void *src, int32_t src_dtype, int64_t i,
                      void *dst, int32_t dst_dtype, int64_t j)
{
    if (src_dtype == dst_dtype) {
        size_t w = src_dtype == ORC_BF16 ? 2 : 4;
        memcpy((char *)dst + (size_t)j * w, (const char *)src + (size_t)i * w, w);
        return;
    }
    store_elem(dst, dst_dtype, j, load_elem(src, src_dtype, i));
}

/* pack (copy-in), with the mixed-precision cast fused: buf[l_t + i] =
 * cast(src_t[i]) for every tensor t [FSDP-1, §5 DBuffer group-level operators
 * and zero-copy access; FSDP-2, native mixed precision].  Padding between
 * tensors is not touched. */
void orc_pack(int32_t n, const int64_t *offsets, const int64_t *numel,
              const void *const *src, int32_t src_dtype, void *buf, int32_t buf_dtype)
{
    for (int32_t t = 0; t < n; ++t)
        for (int64_t i = 0; i < numel[t]; ++i)
            move_elem(src[t], src_dtype, i, buf, buf_dtype, offsets[t] + i);
}

/* unpack (copy-out / reconstruct a tensor from the flat buffer):
 * dst_t[i] = cast(buf[l_t + i]). */
void orc_unpack(int32_t n, const int64_t *offsets, const int64_t *numel,
                const void *buf, int32_t buf_dtype, void *const *dst, int32_t dst_dtype)
{
    for (int32_t t = 0; t < n; ++t)
        for (int64_t i = 0; i < numel[t]; ++i)
            move_elem(buf, buf_dtype, offsets[t] + i, dst[t], dst_dtype, i);
}

/* Gradient scale, accumulate and zero over the tensor ranges, in buffer order:
 * acc = acc + (g * s) with each product and sum rounded to fp32, then g = +0.
 * [FSDP-1, §5 DBuffer group-level operators: add, scale, zero fused;
 *  FSDP-2, gradient accumulation without communication]. */
void orc_scale_accum_zero(int32_t n, const int64_t *offsets, const int64_t *numel,
                          void *grad, int32_t grad_dtype, float *acc, float scale)
{
    for (int32_t t = 0; t < n; ++t)
        for (int64_t i = 0; i < numel[t]; ++i) {
            int64_t j = offsets[t] + i;
            float g = load_elem(grad, grad_dtype, j);
            float prod = g * scale;
            acc[j] = acc[j] + prod;
            if (grad_dtype == ORC_BF16) ((uint16_t *)grad)[j] = 0;
            else ((float *)grad)[j] = 0.0f;
        }
}

/* Per-tensor L2 norms over ragged shards, the global norm and the non-finite
 * flag [veScale-3, OpDispatcher: ragged norm and found_inf handlers; FSDP-2,
 * sharded gradient scaler; known limitation on per-parameter norms].
 * Sum of squares in fp64 in index order, square root in fp64; the global norm
 * is the square root of the per-tensor sums added in tensor order. */
void orc_norm_nonfinite(int32_t n, const int64_t *offsets, const int64_t *numel,
                        const void *buf, int32_t dtype, double *tensor_norms,
                        double *total_norm, int32_t *nonfinite)
{
    double total = 0.0;
    int32_t flag = 0;
    for (int32_t t = 0; t < n; ++t) {
        double s = 0.0;
        for (int64_t i = 0; i < numel[t]; ++i) {
            float x = load_elem(buf, dtype, offsets[t] + i);
            if (!isfinite(x)) flag = 1;
            s += (double)x * (double)x;
        }
        tensor_norms[t] = sqrt(s);
        total += s;
    }
    *total_norm = sqrt(total);
    *nonfinite = flag;
}

/* Number of quantisation blocks of one tensor; block extents <= 0 mean the
 * whole dimension.  Edge blocks are clipped to the tensor. */
static int64_t nblocks_dim(int64_t extent, int64_t blk)
{
    if (blk <= 0) blk = extent;
    if (extent == 0) return 0;
    return (extent + blk - 1) / blk;
}

/* Block-wise absmax quantisation of fp32 values in the flat buffer, with
 * blocks that never cross a shard boundary [FSDP-1, §4 Block-wise RaggedShard;
 * §6.3 8-bit Adam].  Per block: amax = max |x| in fp32; scale = amax / qmax as
 * one fp32 division (qmax = 448 for E4M3, 127 for INT8), replaced by 1.0 when
 * it is not positive (an all-zero block); every code is enc(x / scale) with x /
 * scale one fp32 division.  codes share the buffer's layout (1 byte per
 * element); scales are stored tensor by tensor in row-major block order.
 * Tensors with quant = none are skipped.  Returns the number of scales. */
int64_t orc_block_quant(int32_t n, const int64_t *offsets, const int64_t *rows,
                        const int64_t *cols, const int64_t *qrows, const int64_t *qcols,
                        const int32_t *quant, const float *buf, uint8_t *codes,
                        float *scales)
{
    int64_t s_off = 0;
    for (int32_t t = 0; t < n; ++t) {
        if (quant[t] == ORC_QNONE) continue;
        int64_t R = rows[t], C = cols[t];
        int64_t qr = qrows[t] > 0 ? qrows[t] : R;
        int64_t qc = qcols[t] > 0 ? qcols[t] : C;
        int64_t nbr = nblocks_dim(R, qr), nbc = nblocks_dim(C, qc);
        float qmax = (quant[t] == ORC_QE4M3) ? 448.0f : 127.0f;
        const float *x = buf + offsets[t];
        uint8_t *y = codes + offsets[t];
        for (int64_t bi = 0; bi < nbr; ++bi)
            for (int64_t bj = 0; bj < nbc; ++bj) {
                int64_t r0 = bi * qr, r1 = r0 + qr < R ? r0 + qr : R;
                int64_t c0 = bj * qc, c1 = c0 + qc < C ? c0 + qc : C;
                float amax = 0.0f;
                for (int64_t r = r0; r < r1; ++r)
                    for (int64_t c = c0; c < c1; ++c) {
                        float a = fabsf(x[r * C + c]);
                        if (a > amax) amax = a;
                    }
                float scale = amax / qmax;
                if (!(scale > 0.0f)) scale = 1.0f;
                scales[s_off + bi * nbc + bj] = scale;
                for (int64_t r = r0; r < r1; ++r)
                    for (int64_t c = c0; c < c1; ++c) {
                        float v = x[r * C + c] / scale;
                        y[r * C + c] = (quant[t] == ORC_QE4M3)
                                           ? orc_f32_to_e4m3(v)
                                           : (uint8_t)orc_f32_to_int8(v);
                    }
            }
        s_off += nbr * nbc;
    }
    return s_off;
}

/* Scale offsets: where each tensor's scales start (tensors without quant add
 * no scales).  Returns the total number of scales. */
int64_t orc_scale_offsets(int32_t n, const int64_t *rows, const int64_t *cols,
                          const int64_t *qrows, const int64_t *qcols,
                          const int32_t *quant, int64_t *scale_offsets)
{
    int64_t s = 0;
    for (int32_t t = 0; t < n; ++t) {
        scale_offsets[t] = s;
        if (quant[t] == ORC_QNONE) continue;
        s += nblocks_dim(rows[t], qrows[t] > 0 ? qrows[t] : rows[t]) *
             nblocks_dim(cols[t], qcols[t] > 0 ? qcols[t] : cols[t]);
    }
    return s;
}

/* ------------------------------------------------------------------------ */
/* Fused group optimizer step: AdamW over the flat buffer                    */
/* ------------------------------------------------------------------------ */

/* The scalars every element uses, each one fp32 operation in a fixed order. */
typedef struct {
    float coef;      /* gradient clip coefficient (1 when not clipping) */
    float decay;     /* 1 - lr*wd */
    float step;      /* lr / (1 - beta1^t) */
    float omb1;      /* 1 - beta1 */
    float omb2;      /* 1 - beta2 */
} orc_adamw_scalars;

/* Clip coefficient min(1, max_norm / (total_norm + 1e-6)) of gradient-norm
 * clipping; no clipping when max_norm <= 0. */
float orc_clip_coef(float max_norm, float total_norm)
{
    if (!(max_norm > 0.0f)) return 1.0f;
    float denom = total_norm + 1e-6f;
    float c = max_norm / denom;
    return c < 1.0f ? c : 1.0f;
}

/* Bias correction 1 - beta^t of Adam's moment estimates for step t >= 1: the
 * power of the fp32 beta taken in fp64 by the C library's pow, subtracted from
 * 1 in fp64, rounded once to fp32 (the reading of this library: the pages give
 * no formula). */
float orc_bias_correction(float beta, int64_t step)
{
    double c = 1.0 - pow((double)beta, (double)step);
    return (float)c;
}

/* One AdamW step with decoupled weight decay over every tensor range of the
 * flat buffer [veScale-3, OpDispatcher: fused AdamW handler on the local shard;
 * veScale-FSDP, §5 DBuffer group-level operators].  The pages name the fused
 * optimizer but not its formula; this is the standard AdamW update, every
 * operation rounded to fp32 in this order:
 *   g = grad * coef;  p = p * (1 - lr*wd)
 *   m = beta1*m + (1-beta1)*g;  v = beta2*v + ((1-beta2)*g)*g
 *   p = p - (lr/bc1) * (m / (sqrt(v / bc2) + eps))
 * with bc1 = 1 - beta1^t and bc2 = 1 - beta2^t for step t (orc_bias_correction).  When
 * `nonfinite` is non-zero the step is skipped (nothing is written), as a
 * gradient scaler skips a step with inf/NaN gradients. */
void orc_adamw(int32_t n, const int64_t *offsets, const int64_t *numel, float *p,
               const float *grad, float *m, float *v, float lr, float beta1, float beta2,
               float eps, float wd, int64_t step, float max_norm, float total_norm,
               int32_t nonfinite)
{
    if (nonfinite) return;
    float bc1 = orc_bias_correction(beta1, step);
    float bc2 = orc_bias_correction(beta2, step);
    orc_adamw_scalars s;
    s.coef = orc_clip_coef(max_norm, total_norm);
    s.decay = 1.0f - lr * wd;
    s.step = lr / bc1;
    s.omb1 = 1.0f - beta1;
    s.omb2 = 1.0f - beta2;
    for (int32_t t = 0; t < n; ++t)
        for (int64_t i = 0; i < numel[t]; ++i) {
            int64_t j = offsets[t] + i;
            float g = grad[j] * s.coef;
            float pj = p[j] * s.decay;
            float mj = beta1 * m[j] + s.omb1 * g;
            float vj = beta2 * v[j] + (s.omb2 * g) * g;
            float denom = sqrtf(vj / bc2) + eps;
            p[j] = pj - s.step * (mj / denom);
            m[j] = mj;
            v[j] = vj;
        }
}

/* Layout of the fp32 moments that 8-bit AdamW keeps for tensors without a
 * quantisation block (vectors, norms): those tensors in group order, each
 * starting at a multiple of 4 elements (16 bytes); -1 for quantised tensors.
 * Returns the number of fp32 elements per moment. */
int64_t orc_state_offsets(int32_t n, const int64_t *numel, const int32_t *quant,
                          int64_t *state_offsets)
{
    int64_t s = 0;
    for (int32_t t = 0; t < n; ++t) {
        if (quant[t] != ORC_QNONE) { state_offsets[t] = -1; continue; }
        state_offsets[t] = s;
        s += (numel[t] + 3) / 4 * 4;
    }
    return s;
}

/* The second moment's 8-bit code (unsigned): the linear absmax map without a
 * zero level, code c stands for (c + 1) * scale with scale = block amax / 256,
 * so a positive v never dequantises to 0 (a zero denominator would turn the
 * update into m / eps).  c = clamp(rint(v / scale), 1, 256) - 1 with v / scale
 * one fp32 division; an all-zero block has scale 0 and codes 0. */
uint8_t orc_v_code(float v, float scale)
{
    if (!(scale > 0.0f) || isnan(v)) return 0;
    float r = rintf(v / scale);
    if (r < 1.0f) r = 1.0f;
    if (r > 256.0f) r = 256.0f;
    return (uint8_t)((int)r - 1);
}

/* 8-bit AdamW: the same step with block-wise 8-bit moments [veScale-FSDP, §6.3
 * 8-bit Adam: block-wise INT8 quantisation of the optimizer's gradient
 * statistics; blocks never cross a shard, so each shard quantises locally].
 * The pages do not give the code maps.  Reading: the first moment m takes the
 * signed absmax INT8 map of orc_block_quant (scale = amax / 127, 1 when not
 * positive; code = clamp(rint(m / scale), -127, 127); m = code * scale); the
 * second moment v >= 0 takes orc_v_code's zero-free unsigned map (v = (c + 1) *
 * scale).  Per block of each quantised tensor's quantisation shape: dequantise
 * (one fp32 multiply each), the AdamW step of orc_adamw, new block scales from
 * the new moments' amax, re-encode.  The codes share the flat buffer's layout;
 * scales are indexed like orc_block_quant's.  Tensors with quant = none keep
 * fp32 moments in m32 / v32 at their state offset (orc_state_offsets).  A set
 * non-finite flag skips the step. */
void orc_adamw8(int32_t n, const int64_t *offsets, const int64_t *rows, const int64_t *cols,
                const int64_t *qrows, const int64_t *qcols, const int32_t *quant,
                const int64_t *state_offsets, float *p, const float *grad, uint8_t *m_codes,
                uint8_t *v_codes, float *m_scales, float *v_scales, float *m32, float *v32,
                float lr, float beta1, float beta2, float eps, float wd, int64_t step,
                float max_norm, float total_norm, int32_t nonfinite)
{
    if (nonfinite) return;
    float bc1 = orc_bias_correction(beta1, step);
    float bc2 = orc_bias_correction(beta2, step);
    orc_adamw_scalars s;
    s.coef = orc_clip_coef(max_norm, total_norm);
    s.decay = 1.0f - lr * wd;
    s.step = lr / bc1;
    s.omb1 = 1.0f - beta1;
    s.omb2 = 1.0f - beta2;
    int64_t s_off = 0;
    for (int32_t t = 0; t < n; ++t) {
        int64_t R = rows[t], C = cols[t];
        if (quant[t] == ORC_QNONE) {
            for (int64_t i = 0; i < R * C; ++i) {
                int64_t j = offsets[t] + i, k = state_offsets[t] + i;
                float g = grad[j] * s.coef;
                float pj = p[j] * s.decay;
                float mj = beta1 * m32[k] + s.omb1 * g;
                float vj = beta2 * v32[k] + (s.omb2 * g) * g;
                float denom = sqrtf(vj / bc2) + eps;
                p[j] = pj - s.step * (mj / denom);
                m32[k] = mj;
                v32[k] = vj;
            }
            continue;
        }
        int64_t qr = qrows[t] > 0 ? qrows[t] : R;
        int64_t qc = qcols[t] > 0 ? qcols[t] : C;
        int64_t nbr = nblocks_dim(R, qr), nbc = nblocks_dim(C, qc);
        for (int64_t bi = 0; bi < nbr; ++bi)
            for (int64_t bj = 0; bj < nbc; ++bj) {
                int64_t r0 = bi * qr, r1 = r0 + qr < R ? r0 + qr : R;
                int64_t c0 = bj * qc, c1 = c0 + qc < C ? c0 + qc : C;
                int64_t si = s_off + bi * nbc + bj;
                float ms_old = m_scales[si], vs_old = v_scales[si];
                float mamax = 0.0f, vamax = 0.0f;
                /* pass 1: dequantise and step the moments to find the new block
                 * amax (pass 2 repeats the identical operations) */
                for (int64_t r = r0; r < r1; ++r)
                    for (int64_t c = c0; c < c1; ++c) {
                        int64_t j = offsets[t] + r * C + c;
                        float mo = (float)(int8_t)m_codes[j] * ms_old;
                        float vo = ((float)v_codes[j] + 1.0f) * vs_old;
                        float g = grad[j] * s.coef;
                        float mj = beta1 * mo + s.omb1 * g;
                        float vj = beta2 * vo + (s.omb2 * g) * g;
                        if (fabsf(mj) > mamax) mamax = fabsf(mj);
                        if (fabsf(vj) > vamax) vamax = fabsf(vj);
                    }
                float ms_new = mamax / 127.0f;
                if (!(ms_new > 0.0f)) ms_new = 1.0f;
                float vs_new = vamax / 256.0f;
                /* pass 2: the same step again (identical operations), update the
                 * parameters, encode the new moments */
                for (int64_t r = r0; r < r1; ++r)
                    for (int64_t c = c0; c < c1; ++c) {
                        int64_t j = offsets[t] + r * C + c;
                        float mo = (float)(int8_t)m_codes[j] * ms_old;
                        float vo = ((float)v_codes[j] + 1.0f) * vs_old;
                        float g = grad[j] * s.coef;
                        float pj = p[j] * s.decay;
                        float mj = beta1 * mo + s.omb1 * g;
                        float vj = beta2 * vo + (s.omb2 * g) * g;
                        float denom = sqrtf(vj / bc2) + eps;
                        p[j] = pj - s.step * (mj / denom);
                        m_codes[j] = (uint8_t)orc_f32_to_int8(mj / ms_new);
                        v_codes[j] = orc_v_code(vj, vs_new);
                    }
                m_scales[si] = ms_new;
                v_scales[si] = vs_new;
            }
        s_off += nbr * nbc;
    }
}

/* Shard holding flat position pos: the k with bounds[k] <= pos < bounds[k+1]. */
static int32_t shard_of(int32_t m, const int64_t *bounds, int64_t pos)
{
    int32_t k = 0;
    while (k + 1 < m && bounds[k + 1] <= pos) ++k;
    return k;
}

/* Whole-matrix gather for Muon-style updates [veScale-FSDP, §6.3 Distributed
 * Muon: each matrix is redistributed to a root as the full 2-D matrix, updated
 * there, and the update redistributed back (Algorithm 2)].  The m shards are
 * separate buffers: shard k holds flat positions [bounds[k], bounds[k+1]) at
 * local offsets 0..; element i of tensor t (flat position offsets[t] + i) is
 * copied to dst[t][i].  Tensors with dst[t] == NULL are skipped.  Elements are
 * moved as raw bytes of the dtype (no conversion). */
void orc_gather(int32_t n, const int64_t *offsets, const int64_t *numel, int32_t m,
                const int64_t *bounds, void *const *shards, int32_t dtype, void *const *dst)
{
    size_t es = dtype == ORC_BF16 ? 2 : 4;
    for (int32_t t = 0; t < n; ++t) {
        if (!dst[t]) continue;
        for (int64_t i = 0; i < numel[t]; ++i) {
            int64_t pos = offsets[t] + i;
            int32_t k = shard_of(m, bounds, pos);
            memcpy((char *)dst[t] + (size_t)i * es,
                   (const char *)shards[k] + (size_t)(pos - bounds[k]) * es, es);
        }
    }
}

/* The way back: element i of src[t] goes to its shard position.  Tensors with
 * src[t] == NULL are left as they are; shard bytes outside tensor ranges are
 * never written. */
void orc_scatter(int32_t n, const int64_t *offsets, const int64_t *numel, int32_t m,
                 const int64_t *bounds, const void *const *src, int32_t dtype,
                 void *const *shards)
{
    size_t es = dtype == ORC_BF16 ? 2 : 4;
    for (int32_t t = 0; t < n; ++t) {
        if (!src[t]) continue;
        for (int64_t i = 0; i < numel[t]; ++i) {
            int64_t pos = offsets[t] + i;
            int32_t k = shard_of(m, bounds, pos);
            memcpy((char *)shards[k] + (size_t)(pos - bounds[k]) * es,
                   (const char *)src[t] + (size_t)i * es, es);
        }
    }
}
