// C ABI entry points of libdbuf: argument checks (synchronous, before any launch),
// descriptor-table upload, and dispatch to the group-operator launchers.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>

#include "dbuf_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = int(e);
    return DBUF_ECUDA;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool dtype_ok(int32_t dt) { return dt == DBUF_F32 || dt == DBUF_BF16; }

// Common checks of every operator: plan uploaded, device current.
int check_plan(const dbuf_plan_t *p) {
    if (!p) return DBUF_EINVAL;
    if (!p->uploaded) return DBUF_ENOTUPLOADED;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev != p->dev.device) return DBUF_EDEVICE;
    return DBUF_OK;
}

int finish(int e) { return e == cudaSuccess ? DBUF_OK : cuda_fail(cudaError_t(e)); }

}  // namespace

extern "C" int dbuf_last_cuda_error(void) { return g_last_cuda_error; }

void dbuf::record_cuda_error(int e) { g_last_cuda_error = e; }

extern "C" int dbuf_plan_upload(dbuf_plan_t *p, void *stream) {
    if (!p) return DBUF_EINVAL;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (p->uploaded) return dev == p->dev.device ? DBUF_OK : DBUF_EDEVICE;

    const size_t b_t = align256(sizeof(dbuf::TensorDesc) * p->tdesc.size());
    const size_t b_c = align256(sizeof(dbuf::Chunk) * p->chunks.size());
    const size_t b_r = align256(sizeof(dbuf::RowItem) * p->row_items.size());
    const size_t b_q = align256(sizeof(dbuf::QItem) * p->tile_items.size());
    const size_t b_p = align256(sizeof(dbuf::TileItem) * p->pipe_items.size());
    const size_t b_o = align256(sizeof(dbuf::OptItem) * p->opt_items.size());
    const size_t b_a = align256(sizeof(int32_t) * p->opt_plain.size());
    const size_t b_g = align256(sizeof(dbuf::Piece) * p->pieces.size());
    const size_t b_8 = align256(sizeof(dbuf::P8Item) * p->p8_items.size());
    const size_t b_b = align256(sizeof(dbuf::P8Item) * p->big_items.size());
    const size_t bytes = b_t + b_c + b_r + b_q + b_p + b_o + b_a + b_g + b_8 + b_b + 256;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e);
    int prep = dbuf::prepare_quant_kernels();
    if (prep == int(cudaSuccess)) prep = dbuf::prepare_optim_kernels();
    if (prep != int(cudaSuccess)) return cuda_fail(cudaError_t(prep));
    void *base = nullptr;
    e = cudaMalloc(&base, bytes);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return e == cudaErrorMemoryAllocation ? DBUF_ENOMEM : cuda_fail(e);
    }
    char *c = static_cast<char *>(base);
    dbuf::DeviceTables t;
    t.base = base;
    t.bytes = bytes;
    t.device = dev;
    t.tensors = reinterpret_cast<dbuf::TensorDesc *>(c);
    t.chunks = reinterpret_cast<dbuf::Chunk *>(c + b_t);
    t.row_items = reinterpret_cast<dbuf::RowItem *>(c + b_t + b_c);
    t.tile_items = reinterpret_cast<dbuf::QItem *>(c + b_t + b_c + b_r);
    t.pipe_items = reinterpret_cast<dbuf::TileItem *>(c + b_t + b_c + b_r + b_q);
    t.opt_items = reinterpret_cast<dbuf::OptItem *>(c + b_t + b_c + b_r + b_q + b_p);
    t.opt_plain = reinterpret_cast<int32_t *>(c + b_t + b_c + b_r + b_q + b_p + b_o);
    t.pieces = reinterpret_cast<dbuf::Piece *>(c + b_t + b_c + b_r + b_q + b_p + b_o + b_a);
    t.p8_items = reinterpret_cast<dbuf::P8Item *>(c + b_t + b_c + b_r + b_q + b_p + b_o + b_a + b_g);
    t.big_items =
        reinterpret_cast<dbuf::P8Item *>(c + b_t + b_c + b_r + b_q + b_p + b_o + b_a + b_g + b_8);
    t.status = reinterpret_cast<int32_t *>(c + b_t + b_c + b_r + b_q + b_p + b_o + b_a + b_g + b_8 +
                                           b_b);
    t.num_sms = sms;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(t.status, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) {
        cudaFree(base);
        return cuda_fail(e);
    }
    struct Piece {
        void *dst;
        const void *src;
        size_t n;
    } pieces[10] = {
        {t.tensors, p->tdesc.data(), sizeof(dbuf::TensorDesc) * p->tdesc.size()},
        {t.chunks, p->chunks.data(), sizeof(dbuf::Chunk) * p->chunks.size()},
        {t.row_items, p->row_items.data(), sizeof(dbuf::RowItem) * p->row_items.size()},
        {t.tile_items, p->tile_items.data(), sizeof(dbuf::QItem) * p->tile_items.size()},
        {t.pipe_items, p->pipe_items.data(), sizeof(dbuf::TileItem) * p->pipe_items.size()},
        {t.opt_items, p->opt_items.data(), sizeof(dbuf::OptItem) * p->opt_items.size()},
        {t.opt_plain, p->opt_plain.data(), sizeof(int32_t) * p->opt_plain.size()},
        {t.pieces, p->pieces.data(), sizeof(dbuf::Piece) * p->pieces.size()},
        {t.p8_items, p->p8_items.data(), sizeof(dbuf::P8Item) * p->p8_items.size()},
        {t.big_items, p->big_items.data(), sizeof(dbuf::P8Item) * p->big_items.size()},
    };
    for (const Piece &pc : pieces) {
        if (!pc.n) continue;
        e = cudaMemcpyAsync(pc.dst, pc.src, pc.n, cudaMemcpyHostToDevice, st);
        if (e != cudaSuccess) {
            cudaFree(base);
            return cuda_fail(e);
        }
    }
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
        cudaFree(base);
        return cuda_fail(e);
    }
    p->dev = t;
    p->uploaded = true;
    return DBUF_OK;
}

extern "C" void dbuf_plan_free(dbuf_plan_t *p) {
    if (!p) return;
    if (p->uploaded && p->dev.base) {
        int cur = -1;
        cudaGetDevice(&cur);
        if (cur != p->dev.device) cudaSetDevice(p->dev.device);
        cudaFree(p->dev.base);
        if (cur != p->dev.device && cur >= 0) cudaSetDevice(cur);
    }
    delete p;
}

extern "C" int dbuf_pack_cast(const dbuf_plan_t *p, const void *const *src, int32_t src_dtype,
                              void *buf, int32_t buf_dtype, void *stream) {
    int rc = check_plan(p);
    if (rc) return rc;
    if (!dtype_ok(src_dtype) || !dtype_ok(buf_dtype)) return DBUF_EINVAL;
    if ((p->n > 0 && !src) || (p->total > 0 && !buf)) return DBUF_EINVAL;
    return finish(dbuf::launch_pack(p, src, src_dtype, buf, buf_dtype, stream));
}

extern "C" int dbuf_unpack(const dbuf_plan_t *p, const void *buf, int32_t buf_dtype,
                           void *const *dst, int32_t dst_dtype, void *stream) {
    int rc = check_plan(p);
    if (rc) return rc;
    if (!dtype_ok(buf_dtype) || !dtype_ok(dst_dtype)) return DBUF_EINVAL;
    if ((p->n > 0 && !dst) || (p->total > 0 && !buf)) return DBUF_EINVAL;
    return finish(dbuf::launch_unpack(p, buf, buf_dtype, dst, dst_dtype, stream));
}

extern "C" int dbuf_scale_accum_zero(const dbuf_plan_t *p, void *grad, int32_t grad_dtype,
                                     float *acc, float scale, void *stream) {
    int rc = check_plan(p);
    if (rc) return rc;
    if (!dtype_ok(grad_dtype)) return DBUF_EINVAL;
    if (p->total > 0 && (!grad || !acc)) return DBUF_EINVAL;
    return finish(dbuf::launch_sac(p, grad, grad_dtype, acc, scale, stream));
}

extern "C" int dbuf_norm_nonfinite(const dbuf_plan_t *p, const void *buf, int32_t dtype,
                                   float *tensor_norms, float *total_norm, int32_t *nonfinite,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_plan(p);
    if (rc) return rc;
    if (!dtype_ok(dtype)) return DBUF_EINVAL;
    if (!total_norm || !nonfinite || !workspace) return DBUF_EINVAL;
    if ((p->n > 0 && !tensor_norms) || (p->total > 0 && !buf)) return DBUF_EINVAL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DBUF_EINVAL;
    if (workspace_bytes < dbuf::norm_workspace_bytes(p)) return DBUF_EINVAL;
    return finish(dbuf::launch_norm(p, buf, dtype, tensor_norms, total_norm, nonfinite, workspace,
                                    stream));
}

extern "C" int dbuf_norm_sumsq(const dbuf_plan_t *p, const void *buf, int32_t dtype,
                               double *tensor_sumsq, int32_t *nonfinite, void *workspace,
                               size_t workspace_bytes, void *stream) {
    int rc = check_plan(p);
    if (rc) return rc;
    if (!dtype_ok(dtype)) return DBUF_EINVAL;
    if (!nonfinite || !workspace) return DBUF_EINVAL;
    if ((p->n > 0 && !tensor_sumsq) || (p->total > 0 && !buf)) return DBUF_EINVAL;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DBUF_EINVAL;
    if (workspace_bytes < dbuf::norm_workspace_bytes(p)) return DBUF_EINVAL;
    return finish(dbuf::launch_norm(p, buf, dtype, nullptr, nullptr, nonfinite, workspace, stream,
                                    tensor_sumsq));
}

extern "C" int dbuf_norm_finish(const dbuf_plan_t *p, const double *tensor_sumsq,
                                float *tensor_norms, float *total_norm, void *stream) {
    int rc = check_plan(p);
    if (rc) return rc;
    if (!total_norm) return DBUF_EINVAL;
    if (p->n > 0 && (!tensor_sumsq || !tensor_norms)) return DBUF_EINVAL;
    return finish(dbuf::launch_norm_finish(p, tensor_sumsq, tensor_norms, total_norm, stream));
}

extern "C" int dbuf_block_quant(const dbuf_plan_t *p, const float *buf, uint8_t *codes,
                                float *scales, void *stream) {
    int rc = check_plan(p);
    if (rc) return rc;
    if (p->n_scales > 0 && (!buf || !codes || !scales)) return DBUF_EINVAL;
    return finish(dbuf::launch_quant(p, buf, codes, scales, stream));
}

extern "C" int dbuf_device_status(const dbuf_plan_t *p, int32_t *status, void *stream) {
    int rc = check_plan(p);
    if (rc) return rc;
    if (!status) return DBUF_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, p->dev.status, sizeof(v), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (v != 0) {
        e = cudaMemsetAsync(p->dev.status, 0, sizeof(int32_t), st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    *status = v;
    return DBUF_OK;
}

bool dbuf::adam_params(const dbuf_adamw_hparams &hp, AdamParams *out) {
    if (hp.step < 1) return false;
    const double t = double(hp.step);
    const float bc1 = float(1.0 - std::pow(double(hp.beta1), t));
    const float bc2 = float(1.0 - std::pow(double(hp.beta2), t));
    if (!(bc1 > 0.0f) || !(bc2 > 0.0f) || !std::isfinite(bc1) || !std::isfinite(bc2))
        return false;
    *out = AdamParams{hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, bc1, bc2, hp.max_norm};
    return true;
}

extern "C" int dbuf_adamw_step(const dbuf_plan_t *p, float *params, const float *grads,
                               float *exp_avg, float *exp_avg_sq, const dbuf_adamw_hparams *hp,
                               const float *total_norm, const int32_t *nonfinite, void *stream) {
    dbuf::AdamParams ap;
    if (!p || !hp || !dbuf::adam_params(*hp, &ap)) return DBUF_EINVAL;
    int rc = check_plan(p);
    if (rc) return rc;
    if (p->total > 0 && (!params || !grads || !exp_avg || !exp_avg_sq)) return DBUF_EINVAL;
    return finish(dbuf::launch_adamw(p, params, grads, exp_avg, exp_avg_sq, ap, total_norm,
                                     nonfinite, stream));
}

extern "C" int dbuf_adamw8_step(const dbuf_plan_t *p, float *params, const float *grads,
                                uint8_t *exp_avg_codes, uint8_t *exp_avg_sq_codes,
                                float *exp_avg_scales, float *exp_avg_sq_scales,
                                float *exp_avg_fp32, float *exp_avg_sq_fp32,
                                const dbuf_adamw_hparams *hp, const float *total_norm,
                                const int32_t *nonfinite, void *stream) {
    dbuf::AdamParams ap;
    if (!p || !hp || !dbuf::adam_params(*hp, &ap)) return DBUF_EINVAL;
    int rc = check_plan(p);
    if (rc) return rc;
    if (p->total > 0 && (!params || !grads)) return DBUF_EINVAL;
    if (p->n_scales > 0 &&
        (!exp_avg_codes || !exp_avg_sq_codes || !exp_avg_scales || !exp_avg_sq_scales))
        return DBUF_EINVAL;
    if (p->n_state > 0 && (!exp_avg_fp32 || !exp_avg_sq_fp32)) return DBUF_EINVAL;
    return finish(dbuf::launch_adamw8(p, params, grads, exp_avg_codes, exp_avg_sq_codes,
                                      exp_avg_scales, exp_avg_sq_scales, exp_avg_fp32,
                                      exp_avg_sq_fp32, ap, total_norm, nonfinite, stream));
}

extern "C" int dbuf_gather(const dbuf_plan_t *p, void *const *shards, int32_t dtype,
                           void *const *dst, void *stream) {
    if (p && p->slice_k >= 0) return DBUF_EINVAL;  // needs every shard
    int rc = check_plan(p);
    if (rc) return rc;
    if (!dtype_ok(dtype)) return DBUF_EINVAL;
    if (p->n > 0 && (!shards || !dst)) return DBUF_EINVAL;
    return finish(dbuf::launch_gather(p, shards, dtype, dst, stream));
}

extern "C" int dbuf_scatter(const dbuf_plan_t *p, const void *const *src, int32_t dtype,
                            void *const *shards, void *stream) {
    if (p && p->slice_k >= 0) return DBUF_EINVAL;  // needs every shard
    int rc = check_plan(p);
    if (rc) return rc;
    if (!dtype_ok(dtype)) return DBUF_EINVAL;
    if (p->n > 0 && (!shards || !src)) return DBUF_EINVAL;
    return finish(dbuf::launch_scatter(p, src, dtype, shards, stream));
}
