// Internal layout of a plan and of its device descriptor tables.
// Shared by the host planner (planner.cpp) and the CUDA operators (*.cu).
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/dbuf.h"

namespace dbuf {

// Elements per chunk of the elementwise operators.  A chunk never spans two
// tensors, so every chunk has one source and one destination range; chunk
// starts are multiples of kChunkElems inside a tensor.
constexpr int64_t kChunkElems = 16384;

// Blocks per work item of the row-block (1 x qc) quantisation kernel.
constexpr int32_t kRowItemBlocks = 64;

// One tensor of the group, as the kernels see it (80 bytes).  In a slice plan
// (one shard of a parent plan as a rank's local buffer) a tensor is its piece
// inside the slice: buf_off is local and src_off is the piece's first element
// within the user tensor (0 in a full plan).
struct TensorDesc {
    int64_t buf_off;    // l_t
    int64_t numel;      // n_t
    int64_t src_off;    // first element of this (piece of the) tensor in the user tensor
    int64_t rows;
    int64_t cols;
    int64_t scale_off;  // first block scale of this tensor
    int64_t state_off;  // first fp32 moment in the compact 8-bit-optimizer state, or -1
    int32_t qrows;      // effective quantisation block rows (>= 1)
    int32_t qcols;      // effective quantisation block cols (>= 1)
    int32_t quant;      // DBUF_QUANT_*
    int32_t nbc;        // quantisation blocks per block-row
    int32_t chunk_begin;
    int32_t chunk_end;
};
static_assert(sizeof(TensorDesc) == 80, "TensorDesc layout");

// A contiguous piece of one tensor: elements [off, off+len) of tensor `tensor`.
struct Chunk {
    int64_t off;
    int32_t tensor;
    int32_t len;
};
static_assert(sizeof(Chunk) == 16, "Chunk layout");

// A run of `count` consecutive quantisation blocks (row-major block order) of
// one tensor, starting at block `first`.
struct QItem {
    int64_t first;
    int32_t tensor;
    int32_t count;
};
static_assert(sizeof(QItem) == 16, "QItem layout");

// A run of `count` consecutive 1 x qc blocks (row-major block order) of one
// tensor, starting at block column bj0 of block row bi0.
struct RowItem {
    int32_t tensor;
    int32_t bi0;
    int32_t bj0;
    int32_t count;
};
static_assert(sizeof(RowItem) == 16, "RowItem layout");

// One quantisation tile for the pipelined tile kernel: block (bi, bj) of a
// tensor whose tiles a 2-D tensor-memory-access copy can fetch (at most
// 128 x 128 fp32, rows and tile widths multiples of 16 bytes, the tensor at a
// 16-byte-aligned offset of a 16-byte-aligned buffer).  `slot` is the tensor's
// index in the per-call table of tensor maps.
struct TileItem {
    int32_t tensor;
    int32_t bi;
    int32_t bj;
    int32_t slot;
};
static_assert(sizeof(TileItem) == 16, "TileItem layout");

// A run of `count` consecutive quantisation blocks (row-major block order) of
// one tensor for the 8-bit optimizer step, starting at block (bi0, bj0);
// `lanes` threads (a power of two from 4 to 256) work on one block.
struct OptItem {
    int32_t tensor;
    int32_t bi0;
    int32_t bj0;
    int16_t count;
    int16_t lanes;
};
static_assert(sizeof(OptItem) == 16, "OptItem layout");

// A piece of one tensor inside one shard, for the whole-matrix gather and
// scatter: elements [off, off+len) of tensor `tensor` sit at [shard_off,
// shard_off+len) of shard `shard`.  Pieces are chunks split at shard bounds.
struct Piece {
    int64_t off;
    int64_t shard_off;
    int32_t tensor;
    int32_t len;
    int32_t shard;
    int32_t reserved;
};
static_assert(sizeof(Piece) == 32, "Piece layout");

// One stage of the pipelined 8-bit optimizer: the box of blocks [bi0, bi0 +
// Rb) x [bj0, bj0 + K) of tensor `tensor` (tensor-map slot `slot`), 4096
// elements; Rb and K follow from the tensor's block shape.
struct P8Item {
    int32_t slot;    // within its launch: the plan's p8 tensor index mod kP8MaxTensors
    int32_t tensor;
    int32_t bi0;
    int32_t bj0;
};
static_assert(sizeof(P8Item) == 16, "P8Item layout");

constexpr int kP8MaxTensors = 16;      // tensors with tensor maps per launch (4 maps each);
                                       // a group with more takes one launch per 16
constexpr int kP8ComputeWarps = 16;    // compute warps per CTA of the pipelined kernel
constexpr int kP8UnitsPerThread = 4;   // units of 4 elements per compute thread and stage
constexpr int kP8StageElems = kP8ComputeWarps * 32 * 4 * kP8UnitsPerThread;  // elements per stage

// Moment units (4 elements on the vector path) that one thread of the 8-bit
// optimizer keeps in registers; larger blocks are recomputed in a second pass.
constexpr int kOptUnitsPerLane = 2;
// Target elements per 8-bit optimizer work item.
constexpr int64_t kOptItemElems = 16384;

// Blocks of exactly this many elements (128 x 128, 64 x 256, 256 x 64), twice a
// stage of the pipelined 8-bit optimizer, take their own pipelined kernel.
constexpr int64_t kBigBlockElems = 16384;

constexpr int kPipeMaxRows = 128;
constexpr int kPipeMaxCols = 128;
constexpr int kPipeMaxTensors = 32;  // tensor maps passed per launch; more tensors take more launches

// The scalars of one AdamW step as the kernels take them: the caller's
// hyperparameters with the bias corrections formed (see bias_corrections).
struct AdamParams {
    float lr;
    float beta1;
    float beta2;
    float eps;
    float weight_decay;
    float bias_correction1;  // 1 - beta1^t
    float bias_correction2;  // 1 - beta2^t
    float max_norm;
};

// AdamParams from the ABI struct: bc = (float)(1 - pow((double)beta, (double)t)).
// Returns false for t < 1 or a correction that is not a positive finite float.
bool adam_params(const dbuf_adamw_hparams &hp, AdamParams *out);

struct DeviceTables {
    TensorDesc *tensors = nullptr;
    Chunk *chunks = nullptr;
    RowItem *row_items = nullptr;    // blocks with qrows == 1
    QItem *tile_items = nullptr;     // other blocks with qrows > 1 (one block per item)
    TileItem *pipe_items = nullptr;  // tiles for the pipelined kernel
    OptItem *opt_items = nullptr;    // 8-bit optimizer: blocks of quantised tensors
    int32_t *opt_plain = nullptr;    // 8-bit optimizer: chunks of the other tensors
    Piece *pieces = nullptr;         // gather / scatter: chunks split at shard bounds
    P8Item *p8_items = nullptr;      // pipelined 8-bit optimizer stages
    P8Item *big_items = nullptr;     // pipelined 8-bit optimizer, one block of kBigBlockElems each
    int32_t *status = nullptr;       // device status word (0, or DBUF_ETIMEOUT)
    void *base = nullptr;
    size_t bytes = 0;
    int device = -1;
    int num_sms = 0;
};

// Launchers (one kernel launch over the whole group each; the norm adds a
// small fixed-order finalisation launch).  They return a cudaError_t value.
int launch_pack(const dbuf_plan_t *p, const void *const *src, int src_dt, void *buf, int buf_dt,
                void *stream);
int launch_unpack(const dbuf_plan_t *p, const void *buf, int buf_dt, void *const *dst, int dst_dt,
                  void *stream);
int launch_sac(const dbuf_plan_t *p, void *grad, int grad_dt, float *acc, float scale,
               void *stream);
// tensor_norms and total_norm may be null; tensor_sumsq (optional) receives each
// tensor's fp64 sum of squares.
int launch_norm(const dbuf_plan_t *p, const void *buf, int dt, float *tensor_norms,
                float *total_norm, int32_t *nonfinite, void *workspace, void *stream,
                double *tensor_sumsq = nullptr);
int launch_norm_finish(const dbuf_plan_t *p, const double *sumsq, float *tensor_norms,
                       float *total_norm, void *stream);
int launch_quant(const dbuf_plan_t *p, const float *buf, uint8_t *codes, float *scales,
                 void *stream);

int launch_adamw(const dbuf_plan_t *p, float *params, const float *grads, float *exp_avg,
                 float *exp_avg_sq, const AdamParams &hp, const float *total_norm,
                 const int32_t *nonfinite, void *stream);

int launch_adamw8(const dbuf_plan_t *p, float *params, const float *grads, uint8_t *m_codes,
                  uint8_t *v_codes, float *m_scales, float *v_scales, float *m32, float *v32,
                  const AdamParams &hp, const float *total_norm, const int32_t *nonfinite,
                  void *stream);

int launch_gather(const dbuf_plan_t *p, void *const *shards, int dt, void *const *dst,
                  void *stream);
int launch_scatter(const dbuf_plan_t *p, const void *const *src, int dt, void *const *shards,
                   void *stream);

size_t norm_workspace_bytes(const dbuf_plan_t *p);
// Where the norm's completion tickets (n + 1 uint32) sit in its workspace.
size_t norm_ticket_offset(const dbuf_plan_t *p);
size_t norm_ticket_bytes(const dbuf_plan_t *p);

// One-time per-device set-up of the quantisation kernels (shared memory
// limits); called from dbuf_plan_upload.  Returns a cudaError_t value.
int prepare_quant_kernels();
int prepare_optim_kernels();

// Keeps a cudaError_t for dbuf_last_cuda_error() (per host thread).
void record_cuda_error(int e);

}  // namespace dbuf

struct dbuf_plan {
    int32_t n = 0;
    int32_t m = 0;
    int64_t align = 1;
    bool even = true;
    std::vector<int32_t> units;  // m shares (all 1 when even)
    std::vector<dbuf_tensor_spec> specs;

    int64_t S = 0;
    int64_t total = 0;
    std::vector<int64_t> offsets;        // [n]
    std::vector<int64_t> bounds;         // [m+1]
    std::vector<int64_t> scale_offsets;  // [n]
    int64_t n_scales = 0;

    std::vector<dbuf::TensorDesc> tdesc;
    std::vector<dbuf::Chunk> chunks;
    std::vector<dbuf::RowItem> row_items;
    std::vector<dbuf::QItem> tile_items;
    std::vector<dbuf::TileItem> pipe_items;
    std::vector<int32_t> pipe_tensors;  // plan slot -> tensor id (launch slot = plan slot % 32)
    std::vector<size_t> pipe_item_start;  // [slots + 1]: first pipelined tile of each slot
    std::vector<dbuf::OptItem> opt_items;
    std::vector<int32_t> opt_plain;      // chunk ids of tensors without quantisation
    std::vector<dbuf::Piece> pieces;
    std::vector<dbuf::P8Item> p8_items;
    std::vector<int32_t> p8_tensors;     // slot -> tensor id
    std::vector<size_t> p8_item_start;   // [slots + 1]: first p8 item of each slot
    std::vector<dbuf::P8Item> big_items;   // one item per kBigBlockElems block (slot, tensor, bi, bj)
    std::vector<int32_t> big_tensors;      // slot -> tensor
    std::vector<size_t> big_item_start;    // [slots + 1]
    size_t n_opt_rest = 0;               // opt_items[0, n_opt_rest): tensors without pipelined items
    std::vector<int64_t> state_offsets;  // [n], -1 for quantised tensors
    int64_t n_state = 0;

    // Slice plans (dbuf_plan_slice): shard slice_k of a parent plan, whose
    // global positions [slice_base, slice_base + total) are this plan's local
    // positions [0, total).  slice_k = -1 for a full plan.
    int32_t slice_k = -1;
    int64_t slice_base = 0;
    int64_t scale_base = 0;              // global index of the slice's first block scale
    std::vector<int64_t> src_offsets;    // [n] piece start within each user tensor (slices)

    bool uploaded = false;
    dbuf::DeviceTables dev;
};
