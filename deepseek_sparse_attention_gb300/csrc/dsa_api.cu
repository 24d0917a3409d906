// dsa_api.cu -- the extern "C" entry points of libdsa: host-side validation,
// workspace layout, and the order in which the kernels are enqueued.
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "dsa.h"
#include "dsa_kernels.cuh"

namespace dsa {
namespace {

constexpr size_t kAlign = 256;
constexpr uint32_t kKnownFlags = DSA_FLAG_TWO_LAUNCH | DSA_FLAG_DESC_ORDER | DSA_FLAG_DENSE;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

}  // namespace

size_t ws_zero_bytes() { return kWsHeaderBytes + index_select_fused_state_bytes(); }

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The address at which the current device reaches a caller's buffer: the
// pointer itself for device or managed memory, the mapped address for
// page-locked host memory; nullptr for memory the device cannot address
// (pageable host memory) or a pointer the runtime cannot classify.
const void* device_address(const void* p) {
    if (p == nullptr) return nullptr;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();                       // leave no error behind for the caller
        return nullptr;
    }
    switch (a.type) {
        case cudaMemoryTypeDevice:
        case cudaMemoryTypeManaged: return p;
        case cudaMemoryTypeHost: return a.devicePointer;
        default: return nullptr;
    }
}

bool trace_on() {
    static const bool on = [] {
        const char* e = getenv("DSA_TRACE");
        return e != nullptr && e[0] != '\0' && e[0] != '0';
    }();
    return on;
}

dsa_status check_shape(const dsa_shape* s, Shape* out) {
    if (s == nullptr) return DSA_ERR_INVALID_ARG;
    if (s->idx_heads <= 0 || s->idx_dim <= 0 || s->heads <= 0 || s->kv_lora <= 0 ||
        s->rope_dim < 0 || s->top_k <= 0 || s->kpool <= 0)
        return DSA_ERR_INVALID_ARG;
    if (s->top_k % s->kpool != 0) return DSA_ERR_INVALID_ARG;
    if (!isfinite(s->scale) || !(s->scale > 0.f)) return DSA_ERR_INVALID_ARG;
    if (s->dtype != DSA_F32 && s->dtype != DSA_BF16) return DSA_ERR_INVALID_ARG;
    // What this build implements: the layer geometry of the pages.
    if (s->idx_heads > 64 || s->idx_dim != 128 || s->heads != 64 || s->kv_lora != 512 ||
        (s->rope_dim != 0 && s->rope_dim != 64) || s->kpool > 16 || s->top_k > 65536)
        return DSA_ERR_UNSUPPORTED;
    *out = Shape{s->idx_heads, s->idx_dim, s->heads, s->kv_lora, s->rope_dim,
                 s->top_k, s->kpool, s->scale, s->dtype};
    return DSA_OK;
}

// max_n_q: the query count this entry point's grids take (the queries of the
// pool compression are the new tokens, which a prompt may have millions of).
dsa_status check_batch(const dsa_batch* b, const Shape& sh, BatchDev* out,
                       int64_t max_n_q = 65535) {
    if (b == nullptr) return DSA_ERR_INVALID_ARG;
    if (b->n_seq < 0 || b->n_q < 0 || b->max_q_len < 0 || b->max_kv_len < 0 ||
        (b->flags & ~kKnownFlags) != 0 || b->total_rows < 0 || b->total_keys < 0)
        return DSA_ERR_INVALID_ARG;
    if (b->n_q > 0) {
        if (b->n_seq < 1 || b->row_off == nullptr || b->key_off == nullptr || b->q_off == nullptr)
            return DSA_ERR_INVALID_ARG;
        if (b->max_q_len < 1 || b->max_kv_len < b->max_q_len) return DSA_ERR_INVALID_ARG;
        if ((int64_t)b->max_q_len > (int64_t)b->n_q) return DSA_ERR_INVALID_ARG;
        if (b->total_rows < 1) return DSA_ERR_INVALID_ARG;
    }
    if (b->max_kv_len >= ((int64_t)1 << 31)) return DSA_ERR_UNSUPPORTED;
    if (b->n_q > max_n_q) return DSA_ERR_UNSUPPORTED;
    // descending order sorts a query's selected units in shared memory
    if ((b->flags & DSA_FLAG_DESC_ORDER) && sh.top_k / sh.kpool > 16384) return DSA_ERR_UNSUPPORTED;
    *out = BatchDev{b->row_off,    b->key_off,    b->q_off,      b->n_seq,      b->n_q,
                    b->max_q_len,  b->max_kv_len, b->total_rows, b->total_keys, sh.kpool,
                    b->flags};
    return DSA_OK;
}

// The host scalars of a batch, for sizing and planning (no device pointers).
BatchDev host_batch(const dsa_batch* batch, const Shape& sh) {
    return BatchDev{nullptr,           nullptr,           nullptr,           batch->n_seq,
                    batch->n_q,        batch->max_q_len,  batch->max_kv_len, batch->total_rows,
                    batch->total_keys, sh.kpool,          batch->flags};
}

// Keys a query may score at most, and the default score row stride.
int64_t max_keys(const Shape& sh, const BatchDev& b) { return b.max_kv_len / sh.kpool; }
int64_t default_ld(const Shape& sh, const BatchDev& b) {
    const int64_t k = max_keys(sh, b);
    return k < 4 ? 4 : (k + 3) / 4 * 4;
}

struct StepLayout {
    size_t sel, idx_plan, scores, idx, n_sel, attn, total;
};

// Decode-step workspace: header | fused selection state (fixed size, kept zero
// between launches) | indexer plan | scores | selections | counts | attention.
StepLayout step_layout(const Shape& sh, const BatchDev& b) {
    StepLayout L{};
    size_t off = kWsHeaderBytes;
    L.sel = off;
    off = align_up(off + index_select_fused_state_bytes());
    L.idx_plan = off;
    off = align_up(off + index_scores_scratch_bytes(sh, b));
    L.scores = off;
    off = align_up(off + (size_t)b.n_q * default_ld(sh, b) * sizeof(float));
    L.idx = off;
    off = align_up(off + (size_t)b.n_q * sh.index_row_width() * sizeof(int32_t));
    L.n_sel = off;
    off = align_up(off + (size_t)b.n_q * sizeof(int32_t));
    L.attn = off;
    off = align_up(off + sparse_mla_scratch_bytes(sh, b));
    L.total = off;
    return L;
}

// Host-fed decode step: the step's workspace, then the staged query-side
// inputs (indexer queries, head weights, absorbed queries).
struct StageLayout {
    size_t q_idx, w, q_abs, total;
};
StageLayout stage_layout(const Shape& sh, const BatchDev& b) {
    StageLayout L{};
    size_t off = step_layout(sh, b).total;
    L.q_idx = off;
    off = align_up(off + (size_t)b.n_q * sh.idx_heads * sh.idx_dim * sh.elem_bytes());
    L.w = off;
    off = align_up(off + (size_t)b.n_q * sh.idx_heads * sizeof(float));
    L.q_abs = off;
    off = align_up(off + (size_t)b.n_q * sh.heads * sh.width() * sh.elem_bytes());
    L.total = off;
    return L;
}

// Where the scratch of the single-step entry points begins: after the prefix
// the fused decode launch keeps zero, so that one workspace can serve every
// entry point in turn.
size_t scratch_off() { return align_up(ws_zero_bytes()); }

size_t op_bytes(const Shape& sh, const BatchDev& b, int32_t op) {
    switch (op) {
        case DSA_OP_INDEX_SCORES:
            return align_up(scratch_off() + index_scores_scratch_bytes(sh, b));
        case DSA_OP_TOPK_SELECT: return kWsHeaderBytes;
        case DSA_OP_SPARSE_MLA:
            return align_up(scratch_off() + sparse_mla_scratch_bytes(sh, b));
        case DSA_OP_DECODE_STEP: return step_layout(sh, b).total;
        case DSA_OP_DECODE_STEP_HOST: return stage_layout(sh, b).total;
        case DSA_OP_INDEX_SELECT: return step_layout(sh, b).attn;
        case DSA_OP_POOL_COMPRESS: return kWsHeaderBytes;
        case DSA_OP_PROJECT: return kWsHeaderBytes;
        default: return 0;
    }
}

dsa_status check_ws(void* ws, size_t ws_bytes, size_t need) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0 || ws_bytes < need)
        return DSA_ERR_WORKSPACE;
    return DSA_OK;
}

dsa_status cuda_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return DSA_OK;
    if (trace_on()) fprintf(stderr, "[dsa] %s: %s\n", what, cudaGetErrorString(e));
    return DSA_ERR_CUDA;
}

unsigned char* bytes(void* p) { return static_cast<unsigned char*>(p); }

// Steps 1 and 2 into idx / n_sel: the fused launch where it applies, else the
// indexer and the selection; with DSA_FLAG_DESC_ORDER each row is then put in
// descending score order.
cudaError_t enqueue_index_select(const Shape& sh, const BatchDev& b, const StepLayout& lay,
                                 void* ws, const void* q_idx, const float* w, const void* k_idx,
                                 int32_t* idx, int32_t* n_sel, const void* cache,
                                 cudaStream_t st, const char** what) {
    int32_t* err = static_cast<int32_t*>(ws);
    float* scores = reinterpret_cast<float*>(bytes(ws) + lay.scores);
    const int64_t ld = default_ld(sh, b);
    if (index_select_fused_eligible(sh, b)) {
        *what = "index_select_fused";
        return launch_index_select_fused(sh, b, q_idx, w, k_idx, scores, ld, idx, n_sel,
                                         bytes(ws) + lay.sel,
                                         reinterpret_cast<uint32_t*>(bytes(ws) + kWsGridBarOffset),
                                         cache, (int64_t)sh.width() * (int64_t)sh.elem_bytes(),
                                         err, st);
    }
    *what = "index_scores";
    cudaError_t e = launch_index_scores(sh, b, max_keys(sh, b), q_idx, w, k_idx, scores, ld,
                                        bytes(ws) + lay.idx_plan, err, st);
    if (e != cudaSuccess) return e;
    *what = "topk_select";
    e = launch_topk_select(sh, b, scores, ld, idx, n_sel, err, st);
    if (e != cudaSuccess || !(b.flags & DSA_FLAG_DESC_ORDER)) return e;
    *what = "select_order";
    return launch_select_order_desc(sh, b, scores, ld, idx, n_sel, err, st);
}

// Kernels one call of `op` enqueues for this shape and batch bound.
int32_t plan_launches(const Shape& sh, const BatchDev& bh, int32_t op, int32_t splits) {
    if (bh.n_q <= 0) return 0;
    // attention, then the split merge -- except for two tensor-core splits,
    // which merge inside the attention launch (a CTA pair)
    const int32_t attn = splits > 2 || (splits == 2 && !sparse_mla_tc_eligible(sh, bh)) ? 2 : 1;
    const int32_t idx = bh.max_kv_len / sh.kpool > 0
                            ? (index_scores_tc_eligible(sh, bh) ? index_scores_tc_launches(sh, bh) : 1)
                            : 0;
    const int32_t order = (bh.flags & DSA_FLAG_DESC_ORDER) ? 1 : 0;
    const int32_t sel = index_select_fused_eligible(sh, bh) ? 1 : idx + 1 + order;
    switch (op) {
        case DSA_OP_INDEX_SCORES: return idx;
        case DSA_OP_TOPK_SELECT: return 1 + order;
        case DSA_OP_SPARSE_MLA: return attn;
        case DSA_OP_INDEX_SELECT: return sel;
        case DSA_OP_POOL_COMPRESS: return sh.kpool > 1 ? 1 : 0;
        case DSA_OP_PROJECT: return 1;
        case DSA_OP_DECODE_STEP_HOST:                      // the input copy, then the step
            return 1 + ((bh.flags & DSA_FLAG_DENSE) ? attn : sel + attn);
        default: return (bh.flags & DSA_FLAG_DENSE) ? attn : sel + attn;
    }
}

}  // namespace

// Host validation of dsa_decode_step's arguments, everything but the
// workspace: shapes, pointers, alignment, flags.  *ws_need receives the bytes
// of workspace the step needs and *n_q its query count.
dsa_status decode_step_check(const dsa_shape* shape, const dsa_batch* batch, const void* q_idx,
                             const float* w, const void* k_idx, const void* q_abs,
                             const void* cache, const float* out, const float* lse,
                             const int32_t* idx_out, const int32_t* n_sel_out, size_t* ws_need,
                             int32_t* n_q) {
    Shape sh;
    BatchDev b;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    if ((s = check_batch(batch, sh, &b)) != DSA_OK) return s;
    const bool dense = (b.flags & DSA_FLAG_DENSE) != 0;
    if (dense && (idx_out != nullptr || n_sel_out != nullptr)) return DSA_ERR_INVALID_ARG;
    if (b.n_q > 0 && (q_abs == nullptr || cache == nullptr || out == nullptr ||
                      (!dense && (q_idx == nullptr || w == nullptr || k_idx == nullptr))))
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(k_idx) || !aligned16(q_abs) ||
        !aligned16(cache) || !aligned16(out) || !aligned16(idx_out) || !aligned16(n_sel_out) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
        return DSA_ERR_INVALID_ARG;
    if (ws_need != nullptr) *ws_need = step_layout(sh, b).total;
    if (n_q != nullptr) *n_q = b.n_q;
    return DSA_OK;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

int dsa_version(void) { return DSA_ABI_VERSION; }

const char* dsa_status_string(int32_t status) {
    switch (status) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported shape or size";
        case DSA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
        case DSA_ERR_CUDA: return "CUDA runtime or launch error";
        case DSA_ERR_DEVICE: return "a kernel reported invalid data";
        case DSA_ERR_TIMEOUT: return "a bounded device wait timed out";
        default: return "unknown status";
    }
}

int64_t dsa_index_row_width(const dsa_shape* shape) {
    Shape sh;
    if (check_shape(shape, &sh) != DSA_OK) return -1;
    return sh.index_row_width();
}

dsa_status dsa_workspace_size(const dsa_shape* shape, const dsa_batch* batch, int32_t op,
                              size_t* out_bytes) {
    Shape sh;
    if (out_bytes == nullptr) return DSA_ERR_INVALID_ARG;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    // Sizing needs only the host scalars of the batch.
    if (batch == nullptr || batch->n_q < 0 || batch->max_kv_len < 0 ||
        (batch->flags & ~kKnownFlags) != 0)
        return DSA_ERR_INVALID_ARG;
    if (batch->max_kv_len >= ((int64_t)1 << 31) ||
        (batch->n_q > 65535 && op != DSA_OP_POOL_COMPRESS))
        return DSA_ERR_UNSUPPORTED;
    if (op < DSA_OP_INDEX_SCORES || op > DSA_OP_DECODE_STEP_HOST) return DSA_ERR_INVALID_ARG;
    *out_bytes = op_bytes(sh, host_batch(batch, sh), op);
    return DSA_OK;
}

dsa_status dsa_plan(const dsa_shape* shape, const dsa_batch* batch, int32_t op,
                    dsa_plan_info* info) {
    Shape sh;
    if (info == nullptr || batch == nullptr) return DSA_ERR_INVALID_ARG;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    if (batch->n_q < 0 || batch->max_kv_len < 0 || (batch->flags & ~kKnownFlags) != 0)
        return DSA_ERR_INVALID_ARG;
    if (op < DSA_OP_INDEX_SCORES || op > DSA_OP_DECODE_STEP_HOST) return DSA_ERR_INVALID_ARG;
    const BatchDev bh = host_batch(batch, sh);
    int32_t rps = 0, splits = 0;
    plan_attention_splits(sh, bh, &rps, &splits);
    *info = dsa_plan_info{plan_launches(sh, bh, op, splits), splits, rps, 0};
    return DSA_OK;
}

dsa_status dsa_index_scores(const dsa_shape* shape, const dsa_batch* batch, const void* q_idx,
                            const float* w, const void* k_idx, float* scores, int64_t ld,
                            void* ws, size_t ws_bytes, void* stream) {
    Shape sh;
    BatchDev b;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    if ((s = check_batch(batch, sh, &b)) != DSA_OK) return s;
    if (b.n_q > 0 && (q_idx == nullptr || w == nullptr || k_idx == nullptr || scores == nullptr))
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_idx) || !aligned16(k_idx) || !aligned16(w) || !aligned16(scores))
        return DSA_ERR_INVALID_ARG;
    if (ld < max_keys(sh, b) || ld < 1) return DSA_ERR_INVALID_ARG;
    if ((s = check_ws(ws, ws_bytes, op_bytes(sh, b, DSA_OP_INDEX_SCORES))) != DSA_OK) return s;
    int32_t* err = static_cast<int32_t*>(ws);
    return cuda_status(launch_index_scores(sh, b, max_keys(sh, b), q_idx, w, k_idx, scores, ld,
                                           bytes(ws) + scratch_off(), err,
                                           static_cast<cudaStream_t>(stream)),
                       "index_scores");
}

dsa_status dsa_topk_select(const dsa_shape* shape, const dsa_batch* batch, const float* scores,
                           int64_t ld, int32_t* idx, int32_t* n_sel, void* ws, size_t ws_bytes,
                           void* stream) {
    Shape sh;
    BatchDev b;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    if ((s = check_batch(batch, sh, &b)) != DSA_OK) return s;
    if (b.flags & DSA_FLAG_DENSE) return DSA_ERR_INVALID_ARG;   // no selection to make
    if (b.n_q > 0 && (scores == nullptr || idx == nullptr || n_sel == nullptr))
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(scores) || !aligned16(idx) || !aligned16(n_sel)) return DSA_ERR_INVALID_ARG;
    if (ld < max_keys(sh, b) || ld < 1) return DSA_ERR_INVALID_ARG;
    if ((s = check_ws(ws, ws_bytes, op_bytes(sh, b, DSA_OP_TOPK_SELECT))) != DSA_OK) return s;
    int32_t* err = static_cast<int32_t*>(ws);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_topk_select(sh, b, scores, ld, idx, n_sel, err, st);
    if (e == cudaSuccess && (b.flags & DSA_FLAG_DESC_ORDER))
        e = launch_select_order_desc(sh, b, scores, ld, idx, n_sel, err, st);
    return cuda_status(e, "topk_select");
}

dsa_status dsa_sparse_mla_attn(const dsa_shape* shape, const dsa_batch* batch, const void* q_abs,
                               const void* cache, const int32_t* idx, const int32_t* n_sel,
                               float* out, float* lse, void* ws, size_t ws_bytes, void* stream) {
    Shape sh;
    BatchDev b;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    if ((s = check_batch(batch, sh, &b)) != DSA_OK) return s;
    const bool dense = (b.flags & DSA_FLAG_DENSE) != 0;
    if (b.n_q > 0 && (q_abs == nullptr || cache == nullptr || out == nullptr ||
                      (!dense && (idx == nullptr || n_sel == nullptr))))
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_abs) || !aligned16(cache) || !aligned16(out) || !aligned16(idx))
        return DSA_ERR_INVALID_ARG;
    const size_t need = op_bytes(sh, b, DSA_OP_SPARSE_MLA);
    if ((s = check_ws(ws, ws_bytes, need)) != DSA_OK) return s;
    int32_t* err = static_cast<int32_t*>(ws);
    // The previous kernel in the stream is the caller's: the query is read
    // only after it has completed.
    return cuda_status(launch_sparse_mla(sh, b, q_abs, cache, dense ? nullptr : idx,
                                         dense ? nullptr : n_sel, out, lse,
                                         bytes(ws) + scratch_off(), need - scratch_off(), err,
                                         /*q_early=*/false, static_cast<cudaStream_t>(stream)),
                       "sparse_mla_attn");
}

dsa_status dsa_index_prepare(const dsa_shape* shape, int64_t n_vec, const float* x,
                             const int64_t* pos, int32_t rope_dims, double rope_base, void* out,
                             void* stream) {
    Shape sh;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    if (n_vec < 0 || rope_dims < 0 || rope_dims > sh.idx_dim || (rope_dims & 1) ||
        !isfinite(rope_base) || !(rope_base > 0.0))
        return DSA_ERR_INVALID_ARG;
    if (n_vec > 0 && (x == nullptr || out == nullptr || (rope_dims > 0 && pos == nullptr)))
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || (reinterpret_cast<uintptr_t>(pos) & 7) != 0)
        return DSA_ERR_INVALID_ARG;
    return cuda_status(launch_index_prepare(sh, n_vec, x, pos, rope_dims, rope_base, out,
                                            static_cast<cudaStream_t>(stream)),
                       "index_prepare");
}

dsa_status dsa_pool_compress(const dsa_shape* shape, const dsa_batch* batch, const void* cells,
                             const float* pos, void* pool_keys, void* ws, size_t ws_bytes,
                             void* stream) {
    Shape sh;
    BatchDev b;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    if (sh.kpool < 2) return DSA_ERR_INVALID_ARG;          // token mode has no pools
    if ((s = check_batch(batch, sh, &b, 0x7fffffff)) != DSA_OK) return s;
    if (b.n_seq > 65535) return DSA_ERR_UNSUPPORTED;
    if (b.n_q > 0 && (cells == nullptr || pos == nullptr || pool_keys == nullptr))
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(cells) || !aligned16(pos) || !aligned16(pool_keys)) return DSA_ERR_INVALID_ARG;
    if ((s = check_ws(ws, ws_bytes, op_bytes(sh, b, DSA_OP_POOL_COMPRESS))) != DSA_OK) return s;
    if (b.n_q == 0) return DSA_OK;
    int32_t* err = static_cast<int32_t*>(ws);
    return cuda_status(launch_pool_compress(sh, b, cells, pos, pool_keys, err,
                                            static_cast<cudaStream_t>(stream)),
                       "pool_compress");
}

// The projections' common checks: sizes, pointers (16-byte aligned), workspace.
static dsa_status check_projection(const dsa_shape* shape, int32_t n_q, int32_t k_dim, int32_t k_unit,
                            const void* in, const void* w, const void* out, void* ws,
                            size_t ws_bytes, Shape* sh) {
    dsa_status s = check_shape(shape, sh);
    if (s != DSA_OK) return s;
    if (n_q < 0 || k_dim < k_unit || k_dim % k_unit != 0) return DSA_ERR_INVALID_ARG;
    if (k_dim > 512 || n_q > (1 << 24)) return DSA_ERR_UNSUPPORTED;
    if (n_q > 0 && (in == nullptr || w == nullptr || out == nullptr)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(in) || !aligned16(w) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
    return check_ws(ws, ws_bytes, kWsHeaderBytes);
}

dsa_status dsa_absorb_q(const dsa_shape* shape, int32_t n_q, int32_t nope_dim, const void* q,
                        const void* w_uk, void* q_abs, void* ws, size_t ws_bytes, void* stream) {
    Shape sh;
    dsa_status s = check_projection(shape, n_q, nope_dim, 64, q, w_uk, q_abs, ws, ws_bytes, &sh);
    if (s != DSA_OK) return s;
    return cuda_status(launch_absorb_q(sh, n_q, nope_dim, q, w_uk, q_abs,
                                       static_cast<int32_t*>(ws),
                                       static_cast<cudaStream_t>(stream)),
                       "absorb_q");
}

dsa_status dsa_up_project(const dsa_shape* shape, int32_t n_q, int32_t v_dim, const float* o,
                          const void* w_uv, float* out, void* ws, size_t ws_bytes, void* stream) {
    Shape sh;
    dsa_status s = check_projection(shape, n_q, v_dim, 128, o, w_uv, out, ws, ws_bytes, &sh);
    if (s != DSA_OK) return s;
    return cuda_status(launch_up_project(sh, n_q, v_dim, o, w_uv, out, static_cast<int32_t*>(ws),
                                         static_cast<cudaStream_t>(stream)),
                       "up_project");
}

dsa_status dsa_decode_step(const dsa_shape* shape, const dsa_batch* batch, const void* q_idx,
                           const float* w, const void* k_idx, const void* q_abs,
                           const void* cache, float* out, float* lse, int32_t* idx_out,
                           int32_t* n_sel_out, void* ws, size_t ws_bytes, void* stream) {
    size_t need = 0;
    int32_t n_q = 0;
    dsa_status s = decode_step_check(shape, batch, q_idx, w, k_idx, q_abs, cache, out, lse,
                                     idx_out, n_sel_out, &need, &n_q);
    if (s != DSA_OK) return s;
    if ((s = check_ws(ws, ws_bytes, need)) != DSA_OK) return s;
    if (n_q == 0) return DSA_OK;
    Shape sh;
    BatchDev b;
    check_shape(shape, &sh);
    check_batch(batch, sh, &b);
    const StepLayout lay = step_layout(sh, b);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t* err = static_cast<int32_t*>(ws);
    if (trace_on())
        fprintf(stderr, "[dsa] decode_step n_q=%d max_kv=%lld flags=%u ws=%zu\n", b.n_q,
                (long long)b.max_kv_len, b.flags, lay.total);
    if (b.flags & DSA_FLAG_DENSE) {
        // the indexer's A/B switch: every visible row, no scoring or selection
        return cuda_status(launch_sparse_mla(sh, b, q_abs, cache, nullptr, nullptr, out, lse,
                                             bytes(ws) + lay.attn, lay.total - lay.attn, err,
                                             /*q_early=*/false, st),
                           "decode_step/dense attention");
    }
    int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(bytes(ws) + lay.idx);
    int32_t* n_sel = n_sel_out ? n_sel_out : reinterpret_cast<int32_t*>(bytes(ws) + lay.n_sel);
    const char* what = "";
    cudaError_t e = enqueue_index_select(sh, b, lay, ws, q_idx, w, k_idx, idx, n_sel, cache, st,
                                         &what);
    if (e != cudaSuccess) return cuda_status(e, what);
    // The kernel before the attention is this step's selection, which released
    // its dependents only after waiting for the caller's kernels: the query
    // may be loaded before the attention waits for the selection.
    e = launch_sparse_mla(sh, b, q_abs, cache, idx, n_sel, out, lse, bytes(ws) + lay.attn,
                          lay.total - lay.attn, err, /*q_early=*/true, st);
    return cuda_status(e, "decode_step/sparse_mla_attn");
}

dsa_status dsa_decode_step_host(const dsa_shape* shape, const dsa_batch* batch,
                                const void* h_q_idx, const float* h_w, const void* k_idx,
                                const void* h_q_abs, const void* cache, float* h_out,
                                float* h_lse, int32_t* idx_out, int32_t* n_sel_out, void* ws,
                                size_t ws_bytes, void* stream) {
    Shape sh;
    BatchDev b;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    if ((s = check_batch(batch, sh, &b)) != DSA_OK) return s;
    const bool dense = (b.flags & DSA_FLAG_DENSE) != 0;
    // the device's view of the caller's per-step buffers
    const void *q_idx = nullptr, *w = nullptr, *q_abs = nullptr;
    float *out = nullptr, *lse = nullptr;
    if (b.n_q > 0) {
        if (h_q_abs == nullptr || h_out == nullptr || (!dense && (h_q_idx == nullptr || h_w == nullptr)))
            return DSA_ERR_INVALID_ARG;
        q_abs = device_address(h_q_abs);
        out = static_cast<float*>(const_cast<void*>(device_address(h_out)));
        if (q_abs == nullptr || out == nullptr) return DSA_ERR_INVALID_ARG;
        if (!dense) {
            q_idx = device_address(h_q_idx);
            w = device_address(h_w);
            if (q_idx == nullptr || w == nullptr) return DSA_ERR_INVALID_ARG;
        }
        if (h_lse != nullptr) {
            lse = static_cast<float*>(const_cast<void*>(device_address(h_lse)));
            if (lse == nullptr) return DSA_ERR_INVALID_ARG;
        }
    }
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(q_abs)) return DSA_ERR_INVALID_ARG;
    const StageLayout sl = stage_layout(sh, b);
    void* s_q_idx = dense ? nullptr : bytes(ws) + sl.q_idx;
    float* s_w = dense ? nullptr : reinterpret_cast<float*>(bytes(ws) + sl.w);
    void* s_q_abs = bytes(ws) + sl.q_abs;
    int32_t n_q = 0;
    s = decode_step_check(shape, batch, s_q_idx, s_w, k_idx, s_q_abs, cache, out, lse, idx_out,
                          n_sel_out, nullptr, &n_q);
    if (s != DSA_OK) return s;
    if ((s = check_ws(ws, ws_bytes, sl.total)) != DSA_OK) return s;
    if (n_q == 0) return DSA_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int64_t q_idx_vecs =
        dense ? 0 : (int64_t)b.n_q * sh.idx_heads * sh.idx_dim * (int64_t)sh.elem_bytes() / 16;
    const int64_t q_abs_vecs = (int64_t)b.n_q * sh.heads * sh.width() * (int64_t)sh.elem_bytes() / 16;
    const StageSeg a{static_cast<const uint4*>(q_idx), static_cast<uint4*>(s_q_idx), q_idx_vecs};
    const StageSeg c{static_cast<const uint4*>(q_abs), static_cast<uint4*>(s_q_abs), q_abs_vecs};
    const int64_t w_words = dense ? 0 : (int64_t)b.n_q * sh.idx_heads;
    cudaError_t e = launch_stage_inputs(a, c, static_cast<const uint32_t*>(w),
                                        reinterpret_cast<uint32_t*>(s_w), w_words, st);
    if (e != cudaSuccess) return cuda_status(e, "decode_step_host/stage_inputs");
    return dsa_decode_step(shape, batch, s_q_idx, s_w, k_idx, s_q_abs, cache, out, lse, idx_out,
                           n_sel_out, ws, ws_bytes, stream);
}

dsa_status dsa_index_select(const dsa_shape* shape, const dsa_batch* batch, const void* q_idx,
                            const float* w, const void* k_idx, int32_t* idx, int32_t* n_sel,
                            void* ws, size_t ws_bytes, void* stream) {
    Shape sh;
    BatchDev b;
    dsa_status s = check_shape(shape, &sh);
    if (s != DSA_OK) return s;
    if ((s = check_batch(batch, sh, &b)) != DSA_OK) return s;
    if (b.flags & DSA_FLAG_DENSE) return DSA_ERR_INVALID_ARG;   // no selection to make
    if (b.n_q > 0 && (q_idx == nullptr || w == nullptr || k_idx == nullptr || idx == nullptr ||
                      n_sel == nullptr))
        return DSA_ERR_INVALID_ARG;
    if (!aligned16(q_idx) || !aligned16(w) || !aligned16(k_idx) || !aligned16(idx) ||
        !aligned16(n_sel))
        return DSA_ERR_INVALID_ARG;
    const StepLayout lay = step_layout(sh, b);
    if ((s = check_ws(ws, ws_bytes, lay.attn)) != DSA_OK) return s;
    if (b.n_q == 0) return DSA_OK;
    const char* what = "";
    const cudaError_t e = enqueue_index_select(sh, b, lay, ws, q_idx, w, k_idx, idx, n_sel,
                                               nullptr, static_cast<cudaStream_t>(stream), &what);
    return cuda_status(e, what);
}

dsa_status dsa_check_device_error(void* ws, size_t ws_bytes, void* stream, int32_t* code) {
    if (ws == nullptr) {
        // the no-allocation entry point's scratch array on the current device
        dsa_status s = noalloc_scratch(&ws);
        if (s != DSA_OK) return s;
        ws_bytes = DSA_NOALLOC_SCRATCH_BYTES;
    }
    if (ws_bytes < kWsHeaderBytes) return DSA_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_status(e, "check_device_error/sync");
    int32_t words[3] = {0, 0, 0};
    e = cudaMemcpy(words, ws, sizeof(words), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e, "check_device_error/read");
    if (code != nullptr) *code = words[0];
    if (words[0] == 0) return DSA_OK;
    if (trace_on())
        fprintf(stderr, "[dsa] device error %d (detail %d, kernel %d)\n", words[0], words[1],
                words[2]);
    // an interrupted launch may leave the selection state and the grid
    // barrier dirty: start them from zero again
    e = cudaMemset(ws, 0, ws_bytes < ws_zero_bytes() ? ws_bytes : ws_zero_bytes());
    if (e != cudaSuccess) return cuda_status(e, "check_device_error/clear");
    return words[0] == kDevTimeout ? DSA_ERR_TIMEOUT : DSA_ERR_DEVICE;
}

dsa_status dsa_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (ws == nullptr || ws_bytes < kWsHeaderBytes ||
        (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
        return DSA_ERR_WORKSPACE;
    const size_t n = ws_bytes < ws_zero_bytes() ? ws_bytes : ws_zero_bytes();
    return cuda_status(cudaMemsetAsync(ws, 0, n, static_cast<cudaStream_t>(stream)),
                       "workspace_init");
}

dsa_status dsa_workspace_set_wait_budget(void* ws, size_t ws_bytes, uint64_t ns, void* stream) {
    if (ws == nullptr || ws_bytes < kWsHeaderBytes ||
        (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0)
        return DSA_ERR_WORKSPACE;
    // from pageable host memory: staged before the call returns
    const uint64_t v = ns;
    return cuda_status(cudaMemcpyAsync(bytes(ws) + kWsWaitBudgetOffset, &v, sizeof(v),
                                       cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)),
                       "workspace_set_wait_budget");
}

}  // extern "C"
