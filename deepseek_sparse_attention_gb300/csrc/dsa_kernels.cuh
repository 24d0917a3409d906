// dsa_kernels.cuh -- host-side launchers of the DSA kernels (internal to libdsa).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dsa_common.cuh"

namespace dsa {

// Launches `kern` on `st` with programmatic stream serialization allowed, so
// its prologue may overlap the previous kernel's tail (the kernel itself waits,
// with griddepcontrol.wait, before it touches memory the previous kernel
// writes or reads).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Launches `kern` on `st` and returns that launch's own status (unlike a
// <<<>>> launch checked with cudaGetLastError, which would also report an
// error some earlier runtime call left on this thread).
template <typename... KArgs, typename... Args>
cudaError_t launch_plain(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t st, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Bytes at the start of a workspace that must be zero before a decode step:
// the header and the fused selection state (dsa_api.cu).
size_t ws_zero_bytes();

// Host validation of dsa_decode_step's arguments other than the workspace
// (dsa_api.cu); *ws_need gets the workspace bytes the step needs, *n_q its
// query count.
dsa_status decode_step_check(const dsa_shape* shape, const dsa_batch* batch, const void* q_idx,
                             const float* w, const void* k_idx, const void* q_abs,
                             const void* cache, const float* out, const float* lse,
                             const int32_t* idx_out, const int32_t* n_sel_out, size_t* ws_need,
                             int32_t* n_q);

// Device address of the no-allocation entry point's scratch array on the
// current device (dsa_noalloc.cu), looked up once per device.
dsa_status noalloc_scratch(void** out);

// Streaming multiprocessors of the current device (index_scores_tc.cu); grid
// and wave sizes derive from it.
int sm_count();
// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) of `func` on the current
// device unless a limit at least as large was set there before.
cudaError_t ensure_dyn_smem(const void* func, int bytes);

// A tiled TMA descriptor over a bfloat16 tensor of `rank` dimensions, the
// innermost first: dims[rank] in elements, strides[rank - 1] the byte strides
// of dimensions 1.., box[rank] in elements, the 128-byte swizzle, out-of-range
// elements read as zero (index_scores_tc.cu).  False when the driver's encoder
// is missing or refuses the arguments.
bool encode_bf16_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box);

// Validated layer geometry (see dsa_shape in dsa.h).
struct Shape {
    int32_t idx_heads, idx_dim, heads, kv_lora, rope, top_k, kpool;
    float scale;
    int32_t dtype;                                   // DSA_F32 or DSA_BF16
    int32_t width() const { return kv_lora + rope; } // cache row / q_abs head width
    int64_t index_row_width() const { return (int64_t)top_k + kpool - 1; }
    size_t elem_bytes() const { return dtype == DSA_F32 ? 4 : 2; }
};

// Step 1.  scores[q, t] for t < n_keys(q).  bf16 inputs with 32 indexer heads
// run on the tensor cores (index_scores_tc.cu), everything else on CUDA cores
// (index_scores.cu).  `scratch` holds index_scores_scratch_bytes() bytes.
size_t index_scores_scratch_bytes(const Shape& sh, const BatchDev& b);
cudaError_t launch_index_scores(const Shape& sh, const BatchDev& b, int64_t max_keys,
                                const void* q_idx, const float* w, const void* k_idx,
                                float* scores, int64_t ld, void* scratch, int32_t* err,
                                cudaStream_t st);
bool index_scores_tc_eligible(const Shape& sh, const BatchDev& b);
size_t index_scores_tc_scratch_bytes(int32_t n_seq, int32_t n_q);
int32_t index_scores_tc_launches(const Shape& sh, const BatchDev& b);
cudaError_t launch_index_scores_tc(const Shape& sh, const BatchDev& b, const void* q_idx,
                                   const float* w, const void* k_idx, float* scores, int64_t ld,
                                   void* scratch, int32_t* err, cudaStream_t st);

// Step 2.  One selection row per query: one CTA per query (topk_select.cu), or
// a 16-CTA cluster per query when there are few queries (topk_select_cluster.cu).
bool topk_cluster_eligible(const Shape& sh, const BatchDev& b);
cudaError_t launch_topk_select_cluster(const Shape& sh, const BatchDev& b, const float* scores,
                                       int64_t ld, int32_t* idx, int32_t* n_sel, int32_t* err,
                                       cudaStream_t st);
cudaError_t launch_topk_select(const Shape& sh, const BatchDev& b, const float* scores,
                               int64_t ld, int32_t* idx, int32_t* n_sel, int32_t* err,
                               cudaStream_t st);

// Selections in descending score order (select_order.cu): each query's row
// of ascending selections, reordered by (score descending, index ascending);
// in k-pool mode by pool, each pool's rows kept together, the tail last.
cudaError_t launch_select_order_desc(const Shape& sh, const BatchDev& b, const float* scores,
                                     int64_t ld, int32_t* idx, const int32_t* n_sel, int32_t* err,
                                     cudaStream_t st);

// Steps 1 and 2 fused for decode batches (index_select_fused.cu): one
// cooperative launch of the tensor-core indexer that also selects, for at most
// kFusedMaxQ queries each scored as its own group.  `state` holds
// index_select_fused_state_bytes() bytes that must be zero before the first
// launch (each launch leaves them zero); `gbar` two zeroed words for the grid
// barrier, followed in the header by the wait budget.  DSA_FLAG_TWO_LAUNCH
// and DSA_FLAG_DESC_ORDER turn the path off.  `cache` (may be null) is the
// latent cache the step attends over next, rows of `row_bytes`: the rows
// surely selected are prefetched into L2.
constexpr int kFusedMaxQ = 16;
constexpr int kFusedMaxGrid = 256;
bool index_select_fused_eligible(const Shape& sh, const BatchDev& b);
size_t index_select_fused_state_bytes();
cudaError_t launch_index_select_fused(const Shape& sh, const BatchDev& b, const void* q_idx,
                                      const float* w, const void* k_idx, float* scores,
                                      int64_t ld, int32_t* idx, int32_t* n_sel, void* state,
                                      uint32_t* gbar, const void* cache, int64_t row_bytes,
                                      int32_t* err, cudaStream_t st);

// Indexer query / key preparation (index_prepare.cu): out[v] = H rope(x[v],
// pos[v]) for n_vec float32 vectors of 128, rounded to the shape's dtype.
cudaError_t launch_index_prepare(const Shape& sh, int64_t n_vec, const float* x,
                                 const int64_t* pos, int32_t rope_dims, double base, void* out,
                                 cudaStream_t st);

// Pool-key compression (pool_compress.cu): the complete pools of each sequence
// whose last token is one of its new tokens (q_off), from the per-row cells
// [key | gate] (2 x 128 values, dtype) and the per-slot embedding pos
// [kpool, 128] float32, into pool_keys at key_off (dtype).
cudaError_t launch_pool_compress(const Shape& sh, const BatchDev& b, const void* cells,
                                 const float* pos, void* pool_keys, int32_t* err,
                                 cudaStream_t st);

// The projections around the attention (proj.cu): query absorption
// q_abs[q,h] = (q[q,h,:nope] . w_uk[h], q[q,h,nope:]) and the output
// up-projection out[q,h] = w_uv[h] . o[q,h]; bf16 on the tensor cores, float32
// on CUDA cores.
cudaError_t launch_absorb_q(const Shape& sh, int32_t n_q, int32_t nope, const void* q,
                            const void* w_uk, void* q_abs, int32_t* err, cudaStream_t st);
cudaError_t launch_up_project(const Shape& sh, int32_t n_q, int32_t v_dim, const float* o,
                              const void* w_uv, float* out, int32_t* err, cudaStream_t st);

// The per-query inputs of a host-fed decode step copied into the workspace by
// a kernel (stage_inputs.cu): the 16-byte vectors of two segments and the
// 4-byte words of a third, after the wait for the previous kernel.
struct StageSeg {
    const uint4* src;
    uint4* dst;
    int64_t n;                                        // 16-byte vectors
};
cudaError_t launch_stage_inputs(StageSeg a, StageSeg b, const uint32_t* w_src, uint32_t* w_dst,
                                int64_t w_n, cudaStream_t st);

// Step 3.  bf16 rows run on the tensor cores (sparse_mla_tc.cu), float32 rows
// on CUDA cores (sparse_mla.cu).  Row splits per query and the scratch for the
// split-row partials (bytes; 0 if none is needed).  idx == nullptr (and
// n_sel == nullptr) attends over every visible row (DSA_FLAG_DENSE).
// q_early: the query may be loaded before the kernel waits for the previous
// one (only when that kernel is this library's and released its dependents
// after waiting for its own predecessors).
void plan_attention_splits(const Shape& sh, const BatchDev& b, int32_t* rows_per_split,
                           int32_t* n_split);
size_t sparse_mla_scratch_bytes(const Shape& sh, const BatchDev& b);
cudaError_t launch_merge_splits(int32_t n_q, int32_t n_split, const float* part_o,
                                const float* part_ml, float* out, float* lse, cudaStream_t st);
bool sparse_mla_tc_eligible(const Shape& sh, const BatchDev& b);
// Splits of whole row tiles sized by main_rows; rows past them (up to
// max_rows) go to further splits of the same size.
void plan_attention_splits_tc(int32_t n_q, int64_t main_rows, int64_t max_rows,
                              int32_t* rows_per_split, int32_t* n_split);
cudaError_t launch_sparse_mla_tc(const Shape& sh, const BatchDev& b, const void* q_abs,
                                 const void* cache, const int32_t* idx, const int32_t* n_sel,
                                 float* out, float* lse, float* part_o, float* part_ml,
                                 int32_t rps, int32_t n_split, int32_t* err, bool q_early,
                                 cudaStream_t st);
cudaError_t launch_sparse_mla(const Shape& sh, const BatchDev& b, const void* q_abs,
                              const void* cache, const int32_t* idx, const int32_t* n_sel,
                              float* out, float* lse, void* scratch, size_t scratch_bytes,
                              int32_t* err, bool q_early, cudaStream_t st);

}  // namespace dsa
