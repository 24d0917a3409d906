/*
 * dsa.h -- C ABI of the GB300 DeepSeek-Sparse-Attention hot path (libdsa.so).
 *
 * The hot path of one DSA attention layer, for a batch of queries over their
 * sequences' caches:
 *
 *   1. lightning-indexer scores   s_t = sum_h w_h * relu(q_h . k_t)
 *   2. per-query top-k selection  (or top k/kpool pools + the unfilled tail)
 *   3. absorbed-MLA attention     over only the selected 576-wide (512 latent +
 *      64 rope) or 512-wide (NoPE) cache rows, output in the 512-wide latent
 *
 * and two producers of the indexer's inputs: dsa_index_prepare (rope, then the
 * Walsh-Hadamard rotation of projected indexer queries and keys, rounded to the
 * cache's dtype) and dsa_pool_compress (the k-pool keys, one per 4 tokens, from
 * the tokens' [key | gate] cells).
 *
 * Sources (page title -- section):
 *   "GLM-5.x (glm-dsa, glm5next)" (TensorSharp model notes) -- "The block"
 *     (64 query heads, one 576-wide cache row per token, indexer 32 x 128,
 *     top-k 2048, softmax scale 1/16); "The sparse-attention path" (dense
 *     below top-k, mask unmasked at the selected positions); "GLM-5.3-Flash"
 *     table, row "Pooled indexer" (4-token pools, dense below 2051 tokens).
 *   "GLM-5.3-Flash on WASTE" -- "DeepSeek Sparse Attention, k-pool flavour".
 *   "GLM 5.2 in one C file" (blog) -- "Attention: Multi head Latent Attention
 *     With a Tiny KV Cache" (absorbed decode path); "The Lightning Indexer".
 *   "Add GLM-5.3-Flash support" (Strata pull request) -- absorbed NoPE MLA
 *     (K and V are the same 512-wide latent, scale 1/sqrt(256)).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a DEVICE pointer owned by the caller, row-major and
 *   densely packed as documented; the library never allocates, frees or keeps a
 *   pointer past the call.  Scratch memory is the caller's workspace `ws` of
 *   `ws_bytes` bytes (256-byte aligned), sized by dsa_workspace_size().
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Calls only enqueue work on it: they never synchronise, except
 *   dsa_check_device_error().
 * - Arguments are validated on the host before anything is enqueued; a bad
 *   argument returns DSA_ERR_INVALID_ARG (malformed) or DSA_ERR_UNSUPPORTED
 *   (well formed but outside what this build implements) and enqueues nothing.
 *   A failed launch returns DSA_ERR_CUDA.  Conditions only the device can see
 *   (an index out of range, a sequence shorter than its queries) set an error
 *   word in the workspace and the affected output is left as written by the
 *   kernel; dsa_check_device_error() reads and clears it.
 * - No exceptions cross the ABI.  There is no global mutable state beyond
 *   per-device attribute caches, so calls on different streams may run
 *   concurrently as long as they use distinct workspaces.
 *
 * Batch layout (varlen, causal, aligned to the end of each sequence)
 * ------------------------------------------------------------------
 * Sequence s owns cache rows row_off[s] .. row_off[s+1]-1 (kv_len_s rows),
 * indexer keys key_off[s] .. key_off[s+1]-1 and queries q_off[s] .. q_off[s+1]-1
 * (q_len_s queries, q_len_s <= kv_len_s).  Query i of sequence s sees
 *     L = kv_len_s - q_len_s + 1 + i
 * rows, its own row included: decode is q_len_s = 1 (L = kv_len_s); a chunk of
 * prefill is q_len_s > 1.  With kpool == 1 a sequence has one indexer key per
 * row (key_off may equal row_off); with kpool > 1 it has floor(kv_len_s/kpool)
 * pool keys and a query scores the first floor(L/kpool) of them.
 * Selected indices are row indices RELATIVE TO THE SEQUENCE.
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_ABI_VERSION 2

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent shape */
    DSA_ERR_UNSUPPORTED = 2,   /* valid, but outside what this build implements  */
    DSA_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small      */
    DSA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed            */
    DSA_ERR_DEVICE = 5,        /* a kernel reported bad data (error word set)     */
    DSA_ERR_TIMEOUT = 6        /* a bounded device-side wait gave up              */
} dsa_status;

typedef enum {
    DSA_F32 = 0,               /* float32 q_idx, k_idx, q_abs, cache              */
    DSA_BF16 = 1               /* bfloat16 q_idx, k_idx, q_abs, cache             */
} dsa_dtype;

/* Layer geometry.  The weights w and all outputs are float32 in both dtypes. */
typedef struct {
    int32_t idx_heads;         /* indexer heads Hi (32)                           */
    int32_t idx_dim;           /* indexer head width Di (128)                     */
    int32_t heads;             /* MLA query heads H (64); one shared KV head      */
    int32_t kv_lora;           /* latent width, the value width (512)             */
    int32_t rope_dim;          /* rope tail of a cache row (64), 0 for NoPE       */
    int32_t top_k;             /* tokens kept per query (2048)                    */
    int32_t kpool;             /* 1 = token mode; 4 = one pool key per 4 tokens   */
    float scale;               /* softmax scale (1/16 = 1/sqrt(256))              */
    int32_t dtype;             /* a dsa_dtype                                     */
} dsa_shape;

/* Options of a call, in dsa_batch.flags (0 = the defaults; an unknown bit is
 * DSA_ERR_INVALID_ARG):
 *   DSA_FLAG_TWO_LAUNCH  steps 1 and 2 as two launches (the indexer, then the
 *                        selection) even where one cooperative launch would
 *                        run them; the results are the same.
 *   DSA_FLAG_DESC_ORDER  selections in descending score order instead of
 *                        ascending row order ("Add GLM-5.3-Flash support", DSA
 *                        verification: the descending-score order of a selection
 *                        list is a promise of its own): by (score descending,
 *                        index ascending); in k-pool mode by pool, each pool's
 *                        rows together in ascending order, the unfilled tail
 *                        last.  Same set, same count; dense selections too.
 *                        Implies the two-launch plan.  top_k / kpool <= 16384.
 *   DSA_FLAG_DENSE       the indexer's A/B switch ("GLM-5.x (glm-dsa,
 *                        glm5next)", environment knobs: top-k 0 attends densely
 *                        even past the indexer's top-k): attention over every
 *                        visible row of each query, no scoring or selection.
 *                        dsa_decode_step then ignores q_idx, w and k_idx (may be
 *                        NULL) and takes idx_out = n_sel_out = NULL;
 *                        dsa_sparse_mla_attn ignores idx and n_sel;
 *                        dsa_topk_select and dsa_index_select refuse it. */
#define DSA_FLAG_TWO_LAUNCH 0x1u
#define DSA_FLAG_DESC_ORDER 0x2u
#define DSA_FLAG_DENSE 0x4u

/* Batch description.  The three offset arrays are DEVICE arrays of n_seq+1
 * non-decreasing int64 values starting at 0; the host scalars must bound them
 * (they size grids and tensor maps, and the kernels check the offsets against
 * them, setting the error word and skipping a sequence that breaks a bound). */
typedef struct {
    int32_t n_seq;             /* sequences                                        */
    int32_t n_q;               /* queries in total, = q_off[n_seq]                 */
    int32_t max_q_len;         /* host bound: max_s q_len_s                        */
    uint32_t flags;            /* DSA_FLAG_* options of the call (0: defaults)     */
    int64_t max_kv_len;        /* host bound: max_s kv_len_s (< 2^31)              */
    int64_t total_rows;        /* rows of `cache` (bounds row_off[n_seq])          */
    int64_t total_keys;        /* rows of `k_idx` (bounds key_off[n_seq])          */
    const int64_t *row_off;    /* device [n_seq+1] cache-row offsets               */
    const int64_t *key_off;    /* device [n_seq+1] indexer-key / pool-key offsets  */
    const int64_t *q_off;      /* device [n_seq+1] query offsets                   */
} dsa_batch;

/* Library version (DSA_ABI_VERSION) and a static description of a status. */
int dsa_version(void);
const char *dsa_status_string(int32_t status);

/* Width of one query's index row: top_k + kpool - 1 when the query's selection
 * is sparse, and the dense selection of a query with L <= that bound also fits. */
int64_t dsa_index_row_width(const dsa_shape *shape);

/* Bytes of workspace each entry point needs for this shape and batch bound
 * (host-only, enqueues nothing).  `op` is one of the DSA_OP_* values.  The
 * same workspace may be reused by consecutive calls on one stream. */
#define DSA_OP_INDEX_SCORES 0
#define DSA_OP_TOPK_SELECT 1
#define DSA_OP_SPARSE_MLA 2
#define DSA_OP_DECODE_STEP 3
#define DSA_OP_INDEX_SELECT 4
#define DSA_OP_POOL_COMPRESS 5
#define DSA_OP_PROJECT 6
#define DSA_OP_DECODE_STEP_HOST 7
dsa_status dsa_workspace_size(const dsa_shape *shape, const dsa_batch *batch, int32_t op,
                              size_t *bytes);

/* Execution plan of one entry point for this shape and batch bound (host-only,
 * enqueues nothing): how many kernels it launches, and into how many row
 * splits the attention step divides each query's selection. */
typedef struct {
    int32_t kernel_launches;   /* kernels one call enqueues                        */
    int32_t attn_splits;       /* row splits per query in the attention step       */
    int32_t attn_rows_per_split;
    int32_t reserved;
} dsa_plan_info;
dsa_status dsa_plan(const dsa_shape *shape, const dsa_batch *batch, int32_t op,
                    dsa_plan_info *info);

/* Zeroes the start of the workspace on `stream`: the 256-byte header (device
 * error word, grid barrier, wait budget, launch count) and the decode step's selection state
 * that follows it (DSA_WS_ZERO_BYTES in all, or the whole of a smaller workspace).
 * Call once on a freshly allocated workspace that was not allocated
 * zero-filled; after that every completed call leaves this region as it must
 * be (no entry point uses it as scratch, so one workspace may serve all of
 * them in turn), and dsa_check_device_error() re-zeroes it when a kernel
 * reported an error.  `ws` must be 256-byte aligned and at least 256 bytes. */
#define DSA_WS_ZERO_BYTES (256u + 16u * 25604u * 4u + 16u * 256u * 8u)
dsa_status dsa_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Step 1: lightning-indexer scores ("GLM 5.2 in one C file", "The Lightning
 * Indexer"; "GLM-5.x", "The block", row "DSA indexer").
 *   q_idx  [n_q, idx_heads, idx_dim]   dtype
 *   w      [n_q, idx_heads]            float32
 *   k_idx  [key_off[n_seq], idx_dim]   dtype (token keys, or pool keys)
 *   scores [n_q, ld] float32 out: scores[q, t] = sum_h w[q,h] *
 *          relu(q_idx[q,h,:] . k_idx[key_off[s]+t, :]) for t < n_keys(q),
 *          where n_keys(q) = floor(L/kpool); entries t >= n_keys(q) are not written.
 *   ld >= floor(max_kv_len / kpool).  The page's positive factors 1/sqrt(Di) and
 *   1/sqrt(Hi) are not applied: they fold into w and do not change a selection. */
dsa_status dsa_index_scores(const dsa_shape *shape, const dsa_batch *batch, const void *q_idx,
                            const float *w, const void *k_idx, float *scores, int64_t ld,
                            void *ws, size_t ws_bytes, void *stream);

/* Step 2: per-query selection from the scores of step 1.
 *   kpool == 1: if L <= top_k every row 0..L-1; else the top_k rows in the
 *   order (score descending, index ascending) -- ties go to the lower index.
 *   kpool > 1 ("GLM-5.3-Flash on WASTE", k-pool flavour): with n_pool =
 *   floor(L/kpool) and tail = L mod kpool, if n_pool <= top_k/kpool every row
 *   0..L-1; else the top top_k/kpool pools in the same order, expanded to their
 *   kpool rows, followed by the tail rows kpool*n_pool .. L-1.
 *   idx   [n_q, dsa_index_row_width(shape)] int32 out: ascending row indices,
 *         unused slots set to -1;
 *   n_sel [n_q] int32 out: number of valid entries (dense: L; sparse: top_k
 *         plus the tail).
 * A dense selection always fits the row width: it has L <= top_k + kpool - 1
 * rows. */
dsa_status dsa_topk_select(const dsa_shape *shape, const dsa_batch *batch, const float *scores,
                           int64_t ld, int32_t *idx, int32_t *n_sel, void *ws, size_t ws_bytes,
                           void *stream);

/* Steps 1 and 2 together: the selection dsa_topk_select makes from the scores
 * dsa_index_scores computes, without returning the scores (they stay in the
 * workspace, or never leave the chip).  Arguments as for those two calls;
 * idx / n_sel as for dsa_topk_select; the workspace is sized with
 * DSA_OP_INDEX_SELECT.  Decode batches of at most 16 queries with bf16 inputs
 * and 32 indexer heads run as one cooperative launch, under the conditions
 * stated at dsa_decode_step; other batches as the two launches. */
dsa_status dsa_index_select(const dsa_shape *shape, const dsa_batch *batch, const void *q_idx,
                            const float *w, const void *k_idx, int32_t *idx, int32_t *n_sel,
                            void *ws, size_t ws_bytes, void *stream);

/* Indexer query / key preparation ("GLM-5.x (glm-dsa, glm5next)", "The
 * sparse-attention path": past top-k the indexer applies rope, then a
 * Walsh-Hadamard rotation -- an orthonormal involution on both sides of the dot
 * product, so the scores are unchanged in exact arithmetic while the rounding of
 * the 16-bit key cache is spread evenly over the 128 dimensions; "The block",
 * row "RoPE": NORM mode, base 8e6).
 *   x   [n_vec, idx_dim] float32: projected indexer vectors -- keys (one per
 *       token) or queries (one row per head, idx_heads rows per query)
 *   pos [n_vec] int64: each row's token position (a query's heads share one);
 *       may be NULL when rope_dims == 0
 *   out [n_vec, idx_dim] dtype: H . rope(x[v], pos[v]), rounded -- the q_idx or
 *       k_idx layout of the other entry points
 * rope rotates the adjacent pairs (2i, 2i+1) of the first rope_dims dimensions
 * (even, 0..idx_dim) by pos * rope_base^(-2i / rope_dims); H is the orthonormal
 * Sylvester-Hadamard matrix of order idx_dim, H[i][j] = (-1)^popcount(i & j) /
 * sqrt(idx_dim).  Which of the indexer's 128 dimensions carry rope is not stated
 * on the pages: it is the caller's rope_dims (64 = the first half, the MLA rope
 * width, is the reading this library's tests use).  float32 arithmetic; the
 * rope angle is exact modulo one turn (each pair's rate theta_i / 2 pi as a
 * 64-bit binary fraction, times the position), so large positions lose nothing.
 * x and out 16-byte aligned, pos 8-byte aligned (else DSA_ERR_INVALID_ARG).  No
 * workspace; nothing the device can find wrong. */
dsa_status dsa_index_prepare(const dsa_shape *shape, int64_t n_vec, const float *x,
                             const int64_t *pos, int32_t rope_dims, double rope_base, void *out,
                             void *stream);

/* Pool-key compression for the k-pool indexer ("GLM-5.x (glm-dsa, glm5next)",
 * table "GLM-5.3-Flash", row "Pooled indexer": each cell caches [key|gate], and
 * a softmax over the gates plus a per-slot position embedding compresses each
 * pool; "GLM-5.3-Flash on WASTE", "DeepSeek Sparse Attention, k-pool flavour":
 * one 128-wide key per pool of kpool tokens, computed once, when the pool's last
 * token arrives).  Requires kpool >= 2.
 *   cells     [total_rows, 2 * idx_dim] dtype: one cell per cache row (token),
 *             its key then its gate; the cells of sequence s start at
 *             row_off[s], like its cache rows
 *   pos       [kpool, idx_dim] float32: position embedding of slot i, the
 *             place of a token in its pool
 *   pool_keys [total_keys, idx_dim] dtype, in/out: the k_idx array of the
 *             k-pool entry points (pool j of sequence s at key_off[s] + j)
 * For every sequence s (kv_len_s rows, the last q_len_s of them new) and every
 * pool j with floor((kv_len_s - q_len_s) / kpool) <= j < floor(kv_len_s / kpool)
 * -- the complete pools whose last token is new --
 *     z_i[c] = gate(kpool*j + i)[c] + pos[i][c]            (i < kpool)
 *     pool_keys[key_off[s] + j][c] = sum_i softmax_i(z[c]) * key(kpool*j + i)[c]
 * computed in float32 and rounded to dtype; no other pool key is written and no
 * other cell is read.  A gate of -inf masks its slot (weight 0), and a channel
 * whose slots are all masked gets 0; gates are otherwise finite (+inf and NaN
 * give NaN).  A decode step (q_len 1) writes a key exactly when its
 * token completes a pool; a chunk writes the pools it completes; q_len_s =
 * kv_len_s writes them all.  The batch's queries are only the new tokens here:
 * n_q = q_off[n_seq] (not limited to 65535 for this entry point), max_q_len
 * bounds each q_len_s.  A sequence whose offsets
 * break the host bounds is skipped and sets the error word.  The gate has the
 * key's width and the embedding is added to the gate logits: the pages name the
 * parts of the compressor, not its formula.  Workspace: dsa_workspace_size
 * (DSA_OP_POOL_COMPRESS), the 256-byte header (the error word). */
dsa_status dsa_pool_compress(const dsa_shape *shape, const dsa_batch *batch, const void *cells,
                             const float *pos, void *pool_keys, void *ws, size_t ws_bytes,
                             void *stream);

/* Query absorption, the producer of step 3's query ("GLM-5.x (glm-dsa,
 * glm5next)", "The block": the per-head key decompression of MLA is folded into
 * the query, attn_k_b; "GLM 5.2 in one C file", "Attention: Multi head Latent
 * Attention With a Tiny KV Cache": the key up-projection is absorbed into the
 * query, which then scores the cached latents directly).
 *   q     [n_q, heads, nope_dim + rope_dim] dtype: per head the no-rope part
 *         of the query, then its (already rotated) rope part
 *   w_uk  [heads, nope_dim, kv_lora] dtype: row d of head h is the latent-space
 *         image of no-rope dimension d
 *   q_abs [n_q, heads, kv_lora + rope_dim] dtype out: the q_abs of step 3,
 *         q_abs[q,h,i] = sum_d q[q,h,d] * w_uk[h,d,i] for i < kv_lora, rounded
 *         to dtype; then the rope part copied
 * nope_dim a multiple of 64 up to 512 (192 for GLM-5.x: a 256-wide key head is
 * 192 no-rope + 64 rope dimensions).  float32 accumulation.  Pointers 16-byte
 * aligned.  Workspace: DSA_OP_PROJECT (the error word). */
dsa_status dsa_absorb_q(const dsa_shape *shape, int32_t n_q, int32_t nope_dim, const void *q,
                        const void *w_uk, void *q_abs, void *ws, size_t ws_bytes, void *stream);

/* Output up-projection, the consumer of step 3's output ("GLM-5.x", "The
 * block": the value decompression folded into the output, attn_v_b; "GLM 5.2
 * in one C file": the pooled latent is projected to the head's value space).
 *   o     [n_q, heads, kv_lora] float32: step 3's out
 *   w_uv  [heads, v_dim, kv_lora] dtype: row v of head h maps the latent to
 *         value dimension v
 *   out   [n_q, heads, v_dim] float32 out: out[q,h,v] = sum_i w_uv[h,v,i] * o[q,h,i]
 * v_dim a multiple of 128 up to 512 (256 for GLM-5.x).  bf16 weights multiply
 * o split into two bf16 parts (o to about 2^-16 relative), float32
 * accumulation.  Pointers 16-byte aligned.  Workspace: DSA_OP_PROJECT. */
dsa_status dsa_up_project(const dsa_shape *shape, int32_t n_q, int32_t v_dim, const float *o,
                          const void *w_uv, float *out, void *ws, size_t ws_bytes, void *stream);

/* Step 3: absorbed-MLA attention over the selected rows ("GLM 5.2 in one C
 * file", MLA decode path; "GLM-5.x", "The block").
 *   q_abs [n_q, heads, kv_lora + rope_dim] dtype (absorbed latent part, then rope)
 *   cache [row_off[n_seq], kv_lora + rope_dim] dtype
 *   idx, n_sel as produced by dsa_topk_select (any order is accepted; each
 *   index must satisfy 0 <= idx < L, otherwise the error word is set and the
 *   row is skipped)
 *   out [n_q, heads, kv_lora] float32: o = sum_j softmax_j(z)_j * latent_j with
 *       z_j = scale * (q_abs . row_j) over the full row width
 *   lse [n_q, heads] float32 or NULL: log sum_j exp(z_j).
 * A query with n_sel == 0 gets out = 0 and lse = -inf.  With DSA_FLAG_DENSE
 * every visible row 0..L-1 is attended over and idx / n_sel are not read.
 * `lse` may be unaligned only to 4 bytes. */
dsa_status dsa_sparse_mla_attn(const dsa_shape *shape, const dsa_batch *batch, const void *q_abs,
                               const void *cache, const int32_t *idx, const int32_t *n_sel,
                               float *out, float *lse, void *ws, size_t ws_bytes, void *stream);

/* The whole hot path for every query of the batch: steps 1-3 in one call.
 * Scores and selections live in the workspace unless idx_out / n_sel_out are
 * given (then the selection is also written there, laid out as for
 * dsa_topk_select).  Works for decode and for chunks of prefill alike.
 * Decode batches of at most 16 queries with bf16 inputs and 32 indexer heads
 * run steps 1 and 2 as one cooperative launch whose CTAs wait on one another
 * through the workspace (a grid barrier and per-query histograms and
 * candidate counters that each launch leaves as it found them): the workspace must have been zeroed once
 * (dsa_workspace_init, or allocated zero-filled), and two calls sharing one
 * workspace must not run concurrently.  The launch needs every CTA resident at
 * once; DSA_ERR_CUDA is returned if the device cannot give it that.  Its CTAs'
 * waits on one another give up after the workspace's wait budget
 * (dsa_workspace_set_wait_budget; 2 s by default), recording DSA_ERR_TIMEOUT.
 * DSA_FLAG_TWO_LAUNCH selects the two-launch path (the results are the same);
 * DSA_FLAG_DESC_ORDER orders idx_out by score; DSA_FLAG_DENSE attends over
 * every visible row (see the flags above). */
dsa_status dsa_decode_step(const dsa_shape *shape, const dsa_batch *batch, const void *q_idx,
                           const float *w, const void *k_idx, const void *q_abs,
                           const void *cache, float *out, float *lse, int32_t *idx_out,
                           int32_t *n_sel_out, void *ws, size_t ws_bytes, void *stream);

/* dsa_decode_step fed from host memory: the step's per-query inputs are read
 * from, and its output written to, buffers the host fills and reads each step
 * (the cache, the keys and the batch arrays stay on the device).  The pages
 * have no counterpart: this is a convenience of this library, for a caller
 * whose queries come from the host.
 *   h_q_idx, h_w, h_q_abs  as q_idx, w, q_abs of dsa_decode_step, in
 *       page-locked host memory that the device can address (cudaHostAlloc /
 *       cudaMallocHost, or cudaHostRegister'ed and mapped), or device memory.
 *       The call's first kernel copies them into the workspace -- a kernel,
 *       not a copy-engine transfer, so that the copy is one more link of the
 *       step's chain of programmatically dependent launches -- and the step
 *       reads them there.  16-byte aligned.
 *   h_out, h_lse (may be NULL)  as out, lse, likewise host (or device)
 *       memory: the step's last kernel writes them there directly.
 *   k_idx, cache, idx_out, n_sel_out, flags  as for dsa_decode_step (device
 *       memory).
 * Results are those of dsa_decode_step on the same inputs, bit for bit.  The
 * workspace is sized with DSA_OP_DECODE_STEP_HOST: the step's, then room for
 * the staged inputs; its zeroing and wait budget as for dsa_decode_step.  A
 * buffer the device cannot address (pageable host memory, an unknown pointer)
 * gives DSA_ERR_INVALID_ARG; every argument is checked before anything is
 * enqueued.  The input buffers may be refilled, and the outputs read, once the
 * stream has passed the call. */
dsa_status dsa_decode_step_host(const dsa_shape *shape, const dsa_batch *batch,
                                const void *h_q_idx, const float *h_w, const void *k_idx,
                                const void *h_q_abs, const void *cache, float *h_out,
                                float *h_lse, int32_t *idx_out, int32_t *n_sel_out, void *ws,
                                size_t ws_bytes, void *stream);

/* dsa_decode_step for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a convenience of this library.  Some callers may
 * not call cudaMalloc where they run the layer -- while a framework captures
 * the stream into a CUDA graph, inside a host engine that gives a plugin only
 * its input and output buffers, or in a loop that cannot afford cudaMalloc's
 * implicit device synchronisation.  This entry point takes no workspace: its
 * scratch is one fixed array of DSA_NOALLOC_SCRATCH_BYTES compiled into the
 * library, held by every GPU that loads it until the process exits, and it
 * calls no allocator.
 *   Arguments and results are those of dsa_decode_step without ws/ws_bytes.
 *   Returns DSA_ERR_UNSUPPORTED when the step needs more scratch than the
 *   array holds (dsa_workspace_size(DSA_OP_DECODE_STEP) > the limit; a batch-1
 *   decode at 131072 tokens needs under 6 MiB).
 *   Every argument is checked before anything is enqueued.
 *   The first call on a device looks up the array's device address (with that
 *   device current) and caches it; make that first call before any stream
 *   capture.  All calls share the array and it keeps the previous call's
 *   contents; each call zeroes its first DSA_WS_ZERO_BYTES on `stream` first.  Calls whose
 *   work overlaps on the GPU (other streams, other threads) race on the array:
 *   serialise them.  Device-side checks record into the array's error word:
 *   dsa_check_device_error(NULL, 0, stream, &code) reads and clears it. */
#define DSA_NOALLOC_SCRATCH_BYTES (8u << 20)
dsa_status dsa_decode_step_noalloc(const dsa_shape *shape, const dsa_batch *batch,
                                   const void *q_idx, const float *w, const void *k_idx,
                                   const void *q_abs, const void *cache, float *out, float *lse,
                                   int32_t *idx_out, int32_t *n_sel_out, void *stream);

/* Synchronises `stream`, then reads and clears the workspace error word.
 * *code (may be NULL) receives the first device-side error recorded (0 if
 * none).  Returns DSA_OK, DSA_ERR_DEVICE / DSA_ERR_TIMEOUT when a kernel
 * reported one, or DSA_ERR_CUDA.  After an error it re-zeroes the workspace's
 * first DSA_WS_ZERO_BYTES (an interrupted launch may leave its selection state
 * dirty).  ws == NULL reads the scratch array of dsa_decode_step_noalloc on the
 * current device. */
dsa_status dsa_check_device_error(void *ws, size_t ws_bytes, void *stream, int32_t *code);

/* Sets the budget, in nanoseconds, of every wait of a CTA on other CTAs in the
 * kernels that use this workspace (the fused decode launch's grid barriers);
 * 0 restores the default of 2 s.  A wait that runs out records DSA_ERR_TIMEOUT
 * in the error word and its kernel winds down: nothing waits forever.  The
 * value lives in the workspace header, so dsa_workspace_init and the clearing
 * after an error restore the default.  Enqueued on `stream` (a copy from host
 * memory: not for use while the stream is being captured). */
dsa_status dsa_workspace_set_wait_budget(void *ws, size_t ws_bytes, uint64_t ns, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H */
