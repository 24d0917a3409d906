/*
 * dsa_oracle.h -- host oracle for the DeepSeek-Sparse-Attention hot path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the smoke check
 * of the package entry point and the CPU-baseline leg of the benchmark may load
 * or call this library.  The CUDA library never includes, links or calls it, and
 * it shares no code, header, table or helper with the CUDA library.
 *
 * Every function is a direct, unblocked restatement of what the method computes,
 * accumulated in double precision from float inputs (bf16 inputs are widened to
 * float exactly by the caller).  All sizes are element counts; all pointers are
 * host pointers owned by the caller.  Functions return 0 on success and a
 * negative value on a bad argument; they never allocate memory that outlives the
 * call.
 *
 * Sources (page title -- section):
 *   [GLM-DOC]   "GLM-5.x (glm-dsa, glm5next)" (TensorSharp model notes) --
 *               "The block" table; "The sparse-attention path";
 *               "GLM-5.3-Flash (glm5next)" table, row "Pooled indexer".
 *   [WASTE]     "GLM-5.3-Flash on WASTE" -- "DeepSeek Sparse Attention,
 *               k-pool flavour"; "What is checked".
 *   [ONE-C]     "GLM 5.2 in one C file" (blog) -- "Attention: Multi head Latent
 *               Attention With a Tiny KV Cache"; "The Lightning Indexer: Sparse
 *               Attention When It Helps".
 *   [STRATA]    "Add GLM-5.3-Flash support" (Strata pull request) -- "What a
 *               glm5-next block has that nothing else in the engine does";
 *               "Known gaps".
 */
#ifndef DSA_ORACLE_H
#define DSA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Threads the parallel loops below use: sets them to n when n > 0, and
 * returns the number in effect (timing support; no arithmetic). */
int oracle_set_threads(int32_t n);

/* Lightning-indexer score of n_keys keys against one query.
 *   q      [heads * dim]   indexer query, head-major
 *   w      [heads]         per-head weights
 *   keys   [n_keys * dim]  indexer keys (or pool keys), one row per key
 *   scores [n_keys]        out: s_t = sum_h w_h * max(0, sum_i q[h,i]*keys[t,i])
 * [ONE-C] "The Lightning Indexer": ReLU'd per-head dot product, weighted sum over
 * heads.  The page's positive factors 1/sqrt(dim) and 1/sqrt(heads) are omitted:
 * ReLU is positively homogeneous, so they fold into w and cannot change a
 * selection.  [GLM-DOC] "The block", row "DSA indexer": 32 heads x 128. */
int oracle_index_scores(const float *q, const float *w, const float *keys,
                        int64_t n_keys, int32_t heads, int32_t dim, double *scores);

/* Top-k selection over n scores.
 *   If n <= k every index 0..n-1 is selected (the dense shortcut, [GLM-DOC]
 *   "The sparse-attention path"; [ONE-C] "The Lightning Indexer").
 *   Otherwise the k indices that come first in the total order
 *   (score descending, index ascending) -- ties go to the lower index.
 *   idx [>= min(n,k)] receives the selection in ascending index order;
 *   *n_sel receives min(n, k). */
int oracle_topk(const double *scores, int64_t n, int64_t k, int32_t *idx, int64_t *n_sel);

/* k-pool selection for a query that sees L tokens, given the scores of its
 * n_pool = floor(L / kpool) complete pools ([WASTE] "DeepSeek Sparse Attention,
 * k-pool flavour"; [GLM-DOC] row "Pooled indexer").
 *   If n_pool <= k / kpool, every token 0..L-1 is selected (dense).
 *   Otherwise the top k/kpool pools (oracle_topk order) are expanded to their
 *   kpool member tokens and the tail tokens kpool*n_pool .. L-1 of the unfilled
 *   pool are appended ([STRATA] "Known gaps": the tail is appended).
 *   idx [>= k + kpool - 1] receives ascending token indices; *n_sel the count.
 * kpool == 1 is token mode and equals oracle_topk. */
int oracle_kpool_select(const double *pool_scores, int64_t L, int64_t k, int32_t kpool,
                        int32_t *idx, int64_t *n_sel);

/* A selection put in descending score order ([STRATA] "DSA verification":
 * the descending-score order of a selection list is a promise of its own).
 *   unit_scores [n_units]  the query's scores: one per token (kpool == 1) or
 *                          per pool
 *   sel [n_sel]            a selection as oracle_kpool_select emits it
 *                          (ascending; in k-pool mode whole pools, then the
 *                          L mod kpool tail rows)
 *   out [n_sel]            out: the same rows with the units (tokens, or
 *                          pools with their kpool rows in ascending order)
 *                          sorted by score descending, ties by ascending unit
 *                          (the selection's own tie rule), the tail last in
 *                          ascending order. */
int oracle_order_desc(const double *unit_scores, int64_t n_units, const int32_t *sel,
                      int64_t n_sel, int64_t L, int32_t kpool, int32_t *out);

/* Absorbed-MLA attention of one query over the selected cache rows.
 *   q_abs [heads * width]     absorbed query (latent part then rope part)
 *   rows  [n_rows * width]    latent cache, width = kv_lora (+ rope)
 *   idx   [n_sel]             selected row indices (any order, each < n_rows)
 *   out   [heads * dv]        out: o[h,c] = sum_j p[h,j] * rows[idx_j, c], c < dv
 *   lse   [heads] or NULL     out: log sum_j exp(z[h,j])
 * with z[h,j] = scale * sum_{c<width} q_abs[h,c] * rows[idx_j, c] and
 * p = softmax_j(z).  [ONE-C] "Attention: Multi head Latent Attention ...":
 * absorbed score against the latent plus the rope dot, scaled, softmax, pooled
 * latent.  [GLM-DOC] "The block": scale 1/16, cache row 512 + 64.  [STRATA]:
 * the value of a NoPE row is the 512-wide latent itself. */
int oracle_sparse_mla(const float *q_abs, const float *rows, int64_t n_rows, int32_t heads,
                      int32_t width, int32_t dv, double scale, const int32_t *idx,
                      int64_t n_sel, double *out, double *lse);

/* The same attention written the way [GLM-DOC] "The sparse-attention path"
 * states it: dense attention over all n_rows rows with the logit of every row
 * whose mask byte is 0 set to minus infinity. */
int oracle_dense_masked_mla(const float *q_abs, const float *rows, int64_t n_rows,
                            int32_t heads, int32_t width, int32_t dv, double scale,
                            const uint8_t *mask, double *out, double *lse);

/* One query through the whole path: indexer scores over its keys (L token
 * keys when kpool == 1, floor(L/kpool) pool keys otherwise), selection, and
 * attention over the selected rows of its L cache rows.
 *   scores_out [n_keys] or NULL, idx [k + kpool - 1], n_sel, out [heads*dv],
 *   lse [heads] or NULL. */
int oracle_decode_step(const float *q_idx, const float *w, const float *keys,
                       int32_t idx_heads, int32_t idx_dim, const float *q_abs,
                       const float *rows, int64_t L, int32_t heads, int32_t width,
                       int32_t dv, double scale, int64_t k, int32_t kpool,
                       double *scores_out, int32_t *idx, int64_t *n_sel,
                       double *out, double *lse);

/* Pool-key compression ([GLM-DOC] "GLM-5.3-Flash (glm5next)" table, row
 * "Pooled indexer": each cell caches [key|gate], a softmax over the gates plus
 * a per-slot position embedding compresses each pool; [WASTE] "DeepSeek Sparse
 * Attention, k-pool flavour": one 128-wide key per pool of kpool tokens, made
 * once, when the pool's last token arrives).
 *   cells [n_pools * kpool * 2 * dim]  the pools' cells in token order, each
 *                                      cell = key[dim] then gate[dim]
 *   pos   [kpool * dim]                position embedding of slot i (the
 *                                      cell's place in its pool)
 *   out   [n_pools * dim]              out: for pool p and channel c,
 *     z_i = gate_i[c] + pos[i][c]  (i < kpool: the pool's cells in order)
 *     a_i = exp(z_i) / sum_j exp(z_j)          softmax over the slots
 *     out[p][c] = sum_i a_i * key_i[c]
 * A logit of -inf masks its slot (weight 0); a channel whose slots are all
 * masked gets 0 (an empty weighted sum).  Gates are otherwise finite.
 * Readings (the pages name the parts, not the formula): the gate has the key's
 * width and there is one softmax per key dimension -- [STRATA] "Tests" lists
 * one softmax over the whole pool block instead of per key-dim as a rival
 * reading -- and the position embedding is added to the gate logits inside the
 * softmax. */
int oracle_pool_compress(const float *cells, int64_t n_pools, const float *pos, int32_t kpool,
                         int32_t dim, double *out);

/* The pools a call writes for a sequence of L tokens whose last q_len tokens
 * are new ([WASTE]: a pool's key is computed once, when its last token
 * arrives): pools j0 <= j < j1 with j0 = floor((L - q_len) / kpool) and
 * j1 = floor(L / kpool) -- the complete pools whose last token is new. */
int oracle_new_pools(int64_t L, int64_t q_len, int32_t kpool, int64_t *j0, int64_t *j1);

/* Walsh-Hadamard rotation of one n-vector (n a power of two): out = H x with
 * H[i][j] = (-1)^popcount(i & j) / sqrt(n), the orthonormal Sylvester-Hadamard
 * matrix -- symmetric and its own inverse ([GLM-DOC] "The sparse-attention
 * path": the indexer applies a Walsh-Hadamard rotation, an orthonormal
 * involution, to both sides of its dot product before the keys are rounded to
 * the cache's 16-bit format).  The plain matrix-vector product. */
int oracle_hadamard(const double *x, int32_t n, double *out);

/* Rotary position embedding of one dim-vector at position pos ([GLM-DOC] "The
 * block", row "RoPE": NORM mode, base 8e6): for each pair i < rope_dims / 2 of
 * adjacent dimensions (2i, 2i+1), theta_i = base^(-2i / rope_dims) and
 * a = pos * theta_i,
 *     out[2i]   = x[2i] cos a - x[2i+1] sin a
 *     out[2i+1] = x[2i] sin a + x[2i+1] cos a;
 * dimensions rope_dims .. dim-1 are copied. */
int oracle_rope(const float *x, int32_t dim, int32_t rope_dims, double base, int64_t pos,
                double *out);

/* Indexer query / key preparation ([GLM-DOC] "The sparse-attention path": past
 * top-k the indexer applies rope, then the Walsh-Hadamard rotation, then
 * scores): out[v] = H (rope(x[v], pos[v])) for each of n vectors of dim. */
int oracle_index_prepare(const float *x, const int64_t *pos, int64_t n, int32_t dim,
                         int32_t rope_dims, double base, double *out);

/* Query absorption ([ONE-C] "Attention: Multi head Latent Attention With a
 * Tiny KV Cache": the key up-projection is absorbed into the query, which then
 * scores the latents directly; [GLM-DOC] "The block": the per-head K
 * decompression is folded into the query, attn_k_b).
 *   q     [heads * (nope + rope)]         per head: the nope part, then the
 *                                         (already rotated) rope part
 *   w_uk  [heads * nope * kv_lora]        per head: row d is the latent-space
 *                                         image of nope dimension d
 *   q_abs [heads * (kv_lora + rope)]      out: q_abs[h][i] = sum_d q[h][d] *
 *                                         w_uk[h][d][i] for i < kv_lora, then the
 *                                         rope part copied */
int oracle_absorb_q(const float *q, const float *w_uk, int32_t heads, int32_t nope, int32_t rope,
                    int32_t kv_lora, double *q_abs);

/* Output up-projection ([ONE-C]: the pooled latent is mapped to the head's value
 * space; [GLM-DOC] "The block": the V decompression folded into the output,
 * attn_v_b).
 *   o     [heads * kv_lora]     attention output in the latent
 *   w_uv  [heads * v_dim * kv_lora]  per head: row v maps the latent to value dim v
 *   out   [heads * v_dim]       out: out[h][v] = sum_i w_uv[h][v][i] * o[h][i] */
int oracle_up_project(const double *o, const float *w_uv, int32_t heads, int32_t kv_lora,
                      int32_t v_dim, double *out);

#ifdef __cplusplus
}
#endif
#endif
