// topk_select.cu -- per-query top-k (and k-pool) selection by radix select.
//
// Token mode: the min(k, L) rows that come first in the order (score
// descending, index ascending); dense when L <= k ("GLM-5.x (glm-dsa,
// glm5next)", "The sparse-attention path"; "GLM 5.2 in one C file", "The
// Lightning Indexer" -- with exactly k kept, not the page's strict threshold).
// k-pool mode: the top k/kpool pools expanded to their rows plus the unfilled
// tail, dense when floor(L/kpool) <= k/kpool ("GLM-5.3-Flash on WASTE",
// "DeepSeek Sparse Attention, k-pool flavour").
//
// Scores are mapped to order-preserving uint32 keys.  Three radix levels (12,
// 10 and 10 bits) over the query's scores find the exact k-th largest key T
// and how many keys equal to T are taken; the emission pass then walks the
// scores in ascending index order and keeps every key > T plus the first
// (lowest-index) keys == T, compacting with block-wide prefix sums, so the
// output is ascending without a sort.  One CTA per query.
#include "dsa_kernels.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kItems = 8;        // consecutive scores per thread in the emission pass

// Exclusive prefix sum over the CTA in thread order; *total gets the sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* warp_sums) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = (lane < nwarps) ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    const int before = wid > 0 ? warp_sums[wid - 1] : 0;
    *total = warp_sums[nwarps - 1];
    __syncthreads();
    return before + x - v;
}

__global__ void __launch_bounds__(kThreads)
topk_select_kernel(BatchDev b, int32_t top_k, int32_t kpool, const float* __restrict__ scores,
                   int64_t ld, int32_t* __restrict__ idx, int32_t* __restrict__ n_sel,
                   int64_t width, int32_t* err) {
    __shared__ uint32_t hist[4096];
    __shared__ int warp_sums[32];
    __shared__ uint32_t s_digit;
    __shared__ int64_t s_above;

    const int tid = threadIdx.x;
    const int64_t q = blockIdx.x;
    int32_t* out = idx + q * width;
    QueryInfo qi;
    if (!query_info(b, q, qi, err, /*where=*/2)) {
        for (int64_t i = tid; i < width; i += kThreads) out[i] = -1;
        if (tid == 0) n_sel[q] = 0;
        return;
    }
    const int64_t L = qi.L;
    const int64_t n = qi.n_keys;            // scores this query ranks (tokens or pools)
    const int64_t keep = top_k / kpool;     // how many of them it keeps

    if (n <= keep) {                        // dense: every visible row
        for (int64_t i = tid; i < width; i += kThreads) out[i] = i < L ? (int32_t)i : -1;
        if (tid == 0) n_sel[q] = (int32_t)L;
        return;
    }

    const float* sc = scores + q * ld;

    // ---- radix levels: exact k-th largest key T, and how many keys == T to take
    uint32_t prefix = 0;
    int pbits = 0;
    int64_t k_rem = keep;
#pragma unroll 1
    for (int lvl = 0; lvl < 3; ++lvl) {
        const int bits = lvl == 0 ? 12 : 10;
        const int nb = 1 << bits;
        for (int i = tid; i < nb; i += kThreads) hist[i] = 0;
        __syncthreads();
        const int shift = 32 - pbits - bits;
        for (int64_t t = tid; t < n; t += kThreads) {
            const uint32_t key = order_key(__ldg(sc + t));
            const bool match = pbits == 0 || (key >> (32 - pbits)) == prefix;
            if (match) atomicAdd(&hist[(key >> shift) & (uint32_t)(nb - 1)], 1u);
        }
        __syncthreads();
        // Thread j owns bins [j*per, (j+1)*per); above_j counts the bins of all
        // higher threads.  The digit d is the bin where the running count from
        // the top first reaches k_rem.
        const int per = nb / kThreads;
        int local = 0;
        for (int r = 0; r < per; ++r) local += (int)hist[tid * per + r];
        int total;
        const int excl = block_exclusive_scan(local, &total, warp_sums);
        int64_t run = (int64_t)total - excl - local;
        for (int r = per - 1; r >= 0; --r) {
            const int bin = tid * per + r;
            const int64_t h = hist[bin];
            if (run < k_rem && run + h >= k_rem) {
                s_digit = (uint32_t)bin;
                s_above = run;
            }
            run += h;
        }
        __syncthreads();
        k_rem -= s_above;
        prefix = (prefix << bits) | s_digit;
        pbits += bits;
        __syncthreads();
    }
    const uint32_t T = prefix;

    // ---- emission in ascending index order
    int64_t eq_base = 0, out_base = 0;
    for (int64_t c0 = 0; c0 < n; c0 += (int64_t)kThreads * kItems) {
        const int64_t t_begin = c0 + (int64_t)tid * kItems;
        uint32_t keys[kItems];
        int n_eq = 0, valid = 0;
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            const int64_t t = t_begin + i;
            if (t < n) {
                keys[i] = order_key(__ldg(sc + t));
                valid |= 1 << i;
                n_eq += keys[i] == T;
            } else {
                keys[i] = 0;
            }
        }
        int eq_total;
        const int eq_excl = block_exclusive_scan(n_eq, &eq_total, warp_sums);
        int64_t eq_rank = eq_base + eq_excl;
        int selmask = 0, n_s = 0;
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            if (!((valid >> i) & 1)) continue;
            const bool gt = keys[i] > T;
            const bool eq = keys[i] == T;
            const bool s = gt || (eq && eq_rank < k_rem);
            eq_rank += eq;
            if (s) { selmask |= 1 << i; ++n_s; }
        }
        int sel_total;
        const int sel_excl = block_exclusive_scan(n_s, &sel_total, warp_sums);
        int64_t pos = out_base + sel_excl;
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            if (!((selmask >> i) & 1)) continue;
            if (pos >= keep) break;                 // never write past the kept count
            const int64_t t = t_begin + i;
            if (kpool == 1) {
                out[pos] = (int32_t)t;
            } else {
                for (int r = 0; r < kpool; ++r) out[pos * kpool + r] = (int32_t)(t * kpool + r);
            }
            ++pos;
        }
        eq_base += eq_total;
        out_base += sel_total;
    }
    if (tid == 0 && out_base != keep) record_error(err, kDevBadIndex, (int32_t)q, /*where=*/2);

    // ---- unfilled tail (k-pool), then padding
    const int64_t body = keep * kpool;
    const int64_t tail = L - n * kpool;
    for (int64_t i = tid; i < tail; i += kThreads) out[body + i] = (int32_t)(n * kpool + i);
    const int64_t total_sel = body + tail;
    for (int64_t i = total_sel + tid; i < width; i += kThreads) out[i] = -1;
    if (tid == 0) n_sel[q] = (int32_t)total_sel;
}

}  // namespace

cudaError_t launch_topk_select(const Shape& sh, const BatchDev& b, const float* scores,
                               int64_t ld, int32_t* idx, int32_t* n_sel, int32_t* err,
                               cudaStream_t st) {
    if (b.n_q == 0) return cudaSuccess;
    topk_select_kernel<<<b.n_q, kThreads, 0, st>>>(b, sh.top_k, sh.kpool, scores, ld, idx, n_sel,
                                                   sh.index_row_width(), err);
    return cudaGetLastError();
}

}  // namespace dsa
