// topk_select_cluster.cu -- per-query top-k selection by a 16-CTA thread-block
// cluster, for batches too small to fill the GPU with one CTA per query.
//
// Same result as topk_select.cu (the min(k, L) rows first in the order score
// descending, index ascending, or the k-pool rule of "GLM-5.3-Flash on WASTE",
// "DeepSeek Sparse Attention, k-pool flavour"); the work of one query is spread
// over the 16 CTAs of a cluster, which exchange data through distributed
// shared memory (DSMEM) and cluster barriers instead of global memory:
//   1  each CTA loads a 1/16 slice of the query's scores as order-preserving
//      keys (kept in registers, each thread a contiguous run) and contributes
//      128 strided keys to a 2048-key cluster-wide sample;
//   2  every CTA bounds the k-th key from below from the sample (two radix
//      levels: the key ranked at 1.5x the kept fraction plus a margin);
//   3  each CTA compacts its keys at or above the bound (candidates, a few
//      percent) in index order; every CTA copies all candidates, in cluster-rank
//      order (= index order), and finds the exact k-th key T and how many keys
//      equal to T are taken (the lowest-index ones);
//   4  each CTA writes its taken candidates at the offset given by the taken
//      candidates of the CTAs before it.
// If the bound admits fewer than k or more candidates than the shared lists
// hold (massively tied scores), rank 0 selects alone with radix passes over
// global memory.
#include <cooperative_groups.h>

#include "dsa_kernels.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kCtas = 16;                       // cluster size
constexpr int kThreads = 512;
constexpr int kBins = 2048;                     // top 11 key bits
constexpr int kLocalCap = 2048;                 // candidates per CTA
constexpr int kCandCap = 8192;                  // candidates per query
constexpr int kMaxSlice = 16384;                // scores per CTA (n <= 262144)
constexpr int kPerMax = kMaxSlice / kThreads;   // scores per thread
constexpr int kSampPer = 128;                   // sampled scores per CTA

struct Smem {
    uint32_t hist[kBins];
    uint32_t samp[kSampPer];
    uint32_t lkey[kLocalCap];
    uint32_t akey[kCandCap];
    uint8_t take[kCandCap];
    int warp_sums[32];
    int32_t cnt_lc[kCtas];
    int64_t above;
    uint32_t digit;
    int32_t n_gt, n_lc;
    int32_t flag;
};

__device__ __forceinline__ int block_excl_scan(int v, int* total, int* warp_sums) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) warp_sums[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        warp_sums[lane] = s;
    }
    __syncthreads();
    const int before = wid > 0 ? warp_sums[wid - 1] : 0;
    *total = warp_sums[nw - 1];
    __syncthreads();
    return before + x - v;
}

// Digit d of histogram h[nb] where the count above d is < k <= that plus h[d].
__device__ void find_digit(const uint32_t* h, int nb, int64_t k, Smem& s) {
    const int per = nb >= kThreads ? nb / kThreads : 1;
    const int first = threadIdx.x * per;
    int local = 0;
    for (int r = 0; r < per; ++r)
        if (first + r < nb) local += (int)h[first + r];
    int total;
    const int excl = block_excl_scan(local, &total, s.warp_sums);
    int64_t run = (int64_t)total - excl - local;
    for (int r = per - 1; r >= 0; --r) {
        const int bin = first + r;
        if (bin >= nb) continue;
        const int64_t c = h[bin];
        if (run < k && run + c >= k) { s.digit = (uint32_t)bin; s.above = run; }
        run += c;
    }
    __syncthreads();
}

__device__ __forceinline__ void put(int32_t* out, int64_t pos, int64_t t, int kpool) {
    if (kpool == 1) {
        out[pos] = (int32_t)t;
    } else {
        for (int r = 0; r < kpool; ++r) out[pos * kpool + r] = (int32_t)(t * kpool + r);
    }
}

// Rank 0's fallback: radix levels over the scores in global memory.
__device__ int64_t select_global(const float* sc, int64_t n, int64_t keep, int kpool, int32_t* out,
                                 Smem& s) {
    uint32_t prefix = 0;
    int pbits = 0;
    int64_t k_rem = keep;
    for (int lvl = 0; lvl < 3; ++lvl) {
        const int bits = lvl == 2 ? 10 : 11;
        const int nb = 1 << bits, shift = 32 - pbits - bits;
        for (int i = threadIdx.x; i < nb; i += kThreads) s.hist[i] = 0;
        __syncthreads();
        for (int64_t t = threadIdx.x; t < n; t += kThreads) {
            const uint32_t key = order_key(sc[t]);
            if (pbits == 0 || (key >> (32 - pbits)) == prefix)
                atomicAdd(&s.hist[(key >> shift) & (uint32_t)(nb - 1)], 1u);
        }
        __syncthreads();
        find_digit(s.hist, nb, k_rem, s);
        k_rem -= s.above;
        prefix = (prefix << bits) | s.digit;
        pbits += bits;
        __syncthreads();
    }
    const uint32_t T = prefix;
    int64_t eq_base = 0, out_base = 0;
    for (int64_t c0 = 0; c0 < n; c0 += kThreads) {
        const int64_t t = c0 + threadIdx.x;
        const uint32_t key = t < n ? order_key(sc[t]) : 0u;
        const int eq = t < n && key == T;
        int eq_tot;
        const int64_t er = eq_base + block_excl_scan(eq, &eq_tot, s.warp_sums);
        const int sel = t < n && (key > T || (eq && er < k_rem));
        int sel_tot;
        const int64_t pos = out_base + block_excl_scan(sel, &sel_tot, s.warp_sums);
        if (sel && pos < keep) put(out, pos, t, kpool);
        eq_base += eq_tot;
        out_base += sel_tot;
    }
    return out_base;
}

__global__ void __cluster_dims__(kCtas, 1, 1) __launch_bounds__(kThreads, 1)
topk_select_cluster(BatchDev b, int32_t top_k, int32_t kpool, const float* __restrict__ scores,
                    int64_t ld, int32_t* __restrict__ idx, int32_t* __restrict__ n_sel,
                    int64_t width, int32_t* err) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& s = *reinterpret_cast<Smem*>(smem_raw);
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t q = blockIdx.y;
    int32_t* out = idx + q * width;
    asm volatile("griddepcontrol.wait;" ::: "memory");      // the scores must be complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    QueryInfo qi;
    const bool qok = query_info(b, q, qi, err, /*where=*/12);
    const int64_t L = qok ? qi.L : 0;
    const int64_t n = qok ? qi.n_keys : 0;
    const int64_t keep = top_k / kpool;
    // decisions that skip the cluster path are uniform across the cluster
    if (!qok || n <= keep) {
        if (rank == 0) {
            for (int64_t i = tid; i < width; i += kThreads) out[i] = (qok && i < L) ? (int32_t)i : -1;
            if (tid == 0) n_sel[q] = qok ? (int32_t)L : 0;
        }
        return;
    }
    const float* sc = scores + q * ld;
    const int64_t s0 = n * rank / kCtas, s1 = n * (rank + 1) / kCtas, ns = s1 - s0;

    // ---- 1: this thread's run of the slice (keys in registers) and this CTA's
    // share of a cluster-wide strided sample.  Thread t owns the contiguous run
    // [t*per, t*per + per) of the slice, so thread order is index order.
    const int per = (int)((ns + kThreads - 1) / kThreads);
    const int64_t my0 = (int64_t)tid * per;
    const int my_n = (int)(my0 >= ns ? 0 : (ns - my0 < per ? ns - my0 : per));
    uint32_t kk[kPerMax];
    {
        float v[kPerMax];
#pragma unroll
        for (int e = 0; e < kPerMax; ++e) v[e] = e < my_n ? __ldg(sc + s0 + my0 + e) : 0.f;
#pragma unroll
        for (int e = 0; e < kPerMax; ++e) kk[e] = order_key(v[e]);
    }
    for (int i = tid; i < kSampPer; i += kThreads)
        s.samp[i] = ns > 0 ? order_key(__ldg(sc + s0 + (int64_t)i * ns / kSampPer)) : 0u;
    cluster.sync();
    // ---- 2: every CTA bounds the k-th key from below from the 2048-key sample:
    // the key (to 22 bits) ranked at 1.5x the kept fraction plus a margin
    for (int i = tid; i < kCtas * kSampPer; i += kThreads)
        s.akey[i] = cluster.map_shared_rank(&s.samp[0], i / kSampPer)[i % kSampPer];
    for (int i = tid; i < kBins; i += kThreads) s.hist[i] = 0;
    __syncthreads();
    constexpr int kSamp = kCtas * kSampPer;
    for (int i = tid; i < kSamp; i += kThreads) atomicAdd(&s.hist[s.akey[i] >> 21], 1u);
    __syncthreads();
    int64_t target = (keep * kSamp * 3 + 2 * n - 1) / (2 * n) + 8;
    target = target < kSamp ? target : kSamp;
    find_digit(s.hist, kBins, target, s);
    const uint32_t sb1 = s.digit;
    target -= s.above;
    __syncthreads();
    for (int i = tid; i < kBins; i += kThreads) s.hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < kSamp; i += kThreads)
        if ((s.akey[i] >> 21) == sb1) atomicAdd(&s.hist[(s.akey[i] >> 10) & (kBins - 1)], 1u);
    __syncthreads();
    find_digit(s.hist, kBins, target, s);
    const uint32_t k_lo = (sb1 << 21) | (s.digit << 10);

    // ---- 3: every key >= k_lo is a candidate, compacted in index order
    int my_c = 0;
#pragma unroll
    for (int e = 0; e < kPerMax; ++e) my_c += e < my_n && kk[e] >= k_lo;
    int my_lpos;                                    // this thread's first local candidate
    {
        int n_lc;
        int pos = block_excl_scan(my_c, &n_lc, s.warp_sums);
        my_lpos = pos;
#pragma unroll
        for (int e = 0; e < kPerMax; ++e) {
            if (e < my_n && kk[e] >= k_lo) {
                if (pos < kLocalCap) s.lkey[pos] = kk[e];
                ++pos;
            }
        }
        if (tid == 0) s.n_lc = n_lc;
    }
    cluster.sync();
    // every CTA: the cluster's counts (one remote read each), then all candidates
    if (tid < kCtas) s.cnt_lc[tid] = cluster.map_shared_rank(&s, tid)->n_lc;
    __syncthreads();
    int cand_before = 0, n_cand = 0;
    bool overflow = false;
    int cand_off[kCtas + 1];
    cand_off[0] = 0;
#pragma unroll
    for (int c = 0; c < kCtas; ++c) {
        const int lc = s.cnt_lc[c];
        overflow |= lc > kLocalCap;
        if (c < rank) cand_before += lc;
        n_cand += lc;
        cand_off[c + 1] = n_cand;
    }
    overflow |= n_cand > kCandCap || n_cand < keep;
    if (!overflow) {
        for (int i = tid; i < n_cand; i += kThreads) {
            int c = 0;
#pragma unroll
            for (int r = 1; r < kCtas; ++r) c += i >= cand_off[r];
            s.akey[i] = cluster.map_shared_rank(&s.lkey[0], c)[i - cand_off[c]];
        }
    }
    cluster.sync();                       // all DSMEM reads of this query are done
    if (overflow) {
        if (rank == 0) {
            const int64_t got = select_global(sc, n, keep, kpool, out, s);
            if (tid == 0 && got != keep) record_error(err, kDevBadIndex, (int32_t)q, /*where=*/12);
        }
    } else {
        // exact k-th key T among the candidates: three radix levels
        uint32_t prefix = 0;
        int pbits = 0;
        int64_t k_rem = keep;
        for (int lvl = 0; lvl < 3; ++lvl) {
            const int bits = lvl == 2 ? 10 : 11;
            const int nb = 1 << bits, shift = 32 - pbits - bits;
            for (int i = tid; i < nb; i += kThreads) s.hist[i] = 0;
            __syncthreads();
            for (int i = tid; i < n_cand; i += kThreads)
                if (pbits == 0 || (s.akey[i] >> (32 - pbits)) == prefix)
                    atomicAdd(&s.hist[(s.akey[i] >> shift) & (uint32_t)(nb - 1)], 1u);
            __syncthreads();
            find_digit(s.hist, nb, k_rem, s);
            k_rem -= s.above;
            prefix = (prefix << bits) | s.digit;
            pbits += bits;
            __syncthreads();
        }
        const uint32_t T = prefix;
        // taken: key > T, or key == T among the first k_rem equal ones (the list is
        // in index order).  When every key equal to T is taken (no tie straddles
        // the threshold), taken is simply key >= T.
        int my_eq = 0, my_ge_before = 0;
        for (int i = tid; i < n_cand; i += kThreads) {
            const uint32_t key = s.akey[i];
            my_eq += key == T;
            my_ge_before += key >= T && i < cand_before;
        }
        int n_eq, taken_before;
        block_excl_scan(my_eq, &n_eq, s.warp_sums);
        block_excl_scan(my_ge_before, &taken_before, s.warp_sums);
        if (n_eq == k_rem) {
            for (int i = tid; i < n_cand; i += kThreads) s.take[i] = s.akey[i] >= T;
        } else {
            taken_before = 0;
            int64_t eq_base = 0;
            for (int c0 = 0; c0 < n_cand; c0 += kThreads) {
                const int i = c0 + tid;
                const uint32_t key = i < n_cand ? s.akey[i] : 0u;
                const int eq = i < n_cand && key == T;
                int eq_tot;
                const int64_t er = eq_base + block_excl_scan(eq, &eq_tot, s.warp_sums);
                const int take = i < n_cand && (key > T || (eq && er < k_rem));
                if (i < n_cand) s.take[i] = (uint8_t)take;
                int tk;
                block_excl_scan(take && i < cand_before, &tk, s.warp_sums);
                taken_before += tk;
                eq_base += eq_tot;
            }
        }
        __syncthreads();
        // ---- 4: emission of this slice's taken candidates, ascending, at its offset
        const int my_cpos = cand_before + my_lpos;
        int my_sel = 0;
        for (int e = 0; e < my_c; ++e) my_sel += s.take[my_cpos + e] != 0;
        int sel_tot;
        int64_t pos = taken_before + block_excl_scan(my_sel, &sel_tot, s.warp_sums);
        int cpos = my_cpos;
#pragma unroll
        for (int e = 0; e < kPerMax; ++e) {
            if (e < my_n && kk[e] >= k_lo) {
                if (s.take[cpos] != 0 && pos < keep) {
                    put(out, pos, s0 + my0 + e, kpool);
                    ++pos;
                }
                ++cpos;
            }
        }
    }
    if (rank == 0) {                           // unfilled tail (k-pool), padding, count
        const int64_t body = keep * kpool, tail = L - n * kpool;
        for (int64_t i = tid; i < tail; i += kThreads) out[body + i] = (int32_t)(n * kpool + i);
        for (int64_t i = body + tail + tid; i < width; i += kThreads) out[i] = -1;
        if (tid == 0) n_sel[q] = (int32_t)(body + tail);
    }
    (void)lane;
    (void)warp;
}

}  // namespace

bool topk_cluster_eligible(const Shape& sh, const BatchDev& b) {
    const int64_t n_max = b.max_kv_len / sh.kpool;
    return b.n_q >= 1 && b.n_q * kCtas <= 2 * sm_count() && n_max >= 32768 &&
           n_max <= (int64_t)kCtas * kMaxSlice;
}

cudaError_t launch_topk_select_cluster(const Shape& sh, const BatchDev& b, const float* scores,
                                       int64_t ld, int32_t* idx, int32_t* n_sel, int32_t* err,
                                       cudaStream_t st) {
    const size_t smem = sizeof(Smem);
    cudaError_t e = ensure_dyn_smem((const void*)topk_select_cluster, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(topk_select_cluster, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_select_cluster, dim3(kCtas, (unsigned)b.n_q), dim3(kThreads), smem, st, b,
                      sh.top_k, sh.kpool, scores, ld, idx, n_sel, sh.index_row_width(), err);
}

}  // namespace dsa
