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
// Scores are mapped to order-preserving uint32 keys; the selection is every
// key above the exact k-th largest key T plus the lowest-index keys equal to T.
// One CTA per query:
//   sample  a strided sample of 2048 scores bounds the k-th largest from below
//           (t_lo: the lower edge of the coarse bin that holds 1.5x the kept
//           fraction of the sample);
//   pass    one streaming read of the scores appends every score >= t_lo
//           (typically a few percent) to a shared-memory candidate list;
//   exact   three radix levels over the candidates alone give T; candidates
//           above T set bits of a shared bitmap, those equal to T of a second;
//   emit    the bitmaps are scanned in ascending order (block prefix sums of
//           popcounts), taking equal keys lowest index first, so the output
//           is ascending without a sort.
// When the sample bound admits fewer than k or more candidates than the list
// holds (many equal or adversarially ordered scores), the CTA falls back to
// three radix levels over the scores in global memory and an emission pass that
// re-reads them; queries too long for the shared bitmaps use that path.
#include <cooperative_groups.h>

#include "dsa_kernels.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

constexpr int kL1Bits = 11;                   // first radix level: top 11 key bits
constexpr int kL1Bins = 1 << kL1Bits;
constexpr int kHistCopies = 2;             // 4096 bins: the first multi-level radix level
constexpr int kCandCap = 8192;
constexpr int kSample = 2048;                 // scores sampled to bound the threshold
constexpr int kSampleLog2 = 11;
constexpr int kItems = 8;                     // scores per thread per emission round (fallback)
constexpr size_t kFixedSmem = (size_t)kHistCopies * kL1Bins * 4 + (size_t)kCandCap * 8 + 256;
static_assert(kSample <= kCandCap, "the sample is staged in the candidate list");
constexpr size_t kMaxSmem = 200 * 1024;
constexpr int kBatch = 16;                    // loads in flight per lane in the streaming passes

// Keys of 32*kBatch consecutive scores starting at `base`: lane l gets
// elements base + l + 32*r, all loads issued before any is used.
__device__ __forceinline__ void load_keys(const float* __restrict__ sc, int64_t base, int64_t n,
                                          int lane, uint32_t (&key)[kBatch]) {
    float v[kBatch];
#pragma unroll
    for (int r = 0; r < kBatch; ++r) {
        const int64_t t = base + lane + 32 * r;
        v[r] = t < n ? __ldg(sc + t) : 0.f;
    }
#pragma unroll
    for (int r = 0; r < kBatch; ++r) key[r] = order_key(v[r]);
}

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

// The digit d of a histogram of nb bins at which the count of keys in bins
// above d is < k_rem <= that count plus hist[d]; *above gets the former.
template <int NT>
__device__ void find_digit(const uint32_t* hist, int nb, int64_t k_rem, int* warp_sums,
                           uint32_t* s_digit, int64_t* s_above) {
    const int per = nb >= NT ? nb / NT : 1;
    const int first = threadIdx.x * per;
    int local = 0;
    for (int r = 0; r < per; ++r)
        if (first + r < nb) local += (int)hist[first + r];
    int total;
    const int excl = block_exclusive_scan(local, &total, warp_sums);
    int64_t run = (int64_t)total - excl - local;
    for (int r = per - 1; r >= 0; --r) {
        const int bin = first + r;
        if (bin >= nb) continue;
        const int64_t h = hist[bin];
        if (run < k_rem && run + h >= k_rem) {
            *s_digit = (uint32_t)bin;
            *s_above = run;
        }
        run += h;
    }
    __syncthreads();
}

// Inverse of order_key.
__device__ __forceinline__ float key_to_float(uint32_t key) {
    const uint32_t u = (key & 0x80000000u) ? (key & 0x7fffffffu) : ~key;
    return __uint_as_float(u);
}

// Writes selected unit t (a row, or a pool of kpool rows) at position pos.
__device__ __forceinline__ void put(int32_t* out, int64_t pos, int64_t t, int kpool) {
    if (kpool == 1) {
        out[pos] = (int32_t)t;
    } else {
        for (int r = 0; r < kpool; ++r) out[pos * kpool + r] = (int32_t)(t * kpool + r);
    }
}

// Selection by three radix levels over the scores in global memory, then an
// emission pass over them in ascending order.  `hist` has 4096 entries.
template <int NT>
__device__ void select_multilevel(const float* __restrict__ sc, int64_t n, int64_t keep, int kpool,
                                  int32_t* out, uint32_t* hist, int* warp_sums, uint32_t* s_digit,
                                  int64_t* s_above, int64_t* n_out) {
    const int tid = threadIdx.x;
    uint32_t prefix = 0;
    int pbits = 0;
    int64_t k_rem = keep;
#pragma unroll 1
    for (int lvl = 0; lvl < 3; ++lvl) {
        const int bits = lvl == 0 ? 12 : 10;
        const int nb = 1 << bits;
        for (int i = tid; i < nb; i += NT) hist[i] = 0;
        __syncthreads();
        const int shift = 32 - pbits - bits;
        const int lane = tid & 31, warp = tid >> 5;
        for (int64_t base = (int64_t)warp * 32 * kBatch; base < n;
             base += (int64_t)(NT / 32) * 32 * kBatch) {
            uint32_t key[kBatch];
            load_keys(sc, base, n, lane, key);
#pragma unroll
            for (int r = 0; r < kBatch; ++r) {
                const bool match = base + lane + 32 * r < n &&
                                   (pbits == 0 || (key[r] >> (32 - pbits)) == prefix);
                if (match) atomicAdd(&hist[(key[r] >> shift) & (uint32_t)(nb - 1)], 1u);
            }
        }
        __syncthreads();
        find_digit<NT>(hist, nb, k_rem, warp_sums, s_digit, s_above);
        k_rem -= *s_above;
        prefix = (prefix << bits) | *s_digit;
        pbits += bits;
        __syncthreads();
    }
    const uint32_t T = prefix;
    int64_t eq_base = 0, out_base = 0;
    for (int64_t c0 = 0; c0 < n; c0 += (int64_t)NT * kItems) {
        const int64_t t_begin = c0 + (int64_t)tid * kItems;
        uint32_t keys[kItems];
        int n_eq = 0, valid = 0;
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            const int64_t t = t_begin + i;
            keys[i] = 0;
            if (t < n) {
                keys[i] = order_key(__ldg(sc + t));
                valid |= 1 << i;
                n_eq += keys[i] == T;
            }
        }
        int eq_total;
        const int eq_excl = block_exclusive_scan(n_eq, &eq_total, warp_sums);
        int64_t eq_rank = eq_base + eq_excl;
        int selmask = 0, n_s = 0;
#pragma unroll
        for (int i = 0; i < kItems; ++i) {
            if (!((valid >> i) & 1)) continue;
            const bool eq = keys[i] == T;
            const bool s = keys[i] > T || (eq && eq_rank < k_rem);
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
            put(out, pos++, t_begin + i, kpool);
        }
        eq_base += eq_total;
        out_base += sel_total;
    }
    *n_out = out_base;
}

// CL CTAs per query (1, or a cluster of 2): CTA rank r streams, marks and
// emits the r-th half of the row; the two exchange their candidates through
// distributed shared memory, so each finds the same threshold, and the second
// starts its output after the first half's selections.
template <int CL, int NT>
__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(NT, 1024 / NT)
topk_select_kernel(BatchDev b, int32_t top_k, int32_t kpool, const float* __restrict__ scores,
                   int64_t ld, int32_t* __restrict__ idx, int32_t* __restrict__ n_sel,
                   int64_t width, int32_t bitmap_words, int32_t* err) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem);                 // [copies][kL1Bins]
    uint32_t* cand_key = hist + kHistCopies * kL1Bins;                  // [kCandCap]
    int32_t* cand_idx = reinterpret_cast<int32_t*>(cand_key + kCandCap);
    int* warp_sums = cand_idx + kCandCap;                               // [32]
    uint32_t* s_digit = reinterpret_cast<uint32_t*>(warp_sums + 32);
    int* s_count = reinterpret_cast<int*>(s_digit + 1);
    int64_t* s_above = reinterpret_cast<int64_t*>(s_digit + 2);
    uint32_t* sel_bits = reinterpret_cast<uint32_t*>(smem + kFixedSmem);   // [bitmap_words]
    uint32_t* eq_bits = sel_bits + bitmap_words;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t q = CL == 1 ? blockIdx.x : blockIdx.y;
    const int rank = CL == 1 ? 0 : (int)cg::this_cluster().block_rank();
    int32_t* out = idx + q * width;
    asm volatile("griddepcontrol.wait;" ::: "memory");      // the scores must be complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    QueryInfo qi;
    // (every CTA of a cluster takes the same branches up to the exchange)
    if (!query_info(b, q, qi, err, /*where=*/2)) {
        if (rank == 0) {
            for (int64_t i = tid; i < width; i += NT) out[i] = -1;
            if (tid == 0) n_sel[q] = 0;
        }
        return;
    }
    const int64_t L = qi.L;
    const int64_t n = qi.n_keys;            // scores this query ranks (tokens or pools)
    const int64_t keep = top_k / kpool;     // how many of them it keeps

    if (n <= keep) {                        // dense: every visible row
        if (rank == 0) {
            for (int64_t i = tid; i < width; i += NT) out[i] = i < L ? (int32_t)i : -1;
            if (tid == 0) n_sel[q] = (int32_t)L;
        }
        return;
    }
    const float* sc = scores + q * ld;
    int64_t n_out = 0;
    // this CTA's part of the row: [lo, hi), a whole number of bitmap words
    const int64_t half = CL == 1 ? n : ((n + 1) / 2 + 31) / 32 * 32;
    const int64_t lo = rank * half;
    const int64_t hi = lo + half < n ? lo + half : n;
    const int64_t words = (hi - lo + 31) / 32;
    const int64_t words_first = ((half < n ? half : n) + 31) / 32;   // the larger part, for
                                                                      // a decision both CTAs share
    bool done = false;
    if (words_first <= bitmap_words) {
        // ---- a lower bound t_lo on the k-th largest score from a strided sample:
        // the key (to 22 bits) of the sample element ranked at 1.5x the kept
        // fraction plus a margin, found by two radix levels over the sample.
        uint32_t* samp = cand_key;                       // the sample lives where candidates will
        for (int i = tid; i < kL1Bins; i += NT) hist[i] = 0;
        if (tid == 0) *s_count = 0;
        const int64_t n_samp = n < kSample ? n : kSample;
        // element i n / n_samp: a shift when the row is long (n_samp = kSample,
        // a power of two), i itself otherwise -- no 64-bit division per element
        static_assert((kSample & (kSample - 1)) == 0, "the sample size is a power of two");
        for (int64_t i = tid; i < n_samp; i += NT)
            samp[i] = order_key(__ldg(sc + (n_samp == kSample ? (i * n) >> kSampleLog2 : i)));
        __syncthreads();
        for (int64_t i = tid; i < n_samp; i += NT) atomicAdd(&hist[samp[i] >> 21], 1u);
        __syncthreads();
        int64_t target = (keep * n_samp * 3 + 2 * n - 1) / (2 * n) + 8;
        target = target < n_samp ? target : n_samp;
        find_digit<NT>(hist, kL1Bins, target, warp_sums, s_digit, s_above);
        const uint32_t sb1 = *s_digit;
        target -= *s_above;
        __syncthreads();
        for (int i = tid; i < kL1Bins; i += NT) hist[i] = 0;
        __syncthreads();
        for (int64_t i = tid; i < n_samp; i += NT)
            if ((samp[i] >> 21) == sb1) atomicAdd(&hist[(samp[i] >> 10) & (kL1Bins - 1)], 1u);
        __syncthreads();
        find_digit<NT>(hist, kL1Bins, target, warp_sums, s_digit, s_above);
        const float t_lo = key_to_float((sb1 << 21) | (*s_digit << 10));
        __syncthreads();

        // ---- one streaming pass over [lo, hi): every score >= t_lo becomes a candidate
        for (int64_t base = lo + (int64_t)warp * 32 * kBatch; base < hi;
             base += (int64_t)(NT / 32) * 32 * kBatch) {
            float v[kBatch];
#pragma unroll
            for (int r = 0; r < kBatch; ++r) {
                const int64_t t = base + lane + 32 * r;
                v[r] = t < hi ? __ldg(sc + t) : -INFINITY;
            }
            // the round's hits counted per lane, a warp prefix sum for each
            // lane's first slot, one slot allocation per warp for all of them
            int my = 0;
#pragma unroll
            for (int r = 0; r < kBatch; ++r) my += v[r] >= t_lo;
            int incl = my;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const int n_hit = __shfl_sync(0xffffffffu, incl, 31);
            if (n_hit) {
                int slot = 0;
                if (lane == 0) slot = atomicAdd(s_count, n_hit);
                slot = __shfl_sync(0xffffffffu, slot, 0) + incl - my;
#pragma unroll
                for (int r = 0; r < kBatch; ++r) {
                    if (v[r] >= t_lo) {
                        if (slot < kCandCap) {
                            cand_key[slot] = order_key(v[r]);
                            cand_idx[slot] = (int32_t)(base + lane + 32 * r);
                        }
                        ++slot;
                    }
                }
            }
        }
        for (int64_t w = tid; w < words; w += NT) { sel_bits[w] = 0; eq_bits[w] = 0; }
        __syncthreads();
        int n_cand = *s_count;
        if (CL == 2) {
            // the peer's candidates after this CTA's own: both hold the whole list
            cg::cluster_group cluster = cg::this_cluster();
            cluster.sync();                              // both passes are complete
            const int* peer_count = cluster.map_shared_rank(s_count, rank ^ 1);
            const int n_peer = *peer_count;
            const int n_all = n_cand + n_peer;
            if (n_cand <= kCandCap && n_all <= kCandCap) {
                const uint32_t* pk = cluster.map_shared_rank(cand_key, rank ^ 1);
                const int32_t* pi = cluster.map_shared_rank(cand_idx, rank ^ 1);
                for (int i = tid; i < n_peer; i += NT) {
                    cand_key[n_cand + i] = pk[i];
                    cand_idx[n_cand + i] = pi[i];
                }
            }
            cluster.sync();                              // no DSMEM reads after this
            n_cand = n_all;
        }
        __syncthreads();
        if (n_cand >= keep && n_cand <= kCandCap) {
            // ---- exact k-th key T among the candidates (three radix levels)
            uint32_t prefix = 0;
            int pbits = 0;
            int64_t k_rem = keep;
#pragma unroll 1
            for (int lvl = 0; lvl < 3; ++lvl) {
                const int bits = lvl == 2 ? 10 : 11;
                const int nb = 1 << bits;
                const int shift = 32 - pbits - bits;
                for (int i = tid; i < nb; i += NT) hist[i] = 0;
                __syncthreads();
                for (int i = tid; i < n_cand; i += NT) {
                    const uint32_t key = cand_key[i];
                    if (pbits == 0 || (key >> (32 - pbits)) == prefix)
                        atomicAdd(&hist[(key >> shift) & (uint32_t)(nb - 1)], 1u);
                }
                __syncthreads();
                find_digit<NT>(hist, nb, k_rem, warp_sums, s_digit, s_above);
                k_rem -= *s_above;
                prefix = (prefix << bits) | *s_digit;
                pbits += bits;
                __syncthreads();
            }
            const uint32_t T = prefix;
            // this part's candidates into the bitmaps; the earlier part's
            // selections (keys above T, and how many equal to T) for the offsets
            int gt_before = 0, eq_before = 0;
            for (int i = tid; i < n_cand; i += NT) {
                const uint32_t key = cand_key[i];
                const int32_t t = cand_idx[i];
                if (t < lo) {
                    gt_before += key > T;
                    eq_before += key == T;
                } else if (t < hi) {
                    const int32_t u = (int32_t)(t - lo);
                    if (key > T) atomicOr(&sel_bits[u >> 5], 1u << (u & 31));
                    else if (key == T) atomicOr(&eq_bits[u >> 5], 1u << (u & 31));
                }
            }
            int64_t eq_base = 0, out_base = 0;
            if (CL == 2 && rank > 0) {
                int tot;
                block_exclusive_scan(gt_before, &tot, warp_sums);
                gt_before = tot;
                block_exclusive_scan(eq_before, &tot, warp_sums);
                eq_before = tot;
                eq_base = eq_before;
                out_base = gt_before + (eq_before < k_rem ? eq_before : k_rem);
            }
            __syncthreads();
            // ---- emission in ascending order: keys > T, then the first k_rem keys == T
            for (int64_t w0 = 0; w0 < words; w0 += NT) {
                const int64_t w = w0 + tid;
                const uint32_t sw = w < words ? sel_bits[w] : 0u;
                const uint32_t ew = w < words ? eq_bits[w] : 0u;
                // one scan of both counts (each below 2^16 per round): keys
                // above T in the high half, keys equal to T in the low half
                int tot;
                const int excl = block_exclusive_scan((__popc(sw) << 16) | __popc(ew), &tot,
                                                      warp_sums);
                const int gt_excl = excl >> 16, eq_excl = excl & 0xffff;
                const int gt_total = tot >> 16, eq_total = tot & 0xffff;
                // keys equal to T are taken in word order while k_rem lasts
                int64_t room = k_rem - eq_base;
                room = room < 0 ? 0 : room;
                int64_t take = room - eq_excl;
                take = take < 0 ? 0 : (take > __popc(ew) ? __popc(ew) : take);
                uint32_t m = ew, taken = 0;
                for (int i = 0; i < take; ++i) { taken |= m & (~m + 1u); m &= m - 1u; }
                uint32_t comb = sw | taken;
                const int64_t taken_before = room < eq_excl ? room : eq_excl;
                const int sel_total = gt_total + (int)(room < eq_total ? room : eq_total);
                int64_t pos = out_base + gt_excl + taken_before;
                while (comb != 0u && pos < keep) {
                    const int bit = __ffs(comb) - 1;
                    comb &= comb - 1u;
                    put(out, pos++, lo + w * 32 + bit, kpool);
                }
                eq_base += eq_total;
                out_base += sel_total;
            }
            n_out = out_base;
            done = true;
        }
    }
    if (!done) {                            // the whole row, by the first CTA alone
        if (rank > 0) return;
        select_multilevel<NT>(sc, n, keep, kpool, out, hist, warp_sums, s_digit, s_above, &n_out);
    }
    if (tid == 0 && rank == (done ? CL - 1 : 0) && n_out != keep)
        record_error(err, kDevBadIndex, (int32_t)q, /*where=*/2);
    if (rank > 0) return;

    // ---- unfilled tail (k-pool), then padding
    const int64_t body = keep * kpool;
    const int64_t tail = L - n * kpool;
    for (int64_t i = tid; i < tail; i += NT) out[body + i] = (int32_t)(n * kpool + i);
    const int64_t total_sel = body + tail;
    for (int64_t i = total_sel + tid; i < width; i += NT) out[i] = -1;
    if (tid == 0) n_sel[q] = (int32_t)total_sel;
}

}  // namespace

// Two CTAs per query when that still fits one wave and the rows are long
// enough for the halves to pay for the exchange.
bool topk_pair_eligible(const Shape& sh, const BatchDev& b) {
    return b.n_q >= 1 && 2 * (int64_t)b.n_q <= sm_count() && b.max_kv_len / sh.kpool >= 16384;
}

cudaError_t launch_topk_select(const Shape& sh, const BatchDev& b, const float* scores,
                               int64_t ld, int32_t* idx, int32_t* n_sel, int32_t* err,
                               cudaStream_t st) {
    if (b.n_q == 0) return cudaSuccess;
    if (topk_cluster_eligible(sh, b))
        return launch_topk_select_cluster(sh, b, scores, ld, idx, n_sel, err, st);
    const bool pair = topk_pair_eligible(sh, b);
    // Bitmaps for the longest query's (first) part if they fit; otherwise
    // every query that needs more takes the multi-level path.
    const int64_t n_max = b.max_kv_len / sh.kpool;
    const int64_t part = pair ? ((n_max + 1) / 2 + 31) / 32 * 32 : n_max;
    int64_t words = (part + 31) / 32;
    if (kFixedSmem + (size_t)words * 8 > kMaxSmem) words = 0;
    const size_t smem = kFixedSmem + (size_t)words * 8;
    // A pair has 1024 threads per CTA (one wave: latency wants threads); one
    // CTA per query has 512, two CTAs per SM overlapping their latency chains
    // across the many waves of a prefill chunk.
    auto kern = pair ? topk_select_kernel<2, 1024> : topk_select_kernel<1, 512>;
    const int nt = pair ? 1024 : 512;
    cudaError_t e = ensure_dyn_smem((const void*)kern, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid = pair ? dim3(2, (unsigned)b.n_q) : dim3((unsigned)b.n_q);
    return launch_pdl(kern, grid, dim3(nt), smem, st, b, sh.top_k, sh.kpool, scores, ld, idx,
                      n_sel, sh.index_row_width(), (int32_t)words, err);
}

}  // namespace dsa
