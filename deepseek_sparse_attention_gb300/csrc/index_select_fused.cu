// index_select_fused.cu -- decode scoring and top-k selection in one
// cooperative launch.
//
// The lightning indexer's scores s_t = sum_h w_h * relu(q_h . k_t) ("GLM 5.2 in
// one C file", "The Lightning Indexer") and the per-query selection of the
// min(k, L) best rows -- score descending, ties to the lower index, emitted in
// ascending row order; in k-pool mode the best k/kpool pools expanded to their
// rows plus the unfilled tail ("GLM-5.x (glm-dsa, glm5next)", "The
// sparse-attention path"; "GLM-5.3-Flash on WASTE", "DeepSeek Sparse
// Attention, k-pool flavour").
//
// A decode batch with a long context has few queries and many keys: one query
// would leave all but one SM idle in a per-query selection kernel, and a
// separate launch costs its own ramp-up.  Here the persistent indexer grid (one
// CTA per SM, a contiguous range of (query, key tile) units each) keeps its
// scores and selects in place, all CTAs of a query cooperating through global
// histograms and grid barriers:
//   score   the tensor-core indexer pipeline (index_pipeline.cuh) writes the
//           CTA's scores; they come back (from L2) as order-preserving keys
//           into the shared memory the pipeline's ring used;
//   level 1 histogram of key bits 31..21 per query (shared, then added into
//           the query's global histogram); barrier; every CTA of the query
//           finds the bin b1 that holds the k-th largest key;
//   level 2 the same over bits 20..10 of the keys in b1; barrier;
//   level 3 bits 9..0 of the keys in (b1, b2); barrier: the k-th largest key T
//           is known exactly, and how many keys above it the query has;
//   counts  each CTA publishes how many of its keys are > T and == T; barrier;
//   emit    a CTA's output offset is the count of selected keys of the CTAs
//           before it (keys equal to T go to the lowest indices first); a block
//           scan over its keys writes its selections in ascending order.
// The global histograms are cleared by the launch that used them, as soon as
// every CTA has read them, so they are zero again for the next launch.
#include "index_pipeline.cuh"

namespace dsa {

namespace {

using namespace sm100;
using namespace idxp;

using C = Cfg<1>;
constexpr int kThreads = C::kThreads;                 // 256
constexpr int kWarps = kThreads / 32;
constexpr int kBins1 = 2048;                          // key bits 31..21
constexpr int kBins2 = 2048;                          // key bits 20..10
constexpr int kBins3 = 1024;                          // key bits 9..0
constexpr int kHistWords = kBins1 + kBins2 + kBins3;  // per query
constexpr int kItems = 8;                             // keys per thread per emission round

// Shared memory after the indexer pipeline: the ring (C::kOffA .. C::kOffB)
// holds the CTA's keys, a histogram, per-query state and scan scratch.
constexpr uint32_t kOffHist = C::kOffB - 16384;
constexpr uint32_t kMaxCtaKeys = kOffHist / 4;
constexpr uint32_t kMaxCtaTiles = kMaxCtaKeys / kTileKeys;
constexpr uint32_t kOffSeg = kOffHist + kBins1 * 4;
struct SegState {          // one query's part of this CTA's unit range
    int32_t q;
    int32_t n;             // keys (tokens or pools) in the part
    int32_t koff;          // first key's slot in shared memory
    int32_t t_lo;          // first key's index in the query
    uint32_t prefix;       // resolved high bits of T, then T
    int32_t above;         // keys of the query above the resolved prefix
    int32_t need_eq;       // keys equal to T the query keeps
    int32_t eq;            // keys of this part equal to T
};
constexpr uint32_t kOffRed = kOffSeg + kFusedMaxQ * sizeof(SegState);
static_assert(kOffRed + 256 <= C::kOffB, "selection state must fit in the ring");
static_assert(C::kOffA == 0, "keys start at the ring");
static_assert(kWsHeaderBytes + (size_t)kFusedMaxQ * kHistWords * 4 +
                      (size_t)kFusedMaxQ * kFusedMaxGrid * 8 == DSA_WS_ZERO_BYTES,
              "the zeroed workspace prefix is documented in dsa.h");

// ------------------------------------------------------------ grid barrier

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Every CTA of the grid arrives; the last one resets the count and advances
// the generation word that the others wait on (a bounded wait: on timeout the
// error word is set and false returned).  bar[0] = arrivals, bar[1] = generation.
__device__ bool grid_barrier(uint32_t* bar, volatile int* flag, int32_t* err, int32_t where) {
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const uint32_t gen = ld_acquire_gpu(bar + 1);
        __threadfence();
        const uint32_t arrived = atomicAdd(bar, 1u);
        if (arrived == gridDim.x - 1) {
            atomicExch(bar, 0u);
            __threadfence();
            st_release_gpu(bar + 1, gen + 1);
        } else {
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(bar + 1) == gen) {
                if (globaltimer_ns() - t0 > kWaitNs) {
                    record_error(err, kDevTimeout, where, 6);
                    ok = 0;
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
        *flag = ok;
    }
    __syncthreads();
    return *flag != 0;
}

// ------------------------------------------------------------ block helpers

// Exclusive prefix sum over the CTA in thread order; *total gets the sum.
__device__ int block_excl_scan(int v, int* total, int* red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) red[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int s = lane < kWarps ? red[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, s, off);
            if (lane >= off) s += y;
        }
        if (lane < kWarps) red[lane] = s;
    }
    __syncthreads();
    const int excl = x - v + (wid > 0 ? red[wid - 1] : 0);
    *total = red[kWarps - 1];
    __syncthreads();
    return excl;
}

// In a global histogram of nb bins (nb / kThreads consecutive bins per thread),
// the bin b holding the need-th largest key counted from the top, and the
// count of keys in bins above b.  Result in red[16], red[17].
template <int NB>
__device__ void find_bin(const uint32_t* __restrict__ gh, int need, int* red) {
    constexpr int kPer = NB / kThreads;
    static_assert(kPer == 4 || kPer == 8, "4 or 8 bins per thread");
    uint32_t c[kPer];
    const uint4* src = reinterpret_cast<const uint4*>(gh + threadIdx.x * kPer);
#pragma unroll
    for (int i = 0; i < kPer / 4; ++i) {
        const uint4 v = __ldcg(src + i);
        c[4 * i + 0] = v.x; c[4 * i + 1] = v.y; c[4 * i + 2] = v.z; c[4 * i + 3] = v.w;
    }
    int local = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) local += (int)c[i];
    if (threadIdx.x == 0) { red[16] = 0; red[17] = 0; }
    int total;
    const int excl = block_excl_scan(local, &total, red);
    int above = total - excl - local;                 // keys in the bins of later threads
    if (above < need && above + local >= need) {
#pragma unroll
        for (int i = kPer - 1; i >= 0; --i) {
            if (above + (int)c[i] >= need) {
                red[16] = threadIdx.x * kPer + i;
                red[17] = above;
                break;
            }
            above += (int)c[i];
        }
    }
    __syncthreads();
}

// Adds the shared histogram into the global one and clears it.
template <int NB>
__device__ void flush_hist(uint32_t* hist, uint32_t* __restrict__ gh) {
    __syncthreads();
    for (int i = threadIdx.x; i < NB; i += kThreads) {
        const uint32_t c = hist[i];
        if (c) {
            atomicAdd(gh + i, c);
            hist[i] = 0;
        }
    }
    __syncthreads();
}

// Zeroes words [off, off + len) of every query's global histogram, spread
// over the grid.
__device__ void clear_level(uint32_t* __restrict__ gh, int n_q, int off, int len) {
    const int64_t n = (int64_t)n_q * len;
    for (int64_t e = (int64_t)blockIdx.x * kThreads + threadIdx.x; e < n;
         e += (int64_t)gridDim.x * kThreads)
        gh[(e / len) * kHistWords + off + (e % len)] = 0;
}

__device__ __forceinline__ void put(int32_t* out, int64_t pos, int64_t t, int kpool) {
    if (kpool == 1) {
        out[pos] = (int32_t)t;
    } else {
        for (int r = 0; r < kpool; ++r) out[pos * kpool + r] = (int32_t)(t * kpool + r);
    }
}

// The epilogue policy: scores to the workspace row of the query.
struct ScoreStore {
    float* scores;
    int64_t ld;
    __device__ void begin() {}
    __device__ void emit(const IdxGroup& G, int j, int64_t t_row, bool valid, int64_t, int, float s) {
        if (valid) scores[(int64_t)(G.q0 + j) * ld + t_row] = s;
    }
};

__global__ void __launch_bounds__(kThreads, 1)
index_select_fused(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   const float* __restrict__ w, BatchDev bq, int32_t top_k, int32_t kpool,
                   float* __restrict__ scores, int64_t ld, int32_t* __restrict__ idx,
                   int32_t* __restrict__ n_sel, int64_t width, uint32_t* __restrict__ ghist,
                   int2* __restrict__ gcnt, uint32_t* gbar, int32_t* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int cta = blockIdx.x, grid = gridDim.x;

    const int64_t n_groups = local_decode_plan<C>(smem, bq, kpool, err, /*where=*/6);
    const IdxGroup* gs = reinterpret_cast<const IdxGroup*>(smem + C::kOffPlanG);
    const int64_t* ts = reinterpret_cast<const int64_t*>(smem + C::kOffPlanT);
    const int64_t U = ts[n_groups];
    const int64_t u_begin = (int64_t)cta * U / grid, u_end = (int64_t)(cta + 1) * U / grid;
    const int keep = top_k / kpool;
    const bool fits = u_end - u_begin <= (int64_t)kMaxCtaTiles;
    if (!fits && tid == 0) record_error(err, kDevBadBatch, cta, 6);

    // ---- scores of this CTA's units
    if (u_begin < u_end && fits) {
        ScoreStore epi{scores, ld};
        run<1, C::kStages>(smem, &tm_k, &tm_q, gs, ts, n_groups, u_begin, u_end, w, kpool, epi, err);
    }
    fence_proxy_async_smem();                 // the ring is reused by generic accesses

    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
    SegState* seg = reinterpret_cast<SegState*>(smem + kOffSeg);
    int* red = reinterpret_cast<int*>(smem + kOffRed);
    volatile int* flag = red + 20;
    volatile int* s_nseg = red + 21;

    // ---- this CTA's part of each query (sparse queries only) and whole rows
    for (int i = tid; i < kBins1; i += kThreads) hist[i] = 0;
    if (tid == 0) {
        int ns = 0;
        if (u_begin < u_end && fits) {
            int64_t g = 0;
            while (ts[g + 1] <= u_begin) ++g;
            for (; g < n_groups && ts[g] < u_end; ++g) {
                const int64_t ul = ts[g] > u_begin ? ts[g] : u_begin;
                const int64_t uh = ts[g + 1] < u_end ? ts[g + 1] : u_end;
                if (ul >= uh) continue;
                const int64_t nk = gs[g].L_last / kpool;
                if (nk <= keep) continue;                         // dense: no selection
                const int64_t t_lo = (ul - ts[g]) * kTileKeys;
                int64_t t_hi = (uh - ts[g]) * kTileKeys;
                if (t_hi > nk) t_hi = nk;
                SegState S{};
                S.q = gs[g].q0;
                S.n = (int32_t)(t_hi - t_lo);
                S.koff = (int32_t)((ul - u_begin) * kTileKeys);
                S.t_lo = (int32_t)t_lo;
                seg[ns++] = S;
            }
        }
        *s_nseg = ns;
    }
    // rows one CTA writes whole: failed and dense queries; the tail and the
    // padding of sparse rows (the selected body is written by the emission)
    for (int q = cta; q < bq.n_q; q += grid) {
        const IdxGroup G = gs[q];
        int32_t* out = idx + (int64_t)q * width;
        int64_t from, to_sel, L_sel, n_tot;
        if (G.nq == 0) {
            from = 0; to_sel = 0; L_sel = 0; n_tot = 0;
        } else {
            const int64_t L = G.L_last, nk = L / kpool;
            if (nk <= keep) {
                from = 0; to_sel = L; L_sel = 0; n_tot = L;
            } else {
                from = (int64_t)keep * kpool;
                to_sel = from + (L - nk * kpool);
                L_sel = nk * kpool - from;          // out[i] = i + L_sel on [from, to_sel)
                n_tot = to_sel;
            }
        }
        for (int64_t i = from + tid; i < width; i += kThreads)
            out[i] = i < to_sel ? (int32_t)(i + L_sel) : -1;
        if (tid == 0) n_sel[q] = (int32_t)n_tot;
    }
    __syncthreads();
    const int nseg = *s_nseg;

    // ---- level 1: keys into shared memory, histogram of bits 31..21
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];
        const float* src = scores + (int64_t)S.q * ld + S.t_lo;
        for (int i = tid; i < S.n; i += kThreads) {
            const uint32_t k = order_key(__ldcg(src + i));
            keys[S.koff + i] = k;
            atomicAdd(&hist[k >> 21], 1u);
        }
        flush_hist<kBins1>(hist, ghist + (int64_t)S.q * kHistWords);
    }
    if (!grid_barrier(gbar, flag, err, 61)) return;

    // ---- level 2: bits 20..10 of the keys in b1
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];          // read before the helpers' barriers
        uint32_t* gh = ghist + (int64_t)S.q * kHistWords;
        find_bin<kBins1>(gh, keep, red);
        const uint32_t b1 = (uint32_t)red[16];
        if (tid == 0) { seg[s].prefix = b1; seg[s].above = red[17]; }
        for (int i = tid; i < S.n; i += kThreads) {
            const uint32_t k = keys[S.koff + i];
            if ((k >> 21) == b1) atomicAdd(&hist[(k >> 10) & (kBins2 - 1)], 1u);
        }
        flush_hist<kBins2>(hist, gh + kBins1);
    }
    if (!grid_barrier(gbar, flag, err, 62)) return;
    clear_level(ghist, bq.n_q, 0, kBins1);

    // ---- level 3: bits 9..0 of the keys in (b1, b2)
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];
        uint32_t* gh = ghist + (int64_t)S.q * kHistWords;
        find_bin<kBins2>(gh + kBins1, keep - S.above, red);
        const uint32_t prefix = (S.prefix << 11) | (uint32_t)red[16];
        if (tid == 0) { seg[s].prefix = prefix; seg[s].above = S.above + red[17]; }
        for (int i = tid; i < S.n; i += kThreads) {
            const uint32_t k = keys[S.koff + i];
            if ((k >> 10) == prefix) atomicAdd(&hist[k & (kBins3 - 1)], 1u);
        }
        flush_hist<kBins3>(hist, gh + kBins1 + kBins2);
    }
    if (!grid_barrier(gbar, flag, err, 63)) return;
    clear_level(ghist, bq.n_q, kBins1, kBins2);

    // ---- T exact; this CTA's counts above and at T
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];
        const uint32_t* gh = ghist + (int64_t)S.q * kHistWords;
        find_bin<kBins3>(gh + kBins1 + kBins2, keep - S.above, red);
        const uint32_t T = (S.prefix << 10) | (uint32_t)red[16];
        const int above = S.above + red[17];
        int gt = 0, eq = 0;
        for (int i = tid; i < S.n; i += kThreads) {
            const uint32_t k = keys[S.koff + i];
            gt += k > T;
            eq += k == T;
        }
        int tot_gt, tot_eq;
        block_excl_scan(gt, &tot_gt, red);
        block_excl_scan(eq, &tot_eq, red);
        if (tid == 0) {
            seg[s].prefix = T;
            seg[s].need_eq = keep - above;
            seg[s].eq = tot_eq;
            gcnt[(int64_t)S.q * kFusedMaxGrid + cta] = make_int2(tot_gt, tot_eq);
        }
        __syncthreads();
    }
    if (!grid_barrier(gbar, flag, err, 64)) return;
    clear_level(ghist, bq.n_q, kBins1 + kBins2, kBins3);
    pdl_trigger();

    // ---- emission
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];
        const int64_t q_first_unit = ts[S.q];
        if (warp == 0) {
            // CTAs before this one that hold keys of the query
            int g_before = 0, e_before = 0;
            for (int c = lane; c < cta; c += 32) {
                const int64_t ub = (int64_t)c * U / grid, ue = (int64_t)(c + 1) * U / grid;
                if (ub < ue && ue > q_first_unit) {
                    const int2 v = __ldcg(gcnt + (int64_t)S.q * kFusedMaxGrid + c);
                    g_before += v.x;
                    e_before += v.y;
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                g_before += __shfl_xor_sync(0xffffffffu, g_before, off);
                e_before += __shfl_xor_sync(0xffffffffu, e_before, off);
            }
            if (lane == 0) {
                const int taken_before = e_before < S.need_eq ? e_before : S.need_eq;
                int take = S.need_eq - e_before;
                take = take < 0 ? 0 : (take > S.eq ? S.eq : take);
                red[18] = g_before + taken_before;
                red[19] = take;
            }
        }
        __syncthreads();
        const int base = red[18], take = red[19];
        const bool partial = take > 0 && take < S.eq;     // uniform in the CTA
        const uint32_t T = S.prefix;
        int32_t* out = idx + (int64_t)S.q * width;
        int sel_carry = 0, eq_carry = 0;
        for (int c0 = 0; c0 < S.n; c0 += kThreads * kItems) {
            const int j0 = c0 + tid * kItems;
            uint32_t k[kItems];
#pragma unroll
            for (int r = 0; r < kItems; ++r)
                k[r] = j0 + r < S.n ? keys[S.koff + j0 + r] : 0u;
            int eq_rank = 0;
            if (partial) {
                int ne = 0;
#pragma unroll
                for (int r = 0; r < kItems; ++r) ne += (j0 + r < S.n) && k[r] == T;
                int tot;
                eq_rank = eq_carry + block_excl_scan(ne, &tot, red);
                eq_carry += tot;
            }
            uint32_t selmask = 0;
#pragma unroll
            for (int r = 0; r < kItems; ++r) {
                if (j0 + r >= S.n) continue;
                bool sel = k[r] > T;
                if (k[r] == T) {
                    sel = partial ? eq_rank < take : take > 0;
                    ++eq_rank;
                }
                selmask |= (uint32_t)sel << r;
            }
            int tot;
            int pos = base + sel_carry + block_excl_scan(__popc(selmask), &tot, red);
            sel_carry += tot;
#pragma unroll
            for (int r = 0; r < kItems; ++r) {
                // positions stay below keep when the counts are consistent; the
                // check keeps a corrupted state from writing past the row
                if ((selmask & (1u << r)) && (unsigned)pos < (unsigned)keep)
                    put(out, pos, (int64_t)S.t_lo + j0 + r, kpool);
                pos += (selmask >> r) & 1u;
            }
        }
    }
}

}  // namespace

bool index_select_fused_enabled() {
    const char* v = getenv("DSA_FUSED_SELECT");
    return !(v != nullptr && v[0] == '0');
}

bool index_select_fused_eligible(const Shape& sh, const BatchDev& b) {
    if (!index_select_fused_enabled() || !index_scores_tc_eligible(sh, b)) return false;
    if (!(b.max_q_len <= 1 || b.n_q < 8)) return false;           // one query per group
    if (b.n_q < 1 || b.n_q > kFusedMaxQ || b.max_kv_len >= ((int64_t)1 << 31)) return false;
    const int grid = sm_count();
    if (grid > kFusedMaxGrid) return false;
    // Units (key tiles) of the batch, bounded from the host sizes: decode
    // queries of distinct sequences see disjoint keys.
    const int64_t per_q = b.max_kv_len / sh.kpool / kTileKeys + 1;
    int64_t tiles = (int64_t)b.n_q * per_q;
    if (b.max_q_len <= 1) {
        const int64_t t2 = b.total_keys / kTileKeys + b.n_q;
        if (t2 < tiles) tiles = t2;
    }
    return (tiles + grid - 1) / grid <= (int64_t)kMaxCtaTiles;
}

size_t index_select_fused_state_bytes() {
    return (size_t)kFusedMaxQ * kHistWords * 4 +
           (size_t)kFusedMaxQ * kFusedMaxGrid * sizeof(int2);
}

cudaError_t launch_index_select_fused(const Shape& sh, const BatchDev& b, const void* q_idx,
                                      const float* w, const void* k_idx, float* scores,
                                      int64_t ld, int32_t* idx, int32_t* n_sel, void* state,
                                      uint32_t* gbar, int32_t* err, cudaStream_t st) {
    CUtensorMap tm_k, tm_q;
    if (!make_rows128_map(&tm_k, k_idx, (uint64_t)b.total_keys, kTileKeys) ||
        !make_rows128_map(&tm_q, q_idx, (uint64_t)b.n_q * kIdxHeads, C::N))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(index_select_fused,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, index_select_fused, kThreads,
                                                      C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    uint32_t* ghist = static_cast<uint32_t*>(state);
    int2* gcnt = reinterpret_cast<int2*>(ghist + (size_t)kFusedMaxQ * kHistWords);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sm_count());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, index_select_fused, tm_k, tm_q, w, b, sh.top_k, sh.kpool,
                              scores, ld, idx, n_sel, sh.index_row_width(), ghist, gcnt, gbar,
                              err);
}

}  // namespace dsa
