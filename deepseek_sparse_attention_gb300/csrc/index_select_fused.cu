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
// scores and selects in place.  Scores map to order-preserving uint32 keys; the
// selection is every key above the query's k-th largest key T plus the
// lowest-index keys equal to T.  All CTAs holding keys of a query cooperate
// through global memory and grid barriers:
//   score     the tensor-core indexer pipeline (index_pipeline.cuh) turns the
//             CTA's scores into keys in shared memory (a CTA with more units
//             than that region holds writes them to global memory and reads
//             them back, from L2, into the shared memory the ring used);
//   level 1   histogram of key bits 31..21 (2048 bins) per query, added into
//             the query's global histogram;                         barrier 1
//   bin       every CTA finds the bin b1 that holds the k-th largest key; it
//             publishes how many of its keys lie above b1 and appends its keys
//             in b1 -- the candidates, a few thousand per query -- to the
//             query's global candidate list, counting their bits 20..10 in the
//             query's level-2 histogram of candidates;             barrier 2
//   resolve   every CTA finds the level-2 bin b2 in that histogram, reads the
//             whole candidate list and, in one pass, collects the few keys in
//             (b1, b2) -- ranked by one warp for T and the last index taken at
//             T -- and counts the kept ones before its part;
//   emit      a CTA's output offset is the count of selected keys of the CTAs
//             before it (keys above b1 from the published counts, candidates
//             from the list); a block scan writes its selections in order.
// When a query's candidates overflow the list (heavy ties), the grid instead
// resolves that query by two more histogram levels (bits 20..10 and 9..0) and a
// round of per-CTA counts above and at T, three more barriers.  Global
// histograms are cleared by the launch that used them once every CTA has read
// them, the level-2 histogram of candidates (read after the last barrier) by
// the next launch, which uses the other of two copies; candidate counters are
// cleared before the barrier that precedes their first use.  So the state is
// as the next launch expects it.
#include <atomic>

#include "index_pipeline.cuh"

namespace dsa {

namespace {

using namespace sm100;
using namespace idxp;

using C = Cfg<1, 5>;                                  // five stages: room for the keys below
constexpr int kThreads = C::kThreads;                 // 256
constexpr int kWarps = kThreads / 32;
constexpr int kBits1 = 11, kBits2 = 11, kBits3 = 10;  // 11 + 11 + 10 = 32 key bits
constexpr int kBins1 = 1 << kBits1;
constexpr int kBins2 = 1 << kBits2;
constexpr int kBins3 = 1 << kBits3;
constexpr int kShift1 = 32 - kBits1;                  // 21
constexpr int kShift2 = kBits3;                       // 10
constexpr int kCandCap = 8192;                        // candidates per query
constexpr int kCandSpec = 3072;                       // read before the count is known

// Global state per query (32-bit words; the stride keeps every part 16-byte aligned).
constexpr int kOffH1 = 0;
constexpr int kOffH2 = kOffH1 + kBins1;
constexpr int kOffH3 = kOffH2 + kBins2;
// bits 20..10 of the candidates, counted as they are appended; two copies,
// the launch count's parity picks one and the launch clears the other (the
// previous launch's, complete before this one starts)
constexpr int kOffH2c = kOffH3 + kBins3;
constexpr int kOffCandN = kOffH2c + 2 * kBins2;     // candidate count (+3 words pad)
constexpr int kOffCand = kOffCandN + 4;              // kCandCap x {key, index}
constexpr int kQueryWords = kOffCand + 2 * kCandCap;
static_assert(kQueryWords % 4 == 0 && kOffCand % 2 == 0, "alignment of the state");
static_assert(kCandSpec % 256 == 0 && kCandSpec <= kCandCap, "speculative candidate reads");
static_assert(kCandCap < (1 << 15), "two candidate counts share one 32-bit sum");

struct SegState {          // one query's part of this CTA's unit range (64 bytes)
    int32_t q;
    int32_t n;             // keys (tokens or pools) in the part
    int32_t koff;          // first key's slot in shared memory
    int32_t t_lo;          // first key's index in the query
    uint32_t prefix;       // resolved high bits of T, then T
    int32_t above;         // keys of the query above the resolved prefix
    int32_t need_eq;       // keys equal to T the query keeps
    int32_t eq;            // keys of this part equal to T
    int32_t c_first;       // first CTA holding keys of the query
    int32_t hot_off;       // first slot of the part's hot list, -1 if it has none
    int64_t row0;          // the query's first cache row (for prefetches)
    int32_t n_hot;         // entries of the hot list
    int32_t pad[3];
};
static_assert(sizeof(SegState) == 64, "state layout");

// Shared memory.  Beside the indexer pipeline's layout: a histogram (the
// epilogue's level-1 counts, later every shared-memory level), per-query state
// and scan scratch.  After the pipeline its ring (C::kOffA .. C::kOffB) holds
// the CTA's keys and the staged candidate list.
constexpr uint32_t kOffHist = (C::kOffPlanT + (C::kLocalMaxQ + 1) * 8 + 15) / 16 * 16;
constexpr uint32_t kOffSeg = kOffHist + kBins1 * 4;
constexpr uint32_t kOffRed = kOffSeg + kFusedMaxQ * sizeof(SegState);
constexpr uint32_t kOffRow0 = kOffRed + 256;             // [kFusedMaxQ] int64: first cache rows
constexpr uint32_t kOffSmall = kOffRow0 + kFusedMaxQ * 8;  // [kSmallMax] {key, index}
constexpr int kSmallMax = 32;
// The CTA's keys, written there by the epilogue when its units fit (a
// CTA with more units writes them to global memory and reads them back into
// the ring once scoring is done).
constexpr uint32_t kOffSKeys = kOffSmall + kSmallMax * 8;
constexpr uint32_t kSKeyTiles = 80;
constexpr uint32_t kSmemBytes = kOffSKeys + kSKeyTiles * kTileKeys * 4 + 1024;  // + alignment slack
constexpr uint32_t kOffCandS = C::kOffB - (uint32_t)kCandCap * 8;
constexpr uint32_t kMaxCtaKeys = kOffCandS / 4;
constexpr uint32_t kMaxCtaTiles = kMaxCtaKeys / kTileKeys;
static_assert(C::kOffA == 0, "keys start at the ring");
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(kBins2 <= kBins1 && kBins3 <= kBins1, "one shared histogram serves every level");
static_assert(kWsHeaderBytes + (size_t)kFusedMaxQ * kQueryWords * 4 +
                      (size_t)kFusedMaxQ * kFusedMaxGrid * 8 == DSA_WS_ZERO_BYTES,
              "the zeroed workspace prefix is documented in dsa.h");
static_assert(kWsGridBarOffset % 8 == 0, "64-bit barrier counter");
static_assert(kMaxCtaTiles >= 128, "room for the keys of a CTA");


// Scratch words in `red`: [0, kWarps) scans, then named results.
// [32, 32 + kFusedMaxQ) each query's candidate count.
enum : int { kR0 = 16, kR1 = 17, kR2 = 18, kR3 = 19, kRFlag = 20, kRNseg = 21, kROver = 22,
             kRHistQ = 23, kRSmallN = 24, kRT = 25, kRTLast = 26, kRHotRun = 27,
             kRSmallBefore = 28, kRPar = 29, kROnePart = 30 };
// The hot lists: per part, in index order, the part's keys in or above the
// threshold bin b1 as {key, index in the part} -- every key the selection can
// take -- at the start of the ring, which holds no keys when they went straight
// to shared memory (below the staged candidates).
constexpr int kHotCap = (int)(kOffCandS / 8);
static_assert(32 + kFusedMaxQ <= 64, "scratch words");

// ------------------------------------------------------------ grid barrier

// A plain (relaxed) load at GPU scope: the value only, no ordering -- an
// acquire would hold back every later memory access of the thread until it
// returns.
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Every CTA arrives once on a 64-bit counter that only grows; the barrier is
// complete when the counter reaches the next multiple of the grid size.  The
// counter starts at zero and each launch adds a whole number of grid sizes, so
// the value a CTA reads once its launch may start -- earlier launches done,
// this one's first barrier not yet complete without this CTA -- rounds down to
// the launch's base.  Thread 0 of each CTA keeps the count that completes its
// next barrier.
struct GridBar {
    unsigned long long* ctr;
    unsigned long long seen;     // the counter when the launch began (thread 0)
    unsigned long long next;     // 0 until the first barrier derives it
    uint64_t budget;             // the workspace's wait budget, 0 = default
    unsigned long long target;   // the count that completes the barrier arrived at
};

__device__ __forceinline__ void red_release_add_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Arrival by a releasing reduction (no return trip): every thread's writes
// before it are visible to the CTAs that complete the barrier.  Work that no
// other CTA needs before the barrier may run between the arrival and the wait.
__device__ void grid_arrive(GridBar& gb) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned long long g = gridDim.x;
        if (gb.next == 0) gb.next = gb.seen - gb.seen % g + g;
        gb.target = gb.next;
        gb.next += g;
        red_release_add_u64(gb.ctr, 1ull);
    }
}

// Acquire loads until every CTA has arrived, for at most the wait budget: on
// timeout the error word is set and false returned.
__device__ bool grid_wait(GridBar& gb, int* red, int32_t* err, int32_t where) {
    if (threadIdx.x == 0) {
        int ok = 1;
        const unsigned long long target = gb.target;
        const uint64_t budget_ns = gb.budget != 0 ? gb.budget : kDefaultWaitNs;
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_u64(gb.ctr) < target) {
            if (globaltimer_ns() - t0 > budget_ns) {
                record_error(err, kDevTimeout, where, 6);
                ok = 0;
                break;
            }
        }
        *reinterpret_cast<volatile int*>(red + kRFlag) = ok;
    }
    __syncthreads();
    return *reinterpret_cast<volatile int*>(red + kRFlag) != 0;
}

__device__ __forceinline__ bool grid_barrier(GridBar& gb, int* red, int32_t* err, int32_t where) {
    grid_arrive(gb);
    return grid_wait(gb, red, err, where);
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

__device__ __forceinline__ int block_sum(int v, int* red) {
    int tot;
    block_excl_scan(v, &tot, red);
    return tot;
}

// In a histogram of NB bins (NB / kThreads consecutive bins per thread; global
// memory read through L2, or shared memory), the bin b holding the need-th
// largest key counted from the top, and the count of keys in bins above b:
// red[kR0] = b, red[kR1] = count.  (0, 0) if the histogram holds fewer keys.
template <int NB, bool kGlobal>
__device__ void find_bin(const uint32_t* hist, int need, int* red) {
    constexpr int kPer = NB / kThreads;
    static_assert(kPer % 2 == 0 && kPer >= 2, "bins per thread");
    uint32_t c[kPer];
    if (kGlobal && kPer % 4 == 0) {
        const uint4* src = reinterpret_cast<const uint4*>(hist + threadIdx.x * kPer);
#pragma unroll
        for (int i = 0; i < kPer / 4; ++i) {
            const uint4 v = __ldcg(src + i);
            c[4 * i + 0] = v.x; c[4 * i + 1] = v.y; c[4 * i + 2] = v.z; c[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            c[i] = kGlobal ? __ldcg(hist + threadIdx.x * kPer + i) : hist[threadIdx.x * kPer + i];
    }
    int local = 0;
#pragma unroll
    for (int i = 0; i < kPer; ++i) local += (int)c[i];
    if (threadIdx.x == 0) { red[kR0] = 0; red[kR1] = 0; }
    int total;
    const int excl = block_excl_scan(local, &total, red);
    int above = total - excl - local;                 // keys in the bins of later threads
    if (above < need && above + local >= need) {
#pragma unroll
        for (int i = kPer - 1; i >= 0; --i) {
            if (above + (int)c[i] >= need) {
                red[kR0] = threadIdx.x * kPer + i;
                red[kR1] = above;
                break;
            }
            above += (int)c[i];
        }
    }
    __syncthreads();
}

// Adds the first NB bins of the shared histogram into the global one and
// clears them.
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

// Zeroes words [off, off + len) of every query's global state, spread over the grid.
__device__ void clear_level(uint32_t* __restrict__ gs, int n_q, int off, int len) {
    const int n = n_q * len;                            // at most 16 x 2048
    for (int e = blockIdx.x * kThreads + threadIdx.x; e < n; e += gridDim.x * kThreads)
        gs[(size_t)(e / len) * kQueryWords + off + (e % len)] = 0;
}

__device__ __forceinline__ void put(int32_t* out, int64_t pos, int64_t t, int kpool) {
    if (kpool == 1) {
        out[pos] = (int32_t)t;
    } else {
        for (int r = 0; r < kpool; ++r) out[pos * kpool + r] = (int32_t)(t * kpool + r);
    }
}

// Loads, by warp 0, the published counts of the CTAs c_first .. this one - 1
// (every CTA holding keys of the query before this one; a CTA without units
// publishes zeros): up to 8 per lane, all issued at once.  sum_counts()
// reduces them later.
constexpr int kCntPerLane = kFusedMaxGrid / 32;
struct CountLoads {
    int2 v[kCntPerLane];
};
__device__ __forceinline__ void load_counts(const int2* __restrict__ gcnt_q, int c_first,
                                            CountLoads& cl) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 0; k < kCntPerLane; ++k) {
        const int c = c_first + lane + 32 * k;
        cl.v[k] = c < (int)blockIdx.x ? __ldcg(gcnt_q + c) : make_int2(0, 0);
    }
}
// Warp 0: sums of .x and .y into red[kR2], red[kR3].
__device__ __forceinline__ void sum_counts(const CountLoads& cl, int* red) {
    int a = 0, b = 0;
#pragma unroll
    for (int k = 0; k < kCntPerLane; ++k) { a += cl.v[k].x; b += cl.v[k].y; }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
    }
    if ((threadIdx.x & 31) == 0) { red[kR2] = a; red[kR3] = b; }
}

// Writes this CTA's selections of one query in ascending order from position
// `base`: keys above T, and keys equal to T that are taken -- by index (at most
// t_last) or, when `ranked`, the first `take` of them in this part.  Each
// thread owns a contiguous run of the part's keys (thread order = index
// order): a count, one block scan for the offsets (two when ranked), a write.
__device__ void emit_part(const SegState& S, const uint32_t* keys, uint32_t T, int base,
                          int32_t t_last, bool ranked, int take, int keep, int kpool,
                          int32_t* out, int* red) {
    const int tid = threadIdx.x;
    const int per = (S.n + kThreads - 1) / kThreads;
    const int j_a = tid * per < S.n ? tid * per : S.n;
    const int j_b = j_a + per < S.n ? j_a + per : S.n;
    const uint32_t* k = keys + S.koff;
    int n_gt = 0, n_eq = 0, n_eq_ok = 0;
    for (int j = j_a; j < j_b; ++j) {
        const uint32_t x = k[j];
        n_gt += x > T;
        n_eq += x == T;
        n_eq_ok += x == T && S.t_lo + j <= t_last;
    }
    int eq_rank = 0, tot;
    if (ranked) {
        eq_rank = block_excl_scan(n_eq, &tot, red);
        int t = take - eq_rank;
        n_eq_ok = t < 0 ? 0 : (t > n_eq ? n_eq : t);
    }
    int pos = base + block_excl_scan(n_gt + n_eq_ok, &tot, red);
    for (int j = j_a; j < j_b; ++j) {
        const uint32_t x = k[j];
        bool sel = x > T;
        if (x == T) {
            sel = ranked ? eq_rank < take : S.t_lo + j <= t_last;
            ++eq_rank;
        }
        // positions stay below keep when the counts are consistent; the check
        // keeps a corrupted state from writing past the row
        if (sel) {
            if ((unsigned)pos < (unsigned)keep) put(out, pos, (int64_t)S.t_lo + j, kpool);
            ++pos;
        }
    }
}

// Writes this CTA's selections of one query from the part's hot list (every
// key in or above the threshold bin, in index order): keys above T and keys
// equal to T at index <= t_last, in ascending order from position `base`.
// One block scan per kThreads entries (a few hundred keys out of thousands).
__device__ void emit_hot(const SegState& S, const int2* hot, uint32_t T, int base, int32_t t_last,
                         int keep, int kpool, int32_t* out, int* red) {
    for (int c0 = 0; c0 < S.n_hot; c0 += kThreads) {
        const int i = c0 + threadIdx.x;
        int2 e = make_int2(0, 0);
        bool sel = false;
        if (i < S.n_hot) {
            e = hot[S.hot_off + i];
            const uint32_t x = (uint32_t)e.x;
            sel = x > T || (x == T && S.t_lo + e.y <= t_last);
        }
        int tot;
        const int off = block_excl_scan(sel ? 1 : 0, &tot, red);
        // positions stay below keep when the counts are consistent; the check
        // keeps a corrupted state from writing past the row
        if (sel && (unsigned)(base + off) < (unsigned)keep)
            put(out, base + off, (int64_t)S.t_lo + e.y, kpool);
        base += tot;
    }
}

// Resolves one query from its candidate list (all keys in bin b1, staged in
// shared memory as {key, index}): T, the last index taken at T, and this CTA's
// output offset; then emits.  `need` = keep - (keys above b1); n_cand <= kCandCap.
// The first `staged` entries of the list and (warp 0) the counts `cl` of the
// earlier CTAs may already be loaded, and the level-2 bin b2 with the count of
// candidates above it (have_b2) taken from the query's global level-2
// histogram of its candidates, `h2c`.
__device__ void resolve_from_candidates(const SegState& S, const uint32_t* gsq,
                                        const uint32_t* h2c, const int2* __restrict__ gcnt_q,
                                        int n_cand, int staged, CountLoads& cl,
                                        bool counts_loaded, bool have_b2, uint32_t b2,
                                        int above2, int need, uint32_t b1,
                                        const uint32_t* keys, uint32_t* hist, int2* cand,
                                        const int2* hot, int keep, int kpool, int32_t* out,
                                        int* red) {
    const int tid = threadIdx.x;
    if (tid < 32 && !counts_loaded) load_counts(gcnt_q, S.c_first, cl);
    if (!have_b2) {
        find_bin<kBins2, true>(h2c, need, red);
        b2 = (uint32_t)red[kR0];
        above2 = red[kR1];
    }
    const int2* src = reinterpret_cast<const int2*>(gsq + kOffCand);
    for (int i0 = staged; i0 < n_cand; i0 += 4 * kThreads) {   // four loads in flight
        int2 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = i0 + tid + k * kThreads;
            v[k] = i < n_cand ? __ldcg(src + i) : make_int2(0, 0);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (i0 + tid + k * kThreads < n_cand) cand[i0 + tid + k * kThreads] = v[k];
    }
    if (tid == 0) { red[kRSmallN] = 0; red[kRT] = -1; red[kRTLast] = -1; red[kRSmallBefore] = 0; }
    __syncthreads();
    const uint32_t pre = (b1 << kBits2) | b2;
    // One pass over the list.  The kept keys are the first `need` of the
    // query's candidates in the order (key descending, index ascending).  A
    // candidate above (b1, b2) in its 22 high bits is kept, one below is not;
    // those in (b1, b2) -- usually a handful -- go to a small list, where the
    // last kept one is the (need - above2)-th in that order: its key is T and
    // its index the last one taken at T (every key equal to T is in the list).
    // The pass also counts the kept candidates above (b1, b2) that come
    // before this part's first index.
    int2* small = reinterpret_cast<int2*>(reinterpret_cast<uint8_t*>(red) - kOffRed + kOffSmall);
    int before = 0;
    for (int i = tid; i < n_cand; i += kThreads) {
        const int2 e = cand[i];
        const uint32_t hi = (uint32_t)e.x >> kShift2;
        if (hi == pre) {
            const int slot = atomicAdd(&red[kRSmallN], 1);
            if (slot < kSmallMax) small[slot] = e;
        } else {
            before += hi > pre && e.y < S.t_lo;
        }
    }
    before = block_sum(before, red);
    const int m = red[kRSmallN];
    uint32_t T;
    int32_t t_last;
    if (m <= kSmallMax) {
        if (tid < 32) {                               // one warp ranks the list
            const int2 e = tid < m ? small[tid] : make_int2(0, 0);
            const uint32_t ek = (uint32_t)e.x;
            int rank = 0;
            for (int j = 0; j < m; ++j) {
                const uint32_t kj = __shfl_sync(0xffffffffu, ek, j);
                const int32_t ij = __shfl_sync(0xffffffffu, e.y, j);
                rank += kj > ek || (kj == ek && ij < e.y);
            }
            const unsigned who = __ballot_sync(0xffffffffu, tid < m && rank == need - above2 - 1);
            uint32_t t = 0xffffffffu;
            int32_t tl = -1;
            if (who != 0u) {
                const int w = __ffs(who) - 1;
                t = __shfl_sync(0xffffffffu, ek, w);
                tl = __shfl_sync(0xffffffffu, e.y, w);
            }
            // kept entries of the small list before this part's first index
            const bool kept = tid < m && (ek > t || (ek == t && e.y <= tl));
            const int nb = __popc(__ballot_sync(0xffffffffu, kept && e.y < S.t_lo));
            if (tid == 0) { red[kRT] = (int)t; red[kRTLast] = tl; red[kRSmallBefore] = nb; }
            sum_counts(cl, red);
        }
        __syncthreads();
        T = (uint32_t)red[kRT];
        t_last = red[kRTLast];
        before += red[kRSmallBefore];
    } else {
        // more than kSmallMax keys share 22 bits (exact ties): bits 9..0 by a
        // histogram, then the need_eq-th smallest index among the keys at T
        for (int i = tid; i < n_cand; i += kThreads) {
            const uint32_t k = (uint32_t)cand[i].x;
            if ((k >> kShift2) == pre) atomicAdd(&hist[k & (kBins3 - 1)], 1u);
        }
        __syncthreads();
        find_bin<kBins3, false>(hist, need - above2, red);
        T = (pre << kBits3) | (uint32_t)red[kR0];
        const int need_eq = need - above2 - red[kR1];  // keys equal to T that are kept
        for (int i = tid; i < kBins3; i += kThreads) hist[i] = 0;
        int n_eq = 0;
        for (int i = tid; i < n_cand; i += kThreads) n_eq += (uint32_t)cand[i].x == T;
        n_eq = block_sum(n_eq, red);
        t_last = 0x7fffffff;
        if (need_eq < n_eq) {
            if (tid == 0) red[kR0] = -1;
            __syncthreads();
            for (int i = tid; i < n_cand; i += kThreads) {
                if ((uint32_t)cand[i].x != T) continue;
                const int32_t ti = cand[i].y;
                int rank = 0;
                for (int j = 0; j < n_cand; ++j) rank += (uint32_t)cand[j].x == T && cand[j].y < ti;
                if (rank == need_eq - 1) red[kR0] = ti;
            }
            __syncthreads();
            t_last = red[kR0];
        }
        // kept candidates of the small list's bits before this part's first index
        int b_eq = 0;
        for (int i = tid; i < n_cand; i += kThreads) {
            const uint32_t k = (uint32_t)cand[i].x;
            const int32_t ti = cand[i].y;
            b_eq += (k >> kShift2) == pre && ti < S.t_lo && (k > T || (k == T && ti <= t_last));
        }
        before += block_sum(b_eq, red);
        if (tid < 32) sum_counts(cl, red);
        __syncthreads();
    }
    const int base = red[kR2] + before;
    if (S.hot_off >= 0) emit_hot(S, hot, T, base, t_last, keep, kpool, out, red);
    else emit_part(S, keys, T, base, t_last, false, 0, keep, kpool, out, red);
}

// The epilogue policy: each score as its order-preserving key into the
// workspace row of its query, and into the shared level-1 histogram when the
// key belongs to `hist_q` (the first query this CTA selects for).
struct KeyStore {
    uint32_t* keys;        // global [query][ld], or (skeys) shared [unit - u_begin][128]
    int64_t ld;
    uint32_t* skeys;
    int64_t u_begin;
    uint32_t* hist;
    int32_t hist_q;
    __device__ void begin() {}
    __device__ void emit(const IdxGroup& G, int j, int64_t t_row, bool valid, int64_t u, int row,
                         float s) {
        if (!valid) return;
        const uint32_t k = order_key(s);
        if (skeys != nullptr) skeys[(u - u_begin) * kTileKeys + row] = k;
        else keys[(int64_t)(G.q0 + j) * ld + t_row] = k;
        if (G.q0 + j == hist_q) atomicAdd(&hist[k >> kShift1], 1u);
    }
};

// kSpec: the instantiation for batches whose host scalars imply their plan
// (spec_plan_guess), which guesses its first key tiles before the batch
// offsets are read (spec_issue / spec_settle); other batches run the one
// without that code.
template <bool kSpec>
__global__ void __launch_bounds__(kThreads, 1)
index_select_fused(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   const float* __restrict__ w, BatchDev bq, int32_t top_k, int32_t kpool,
                   uint32_t* __restrict__ gkeys, int64_t ld, int32_t* __restrict__ idx,
                   int32_t* __restrict__ n_sel, int64_t width, uint32_t* __restrict__ gstate,
                   int2* __restrict__ gcnt, unsigned long long* gbar,
                   const uint8_t* __restrict__ pf_cache, int64_t pf_row_bytes, int32_t* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x;
    const int cta = blockIdx.x, grid = gridDim.x;
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);     // re-pointed below when direct
    uint32_t* hist = reinterpret_cast<uint32_t*>(smem + kOffHist);
    int2* cand = reinterpret_cast<int2*>(smem + kOffCandS);
    SegState* seg = reinterpret_cast<SegState*>(smem + kOffSeg);
    int* red = reinterpret_cast<int*>(smem + kOffRed);

    setup<1, C::kStages>(smem, &tm_k, &tm_q);  // local to the CTA: before the wait
    pdl_wait();                               // the inputs of the previous kernels
    // thread 0: the barrier counter's value at the start and the budget of the
    // waits on other CTAs (workspace header); both first used at barrier 1
    GridBar gb{gbar, 0, 0, 0, 0};
    uint32_t* launch_count = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(err) +
                                                         kWsLaunchCountOffset);
    uint32_t n_launch = 0;                    // thread 0: first used after scoring
    if (tid == 0) {
        gb.seen = ld_relaxed_u64(gbar);
        gb.budget = *reinterpret_cast<const volatile uint64_t*>(
            reinterpret_cast<const uint8_t*>(err) + kWsWaitBudgetOffset);
        n_launch = *reinterpret_cast<const volatile uint32_t*>(launch_count);
    }
    // thread 32: a single query's first key tiles, guessed from the batch's
    // bounds, while thread 0 reads the batch offsets (checked after the plan)
    if (kSpec && tid == 32)
        spec_issue<1, C::kStages>(smem, &tm_k, &tm_q, bq, kpool, cta, grid, (int64_t)kMaxCtaTiles);
    int64_t* row0s = reinterpret_cast<int64_t*>(smem + kOffRow0);
    const int64_t n_groups = local_decode_plan<C>(smem, bq, kpool, err, /*where=*/6, row0s);
    const IdxGroup* gs = reinterpret_cast<const IdxGroup*>(smem + C::kOffPlanG);
    const int64_t* ts = reinterpret_cast<const int64_t*>(smem + C::kOffPlanT);
    const int64_t U = ts[n_groups];
    const int64_t u_begin = mul_div(cta, U, grid), u_end = mul_div(cta + 1, U, grid);
    const int keep = top_k / kpool;
    const bool fits = u_end - u_begin <= (int64_t)kMaxCtaTiles;
    const bool direct = u_end - u_begin <= (int64_t)kSKeyTiles;   // keys straight to shared memory
    if (direct) keys = reinterpret_cast<uint32_t*>(smem + kOffSKeys);
    const int64_t u_run = u_begin < u_end && fits ? u_end : u_begin;   // the range scored
    int pre = 0;                              // thread 0: the first key tiles on their way now
    if (tid == 0)
        pre = kSpec ? spec_settle<1, C::kStages>(smem, &tm_k, &tm_q, bq, kpool, gs, ts, n_groups,
                                                 u_begin, u_run, err, /*where=*/64)
                    : issue_first<1, C::kStages>(smem, &tm_k, &tm_q, gs, ts, n_groups, u_begin,
                                                 u_run);

    // ---- before scoring: only what the epilogue needs, the first query this
    // CTA selects for (its level-1 counts are taken while scoring)
    for (int i = tid; i < kBins1; i += kThreads) hist[i] = 0;
    if (tid == 0) {
        int hq = -1;
        if (u_begin < u_end && fits) {
            int64_t g = 0;
            while (ts[g + 1] <= u_begin) ++g;
            for (; g < n_groups && ts[g] < u_end && hq < 0; ++g)
                // floor(L / kpool) > keep, without the division
                if (ts[g + 1] > ts[g] && gs[g].L_last >= (keep + 1) * kpool) hq = gs[g].q0;
        }
        red[kRHistQ] = hq;
    }
    __syncthreads();

    // ---- scores of this CTA's units (keys to global, level-1 counts of hist_q)
    {                                         // an empty range only releases TMEM
        KeyStore epi{gkeys, ld, direct ? keys : nullptr, u_begin, hist, red[kRHistQ]};
        run<1, C::kStages>(smem, &tm_k, &tm_q, gs, ts, n_groups, u_begin, u_run, w, kpool, epi,
                           err, pre);
    }
    fence_proxy_async_smem();                 // the ring is reused by generic accesses

    // ---- before barrier 1 only what the other CTAs read after it: the
    // candidate counters zeroed and this CTA's level-1 counts -- its first
    // query's, taken while scoring, flushed first.  A CTA whose scored range
    // lies in one query's keys then arrives and does the rest while the others
    // arrive; one straddling queries first counts and flushes its other parts.
    const int hq = red[kRHistQ];
    if (tid == 0) {
        for (int q = cta; q < bq.n_q; q += grid) gstate[(int64_t)q * kQueryWords + kOffCandN] = 0;
        int64_t g = 0;
        while (g + 1 < n_groups && ts[g + 1] <= u_begin) ++g;
        red[kROnePart] = u_run <= u_begin || ts[g + 1] >= u_run;
    }
    if (hq >= 0) flush_hist<kBins1>(hist, gstate + (int64_t)hq * kQueryWords + kOffH1);
    else __syncthreads();
    const bool one_part = red[kROnePart] != 0;
    if (one_part) grid_arrive(gb);

    // ---- this CTA's part of each sparse query (the first is hist_q's), whole rows
    if (tid == 0) {
        int ns = 0;
        if (!fits) record_error(err, kDevBadBatch, cta, 6);
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
                // the CTA whose units contain the query's first unit ts[g]:
                // the smallest c with floor((c + 1) U / grid) > ts[g]
                S.c_first = (int32_t)(mul_div(1, (ts[g] + 1) * grid + U - 1, U) - 1);
                S.row0 = pf_cache != nullptr ? row0s[S.q] : -1;
                seg[ns++] = S;
            }
        }
        red[kRNseg] = ns;
        red[kRPar] = (int)(n_launch & 1u);
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
            const int64_t L = G.L_last, nk = G.L_last / kpool;   // 32-bit division
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
    const int nseg = red[kRNseg];
    const int par = red[kRPar];
    // the previous launch's copy, for every query it may have had
    clear_level(gstate, kFusedMaxQ, kOffH2c + (par ^ 1) * kBins2, kBins2);

    // ---- keys back into shared memory (asynchronous copies, 16 bytes each:
    // part starts are tile-aligned and rows padded to 4 keys), the other
    // parts' level-1 counts
    for (int s = 0; s < nseg && !direct; ++s) {
        const SegState S = seg[s];
        const uint32_t* src = gkeys + (int64_t)S.q * ld + S.t_lo;
        const uint32_t dst = smem_u32(keys + S.koff);
        for (int c = tid; c < (S.n + 3) / 4; c += kThreads)
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16 * c),
                         "l"(src + 4 * c)
                         : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    for (int s = 1; s < nseg; ++s) {
        const SegState S = seg[s];
        for (int i = tid; i < S.n; i += kThreads) atomicAdd(&hist[keys[S.koff + i] >> kShift1], 1u);
        flush_hist<kBins1>(hist, gstate + (int64_t)S.q * kQueryWords + kOffH1);
    }
    if (!one_part) grid_arrive(gb);
    if (!grid_wait(gb, red, err, 61)) return;

    // ---- b1; counts above it; candidates in it; the hot lists
    if (tid == 0) red[kRHotRun] = 0;
    int2* hot = reinterpret_cast<int2*>(smem);
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];          // read before the helpers' barriers
        uint32_t* gsq = gstate + (int64_t)S.q * kQueryWords;
        find_bin<kBins1, true>(gsq + kOffH1, keep, red);
        const uint32_t b1 = (uint32_t)red[kR0];
        if (tid == 0) { seg[s].prefix = b1; seg[s].above = red[kR1]; }
        // Pass 1 over this thread's contiguous run of the part (thread order is
        // index order): keys above b1 and in b1.  Keys above b1 are selected
        // whatever the rest of the resolve finds: their cache rows (a pool's
        // kpool rows) go to L2 now, for the attention's gather after this launch.
        const int per = (S.n + kThreads - 1) / kThreads;
        const int j_a = tid * per < S.n ? tid * per : S.n;
        const int j_b = j_a + per < S.n ? j_a + per : S.n;
        int n_above = 0, n_in = 0;
        for (int j = j_a; j < j_b; ++j) {
            const uint32_t bin = keys[S.koff + j] >> kShift1;
            n_above += bin > b1;
            n_in += bin == b1;
            if (bin > b1 && S.row0 >= 0)
                prefetch_l2_bytes(pf_cache + (S.row0 + (int64_t)(S.t_lo + j) * kpool) * pf_row_bytes,
                                  (uint32_t)(kpool * pf_row_bytes));
        }
        // above in the high half, in b1 in the low half (each < 2^16 per CTA)
        int tot;
        const int excl = block_excl_scan((n_above << 16) | n_in, &tot, red);
        if (tid == 0) {
            const int n_in_all = tot & 0xffff, n_hot = (tot >> 16) + n_in_all;
            red[kR2] = n_in_all ? (int)atomicAdd(gsq + kOffCandN, (uint32_t)n_in_all) : 0;
            gcnt[(int64_t)S.q * kFusedMaxGrid + cta] = make_int2(tot >> 16, 0);
            const int run = red[kRHotRun];
            const bool room = direct && run + n_hot <= kHotCap;
            seg[s].hot_off = room ? run : -1;
            seg[s].n_hot = n_hot;
            if (room) red[kRHotRun] = run + n_hot;
        }
        __syncthreads();
        // Pass 2: the hot list and this CTA's candidates in the global list
        if (n_above + n_in > 0) {
            int cpos = red[kR2] + (excl & 0xffff);
            int hpos = seg[s].hot_off >= 0 ? seg[s].hot_off + (excl >> 16) + (excl & 0xffff) : -1;
            int2* dst = reinterpret_cast<int2*>(gsq + kOffCand);
            uint32_t* h2c = gsq + kOffH2c + par * kBins2;
            for (int j = j_a; j < j_b; ++j) {
                const uint32_t k = keys[S.koff + j];
                const uint32_t bin = k >> kShift1;
                if (bin < b1) continue;
                if (hpos >= 0) hot[hpos++] = make_int2((int)k, j);
                if (bin == b1) {
                    if (cpos < kCandCap) dst[cpos] = make_int2((int)k, S.t_lo + j);
                    ++cpos;
                    atomicAdd(h2c + ((k >> kShift2) & (kBins2 - 1)), 1u);
                }
            }
        }
    }
    if (u_begin >= u_end)                   // no units: zero counts for every query
        for (int q = tid; q < bq.n_q; q += kThreads)
            gcnt[(int64_t)q * kFusedMaxGrid + cta] = make_int2(0, 0);
    if (!grid_barrier(gb, red, err, 62)) return;
    clear_level(gstate, bq.n_q, kOffH1, kBins1);

    // this launch's count, for the next one's parity (every CTA read it before barrier 1)
    if (cta == 0 && tid == 0) atomicAdd(launch_count, 1u);

    // ---- one round of loads: every query's candidate count (does any need
    // the histogram levels? grid-uniform), and for the first part the counts of
    // the earlier CTAs, the head of the candidate list and the level-2
    // histogram of the candidates
    int* n_cand_q = red + 32;                         // [kFusedMaxQ]
    CountLoads cl;
    uint32_t b2_0 = 0;
    int above2_0 = 0;
    if (nseg > 0) {
        const int q0 = seg[0].q;
        const uint32_t* gsq0 = gstate + (int64_t)q0 * kQueryWords;
        if (tid < 32) load_counts(gcnt + (int64_t)q0 * kFusedMaxGrid, seg[0].c_first, cl);
        const int2* src = reinterpret_cast<const int2*>(gsq0 + kOffCand);
        int2 v[kCandSpec / kThreads];                 // all in flight at once
#pragma unroll
        for (int k = 0; k < kCandSpec / kThreads; ++k) v[k] = __ldcg(src + tid + k * kThreads);
        // with those loads in flight: the level-2 bin of the first part's query
        find_bin<kBins2, true>(gsq0 + kOffH2c + par * kBins2, keep - seg[0].above, red);
        b2_0 = (uint32_t)red[kR0];
        above2_0 = red[kR1];
#pragma unroll
        for (int k = 0; k < kCandSpec / kThreads; ++k) cand[tid + k * kThreads] = v[k];
    }
    if (tid < 32) {
        int over = 0;
        if (tid < bq.n_q) {
            const uint32_t n = __ldcg(gstate + (int64_t)tid * kQueryWords + kOffCandN);
            n_cand_q[tid] = (int)n;
            over = n > (uint32_t)kCandCap;
        }
        over = __any_sync(0xffffffffu, over);
        if (tid == 0) red[kROver] = over;
    }
    __syncthreads();
    const bool any_over = red[kROver] != 0;

    // ---- resolve from the candidate lists
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];
        const uint32_t* gsq = gstate + (int64_t)S.q * kQueryWords;
        const int n_cand = n_cand_q[S.q];
        if (n_cand > kCandCap) continue;
        const int staged = s == 0 ? (n_cand < kCandSpec ? n_cand : kCandSpec) : 0;
        resolve_from_candidates(S, gsq, gsq + kOffH2c + par * kBins2,
                                gcnt + (int64_t)S.q * kFusedMaxGrid, n_cand, staged, cl, s == 0,
                                s == 0, b2_0, above2_0, keep - S.above, S.prefix, keys, hist, cand,
                                reinterpret_cast<const int2*>(smem), keep, kpool,
                                idx + (int64_t)S.q * width, red);
    }
    if (!any_over) {
        pdl_trigger();
        return;
    }

    // ---- overflow: bits 20..10 of the keys in b1
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];
        uint32_t* gsq = gstate + (int64_t)S.q * kQueryWords;
        if (n_cand_q[S.q] <= kCandCap) continue;
        for (int i = tid; i < S.n; i += kThreads) {
            const uint32_t k = keys[S.koff + i];
            if ((k >> kShift1) == S.prefix) atomicAdd(&hist[(k >> kShift2) & (kBins2 - 1)], 1u);
        }
        flush_hist<kBins2>(hist, gsq + kOffH2);
    }
    if (!grid_barrier(gb, red, err, 63)) return;

    // ---- bits 9..0 of the keys in (b1, b2)
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];
        uint32_t* gsq = gstate + (int64_t)S.q * kQueryWords;
        if (n_cand_q[S.q] <= kCandCap) continue;
        find_bin<kBins2, true>(gsq + kOffH2, keep - S.above, red);
        const uint32_t pre = (S.prefix << kBits2) | (uint32_t)red[kR0];
        if (tid == 0) { seg[s].prefix = pre; seg[s].above = S.above + red[kR1]; }
        for (int i = tid; i < S.n; i += kThreads) {
            const uint32_t k = keys[S.koff + i];
            if ((k >> kShift2) == pre) atomicAdd(&hist[k & (kBins3 - 1)], 1u);
        }
        flush_hist<kBins3>(hist, gsq + kOffH3);
    }
    if (!grid_barrier(gb, red, err, 64)) return;

    // ---- T exact; this CTA's counts above and at T
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];
        const uint32_t* gsq = gstate + (int64_t)S.q * kQueryWords;
        if (n_cand_q[S.q] <= kCandCap) continue;
        find_bin<kBins3, true>(gsq + kOffH3, keep - S.above, red);
        const uint32_t T = (S.prefix << kBits3) | (uint32_t)red[kR0];
        const int above = S.above + red[kR1];
        int gt = 0, eq = 0;
        for (int i = tid; i < S.n; i += kThreads) {
            const uint32_t k = keys[S.koff + i];
            gt += k > T;
            eq += k == T;
        }
        gt = block_sum(gt, red);
        eq = block_sum(eq, red);
        if (tid == 0) {
            seg[s].prefix = T;
            seg[s].need_eq = keep - above;
            seg[s].eq = eq;
            gcnt[(int64_t)S.q * kFusedMaxGrid + cta] = make_int2(gt, eq);
        }
        __syncthreads();
    }
    if (!grid_barrier(gb, red, err, 65)) return;
    clear_level(gstate, bq.n_q, kOffH2, kBins2 + kBins3);
    pdl_trigger();

    // ---- emission of the overflowed queries
    for (int s = 0; s < nseg; ++s) {
        const SegState S = seg[s];
        if (n_cand_q[S.q] <= kCandCap) continue;
        if (tid < 32) {
            CountLoads cl2;
            load_counts(gcnt + (int64_t)S.q * kFusedMaxGrid, S.c_first, cl2);
            sum_counts(cl2, red);
        }
        __syncthreads();
        const int g_before = red[kR2], e_before = red[kR3];
        const int taken_before = e_before < S.need_eq ? e_before : S.need_eq;
        int take = S.need_eq - e_before;
        take = take < 0 ? 0 : (take > S.eq ? S.eq : take);
        __syncthreads();
        // keys equal to T: the first `take` of this part (ranked), or none
        emit_part(S, keys, S.prefix, g_before + taken_before, -1, take > 0, take, keep, kpool,
                  idx + (int64_t)S.q * width, red);
    }
}

}  // namespace

bool index_select_fused_eligible(const Shape& sh, const BatchDev& b) {
    // the two-launch plan on request; descending order needs the scores the
    // two-launch indexer keeps
    if (b.flags & (DSA_FLAG_TWO_LAUNCH | DSA_FLAG_DESC_ORDER | DSA_FLAG_DENSE)) return false;
    if (!index_scores_tc_eligible(sh, b)) return false;
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
    return (size_t)kFusedMaxQ * kQueryWords * 4 +
           (size_t)kFusedMaxQ * kFusedMaxGrid * sizeof(int2);
}

cudaError_t launch_index_select_fused(const Shape& sh, const BatchDev& b, const void* q_idx,
                                      const float* w, const void* k_idx, float* scores,
                                      int64_t ld, int32_t* idx, int32_t* n_sel, void* state,
                                      uint32_t* gbar, const void* cache, int64_t row_bytes,
                                      int32_t* err, cudaStream_t st) {
    CUtensorMap tm_k, tm_q;
    if (!make_rows128_map(&tm_k, k_idx, (uint64_t)b.total_keys, kTileKeys) ||
        !make_rows128_map(&tm_q, q_idx, (uint64_t)b.n_q * kIdxHeads, C::N))
        return cudaErrorInvalidValue;
    int64_t g_nk = 0, g_ns = 0;
    const int spec = spec_plan_guess(b, sh.kpool, &g_nk, &g_ns) ? 1 : 0;
    auto kern = spec ? index_select_fused<true> : index_select_fused<false>;
    cudaError_t e = ensure_dyn_smem((const void*)kern, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    // one CTA must fit an SM (the cooperative grid is one per SM); checked
    // once per device and instantiation
    static std::atomic<int> fits_sm[2][64];
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || fits_sm[spec][dev].load(std::memory_order_relaxed) == 0) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmemBytes);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
        if (dev >= 0 && dev < 64) fits_sm[spec][dev].store(1, std::memory_order_relaxed);
    }
    uint32_t* gstate = static_cast<uint32_t*>(state);
    int2* gcnt = reinterpret_cast<int2*>(gstate + (size_t)kFusedMaxQ * kQueryWords);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sm_count());
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    // Cooperative (every CTA resident: the grid barriers), and with programmatic
    // stream serialization, so that the launch overlaps the previous kernel's
    // tail; the kernel waits for it (griddepcontrol.wait) before reading
    // anything.  Should a driver refuse the pair, the launch is cooperative only.
    static bool pdl_ok = true;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    auto go = [&](unsigned n_attr) {
        cfg.numAttrs = n_attr;
        return cudaLaunchKernelEx(&cfg, kern, tm_k, tm_q, w, b, sh.top_k, sh.kpool,
                                  reinterpret_cast<uint32_t*>(scores), ld, idx, n_sel,
                                  sh.index_row_width(), gstate, gcnt,
                                  reinterpret_cast<unsigned long long*>(gbar),
                                  static_cast<const uint8_t*>(cache), row_bytes, err);
    };
    if (pdl_ok) {
        e = go(2);
        if (e != cudaErrorNotSupported && e != cudaErrorInvalidValue) return e;
        (void)cudaGetLastError();
        pdl_ok = false;
    }
    return go(1);
}

}  // namespace dsa
