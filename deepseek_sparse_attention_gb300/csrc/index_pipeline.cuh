// index_pipeline.cuh -- the warp-specialised tcgen05 indexer pipeline, shared
// by the standalone indexer kernel and the fused decode kernel.
//
// One CTA walks a contiguous range [u_begin, u_end) of (query group, key tile)
// units.  warp 0: TMA producer (key tiles into a shared-memory ring with the
// 128-byte swizzle, the group's query rows once per group); warp 1: one thread
// issues tcgen05.mma (M = 128 keys, N = 32 heads per query, K = 128) into two
// TMEM accumulators; warps 4..: epilogue, one TMEM lane (key) per thread,
// relu and the weighted head sum, handed to an epilogue policy `Epi`:
//   epi.begin()                              once per epilogue thread
//   epi.emit(G, j, t_row, valid, u, row, s)  score s of key t_row of query
//                                            G.q0 + j (valid: t_row is visible)
// All waits are bounded; a timeout sets the error word and winds down.
#pragma once

#include "dsa_kernels.cuh"
#include "sm100.cuh"

namespace dsa {
namespace idxp {

using namespace sm100;

constexpr int kTileKeys = 128;                      // MMA M
constexpr int kIdxDim = 128;                        // MMA K
constexpr int kIdxHeads = 32;
constexpr uint32_t kRowHalfBytes = 128;             // 64 bf16: one swizzle row
constexpr uint32_t kABoxBytes = kTileKeys * kRowHalfBytes;    // 16 KB
constexpr uint32_t kABytes = 2 * kABoxBytes;                  // 32 KB per key tile
constexpr uint64_t kWaitNs = 2000000000ull;         // bounded waits: 2 s

// Host side (index_scores_tc.cu): a tensor map over a row-major [rows, 128]
// bf16 matrix read in boxes of box_rows x 64 columns with the 128-byte swizzle
// (false when the driver entry point is missing or the encoder refuses).
bool make_rows128_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows);

struct IdxGroup {          // consecutive queries of one sequence scored together
    int64_t key0;          // first indexer key of the sequence
    int32_t q0;            // first query of the group
    int32_t nq;            // queries in the group
    int32_t L_last;        // rows seen by the group's last query
    int32_t pad;
};

template <int GQ, int STAGES = (GQ == 1 ? 6 : 4)>
struct Cfg {
    static constexpr int N = kIdxHeads * GQ;
    static constexpr int kStages = STAGES;
    static constexpr uint32_t kBBoxBytes = N * kRowHalfBytes;
    static constexpr uint32_t kBBytes = 2 * kBBoxBytes;
    static constexpr uint32_t kTmemCols = 2 * N;                  // two accumulators
    static constexpr int kEpiWarps = GQ == 1 ? 4 : 16;          // 16: two queries per warpgroup
    static constexpr int kEpiGroups = kEpiWarps / 4;              // warpgroups in the epilogue
    static constexpr int kThreads = (4 + kEpiWarps) * 32;
    static constexpr uint32_t kOffA = 0;
    static constexpr uint32_t kOffB = kStages * kABytes;
    static constexpr uint32_t kOffBar = kOffB + kBBytes;
    // full[S], empty[S], b_full, b_empty, acc_full[2], acc_empty[2], drain
    static constexpr int kNumBars = 2 * kStages + 7;
    static constexpr uint32_t kOffMisc = kOffBar + kNumBars * 8;
    // decode batches plan their (query, key tile) units in shared memory
    static constexpr int kLocalMaxQ = 256;
    // grouped queries: each epilogue warp's copy of its two queries' head weights
    static constexpr uint32_t kOffW = (kOffMisc + 16 + 15) / 16 * 16;
    static constexpr uint32_t kOffPlanG = kOffW + (GQ > 1 ? kEpiWarps * 2 * kIdxHeads * 4 : 0);  // IdxGroup[256]
    static constexpr uint32_t kOffPlanT = kOffPlanG + kLocalMaxQ * 24;             // int64[257]
    static constexpr uint32_t kSmemBytes = kOffPlanT + (kLocalMaxQ + 1) * 8 + 1024;
    static_assert(kTmemCols == 64 || kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512,
                  "TMEM allocation must be a power of two");
};

// Walks (group, tile) units in order.  kCache keeps tile_off[g] and
// tile_off[g + 1] in registers (read once per group: the grouped plan lives in
// global memory); the decode plan is in shared memory and is read directly.
template <bool kCache>
struct Cursor {
    const int64_t* tile_off;
    int64_t g, t;
    int64_t beg, end;                 // kCache: tile_off[g], tile_off[g + 1]
    __device__ int64_t b0() const { return kCache ? beg : tile_off[g]; }
    __device__ int64_t b1() const { return kCache ? end : tile_off[g + 1]; }
    __device__ void seek(int64_t u, int64_t n_groups) {
        int64_t lo = 0, hi = n_groups - 1;           // last g with tile_off[g] <= u
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (tile_off[mid] <= u) lo = mid; else hi = mid - 1;
        }
        g = lo;
        if (kCache) { beg = tile_off[g]; end = tile_off[g + 1]; }
        t = u - tile_off[g];
    }
    __device__ void next() {
        ++t;
        while (b0() + t >= b1()) {
            ++g;
            t = 0;
            if (kCache) { beg = end; end = tile_off[g + 1]; }
        }
    }
    __device__ bool last_of_group() const { return b0() + t + 1 >= b1(); }
};

// One group per query (decode batches of at most Cfg::kLocalMaxQ queries):
// every CTA derives the (group, tile) schedule itself into shared memory --
// groups at kOffPlanG, the exclusive prefix of tiles per group at kOffPlanT --
// and returns the group count.  A query whose offsets fail the batch checks
// gets an empty group (nq = 0, no tiles).  Called by every thread.  `row0`,
// when given, receives each query's first cache row (-1 for a failed query).
template <class C>
__device__ int64_t local_decode_plan(uint8_t* smem, const BatchDev& bq, int32_t kpool,
                                     int32_t* err, int32_t where, int64_t* row0 = nullptr) {
    IdxGroup* gs = reinterpret_cast<IdxGroup*>(smem + C::kOffPlanG);
    int64_t* ts = reinterpret_cast<int64_t*>(smem + C::kOffPlanT);
    if (threadIdx.x < bq.n_q) {
        QueryInfo qi;
        IdxGroup G{0, (int32_t)threadIdx.x, 0, 0, 0};
        const bool ok = query_info(bq, threadIdx.x, qi, err, where);
        if (ok) {
            G.key0 = qi.key0;
            G.nq = 1;
            G.L_last = (int32_t)qi.L;
        }
        if (row0 != nullptr) row0[threadIdx.x] = ok ? qi.row0 : -1;
        gs[threadIdx.x] = G;
        ts[threadIdx.x + 1] = G.nq ? (G.L_last / kpool + kTileKeys - 1) / kTileKeys : 0;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        ts[0] = 0;
        for (int i = 1; i <= bq.n_q; ++i) ts[i] += ts[i - 1];
    }
    __syncthreads();
    return bq.n_q;
}

// Barrier init, TMEM allocation and the tensor maps' prefetch: work local to
// the CTA that reads no global memory, so a kernel does it before it waits
// for its predecessor.  Called by every thread; ends with a CTA barrier.
template <int GQ, int STAGES>
__device__ void setup(uint8_t* smem, const CUtensorMap* tm_k_p, const CUtensorMap* tm_q_p) {
    using C = Cfg<GQ, STAGES>;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::kStages;
    uint64_t* b_full = bars + 2 * C::kStages;
    uint64_t* b_empty = b_full + 1;
    uint64_t* acc_full = b_full + 2;
    uint64_t* acc_empty = b_full + 4;
    uint64_t* drain = b_full + 6;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + C::kOffMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(b_full, 1);
        mbar_init(b_empty, 1);
        for (int i = 0; i < 2; ++i) { mbar_init(&acc_full[i], 1); mbar_init(&acc_empty[i], C::kEpiWarps); }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(tm_k_p);
        prefetch_tensormap(tm_q_p);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// The producer's first loads, by thread 0 alone, as soon as its range is
// known -- before the rest of the CTA's set-up, so that the first bytes are
// on their way while that runs: the query tile of the first unit's group and
// up to STAGES key tiles of that group.  Returns how many key tiles it
// issued (stages 0 .. n - 1, first phase); run() continues after them.
template <int GQ, int STAGES>
__device__ int issue_first(uint8_t* smem, const CUtensorMap* tm_k_p, const CUtensorMap* tm_q_p,
                           const IdxGroup* __restrict__ groups, const int64_t* __restrict__ tile_off,
                           int64_t n_groups, int64_t u_begin, int64_t u_end) {
    using C = Cfg<GQ, STAGES>;
    if (u_begin >= u_end) return 0;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;
    uint64_t* b_full = bars + 2 * C::kStages;
    Cursor<(GQ > 1)> c{tile_off, 0, 0, 0, 0};
    c.seek(u_begin, n_groups);
    const IdxGroup G = groups[c.g];
    uint8_t* bsm = smem + C::kOffB;
    mbar_arrive_expect_tx(b_full, C::kBBytes);
    tma_load_2d(bsm, tm_q_p, b_full, 0, G.q0 * kIdxHeads);
    tma_load_2d(bsm + C::kBBoxBytes, tm_q_p, b_full, 64, G.q0 * kIdxHeads);
    // the first group's tiles left from u_begin, the range's, the ring's
    int64_t n = c.b1() - (c.b0() + c.t);
    if (n > u_end - u_begin) n = u_end - u_begin;
    if (n > C::kStages) n = C::kStages;
    for (int s = 0; s < (int)n; ++s) {
        uint8_t* asm_ = smem + C::kOffA + s * kABytes;
        const int32_t y = (int32_t)(G.key0 + (c.t + s) * kTileKeys);
        mbar_arrive_expect_tx(&full[s], kABytes);
        tma_load_2d(asm_, tm_k_p, &full[s], 0, y);
        tma_load_2d(asm_ + kABoxBytes, tm_k_p, &full[s], 64, y);
    }
    return (int)n;
}

// The decode plan a batch's host scalars imply when they leave it one
// possibility worth guessing: *n_seqs sequences of *nk keys each, one query
// each, the keys of sequence s from row s * nk of k_idx.  Only a single query
// is guessed: its keys start at row 0 (the offsets start at 0) and, when its
// sequence is as long as the batch's bound -- the usual case -- number
// floor(max_kv_len / kpool) (or the keys there are, if fewer).  (For a batch
// of equal sequences at the bound the scalars force every offset too, but
// there the guess measured slower in the whole step: 74.2 -> 75.5 us on the
// 1M-token k-pool decode, with the launch alone 1.4 us faster.)  False when
// no guess is made.  A guess is only ever a guess: the kernels check it
// against the plan they read.
__host__ __device__ inline bool spec_plan_guess(const BatchDev& b, int32_t kpool, int64_t* nk,
                                                int64_t* n_seqs) {
    if (kpool < 1 || b.n_q != 1 || b.n_seq != 1) return false;
    *nk = b.max_kv_len / kpool < b.total_keys ? b.max_kv_len / kpool : b.total_keys;
    *n_seqs = 1;
    return *nk > 0;
}

// A CTA's first key tiles under the guessed plan: spec_issue (one thread other
// than thread 0, right after the wait for the previous kernel, before the
// plan's CTA barriers) issues the query tile and the first key tiles of the
// CTA's guessed range (of `max_tiles` at most) and notes how many in shared
// memory; the batch offsets are read meanwhile.  spec_settle (thread 0, after
// the plan, and followed by a CTA barrier before any thread enters run())
// keeps them when the plan gives the same first tiles, else lets them land,
// re-arms their barriers and issues the real ones.  It returns the key tiles
// on their way: run()'s `pre`.
struct SpecRange {
    int64_t nk, per, ub, ue;          // keys and tiles per sequence, the CTA's guessed units
};

__device__ inline bool spec_range(const BatchDev& b, int32_t kpool, int64_t cta, int64_t grid,
                                  SpecRange* r) {
    int64_t nk = 0, n_seqs = 0;
    if (!spec_plan_guess(b, kpool, &nk, &n_seqs)) return false;
    r->nk = nk;
    r->per = (nk + kTileKeys - 1) / kTileKeys;
    const int64_t u_all = r->per * n_seqs;
    r->ub = mul_div(cta, u_all, grid);
    r->ue = mul_div(cta + 1, u_all, grid);
    return r->ub < r->ue;
}

template <int GQ, int STAGES>
__device__ void spec_issue(uint8_t* smem, const CUtensorMap* tm_k_p, const CUtensorMap* tm_q_p,
                           const BatchDev& bq, int32_t kpool, int64_t cta, int64_t grid,
                           int64_t max_tiles) {
    using C = Cfg<GQ, STAGES>;
    int32_t* note = reinterpret_cast<int32_t*>(smem + C::kOffMisc + 8);
    int spec = 0;
    SpecRange r;
    if (GQ == 1 && spec_range(bq, kpool, cta, grid, &r) && r.ue - r.ub <= max_tiles) {
        const int64_t g = r.ub / r.per;                // the guessed group of the first unit
        const IdxGroup gg{g * r.nk, (int32_t)g, 1, (int32_t)(r.nk * kpool), 0};
        const int64_t t0[2] = {g * r.per, (g + 1) * r.per};
        spec = issue_first<GQ, STAGES>(smem, tm_k_p, tm_q_p, &gg, t0, 1, r.ub, r.ue);
    }
    note[0] = spec;
}

// a wrong guess: its loads land, then their barriers start afresh
static __device__ __noinline__ void spec_drain(uint64_t* bars, int stages, int spec, int32_t* err,
                                        int32_t where) {
    uint64_t* full = bars;
    uint64_t* b_full = bars + 2 * stages;
    bool landed = mbar_wait(b_full, 0, kWaitNs);
#pragma unroll 1
    for (int s = 0; s < spec; ++s) landed = mbar_wait(&full[s], 0, kWaitNs) && landed;
    if (!landed) record_error(err, kDevTimeout, (int32_t)blockIdx.x, where);
    mbar_inval(b_full);
    mbar_init(b_full, 1);
#pragma unroll 1
    for (int s = 0; s < spec; ++s) {
        mbar_inval(&full[s]);
        mbar_init(&full[s], 1);
    }
    fence_mbarrier_init();
}

template <int GQ, int STAGES>
__device__ int spec_settle(uint8_t* smem, const CUtensorMap* tm_k_p, const CUtensorMap* tm_q_p,
                           const BatchDev& bq, int32_t kpool, const IdxGroup* __restrict__ groups,
                           const int64_t* __restrict__ tile_off, int64_t n_groups,
                           int64_t u_begin, int64_t u_end, int32_t* err, int32_t where) {
    using C = Cfg<GQ, STAGES>;
    const int spec = reinterpret_cast<const int32_t*>(smem + C::kOffMisc + 8)[0];
    if (spec > 0) {
        SpecRange r;
        spec_range(bq, kpool, blockIdx.x, gridDim.x, &r);
        if (u_begin == r.ub && u_begin < u_end) {
            // the plan's group of the first unit, and the key tiles
            // issue_first would issue now: that group's from u_begin
            Cursor<false> c{tile_off, 0, 0, 0, 0};
            c.seek(u_begin, n_groups);
            int64_t n_now = tile_off[c.g + 1] - u_begin;
            if (n_now > u_end - u_begin) n_now = u_end - u_begin;
            if (n_now > C::kStages) n_now = C::kStages;
            const int64_t g = r.ub / r.per;
            if (c.g == g && groups[c.g].q0 == g && groups[c.g].key0 == g * r.nk && n_now == spec)
                return spec;                           // the guessed tiles are the first ones
        }
        spec_drain(reinterpret_cast<uint64_t*>(smem + C::kOffBar), C::kStages, spec, err, where);
    }
    return issue_first<GQ, STAGES>(smem, tm_k_p, tm_q_p, groups, tile_off, n_groups, u_begin,
                                   u_end);
}

// The three roles over [u_begin, u_end) (possibly empty), then TMEM release.
// Called by every thread of the CTA (Cfg::kThreads) after setup().
template <int GQ, int STAGES, class Epi>
__device__ void run(uint8_t* smem, const CUtensorMap* tm_k_p, const CUtensorMap* tm_q_p,
                    const IdxGroup* __restrict__ groups, const int64_t* __restrict__ tile_off,
                    int64_t n_groups, int64_t u_begin, int64_t u_end,
                    const float* __restrict__ w, int32_t kpool, Epi& epi, int32_t* err,
                    int pre = 0) {
    using C = Cfg<GQ, STAGES>;
    const CUtensorMap& tm_k = *tm_k_p;
    const CUtensorMap& tm_q = *tm_q_p;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::kStages;
    uint64_t* b_full = bars + 2 * C::kStages;
    uint64_t* b_empty = b_full + 1;
    uint64_t* acc_full = b_full + 2;
    uint64_t* acc_empty = b_full + 4;
    uint64_t* drain = b_full + 6;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + C::kOffMisc + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {                                           // ---- TMA producer
            // (thread 0: `pre` key tiles and their group's query tile may have
            // been issued already by issue_first)
            Cursor<(GQ > 1)> c{tile_off, 0, 0, 0, 0};
            c.seek(u_begin, n_groups);
            int stage = 0;
            uint32_t phase = 0, b_empty_par = 0;
            int64_t b_group = -1;
            int8_t issued_par[C::kStages];
            for (int s = 0; s < C::kStages; ++s) issued_par[s] = s < pre ? 0 : -1;
            if (pre > 0) {
                b_group = c.g;
                stage = pre % C::kStages;
                phase = pre == C::kStages ? 1u : 0u;
                for (int s = 0; s < pre && u_begin + s + 1 < u_end; ++s) c.next();
            }
            bool ok = true;
            for (int64_t u = u_begin + pre; u < u_end && ok; ++u) {
                const IdxGroup G = groups[c.g];
                if (c.g != b_group) {
                    if (b_group >= 0) {
                        ok = mbar_wait(b_empty, b_empty_par, kWaitNs);
                        b_empty_par ^= 1;
                        if (!ok) break;
                    }
                    uint8_t* bsm = smem + C::kOffB;
                    mbar_arrive_expect_tx(b_full, C::kBBytes);
                    tma_load_2d(bsm, &tm_q, b_full, 0, G.q0 * kIdxHeads);
                    tma_load_2d(bsm + C::kBBoxBytes, &tm_q, b_full, 64, G.q0 * kIdxHeads);
                    b_group = c.g;
                }
                ok = mbar_wait(&empty[stage], phase ^ 1, kWaitNs);
                if (!ok) break;
                uint8_t* asm_ = smem + C::kOffA + stage * kABytes;
                const int32_t y = (int32_t)(G.key0 + c.t * kTileKeys);
                mbar_arrive_expect_tx(&full[stage], kABytes);
                tma_load_2d(asm_, &tm_k, &full[stage], 0, y);
                tma_load_2d(asm_ + kABoxBytes, &tm_k, &full[stage], 64, y);
                issued_par[stage] = (int8_t)phase;
                if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                if (u + 1 < u_end) c.next();
            }
            if (!ok) {
                record_error(err, kDevTimeout, blockIdx.x, /*where=*/5);
                *abort_flag = 1;
                // let this CTA's copies in flight land before the CTA retires
                for (int s = 0; s < C::kStages; ++s)
                    if (issued_par[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_par[s], 50000000ull);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {                                           // ---- MMA issuer
            constexpr uint32_t idesc = idesc_bf16_f32(kTileKeys, C::N);
            Cursor<(GQ > 1)> c{tile_off, 0, 0, 0, 0};
            c.seek(u_begin, n_groups);
            int stage = 0, ab = 0;
            uint32_t phase = 0, acc_par = 0, b_full_par = 0;
            int64_t b_group = -1;
            bool ok = true;
            for (int64_t u = u_begin; u < u_end && ok; ++u) {
                if (*abort_flag) { ok = false; break; }
                if (c.g != b_group) {
                    ok = mbar_wait(b_full, b_full_par, kWaitNs);
                    b_full_par ^= 1;
                    b_group = c.g;
                    if (!ok) break;
                }
                ok = mbar_wait(&acc_empty[ab], acc_par ^ 1, kWaitNs) &&
                     mbar_wait(&full[stage], phase, kWaitNs);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(smem + C::kOffA + stage * kABytes);
                const uint32_t b0 = smem_u32(smem + C::kOffB);
                const uint32_t d = tmem_base + (uint32_t)(ab * C::N);
#pragma unroll
                for (int kk = 0; kk < kIdxDim / 16; ++kk) {
                    const uint32_t koff = (uint32_t)(kk & 3) * 32u, half = (uint32_t)(kk >> 2);
                    mma_bf16_ss(d, sdesc_kmajor_sw128(a0 + half * kABoxBytes + koff),
                                sdesc_kmajor_sw128(b0 + half * C::kBBoxBytes + koff), idesc,
                                kk > 0 ? 1u : 0u);
                }
                mma_commit(&empty[stage]);                 // stage reusable once these finish
                mma_commit(&acc_full[ab]);                 // accumulator ready for the epilogue
                if (c.last_of_group()) mma_commit(b_empty);
                if (++stage == C::kStages) { stage = 0; phase ^= 1; }
                if (++ab == 2) { ab = 0; acc_par ^= 1; }
                if (u + 1 < u_end) c.next();
            }
            if (!ok) {
                record_error(err, kDevTimeout, blockIdx.x, /*where=*/6);
                *abort_flag = 1;
            }
            mma_commit(drain);                             // all issued MMAs retired
            mbar_wait(drain, 0, 50000000ull);
        }
    } else if (warp >= 4) {                                        // ---- epilogue
        const int ew = warp - 4;
        const int wg = ew >> 2;                                    // epilogue warpgroup
        const int lane_base = 32 * (warp & 3);                     // this warp's TMEM lanes
        const int row = lane_base + lane;
        // grouped queries: this warp's queries' head weights in its own slice of
        // shared memory, refreshed when the group changes (warp-private: no
        // synchronisation beyond the warp)
        float* w_s = reinterpret_cast<float*>(smem + C::kOffW) + ew * 2 * kIdxHeads;
        Cursor<(GQ > 1)> c{tile_off, 0, 0, 0, 0};
        c.seek(u_begin, n_groups);
        int ab = 0;
        uint32_t acc_par = 0;
        epi.begin();
        int64_t g_loaded = -1;
        IdxGroup G{};
        for (int64_t u = u_begin; u < u_end; ++u) {
            if (GQ == 1 || c.g != g_loaded) {                      // grouped: once per group
                G = groups[c.g];
                g_loaded = c.g;
                if (GQ > 1) {
                    __syncwarp();
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        const int j = wg + r * C::kEpiGroups;
                        w_s[r * kIdxHeads + lane] =
                            j < G.nq ? w[(int64_t)(G.q0 + j) * kIdxHeads + lane] : 0.f;
                    }
                    __syncwarp();
                }
            }
            if (*abort_flag || !mbar_wait(&acc_full[ab], acc_par, kWaitNs)) {
                record_error(err, kDevTimeout, blockIdx.x, /*where=*/7);
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int64_t t_row = c.t * kTileKeys + row;
            for (int j = wg; j < G.nq; j += C::kEpiGroups) {
                float v[32];
                tmem_ld_32cols(tmem_base + ((uint32_t)lane_base << 16) + (uint32_t)(ab * C::N + 32 * j), v);
                // the query's head weights: warp-uniform addresses, one broadcast each
                const float4* w4 =
                    GQ > 1 ? reinterpret_cast<const float4*>(w_s + ((j - wg) / C::kEpiGroups) * kIdxHeads)
                           : reinterpret_cast<const float4*>(w + (int64_t)(G.q0 + j) * kIdxHeads);
                // four partial sums (heads 4i, 4i+1, 4i+2, 4i+3 of each group of
                // four), two packed FMAs per group: short dependency chains
                float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
                for (int h4 = 0; h4 < kIdxHeads / 4; ++h4) {
                    const float4 wv = GQ > 1 ? w4[h4] : __ldg(w4 + h4);
                    fma2(a0, a1, wv.x, wv.y, fmaxf(v[4 * h4 + 0], 0.f), fmaxf(v[4 * h4 + 1], 0.f));
                    fma2(b0, b1, wv.z, wv.w, fmaxf(v[4 * h4 + 2], 0.f), fmaxf(v[4 * h4 + 3], 0.f));
                }
                const float s = (a0 + a1) + (b0 + b1);
                // visible: t_row < floor(rows seen by the query / kpool), without
                // the (emulated) 64-bit division
                const int64_t seen = (int64_t)(G.L_last - (G.nq - 1 - j));
                epi.emit(G, j, t_row, (t_row + 1) * kpool <= seen, u, row, s);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[ab]);
            if (++ab == 2) { ab = 0; acc_par ^= 1; }
            if (u + 1 < u_end) c.next();
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace idxp
}  // namespace dsa
