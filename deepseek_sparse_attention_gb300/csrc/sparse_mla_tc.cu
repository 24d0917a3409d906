// sparse_mla_tc.cu -- absorbed-MLA attention over the selected cache rows on
// the tcgen05 tensor cores.
//
// z[h,j] = scale * q_abs[h,:] . row_j (latent + rope), p = softmax_j(z),
// out[h,c] = sum_j p[h,j] row_j[c] for the 512 latent columns ("GLM 5.2 in one
// C file", "Attention: Multi head Latent Attention With a Tiny KV Cache";
// "GLM-5.x (glm-dsa, glm5next)", "The block": 64 heads, one 576-wide row,
// scale 1/16; "Add GLM-5.3-Flash support": a NoPE row is the 512-wide latent,
// key and value alike).
//
// One CTA handles a range of one query's selected rows in tiles of 64 rows,
// two row buffers deep, so that one tile's gather overlaps the previous
// tile's softmax and value product:
//   warps 0,2,3 and 8-11 gather each tile's rows with 16-byte cp.async copies
//              straight into the 128-byte swizzle layout of buffer t % 2 --
//              thousands of copies in flight per SM, where a TMA gather4 (four
//              128-byte row pieces per request) kept too few (the first two
//              tiles are copied by every thread but warp 1's; thread 0 loads
//              the query once by TMA);
//   warp 1     issues S^T = R . Q^T (M = 64 rows, N = 64 heads, K = the row
//              width) into one of two TMEM score buffers -- the next tile's
//              scores before this tile's values -- then O^T += R^T . P^T
//              (M = 128 latent columns x 4, N = 64 heads, K = 64 rows) with both
//              operands MN-major: the same gathered tile serves as K-major A for
//              the scores and as MN-major A for the values;
// P is split into bf16 hi + lo parts and the value product runs once on each
// (through the same shared-memory buffer), carrying P to ~2^-16 relative where
// bf16 alone (up to 2^-8) would not meet the output tolerance in every case.
//   warps 4-7  softmax across the tile's rows: an M = 64 accumulator puts row
//              16 q + i in lane i of TMEM quadrant q; a 16x64b load gives every
//              lane a row and the 32 heads of one parity; per-head tile maxima
//              by a halving shuffle exchange, a running maximum that is raised
//              (and O^T rescaled in TMEM, after the previous tile's values are
//              in) only when a tile exceeds it by more than 2^8, exp2, P^T
//              written to shared memory (into the buffer's rope block, which
//              the scores no longer need), per-thread partial row sums reduced
//              once at the end; warps 4-11 then read O^T out of TMEM.
// Splits of one query are combined by the log-sum-exp merge: a separate
// launch over the partials in global memory, or, for two splits, inside this
// launch by the two CTAs of a cluster through distributed shared memory.
#include <math.h>

#include <cooperative_groups.h>

#include "dsa_kernels.cuh"
#include "sm100.cuh"

namespace cg = cooperative_groups;

namespace dsa {
namespace {

using namespace sm100;

constexpr int kHeads = 64;
constexpr int kTileRows = 64;                       // rows per tile (MMA M of the scores)
constexpr int kOBlock = 128;                        // latent columns per O^T block (MMA M)
constexpr int kLatent = 512;
constexpr uint32_t kQBlock = kHeads * 128;          // one 64-column block of Q: 8 KB
constexpr uint32_t kRBlock = kTileRows * 128;       // one 64-column block of a row tile: 8 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 0;                       // S^T of buffer b: columns 64 b .. 64 b + 63
constexpr uint32_t kOCol = 128;                     // O^T: 128 .. 383
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kSlack = 8.f;                       // lazy rescale threshold (log2 units)
// Warps 0, 2, 3 and 8-11 gather rows (224 threads), warp 1 issues the MMAs,
// warps 4-7 run the softmax; all but warp 1 copy the first two tiles.
constexpr int kLoaders = 224;
constexpr int kSoftmaxThreads = 128;
constexpr int kThreads = 384;
constexpr int kIssuers = kLoaders + kSoftmaxThreads; // threads that copy rows: 352
constexpr int kRowSlots = kIssuers / 8;             // rows a tile's copy round covers: 44
static_assert(kIssuers % 8 == 0 && 2 * kRowSlots >= 64, "two rows per slot cover a tile");

template <int W>
struct Cfg {
    static constexpr int kCB = W / 64;               // 64-column blocks of a row
    static constexpr uint32_t kOffQ = 0;
    static constexpr uint32_t kOffR = kCB * kQBlock;                 // two row buffers
    static constexpr uint32_t kBufBytes = kCB * kRBlock;
    // P_hi^T [64 rows x 64 heads] bf16 of buffer b: the buffer's rope block when
    // there is one (no longer needed once the scores are formed), else its own.
    static constexpr uint32_t kOffPx = kOffR + 2 * kBufBytes;         // NoPE: two P_hi blocks
    // P_lo^T: one block shared by the two buffers (a tile writes it once the
    // previous tile's value products are done)
    static constexpr uint32_t kOffPlo = W == 576 ? kOffPx : kOffPx + 2 * kRBlock;
    static constexpr uint32_t kOffBar = kOffPlo + kRBlock;
    // q_full, drain, r_full[2], s_full[2], p_full[2], pv_done[2]
    static constexpr uint32_t kOffRed = kOffBar + 128;          // [4][64] int
    static constexpr uint32_t kOffL = kOffRed + 4 * 64 * 4;     // [64] float
    static constexpr uint32_t kOffM = kOffL + 64 * 4;           // [64] float
    static constexpr uint32_t kOffMisc = kOffM + 64 * 4;
    static constexpr uint32_t kSmemBytes = kOffMisc + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    __device__ static uint32_t off_p(int b) {
        return W == 576 ? kOffR + b * kBufBytes + 8 * kRBlock : kOffPx + b * kRBlock;
    }
};

__device__ __forceinline__ int fkey(float f) {           // order-preserving float -> int
    const int i = __float_as_int(f);
    return i >= 0 ? i : i ^ 0x7fffffff;
}
__device__ __forceinline__ float fval(int k) { return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff); }

template <int W>
__global__ void __launch_bounds__(kThreads, 1)
sparse_mla_tc(const __grid_constant__ CUtensorMap tm_q, const void* __restrict__ cache,
              BatchDev b, float scale, const int32_t* __restrict__ idx,
              const int32_t* __restrict__ n_sel, int64_t idx_width, int32_t rows_per_split,
              int32_t n_split, int32_t pair, int32_t q_early, float* __restrict__ out,
              float* __restrict__ lse, float* __restrict__ part_o, float* __restrict__ part_ml,
              int32_t* err) {
    using C = Cfg<W>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t *q_full = bars, *drain = bars + 1, *r_full = bars + 2, *s_full = bars + 4,
             *p_full = bars + 6, *pv_done = bars + 8;
    int* red = reinterpret_cast<int*>(smem + C::kOffRed);
    float* l_fin = reinterpret_cast<float*>(smem + C::kOffL);
    float* m_fin = reinterpret_cast<float*>(smem + C::kOffM);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t q = blockIdx.y;
    const int split = blockIdx.x;
    // Two CTAs per split (gridDim.z == 2) share a tile's gather, scores and
    // softmax -- each computes them -- and divide the value product and the
    // output by latent half: blocks 2 half and 2 half + 1 of the four.
    const int half = blockIdx.z;
    const bool halved = gridDim.z == 2;
    auto owns = [&](int blk) { return !halved || (blk >> 1) == half; };
    // Two splits of a query launched as a cluster (pair != 0): each stages its
    // unnormalised O as [head][latent] in its own shared memory and its row
    // maxima and sums stay in m_fin / l_fin; then each combines half of the
    // heads from both through distributed shared memory and writes the final
    // output -- no partials in global memory and no merge launch.  Every
    // thread of both CTAs calls this once (an empty split too, with l = 0).
    float* stage = reinterpret_cast<float*>(smem);    // the query and row buffers, once free
    auto pair_merge = [&]() {
        cg::cluster_group cl = cg::this_cluster();
        cl.sync();                                    // both stages are written
        const int rank = (int)cl.block_rank();
        const float4* st0 = reinterpret_cast<const float4*>(stage);
        const float4* st1 = reinterpret_cast<const float4*>(cl.map_shared_rank(stage, rank ^ 1));
        const float* m1p = cl.map_shared_rank(m_fin, rank ^ 1);
        const float* l1p = cl.map_shared_rank(l_fin, rank ^ 1);
        float4* o4 = reinterpret_cast<float4*>(out);
        constexpr int kC4 = kLatent / 4;
        for (int i = threadIdx.x; i < (kHeads / 2) * kC4; i += blockDim.x) {
            const int h = (kHeads / 2) * rank + i / kC4, c4 = i % kC4;
            const float l0 = l_fin[h], l1 = l1p[h];
            const float m0 = l0 > 0.f ? m_fin[h] : -INFINITY, m1 = l1 > 0.f ? m1p[h] : -INFINITY;
            const float M = fmaxf(m0, m1);
            const float f0 = l0 > 0.f ? exp2f(m0 - M) : 0.f, f1 = l1 > 0.f ? exp2f(m1 - M) : 0.f;
            const float L = l0 * f0 + l1 * f1;
            float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
            if (L > 0.f) {
                const float inv = 1.f / L;
                const float4 a = l0 > 0.f ? st0[h * kC4 + c4] : r;
                const float4 c = l1 > 0.f ? st1[h * kC4 + c4] : r;
                r = make_float4((a.x * f0 + c.x * f1) * inv, (a.y * f0 + c.y * f1) * inv,
                                (a.z * f0 + c.z * f1) * inv, (a.w * f0 + c.w * f1) * inv);
            }
            o4[(q * kHeads + h) * kC4 + c4] = r;
            if (c4 == 0 && lse != nullptr)
                lse[q * kHeads + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        cl.sync();                                    // the peer's reads of this stage are done
    };
    // Before the selection is waited for: barriers, TMEM, and -- when the
    // previous kernel is this library's selection, launched after the caller's
    // kernels completed -- the query tile.
    if (threadIdx.x < kHeads) m_fin[threadIdx.x] = -INFINITY;   // the running maxima
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(drain, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&r_full[i], kIssuers);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], kSoftmaxThreads);
            mbar_init(&pv_done[i], 1);
        }
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    auto load_query = [&]() {
        mbar_arrive_expect_tx(q_full, C::kCB * kQBlock);
        for (int cb = 0; cb < C::kCB; ++cb)
            tma_load_2d(smem + C::kOffQ + cb * kQBlock, &tm_q, q_full, 64 * cb, (int32_t)(q * kHeads));
    };
    if (threadIdx.x == 0) {
        prefetch_tensormap(&tm_q);
        if (q_early) load_query();
    }
    // A CTA leaving before its pipeline runs: the query tile must have landed
    // and TMEM goes back.
    auto leave_early = [&]() {
        if (threadIdx.x == 0) mbar_wait(q_full, 0, kWaitNs);
        tc_fence_before();
        __syncthreads();
        if (warp == 1) {
            tc_fence_after();
            tmem_dealloc(tmem_base, kTmemCols);
        }
    };
    pdl_wait();                                       // the selection must be complete
    pdl_trigger();
    if (threadIdx.x == 0 && !q_early) load_query();
    // Selected row j of the query: idx[q][j], or row j itself when there is
    // no selection (dense: every visible row).
    const bool dense = idx == nullptr;
    auto sel_row = [&](int64_t j) -> int32_t {
        return dense ? (int32_t)j : idx[q * idx_width + j];
    };
    // Row gather slots: every thread but the MMA warp's copies rows -- eight
    // threads per row (one 16-byte piece of each 64-column block's 128-byte
    // line), kIssuers / 8 rows at a time: slot s takes rows s / 8 and, where
    // it exists, s / 8 + kRowSlots of each tile.
    const int slot = warp == 0 ? lane : (warp < 4 ? 32 * (warp - 1) + lane : threadIdx.x - 32);
    const int rs = slot >> 3, k8 = slot & 7;
    const bool issuer = warp != 1;
    const bool two_rows = rs + kRowSlots < kTileRows;
    // Three independent reads go out together: the selection count, this
    // thread's indices of the first tile (whatever the count; unused past it)
    // and the batch arrays.
    const int64_t j0 = (int64_t)split * rows_per_split;
    int64_t ns = dense ? 0 : n_sel[q];
    int32_t ia = issuer && (dense || j0 + rs < idx_width) ? sel_row(j0 + rs) : 0;
    int32_t ib = issuer && two_rows && (dense || j0 + rs + kRowSlots < idx_width)
                     ? sel_row(j0 + rs + kRowSlots) : 0;
    QueryInfo qi;
    if (!query_info(b, q, qi, err, /*where=*/8)) {
        leave_early();
        return;
    }
    if (dense) ns = qi.L;
    else ns = ns < 0 ? 0 : (ns > idx_width ? idx_width : ns);
    const int64_t j1 = j0 + rows_per_split < ns ? j0 + rows_per_split : ns;
    if (j0 >= j1) {
        if (pair) {                                   // no weight from this half
            if (threadIdx.x < kHeads) { m_fin[threadIdx.x] = -INFINITY; l_fin[threadIdx.x] = 0.f; }
            __syncthreads();
            pair_merge();
        } else if (n_split == 1) {                    // no rows: out = 0, lse = -inf
            for (int i = threadIdx.x; i < kHeads * kLatent; i += blockDim.x)
                out[q * kHeads * kLatent + i] = 0.f;
            if (lse != nullptr && threadIdx.x < kHeads) lse[q * kHeads + threadIdx.x] = -INFINITY;
        } else if (threadIdx.x < kHeads && half == 0) {  // empty split: weight 0 in the merge,
            const int64_t part = q * n_split + split;  // which then never reads its output
            part_ml[(part * kHeads + threadIdx.x) * 2] = -INFINITY;
            part_ml[(part * kHeads + threadIdx.x) * 2 + 1] = 0.f;
        }
        leave_early();
        return;
    }
    const int n_tiles = (int)((j1 - j0 + kTileRows - 1) / kTileRows);


    // Copies of this thread's rows of tile t (indices ra, rb read from the
    // selection) into buffer t % 2 in the 128-byte swizzle layout; the
    // buffer's r_full barrier counts this thread's arrival once they have all
    // landed (cp.async.mbarrier.arrive), so no thread waits for its copies.
    // Rows past the split, and indices out of range (reported), copy row 0 of
    // the sequence, which the softmax gives no weight.
    const unsigned char* cbase = static_cast<const unsigned char*>(cache);
    auto issue_rows = [&](int t, int32_t ra, int32_t rb) {
        const uint32_t rbase = smem_u32(smem + C::kOffR + (t & 1) * C::kBufBytes);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = rs + h * kRowSlots;
            if (r >= kTileRows) continue;
            const int64_t j = j0 + (int64_t)t * kTileRows + r;
            int32_t rr = h == 0 ? ra : rb;
            if (j >= j1) {
                rr = 0;
            } else if (rr < 0 || rr >= qi.L) {
                record_error(err, kDevBadIndex, (int32_t)q, /*where=*/8);
                rr = 0;
            }
            const unsigned char* src = cbase + ((qi.row0 + rr) * W + k8 * 8) * 2;
            const uint32_t dst = rbase + r * 128 + ((k8 ^ (r & 7)) << 4);
#pragma unroll
            for (int cb = 0; cb < C::kCB; ++cb)
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                             ::"r"(dst + cb * kRBlock), "l"(src + cb * 128)
                             : "memory");
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];"
                     ::"r"(smem_u32(&r_full[t & 1]))
                     : "memory");
    };
    // this thread's indices of tile t (read a tile ahead of their copies)
    auto fetch_rows = [&](int t, int32_t& ra, int32_t& rb) {
        const int64_t j = j0 + (int64_t)t * kTileRows + rs;
        ra = j < j1 ? sel_row(j) : 0;
        rb = two_rows && j + kRowSlots < j1 ? sel_row(j + kRowSlots) : 0;
    };
    if (issuer) issue_rows(0, ia, ib);

    if ((warp != 1 && warp < 4) || warp >= 8) {                      // ---- loads
        // warps 0, 2, 3, 8-11: their share of the second tile at once, then
        // tile t + 1 as soon as its buffer is free (the PV of tile t - 1 has
        // completed).
        bool ok = true;
        // From the third tile on the loaders copy whole tiles alone (eight
        // threads per row, 28 rows a pass), keeping the softmax warps' time
        // for the softmax; those arrive on the barrier without copies.
        constexpr int kRowsPerPass = kLoaders / 8;
        constexpr int kPasses = (kTileRows + kRowsPerPass - 1) / kRowsPerPass;
        const int ls = warp == 0 ? lane : (warp < 4 ? 32 * (warp - 1) + lane : 96 + 32 * (warp - 8) + lane);
        const int rsub = ls >> 3, k8l = ls & 7;
        for (int t = 0; t + 1 < n_tiles && ok; ++t) {
            if (t == 0) {
                fetch_rows(1, ia, ib);
                issue_rows(1, ia, ib);
                continue;
            }
            int32_t rr[kPasses];
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps) {
                const int r = kRowsPerPass * ps + rsub;
                const int64_t j = j0 + (int64_t)(t + 1) * kTileRows + r;
                rr[ps] = r < kTileRows && j < j1 ? sel_row(j) : 0;
            }
            ok = mbar_wait(&pv_done[(t + 1) & 1], (uint32_t)(((t - 1) >> 1) & 1), kWaitNs);
            if (!ok) break;
            const uint32_t rbase = smem_u32(smem + C::kOffR + ((t + 1) & 1) * C::kBufBytes);
#pragma unroll
            for (int ps = 0; ps < kPasses; ++ps) {
                const int r = kRowsPerPass * ps + rsub;
                if (r >= kTileRows) continue;
                const int64_t j = j0 + (int64_t)(t + 1) * kTileRows + r;
                int32_t row = rr[ps];
                if (j >= j1) {
                    row = 0;
                } else if (row < 0 || row >= qi.L) {
                    record_error(err, kDevBadIndex, (int32_t)q, /*where=*/8);
                    row = 0;
                }
                const unsigned char* src = cbase + ((qi.row0 + row) * W + k8l * 8) * 2;
                const uint32_t dst = rbase + r * 128 + ((k8l ^ (r & 7)) << 4);
#pragma unroll
                for (int cb = 0; cb < C::kCB; ++cb)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                                 ::"r"(dst + cb * kRBlock), "l"(src + cb * 128)
                                 : "memory");
            }
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];"
                         ::"r"(smem_u32(&r_full[(t + 1) & 1]))
                         : "memory");
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (!ok && ls == 0) record_error(err, kDevTimeout, (int32_t)q, /*where=*/9);
    } else if (warp == 1) {                                           // ---- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(kTileRows, kHeads);
            constexpr uint32_t idesc_pv = idesc_bf16_f32_major(kOBlock, kHeads, 1, 1);
            const uint32_t q0 = smem_u32(smem + C::kOffQ);
            bool ok = mbar_wait(q_full, 0, kWaitNs);
            // Issue whatever is ready, in dependency order: the scores S(s) of
            // tile s once its rows are in (and at most one tile ahead of the
            // values, whose softmax frees the other score buffer), and the
            // value products of tile v -- on P_hi, then on P_lo -- as soon as
            // the softmax hands both over.
            int next_s = 0, next_v = 0;
            uint64_t t_prog = globaltimer_ns();
            while (ok && next_v < n_tiles) {
                bool progressed = false;
                if (next_s < n_tiles && next_s <= next_v + 1 &&
                    mbar_test_wait(&r_full[next_s & 1], (uint32_t)((next_s >> 1) & 1))) {
                    // S^T(s) = R(s) Q^T: M = 64 rows, N = 64 heads, K = the row width.
                    // The rows were written by cp.async (generic proxy): fence
                    // before the tensor core (async proxy) reads them.
                    fence_proxy_async_smem();
                    tc_fence_after();
                    const int bs = next_s & 1;
                    const uint32_t r0 = smem_u32(smem + C::kOffR + bs * C::kBufBytes);
                    for (int cb = 0; cb < C::kCB; ++cb) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            mma_bf16_ss(tmem_base + kSCol + 64 * bs,
                                        sdesc_kmajor_sw128(r0 + cb * kRBlock + kk * 32),
                                        sdesc_kmajor_sw128(q0 + cb * kQBlock + kk * 32), idesc_s,
                                        (cb | kk) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit(&s_full[bs]);
                    ++next_s;
                    progressed = true;
                }
                if (next_v < next_s &&
                    mbar_test_wait(&p_full[next_v & 1], (uint32_t)((next_v >> 1) & 1))) {
                    // A = R^T: MN-major, 64-column blocks 8 KB apart, 8-row
                    // groups 1 KB apart.  B = P^T: MN-major, the 64 heads are one block.
                    tc_fence_after();
                    const int bv = next_v & 1;
                    const uint32_t r0 = smem_u32(smem + C::kOffR + bv * C::kBufBytes);
                    for (int part = 0; part < 2; ++part) {
                        const uint32_t p0 = smem_u32(smem + (part == 0 ? C::off_p(bv) : C::kOffPlo));
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if (!owns(i)) continue;
#pragma unroll
                            for (int kk = 0; kk < kTileRows / 16; ++kk) {
                                mma_bf16_ss(tmem_base + kOCol + 64 * i,
                                            sdesc_sw128(r0 + 2 * i * kRBlock + kk * 2048, kRBlock, 1024),
                                            sdesc_sw128(p0 + kk * 2048, 1024, 1024), idesc_pv,
                                            (next_v > 0 || part > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                    }
                    mma_commit(&pv_done[bv]);
                    ++next_v;
                    progressed = true;
                }
                if (progressed) t_prog = globaltimer_ns();
                else if (globaltimer_ns() - t_prog > kWaitNs) ok = false;
            }
            if (!ok) record_error(err, kDevTimeout, (int32_t)q, /*where=*/10);
            mma_commit(drain);
            mbar_wait(drain, 0, 50000000ull);
        }
    } else {                                                          // ---- softmax
        // warps 4-7, one warpgroup.  The scores of an M = 64 tile sit in lanes
        // 0..15 of TMEM quadrant wq; a 16x64b load gives lane l of warp 4 + wq
        // the row 16 wq + (l >> 2) + 8 (l & 1) and the 32 heads of parity
        // p = (l >> 1) & 1 (p, p + 2, ..., p + 62): every lane a row.
        const int wq = warp & 3;
        const int p = (lane >> 1) & 1;
        const int row = 16 * wq + (lane >> 2) + 8 * (lane & 1);
        const int ts = threadIdx.x - 128;            // 0..127; 0..63 own a head each
        const uint32_t lane_addr = tmem_base + ((uint32_t)(32 * wq) << 16);
        const float c2 = scale * kLog2e;
        // partial row sums of heads 32 p .. 32 p + 31 of this row (the heads a
        // lane holds after the exchange with lane ^ 2, below)
        float l_part[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) l_part[e] = 0.f;
        // running maxima (one writer per head) and rescale factors live in shared memory
        float* m_sh = m_fin;
        float* alpha_s = l_fin;
        bool ok = true;
        // this thread's row index, read a tile ahead so that the load overlaps
        // the previous tile's work (-1: no row)
        auto row_index = [&](int t) -> int32_t {
            const int64_t jrow = j0 + (int64_t)t * kTileRows + row;
            return (t < n_tiles && jrow < j1) ? sel_row(jrow) : -1;
        };
        // this thread's copies of tile 1 (its buffer is free from the start)
        if (n_tiles > 1) {
            fetch_rows(1, ia, ib);
            issue_rows(1, ia, ib);
        }
        int32_t r_cur = row_index(0);
        for (int t = 0; t < n_tiles; ++t) {
            const int bf = t & 1;
            const int32_t r_next = row_index(t + 1);
            // tiles from the third on are copied by the loaders alone: this
            // thread's arrival for tile t + 1 (its buffer's previous phase,
            // tile t - 1, completed before this tile's scores)
            if (t >= 1 && t + 1 < n_tiles) mbar_arrive(&r_full[(t + 1) & 1]);
            if (ok) ok = mbar_wait(&s_full[bf], (uint32_t)((t >> 1) & 1), kWaitNs);
            tc_fence_after();
            // rows past the split, and rows whose index is out of range (reported
            // by the loader), take no weight
            const bool valid = r_cur >= 0 && r_cur < qi.L;
            r_cur = r_next;
            float x[32];                             // x[k]: head p + 2 k
            {
                float v[32];
                tmem_ld_16x64b_32(lane_addr + kSCol + 64 * bf, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] = valid ? v[e] * c2 : -INFINITY;
            }
            // Does any score of the tile exceed its head's running maximum by
            // more than the slack?  If none does (the usual case after the
            // first tiles) the maxima stay and no reduction is needed.
            uint32_t exceed = 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) exceed |= (uint32_t)(x[e] > m_sh[p + 2 * e] + kSlack);
            uint32_t any_exceed;
            asm volatile(
                "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                : "=r"(any_exceed)
                : "r"(exceed), "n"(kSoftmaxThreads)
                : "memory");
            uint32_t any_raised = 0;
            if (any_exceed) {
                // per-head maximum over the warp's 16 rows (the 16 lanes of a
                // parity: lane bits 0, 2, 3, 4), then over the four warps.  A
                // halving exchange: at each step a lane keeps half of its
                // values, swaps the other half with the partner across one lane
                // bit and takes the maximum, so that after four steps each lane
                // holds two heads' maxima (30 shuffles for 32 heads).
                int* rb = red + wq * kHeads;
                float m16[16], m8[8], m4[4], m2[2];
                {
                    const bool b = (lane >> 4) & 1;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float r = __shfl_xor_sync(0xffffffffu, b ? x[i] : x[i + 16], 16);
                        m16[i] = fmaxf(b ? x[i + 16] : x[i], r);
                    }
                }
                {
                    const bool b = (lane >> 3) & 1;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float r = __shfl_xor_sync(0xffffffffu, b ? m16[i] : m16[i + 8], 8);
                        m8[i] = fmaxf(b ? m16[i + 8] : m16[i], r);
                    }
                }
                {
                    const bool b = (lane >> 2) & 1;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float r = __shfl_xor_sync(0xffffffffu, b ? m8[i] : m8[i + 4], 4);
                        m4[i] = fmaxf(b ? m8[i + 4] : m8[i], r);
                    }
                }
                {
                    const bool b = lane & 1;
#pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const float r = __shfl_xor_sync(0xffffffffu, b ? m4[i] : m4[i + 2], 1);
                        m2[i] = fmaxf(b ? m4[i + 2] : m4[i], r);
                    }
                }
                // m2[i]: the maximum of x[e], e = i + 2 (lane & 1) + 4 ((lane >> 2) & 7)
                const int e0 = 2 * (lane & 1) + 4 * ((lane >> 2) & 7);
                rb[p + 2 * e0] = fkey(m2[0]);
                rb[p + 2 * e0 + 2] = fkey(m2[1]);
                asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory");
                uint32_t raised = 0;
                if (ts < kHeads) {                     // head ts: raise its running maximum?
                    const int h = ts;
                    const int mk = max(max(red[h], red[kHeads + h]), max(red[2 * kHeads + h], red[3 * kHeads + h]));
                    const float tmax = fval(mk), m_old = m_sh[h];
                    float a = 1.f;
                    if (tmax > m_old + kSlack) {
                        a = m_old == -INFINITY ? 0.f : exp2f(m_old - tmax);
                        m_sh[h] = tmax;
                        raised = 1;
                    }
                    alpha_s[h] = a;
                }
                asm volatile(
                    "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                    "bar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                    : "=r"(any_raised)
                    : "r"(raised), "n"(kSoftmaxThreads)
                    : "memory");
            }
            if (any_raised) {
#pragma unroll
                for (int e = 0; e < 32; ++e) l_part[e] *= alpha_s[32 * p + e];
            }
            if (any_raised && t > 0) {                 // O^T follows the new maxima
                // the previous tile's PV may still be accumulating into O^T
                const int pb = (t - 1) & 1;
                if (ok) ok = mbar_wait(&pv_done[pb], (uint32_t)(((t - 1) >> 1) & 1), kWaitNs);
                tc_fence_after();
#pragma unroll 1
                for (int i = 0; i < 8; ++i) {          // 4 blocks x two halves of the heads
                    if (!owns(i >> 1)) continue;
                    float v[32];
                    const int hh = 32 * (i & 1);
                    const uint32_t a = lane_addr + kOCol + 64 * (i >> 1) + hh;
                    tmem_ld_32cols(a, v);
#pragma unroll
                    for (int c = 0; c < 32; ++c) v[c] *= alpha_s[hh + c];
                    tmem_st_32cols(a, v);
                }
                tc_fence_before();
                asm volatile("bar.sync 1, %0;" ::"n"(kSoftmaxThreads) : "memory");
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = exp2f(x[e] - m_sh[p + 2 * e]);
            // P^T row: this lane and lane ^ 2 (same row, other parity) swap
            // halves so that this lane holds heads 32 p .. 32 p + 31 as pairs
            // (32 p + 2 k, 32 p + 2 k + 1); 32 bf16 in the 128-byte swizzle layout,
            // twice: p = hi + lo with hi = bf16(p), lo = bf16(p - hi), so that
            // the two value products carry P to ~2^-16 relative.  hi goes to the
            // buffer's P block, lo to the shared P_lo block once the previous
            // tile's value products (which read it) are done.
            uint8_t* prow = smem + C::off_p(bf) + row * 128;
            uint8_t* plow = smem + C::kOffPlo + row * 128;
            uint32_t lo4[4][4];
#pragma unroll
            for (int c16 = 0; c16 < 4; ++c16) {
                uint32_t w4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int k = 4 * c16 + e;
                    const float send = p ? x[k] : x[k + 16];
                    const float r = __shfl_xor_sync(0xffffffffu, send, 2);
                    const float p0 = p ? r : x[k];
                    const float p1 = p ? x[k + 16] : r;
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(p0, p1);
                    const float2 hf = __bfloat1622float2(hi);
                    const __nv_bfloat162 lo = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
                    const float2 lf = __bfloat1622float2(lo);
                    l_part[2 * k] += hf.x + lf.x;
                    l_part[2 * k + 1] += hf.y + lf.y;
                    w4[e] = *reinterpret_cast<const uint32_t*>(&hi);
                    lo4[c16][e] = *reinterpret_cast<const uint32_t*>(&lo);
                }
                const int chunk = 4 * p + c16;
                *reinterpret_cast<uint4*>(prow + ((chunk ^ (row & 7)) << 4)) =
                    make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            if (t > 0 && ok)
                ok = mbar_wait(&pv_done[(t - 1) & 1], (uint32_t)(((t - 1) >> 1) & 1), kWaitNs);
#pragma unroll
            for (int c16 = 0; c16 < 4; ++c16) {
                const int chunk = 4 * p + c16;
                *reinterpret_cast<uint4*>(plow + ((chunk ^ (row & 7)) << 4)) =
                    make_uint4(lo4[c16][0], lo4[c16][1], lo4[c16][2], lo4[c16][3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&p_full[bf]);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        {
            const int tl = n_tiles - 1;
            if (ok) ok = mbar_wait(&pv_done[tl & 1], (uint32_t)((tl >> 1) & 1), kWaitNs);
        }
        if (!ok) record_error(err, kDevTimeout, (int32_t)q, /*where=*/11);
        // row sums: per-thread partials -> shared memory (the row buffers are
        // free once the last PV has completed), summed per head below
        float* lsc = reinterpret_cast<float*>(smem + C::kOffR);
#pragma unroll
        for (int e = 0; e < 32; ++e) lsc[row * (kHeads + 1) + 32 * p + e] = l_part[e];
    }

    // ---- epilogue, warps 4-11: per-head sums, then O^T read out of TMEM
    if (warp >= 4) {
        asm volatile("bar.sync 3, %0;" ::"n"(2 * kSoftmaxThreads) : "memory");
        tc_fence_after();
        const int wq = warp & 3, sg = (warp - 4) >> 2;
        const int hb = 32 * sg;                      // this warp's heads: hb .. hb + 31
        const bool head_owner = warp == 4 || warp == 5;    // head (warp - 4) * 32 + lane
        const int ho = (warp - 4) * 32 + lane;
        const uint32_t lane_addr = tmem_base + ((uint32_t)(32 * wq) << 16);
        const float* lsc = reinterpret_cast<const float*>(smem + C::kOffR);
        if (head_owner) {                          // four independent sums, loads in flight together
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int r = 0; r < kTileRows; ++r) s4[r & 3] += lsc[r * (kHeads + 1) + ho];
            l_fin[ho] = (s4[0] + s4[1]) + (s4[2] + s4[3]);
        }
        asm volatile("bar.sync 3, %0;" ::"n"(2 * kSoftmaxThreads) : "memory");
        // O^T lane 32 wq + lane holds latent columns 32 wq + lane + 128 i (an
        // M = 128 accumulator); this thread writes heads hb ..
        // two latent blocks' TMEM loads in flight per wait
        if (pair) {                                   // staged for the pair merge
#pragma unroll 1
            for (int i = 0; i < 4; i += 2) {
                const int c = 32 * wq + lane + kOBlock * i;
                float v[32], u[32];
                tmem_ld_32cols_x2(lane_addr + kOCol + 64 * i + hb, lane_addr + kOCol + 64 * (i + 1) + hb,
                                  v, u);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    stage[(hb + e) * kLatent + c] = v[e];
                    stage[(hb + e) * kLatent + c + kOBlock] = u[e];
                }
            }
        }
        const bool final_out = n_split == 1;
        const int64_t part = q * n_split + split;
        float* dst = final_out ? out + q * kHeads * kLatent : part_o + part * kHeads * kLatent;
#pragma unroll 1
        for (int i = 0; i < 4 && !pair; i += 2) {
            if (!owns(i)) continue;
            const int c = 32 * wq + lane + kOBlock * i;
            float v[32], u[32];
            tmem_ld_32cols_x2(lane_addr + kOCol + 64 * i + hb, lane_addr + kOCol + 64 * (i + 1) + hb,
                              v, u);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const float l = l_fin[hb + e];
                const float inv = l > 0.f ? 1.f / l : 0.f;
                dst[(hb + e) * kLatent + c] = final_out ? v[e] * inv : v[e];
                dst[(hb + e) * kLatent + c + kOBlock] = final_out ? u[e] * inv : u[e];
            }
        }
        if (head_owner && !pair && half == 0) {
            const int h = ho;
            const float l = l_fin[h];
            const float m = m_fin[h];
            if (final_out) {
                if (lse != nullptr)
                    lse[q * kHeads + h] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
            } else {
                part_ml[(part * kHeads + h) * 2] = l > 0.f ? m * kLn2 : -INFINITY;
                part_ml[(part * kHeads + h) * 2 + 1] = l;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (pair) pair_merge();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Row-major [rows, width] bf16 matrix read in boxes of box_rows x 64 columns
// with the 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t width, uint32_t box_rows) {
    if (rows == 0) return false;
    const uint64_t dims[2] = {(uint64_t)width, rows};
    const uint64_t strides[1] = {(uint64_t)width * 2};
    const uint32_t box[2] = {64, box_rows};
    return encode_bf16_map(m, base, 2, dims, strides, box);
}

template <int W>
cudaError_t launch_w(const Shape& sh, const BatchDev& b, const void* q_abs, const void* cache,
                     const int32_t* idx, const int32_t* n_sel, float* out, float* lse,
                     float* part_o, float* part_ml, int32_t rps, int32_t n_split, int32_t* err,
                     bool q_early, cudaStream_t st) {
    using C = Cfg<W>;
    CUtensorMap tm_q;
    if (!make_map(&tm_q, q_abs, (uint64_t)b.n_q * kHeads, W, kHeads)) return cudaErrorInvalidValue;
    auto kern = sparse_mla_tc<W>;
    cudaError_t e = ensure_dyn_smem((const void*)kern, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    const int32_t pair = n_split == 2 ? 1 : 0;
    if (!pair) {
        // A launch of few CTAs (decode) doubles them to split the value product
        // and the output store by latent half, while it still fits one wave.
        const unsigned halves =
            n_split > 2 && (int64_t)b.n_q * n_split * 2 <= (int64_t)sm_count() ? 2u : 1u;
        e = launch_pdl(kern, dim3((unsigned)n_split, (unsigned)b.n_q, halves), dim3(kThreads), C::kSmemBytes,
                       st, tm_q, cache, b, sh.scale, idx, n_sel, sh.index_row_width(), rps, n_split,
                       pair, (int32_t)q_early, out, lse, part_o, part_ml, err);
        if (e != cudaSuccess || n_split == 1) return e;
        return launch_merge_splits(b.n_q, n_split, part_o, part_ml, out, lse, st);
    }
    // two splits per query: a cluster of two CTAs merges in distributed shared memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, (unsigned)b.n_q);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tm_q, cache, b, sh.scale, idx, n_sel,
                              sh.index_row_width(), rps, n_split, pair, (int32_t)q_early, out, lse,
                              part_o, part_ml, err);
}

}  // namespace

bool sparse_mla_tc_eligible(const Shape& sh, const BatchDev& b) {
    return sh.dtype == DSA_BF16 && sh.heads == kHeads && sh.kv_lora == kLatent &&
           (sh.width() == 576 || sh.width() == 512) && b.total_rows >= 1 &&
           b.total_rows < ((int64_t)1 << 31) && (int64_t)b.n_q * kHeads < ((int64_t)1 << 31);
}

// Tiles of 64 rows; at most one CTA per SM in a single wave.  A split's
// partial output (64 x 512 floats, written and merged) costs about as much as
// gathering a hundred rows, and a second wave of CTAs costs a wave's tiles, so
// a batch takes the most splits per query that still fit one wave (64 ragged
// decode queries: 2 splits, 128 CTAs, measured faster than 4 or 5 over two or
// three waves).  Splits keep two tiles each, except for a lone query, whose
// latency wants every split it can get.
void plan_attention_splits_tc(int32_t n_q, int64_t main_rows, int64_t max_rows,
                              int32_t* rows_per_split, int32_t* n_split) {
    if (max_rows < 1) max_rows = 1;
    if (main_rows < 1 || main_rows > max_rows) main_rows = max_rows;
    const int64_t tiles = (main_rows + kTileRows - 1) / kTileRows;
    const int64_t sms = sm_count();
    int64_t splits = n_q <= sms ? sms / n_q : 1;
    const int64_t max_splits = (n_q == 1 || tiles < 2) ? tiles : tiles / 2;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    const int64_t tiles_per = (tiles + splits - 1) / splits;
    const int64_t rps = tiles_per * kTileRows;
    splits = (max_rows + rps - 1) / rps;
    *rows_per_split = (int32_t)rps;
    *n_split = (int32_t)splits;
}

cudaError_t launch_sparse_mla_tc(const Shape& sh, const BatchDev& b, const void* q_abs,
                                 const void* cache, const int32_t* idx, const int32_t* n_sel,
                                 float* out, float* lse, float* part_o, float* part_ml,
                                 int32_t rps, int32_t n_split, int32_t* err, bool q_early,
                                 cudaStream_t st) {
    if (sh.width() == 576)
        return launch_w<576>(sh, b, q_abs, cache, idx, n_sel, out, lse, part_o, part_ml, rps,
                             n_split, err, q_early, st);
    return launch_w<512>(sh, b, q_abs, cache, idx, n_sel, out, lse, part_o, part_ml, rps, n_split,
                         err, q_early, st);
}

}  // namespace dsa
