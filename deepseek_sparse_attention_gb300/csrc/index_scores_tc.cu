// index_scores_tc.cu -- lightning-indexer scoring on the tcgen05 tensor cores.
//
// s_t = sum_h w_h * relu(q_h . k_t) ("GLM 5.2 in one C file", "The Lightning
// Indexer"; "GLM-5.x (glm-dsa, glm5next)", "The block": 32 heads x 128).
//
// The 32 head dots of a key are a dense contraction: a tile of 128 keys (M)
// against the 32 heads of up to GQ queries of one sequence (N = 32*GQ), K =
// 128.  Queries of a prefill chunk share the keys of their sequence, so a
// group of GQ = 8 consecutive queries is scored per key tile (N = 256); decode
// queries each form their own group (GQ = 1, N = 32).  Per CTA (persistent,
// one per SM, a contiguous range of (group, key tile) units):
//   warp 0     TMA producer: key tiles into a ring of shared-memory stages
//              (128-byte swizzle, two 64-column boxes per tile), the group's
//              query rows once per group;
//   warp 1     MMA issuer: 8 x tcgen05.mma (K = 16 each) per tile into one of
//              two TMEM accumulators, commits that free the stage and hand the
//              accumulator to the epilogue;
//   warps 4..  epilogue: tcgen05.ld of each key's 32 head dots (one TMEM lane
//              per key), relu, weighted head sum, coalesced score stores.
// Decode streams every key once from HBM and is bound by HBM bandwidth; a
// prefill chunk re-reads each key tile for every query group (from L2) and is
// bound by the tensor pipe.
#include "dsa_kernels.cuh"
#include "sm100.cuh"

namespace dsa {
namespace {

using namespace sm100;

constexpr int kTileKeys = 128;                      // MMA M
constexpr int kIdxDim = 128;                        // MMA K
constexpr int kIdxHeads = 32;
constexpr uint32_t kRowHalfBytes = 128;             // 64 bf16: one swizzle row
constexpr uint32_t kABoxBytes = kTileKeys * kRowHalfBytes;    // 16 KB
constexpr uint32_t kABytes = 2 * kABoxBytes;                  // 32 KB per key tile
constexpr uint64_t kWaitNs = 2000000000ull;         // bounded waits: 2 s

struct IdxGroup {          // consecutive queries of one sequence scored together
    int64_t key0;          // first indexer key of the sequence
    int32_t q0;            // first query of the group
    int32_t nq;            // queries in the group
    int32_t L_last;        // rows seen by the group's last query
    int32_t pad;
};

template <int GQ>
struct Cfg {
    static constexpr int N = kIdxHeads * GQ;
    static constexpr int kStages = GQ == 1 ? 6 : 4;
    static constexpr uint32_t kBBoxBytes = N * kRowHalfBytes;
    static constexpr uint32_t kBBytes = 2 * kBBoxBytes;
    static constexpr uint32_t kTmemCols = 2 * N;                  // two accumulators
    static constexpr int kEpiWarps = GQ == 1 ? 4 : 8;
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
    static constexpr uint32_t kOffPlanG = (kOffMisc + 16 + 15) / 16 * 16;           // IdxGroup[256]
    static constexpr uint32_t kOffPlanT = kOffPlanG + kLocalMaxQ * 24;             // int64[257]
    static constexpr uint32_t kSmemBytes = kOffPlanT + (kLocalMaxQ + 1) * 8 + 1024;
    static_assert(kTmemCols == 64 || kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512,
                  "TMEM allocation must be a power of two");
};

// ---------------------------------------------------------------- planning

// Inclusive prefix sum of a[0..n) in place, one CTA.
__device__ void block_inclusive_scan(int64_t* a, int64_t n, int64_t* warp_tot) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int64_t carry = 0;
    for (int64_t base = 0; base < n; base += blockDim.x) {
        const int64_t i = base + threadIdx.x;
        int64_t v = i < n ? a[i] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int64_t y = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += y;
        }
        if (lane == 31) warp_tot[wid] = v;
        __syncthreads();
        if (wid == 0) {
            int64_t s = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int64_t y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += y;
            }
            warp_tot[lane] = s;
        }
        __syncthreads();
        const int64_t incl = v + (wid > 0 ? warp_tot[wid - 1] : 0) + carry;
        if (i < n) a[i] = incl;
        carry += warp_tot[nw - 1];
        __syncthreads();
    }
}

// Splits every sequence's queries into groups of up to GQ and counts the key
// tiles each group needs; tile_off[g] is the first unit of group g.
__global__ void __launch_bounds__(1024)
idx_group_plan(BatchDev b, int32_t gq, int64_t* seq_goff, IdxGroup* groups, int64_t* tile_off,
               int32_t* err) {
    __shared__ int64_t warp_tot[32];
    for (int s = threadIdx.x; s < b.n_seq; s += blockDim.x) {
        const int64_t q_len = b.q_off[s + 1] - b.q_off[s];
        seq_goff[s + 1] = q_len > 0 ? (q_len + gq - 1) / gq : 0;
    }
    if (threadIdx.x == 0) seq_goff[0] = 0;
    __syncthreads();
    block_inclusive_scan(seq_goff + 1, b.n_seq, warp_tot);
    for (int s = threadIdx.x; s < b.n_seq; s += blockDim.x) {
        const int64_t q0 = b.q_off[s], q_len = b.q_off[s + 1] - q0;
        const int64_t r0 = b.row_off[s], kv_len = b.row_off[s + 1] - r0;
        const int64_t k0 = b.key_off[s], n_keys_seq = b.key_off[s + 1] - k0;
        const bool ok = q_len <= kv_len && kv_len <= b.max_kv_len && r0 >= 0 &&
                        b.row_off[s + 1] <= b.total_rows && k0 >= 0 &&
                        n_keys_seq >= kv_len / b.kpool && b.key_off[s + 1] <= b.total_keys &&
                        q0 >= 0 && b.q_off[s + 1] <= b.n_q;
        if (!ok && q_len > 0) record_error(err, kDevBadBatch, s, /*where=*/4);
        int64_t g = seq_goff[s];
        for (int64_t j = 0; j < q_len; j += gq, ++g) {
            IdxGroup G;
            G.key0 = k0;
            G.q0 = (int32_t)(q0 + j);
            G.nq = ok ? (int32_t)(q_len - j < gq ? q_len - j : gq) : 0;
            G.L_last = ok ? (int32_t)(kv_len - q_len + j + G.nq) : 0;
            G.pad = 0;
            groups[g] = G;
            const int64_t nk = G.nq > 0 ? G.L_last / b.kpool : 0;
            tile_off[g + 1] = (nk + kTileKeys - 1) / kTileKeys;
        }
    }
    if (threadIdx.x == 0) tile_off[0] = 0;
    __syncthreads();
    block_inclusive_scan(tile_off + 1, seq_goff[b.n_seq], warp_tot);
}

// ---------------------------------------------------------------- the kernel

struct Cursor {                       // walks (group, tile) units in order
    const int64_t* tile_off;
    int64_t g, t;
    __device__ void seek(int64_t u, int64_t n_groups) {
        int64_t lo = 0, hi = n_groups - 1;           // last g with tile_off[g] <= u
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (tile_off[mid] <= u) lo = mid; else hi = mid - 1;
        }
        g = lo;
        t = u - tile_off[g];
    }
    __device__ void next() {
        ++t;
        while (tile_off[g] + t >= tile_off[g + 1]) { ++g; t = 0; }
    }
    __device__ bool last_of_group() const { return tile_off[g] + t + 1 >= tile_off[g + 1]; }
};

template <int GQ>
__global__ void __launch_bounds__(Cfg<GQ>::kThreads, 1)
index_scores_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                const float* __restrict__ w, const IdxGroup* __restrict__ groups,
                const int64_t* __restrict__ tile_off, const int64_t* __restrict__ seq_goff,
                int32_t n_seq, int32_t kpool, float* __restrict__ scores, int64_t ld,
                BatchDev bq, int32_t local_plan, int32_t* err) {
    using C = Cfg<GQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
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
    pdl_trigger();
    int64_t n_groups;
    if (!local_plan) pdl_wait();                      // the plan kernel's arrays
    if (local_plan) {
        // one group per query (decode); every CTA derives the schedule itself
        IdxGroup* gs = reinterpret_cast<IdxGroup*>(smem + C::kOffPlanG);
        int64_t* ts = reinterpret_cast<int64_t*>(smem + C::kOffPlanT);
        if (threadIdx.x < bq.n_q) {
            QueryInfo qi;
            IdxGroup G{0, (int32_t)threadIdx.x, 0, 0, 0};
            if (query_info(bq, threadIdx.x, qi, err, /*where=*/4)) {
                G.key0 = qi.key0;
                G.nq = 1;
                G.L_last = (int32_t)qi.L;
            }
            gs[threadIdx.x] = G;
            ts[threadIdx.x + 1] = G.nq ? (G.L_last / kpool + kTileKeys - 1) / kTileKeys : 0;
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            ts[0] = 0;
            for (int i = 1; i <= bq.n_q; ++i) ts[i] += ts[i - 1];
        }
        __syncthreads();
        groups = gs;
        tile_off = ts;
        n_groups = bq.n_q;
    } else {
        n_groups = seq_goff[n_seq];
    }
    const int64_t U = tile_off[n_groups];
    const int64_t u_begin = (int64_t)blockIdx.x * U / gridDim.x;
    const int64_t u_end = (int64_t)(blockIdx.x + 1) * U / gridDim.x;
    if (u_begin >= u_end) return;                    // uniform: no barrier or TMEM touched

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
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_q);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {                                           // ---- TMA producer
            Cursor c{tile_off, 0, 0};
            c.seek(u_begin, n_groups);
            int stage = 0;
            uint32_t phase = 0, b_empty_par = 0;
            int64_t b_group = -1;
            int8_t issued_par[C::kStages];
            for (int s = 0; s < C::kStages; ++s) issued_par[s] = -1;
            bool ok = true;
            for (int64_t u = u_begin; u < u_end && ok; ++u) {
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
            Cursor c{tile_off, 0, 0};
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
        Cursor c{tile_off, 0, 0};
        c.seek(u_begin, n_groups);
        int ab = 0;
        uint32_t acc_par = 0;
        pdl_wait();                                    // the score rows may still be read
        for (int64_t u = u_begin; u < u_end; ++u) {
            const IdxGroup G = groups[c.g];
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
                const float4* w4 = reinterpret_cast<const float4*>(w + (int64_t)(G.q0 + j) * kIdxHeads);
                float s = 0.f;
#pragma unroll
                for (int h4 = 0; h4 < kIdxHeads / 4; ++h4) {
                    const float4 wv = __ldg(w4 + h4);
                    s = fmaf(wv.x, fmaxf(v[4 * h4 + 0], 0.f), s);
                    s = fmaf(wv.y, fmaxf(v[4 * h4 + 1], 0.f), s);
                    s = fmaf(wv.z, fmaxf(v[4 * h4 + 2], 0.f), s);
                    s = fmaf(wv.w, fmaxf(v[4 * h4 + 3], 0.f), s);
                }
                const int64_t nk = (int64_t)(G.L_last - (G.nq - 1 - j)) / kpool;
                if (t_row < nk) scores[(int64_t)(G.q0 + j) * ld + t_row] = s;
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

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiledFn) nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// Row-major [rows, 128] bf16 matrix read in boxes of box_rows x 64 columns with
// the 128-byte swizzle.
bool make_rows128_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr || rows == 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)kIdxDim, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)kIdxDim * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    return n;
}

struct PlanArrays {
    int64_t* seq_goff;
    IdxGroup* groups;
    int64_t* tile_off;
};

PlanArrays plan_arrays(void* scratch, int32_t n_seq, int32_t n_q) {
    unsigned char* p = static_cast<unsigned char*>(scratch);
    PlanArrays a;
    a.seq_goff = reinterpret_cast<int64_t*>(p);
    p += ((size_t)(n_seq + 1) * 8 + 255) / 256 * 256;
    a.groups = reinterpret_cast<IdxGroup*>(p);
    p += ((size_t)(n_q > 0 ? n_q : 1) * sizeof(IdxGroup) + 255) / 256 * 256;
    a.tile_off = reinterpret_cast<int64_t*>(p);
    return a;
}

template <int GQ>
cudaError_t launch_tc(const Shape& sh, const BatchDev& b, const void* q_idx, const float* w,
                      const void* k_idx, float* scores, int64_t ld, const PlanArrays& pa,
                      int32_t* err, cudaStream_t st) {
    using C = Cfg<GQ>;
    CUtensorMap tm_k, tm_q;
    if (!make_rows128_map(&tm_k, k_idx, (uint64_t)b.total_keys, kTileKeys) ||
        !make_rows128_map(&tm_q, q_idx, (uint64_t)b.n_q * kIdxHeads, C::N))
        return cudaErrorInvalidValue;
    const bool local = GQ == 1 && b.n_q <= C::kLocalMaxQ;
    cudaError_t e;
    if (!local) {
        idx_group_plan<<<1, 1024, 0, st>>>(b, GQ, pa.seq_goff, pa.groups, pa.tile_off, err);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    auto kern = index_scores_tc<GQ>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmemBytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(sm_count()), dim3(C::kThreads), C::kSmemBytes, st, tm_k, tm_q, w,
                      (const IdxGroup*)pa.groups, (const int64_t*)pa.tile_off,
                      (const int64_t*)pa.seq_goff, b.n_seq, sh.kpool, scores, ld, b,
                      local ? 1 : 0, err);
}

}  // namespace

bool index_scores_tc_eligible(const Shape& sh, const BatchDev& b) {
    // Tensor maps are only built with boxes no larger than the tensor.
    return sh.dtype == DSA_BF16 && sh.idx_heads == kIdxHeads && sh.idx_dim == kIdxDim &&
           b.total_keys >= kTileKeys && b.total_keys < ((int64_t)1 << 31) &&
           (int64_t)b.n_q * kIdxHeads < ((int64_t)1 << 31);
}

int32_t index_scores_tc_launches(const Shape& sh, const BatchDev& b) {
    (void)sh;
    const bool gq1 = b.max_q_len <= 1 || b.n_q < 8;
    return (gq1 && b.n_q <= Cfg<1>::kLocalMaxQ) ? 1 : 2;
}

size_t index_scores_tc_scratch_bytes(int32_t n_seq, int32_t n_q) {
    const size_t a = ((size_t)(n_seq + 1) * 8 + 255) / 256 * 256;
    const size_t g = ((size_t)(n_q > 0 ? n_q : 1) * sizeof(IdxGroup) + 255) / 256 * 256;
    const size_t t = ((size_t)(n_q + 1) * 8 + 255) / 256 * 256;
    return a + g + t;
}

cudaError_t launch_index_scores_tc(const Shape& sh, const BatchDev& b, const void* q_idx,
                                   const float* w, const void* k_idx, float* scores, int64_t ld,
                                   void* scratch, int32_t* err, cudaStream_t st) {
    const PlanArrays pa = plan_arrays(scratch, b.n_seq, b.n_q);
    // Decode queries each form a group; chunks of prefill share key tiles among
    // 8 queries (when there are at least 8 queries, so the query box fits).
    if (b.max_q_len <= 1 || b.n_q < 8)
        return launch_tc<1>(sh, b, q_idx, w, k_idx, scores, ld, pa, err, st);
    return launch_tc<8>(sh, b, q_idx, w, k_idx, scores, ld, pa, err, st);
}

}  // namespace dsa
