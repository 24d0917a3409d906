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
//   warps 4..  epilogue (4 warps for decode, 16 for a group of 8 queries:
//              each warpgroup takes two of them): tcgen05.ld of each key's 32
//              head dots (one TMEM lane per key), relu, weighted head sum with
//              packed FMAs into four partial sums, coalesced score stores.
// Decode streams every key once from HBM and is bound by HBM bandwidth; a
// prefill chunk re-reads each key tile for every query group (from L2) and is
// bound by the tensor pipe.
#include <atomic>
#include <mutex>

#include "index_pipeline.cuh"

namespace dsa {
namespace idxp {

// Row-major [rows, 128] bf16 matrix read in boxes of box_rows x 64 columns with
// the 128-byte swizzle.
bool make_rows128_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
    if (rows == 0) return false;
    const uint64_t dims[2] = {(uint64_t)kIdxDim, rows};
    const uint64_t strides[1] = {(uint64_t)kIdxDim * 2};
    const uint32_t box[2] = {64, box_rows};
    return encode_bf16_map(m, base, 2, dims, strides, box);
}

}  // namespace idxp

namespace {

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

}  // namespace

bool encode_bf16_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr || rank < 1 || rank > 5) return false;
    cuuint64_t d[5], st[4];
    cuuint32_t bx[5], estr[5];
    for (int i = 0; i < rank; ++i) {
        if (dims[i] == 0) return false;
        d[i] = dims[i];
        bx[i] = box[i];
        estr[i] = 1;
        if (i + 1 < rank) st[i] = strides[i];
    }
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), d,
               st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// Host-side per-device facts, looked up once: a decode step is launched
// thousands of times a second and each driver query costs host time.
namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

struct SmemLimit {                       // the largest limit set so far, per (kernel, device)
    const void* func;
    int dev;
    int bytes;
};
std::mutex g_smem_mu;
SmemLimit g_smem[256];
int g_smem_n = 0;
}  // namespace

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < kMaxDevices) {
        n = g_sm_count[dev].load(std::memory_order_relaxed);
        if (n > 0) return n;
    }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        return 148;
    if (dev >= 0 && dev < kMaxDevices) g_sm_count[dev].store(n, std::memory_order_relaxed);
    return n;
}

cudaError_t ensure_dyn_smem(const void* func, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_smem_mu);
    int i = 0;
    while (i < g_smem_n && !(g_smem[i].func == func && g_smem[i].dev == dev)) ++i;
    if (i < g_smem_n && g_smem[i].bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (i < g_smem_n) g_smem[i].bytes = bytes;
    else if (g_smem_n < 256) g_smem[g_smem_n++] = SmemLimit{func, dev, bytes};
    return cudaSuccess;
}

namespace {

using namespace sm100;
using namespace idxp;

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
    // one thread per group (a prefill chunk is one sequence of many groups):
    // its sequence by binary search over the group offsets
    const int64_t n_groups = seq_goff[b.n_seq];
    for (int64_t g = threadIdx.x; g < n_groups; g += blockDim.x) {
        int lo = 0, hi = b.n_seq - 1;                 // last s with seq_goff[s] <= g
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (seq_goff[mid] <= g) lo = mid; else hi = mid - 1;
        }
        const int s = lo;
        const int64_t q0 = b.q_off[s], q_len = b.q_off[s + 1] - q0;
        const int64_t r0 = b.row_off[s], kv_len = b.row_off[s + 1] - r0;
        const int64_t k0 = b.key_off[s], n_keys_seq = b.key_off[s + 1] - k0;
        const bool ok = q_len <= kv_len && kv_len <= b.max_kv_len && r0 >= 0 &&
                        b.row_off[s + 1] <= b.total_rows && k0 >= 0 &&
                        n_keys_seq >= kv_len / b.kpool && b.key_off[s + 1] <= b.total_keys &&
                        q0 >= 0 && b.q_off[s + 1] <= b.n_q;
        const int64_t j = (g - seq_goff[s]) * gq;
        if (!ok && j == 0) record_error(err, kDevBadBatch, s, /*where=*/4);
        IdxGroup G;
        G.key0 = k0;
        G.q0 = (int32_t)(q0 + j);
        G.nq = ok ? (int32_t)(q_len - j < gq ? q_len - j : gq) : 0;
        // L_last < 2^31 (max_kv_len is), so 32-bit divisions
        G.L_last = ok ? (int32_t)(kv_len - q_len + j + G.nq) : 0;
        G.pad = 0;
        groups[g] = G;
        const int32_t nk = G.nq > 0 ? G.L_last / b.kpool : 0;
        tile_off[g + 1] = (nk + kTileKeys - 1) / kTileKeys;
    }
    if (threadIdx.x == 0) tile_off[0] = 0;
    __syncthreads();
    block_inclusive_scan(tile_off + 1, n_groups, warp_tot);
}

// ---------------------------------------------------------------- the kernel

// The standalone indexer's epilogue policy: scores to global memory (the
// kernel has waited for the previous kernel, which may read the score rows).
struct ScoreStore {
    float* scores;
    int64_t ld;
    __device__ void begin() {}
    __device__ void emit(const IdxGroup& G, int j, int64_t t_row, bool valid, int64_t, int, float s) {
        if (valid) scores[(int64_t)(G.q0 + j) * ld + t_row] = s;
    }
};

// kSpec: the instantiation for decode batches whose host scalars imply their
// plan (spec_plan_guess), which guesses its first key tiles before the batch
// offsets are read (spec_issue / spec_settle).
template <int GQ, bool kSpec>
__global__ void __launch_bounds__(Cfg<GQ>::kThreads, 1)
index_scores_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                const float* __restrict__ w, const IdxGroup* __restrict__ groups,
                const int64_t* __restrict__ tile_off, const int64_t* __restrict__ seq_goff,
                int32_t n_seq, int32_t kpool, float* __restrict__ scores, int64_t ld,
                BatchDev bq, int32_t local_plan, int32_t* err) {
    using C = Cfg<GQ>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    pdl_trigger();
    setup<GQ, C::kStages>(smem, &tm_k, &tm_q);       // local to the CTA: before the wait
    // Everything below reads memory an earlier kernel may write -- the batch
    // offsets, the plan kernel's arrays, the queries and keys the TMA loads --
    // so nothing is read before the previous kernel is complete and visible.
    pdl_wait();
    int64_t n_groups;
    if (local_plan) {
        // thread 32: a single query's first key tiles, guessed from the
        // batch's bounds, while thread 0 reads the batch offsets
        if (kSpec && threadIdx.x == 32)
            spec_issue<GQ, C::kStages>(smem, &tm_k, &tm_q, bq, kpool, blockIdx.x, gridDim.x,
                                       INT64_MAX);
        n_groups = local_decode_plan<C>(smem, bq, kpool, err, /*where=*/4);
        groups = reinterpret_cast<const IdxGroup*>(smem + C::kOffPlanG);
        tile_off = reinterpret_cast<const int64_t*>(smem + C::kOffPlanT);
    } else {
        n_groups = seq_goff[n_seq];
    }
    const int64_t U = tile_off[n_groups];
    const int64_t u_begin = mul_div(blockIdx.x, U, gridDim.x);
    const int64_t u_end = mul_div(blockIdx.x + 1, U, gridDim.x);
    int pre = 0;                                     // the first key tiles on their way now
    if (threadIdx.x == 0)
        pre = kSpec && local_plan ? spec_settle<GQ, C::kStages>(smem, &tm_k, &tm_q, bq, kpool, groups,
                                                                tile_off, n_groups, u_begin, u_end,
                                                                err, /*where=*/65)
                         : issue_first<GQ, C::kStages>(smem, &tm_k, &tm_q, groups, tile_off,
                                                       n_groups, u_begin, u_end);
    // a wrong guess re-arms barriers that the other roles wait on in run()
    if (kSpec) __syncthreads();
    ScoreStore epi{scores, ld};                      // an empty range only releases TMEM
    run<GQ, C::kStages>(smem, &tm_k, &tm_q, groups, tile_off, n_groups, u_begin, u_end, w, kpool,
                        epi, err, pre);
}

// ---------------------------------------------------------------- host side

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
        e = launch_plain(idx_group_plan, dim3(1), dim3(1024), 0, st, b, (int32_t)GQ, pa.seq_goff,
                         pa.groups, pa.tile_off, err);
        if (e != cudaSuccess) return e;
    }
    int64_t g_nk = 0, g_ns = 0;
    auto kern = local && spec_plan_guess(b, sh.kpool, &g_nk, &g_ns) ? index_scores_tc<GQ, true>
                                                                    : index_scores_tc<GQ, false>;
    e = ensure_dyn_smem((const void*)kern, (int)C::kSmemBytes);
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
