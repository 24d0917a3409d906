// index_scores.cu -- lightning-indexer scoring, CUDA-core path.
//
// s_t = sum_h w_h * relu(q_h . k_t) for every key a query sees ("GLM 5.2 in one
// C file", "The Lightning Indexer": per-head ReLU'd dot, weighted sum over
// heads; "GLM-5.x (glm-dsa, glm5next)", "The block": 32 heads x 128).
//
// One CTA scores 32 consecutive keys of one query: the query's heads are
// widened to float in shared memory (rows padded by 16 bytes so that the eight
// heads a warp reads at once sit in distinct banks); eight threads share a
// key, each holding the key row in registers and taking every eighth head,
// and their weighted ReLU sums are added by shuffles.  Float accumulation.
// This path serves float32 inputs (exact float products, which the bf16
// tensor-core path cannot give) and indexer head counts other than 32.
#include "dsa_kernels.cuh"

namespace dsa {
namespace {

constexpr int kDim = 128;        // indexer head width this build supports
constexpr int kMaxHeads = 64;
constexpr int kKeysPerCta = 32;
constexpr int kLanesPerKey = 8;
constexpr int kThreads = kKeysPerCta * kLanesPerKey;
constexpr int kQStride4 = kDim / 4 + 1;    // float4s per shared query row (padded)

__device__ __forceinline__ void load_row(const float* __restrict__ src, float* dst) {
    const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
    for (int i = 0; i < kDim / 4; ++i) {
        const float4 v = __ldg(s4 + i);
        dst[4 * i + 0] = v.x; dst[4 * i + 1] = v.y; dst[4 * i + 2] = v.z; dst[4 * i + 3] = v.w;
    }
}

__device__ __forceinline__ void load_row(const __nv_bfloat16* __restrict__ src, float* dst) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < kDim / 8; ++i) {
        const uint4 v = __ldg(s4 + i);
        const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&wds[j]);
            const float2 f = __bfloat1622float2(p);
            dst[8 * i + 2 * j + 0] = f.x;
            dst[8 * i + 2 * j + 1] = f.y;
        }
    }
}

// 16 bytes of a query row (vector v of the query's heads) widened into the
// padded shared layout.
__device__ __forceinline__ void stage16(const float* __restrict__ src, int v, float4* qs) {
    constexpr int kV = kDim / 4;                         // float4s per head
    qs[(v / kV) * kQStride4 + v % kV] = __ldg(reinterpret_cast<const float4*>(src) + v);
}
__device__ __forceinline__ void stage16(const __nv_bfloat16* __restrict__ src, int v, float4* qs) {
    constexpr int kV = kDim / 8;                         // 16-byte vectors per head
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(src) + v);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
    const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.z));
    const float2 d = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.w));
    float4* row = qs + (v / kV) * kQStride4 + 2 * (v % kV);
    row[0] = make_float4(a.x, a.y, b.x, b.y);
    row[1] = make_float4(c.x, c.y, d.x, d.y);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
index_scores_simt(BatchDev b, int32_t hi, const T* __restrict__ q_idx,
                  const float* __restrict__ w, const T* __restrict__ k_idx,
                  float* __restrict__ scores, int64_t ld, int32_t* err) {
    __shared__ float4 qs[kMaxHeads * kQStride4];
    __shared__ float wsh[kMaxHeads];
    const int64_t q = blockIdx.y;
    QueryInfo qi;
    if (!query_info(b, q, qi, err, /*where=*/1)) return;          // uniform in the CTA
    const int64_t t0 = (int64_t)blockIdx.x * kKeysPerCta;
    if (t0 >= qi.n_keys) return;

    // eight consecutive lanes per key: lane group g takes heads g, g + 8, ...;
    // the key row's loads go out before the query is staged
    const int g = threadIdx.x % kLanesPerKey;
    const int64_t t = t0 + threadIdx.x / kLanesPerKey;
    const bool live = t < qi.n_keys;
    float key[kDim];
    if (live) load_row(k_idx + (qi.key0 + t) * kDim, key);

    // the query's heads: 16-byte loads, several in flight per thread
    const T* qsrc = q_idx + q * (int64_t)hi * kDim;
    constexpr int kPer16 = 16 / (int)sizeof(T);
    const int n16 = hi * kDim / kPer16;
#pragma unroll 4
    for (int v = threadIdx.x; v < n16; v += kThreads) stage16(qsrc, v, qs);
    for (int i = threadIdx.x; i < hi; i += blockDim.x) wsh[i] = w[q * hi + i];
    __syncthreads();

    float acc = 0.f;
    if (live) {
        for (int h = g; h < hi; h += kLanesPerKey) {
            float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
            for (int c = 0; c < kDim / 4; ++c) {
                const float4 qv = qs[h * kQStride4 + c];
                d0 = fmaf(qv.x, key[4 * c + 0], d0);
                d1 = fmaf(qv.y, key[4 * c + 1], d1);
                d2 = fmaf(qv.z, key[4 * c + 2], d2);
                d3 = fmaf(qv.w, key[4 * c + 3], d3);
            }
            const float d = (d0 + d1) + (d2 + d3);
            acc = fmaf(wsh[h], fmaxf(d, 0.f), acc);                  // weight * relu
        }
    }
#pragma unroll
    for (int off = kLanesPerKey / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (live && g == 0) scores[q * ld + t] = acc;
}

}  // namespace

size_t index_scores_scratch_bytes(const Shape& sh, const BatchDev& b) {
    return index_scores_tc_eligible(sh, b) ? index_scores_tc_scratch_bytes(b.n_seq, b.n_q) : 0;
}

cudaError_t launch_index_scores(const Shape& sh, const BatchDev& b, int64_t max_keys,
                                const void* q_idx, const float* w, const void* k_idx,
                                float* scores, int64_t ld, void* scratch, int32_t* err,
                                cudaStream_t st) {
    if (b.n_q == 0 || max_keys == 0) return cudaSuccess;
    if (index_scores_tc_eligible(sh, b))
        return launch_index_scores_tc(sh, b, q_idx, w, k_idx, scores, ld, scratch, err, st);
    const dim3 grid((unsigned)((max_keys + kKeysPerCta - 1) / kKeysPerCta), (unsigned)b.n_q);
    if (sh.dtype == DSA_F32)
        return launch_plain(index_scores_simt<float>, grid, dim3(kThreads), 0, st, b,
                            sh.idx_heads, static_cast<const float*>(q_idx), w,
                            static_cast<const float*>(k_idx), scores, ld, err);
    return launch_plain(index_scores_simt<__nv_bfloat16>, grid, dim3(kThreads), 0, st, b,
                        sh.idx_heads, static_cast<const __nv_bfloat16*>(q_idx), w,
                        static_cast<const __nv_bfloat16*>(k_idx), scores, ld, err);
}

}  // namespace dsa
