// pool_compress.cu -- pool-key compression for the k-pool indexer.
//
// Each token caches a cell [key | gate] of 2 x 128 values; a pool of kpool
// consecutive tokens is compressed into one 128-wide key by a softmax over its
// cells' gates plus a per-slot position embedding, weighting their keys, per
// channel ("GLM-5.x (glm-dsa, glm5next)", table "GLM-5.3-Flash", row "Pooled
// indexer").  The key is made once, when the pool's last token arrives
// ("GLM-5.3-Flash on WASTE", "DeepSeek Sparse Attention, k-pool flavour"):
// a call writes, for each sequence, the complete pools whose last token is
// one of the sequence's new tokens (its queries' rows).
//
// HBM-bound streaming: one warp per pool, four channels per lane (8- or
// 16-byte loads of each cell's key and gate quarter, coalesced across the
// warp), a one-pass running softmax over the slots in float32, the key written
// in the cache's dtype.
#include "dsa_kernels.cuh"

namespace dsa {
namespace {

constexpr int kDim = 128;                  // indexer key width
constexpr int kWarpsPerCta = 8;

struct Quad {
    float v[4];
};

__device__ __forceinline__ Quad load4(const float* p) {
    const float4 x = __ldcs(reinterpret_cast<const float4*>(p));
    return Quad{{x.x, x.y, x.z, x.w}};
}
__device__ __forceinline__ Quad load4(const __nv_bfloat16* p) {
    const uint2 x = __ldcs(reinterpret_cast<const uint2*>(p));
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&x.y));
    return Quad{{a.x, a.y, b.x, b.y}};
}
__device__ __forceinline__ void store4(float* p, const Quad& q) {
    *reinterpret_cast<float4*>(p) = make_float4(q.v[0], q.v[1], q.v[2], q.v[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const Quad& q) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(q.v[0], q.v[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(q.v[2], q.v[3]);
    uint2 x;
    x.x = *reinterpret_cast<const uint32_t*>(&a);
    x.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = x;
}

// grid: x = chunks of kWarpsPerCta new pools of one sequence, y = sequence.
// KP > 0: the pool size at compile time (every cell's loads issued before any
// arithmetic); KP = 0: b.kpool at run time.
template <typename T, int KP>
__global__ void __launch_bounds__(32 * kWarpsPerCta)
pool_compress_kernel(BatchDev b, const T* __restrict__ cells, const float* __restrict__ pos,
                     T* __restrict__ pool_keys, int32_t* err) {
    const int s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kpool = KP > 0 ? KP : b.kpool;
    // the sequence: its rows (one cell per row), pool keys and new tokens
    const int64_t q0 = b.q_off[s], q1 = b.q_off[s + 1];
    const int64_t r0 = b.row_off[s], r1 = b.row_off[s + 1];
    const int64_t k0 = b.key_off[s], k1 = b.key_off[s + 1];
    const int64_t kv_len = r1 - r0, q_len = q1 - q0;
    if (q_len < 0 || q_len > kv_len || q_len > b.max_q_len || kv_len > b.max_kv_len || r0 < 0 ||
        r1 > b.total_rows || k0 < 0 || k1 > b.total_keys || k1 - k0 < kv_len / kpool) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, kDevBadBatch, s, /*where=*/20);
        return;
    }
    // the complete pools whose last token is new
    const int64_t j = (kv_len - q_len) / kpool + (int64_t)blockIdx.x * kWarpsPerCta + warp;
    if (j >= kv_len / kpool) return;
    const int c = 4 * lane;                                  // this lane's channels
    const T* cell = cells + (r0 + j * kpool) * (2 * kDim);
    Quad out;
    if constexpr (KP > 0) {
        // all of the pool's key and gate quarters in flight at once
        Quad key[KP > 0 ? KP : 1], gate[KP > 0 ? KP : 1];
#pragma unroll
        for (int i = 0; i < KP; ++i) {
            key[i] = load4(cell + i * 2 * kDim + c);
            gate[i] = load4(cell + i * 2 * kDim + kDim + c);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // softmax over the slots of gate + slot embedding, weighting the keys
            float z[KP > 0 ? KP : 1], zmax = -INFINITY;
#pragma unroll
            for (int i = 0; i < KP; ++i) {
                z[i] = gate[i].v[e] + __ldg(pos + i * kDim + c + e);
                zmax = fmaxf(zmax, z[i]);
            }
            float den = 0.f, num = 0.f;
#pragma unroll
            for (int i = 0; i < KP; ++i) {
                const float w = z[i] == -INFINITY ? 0.f : expf(z[i] - zmax);   // masked slot
                den += w;
                num += w * key[i].v[e];
            }
            out.v[e] = den > 0.f ? num / den : 0.f;          // every slot masked: 0
        }
    } else {
        float m[4], den[4], num[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) { m[e] = -INFINITY; den[e] = 0.f; num[e] = 0.f; }
        for (int i = 0; i < kpool; ++i, cell += 2 * kDim) {
            const Quad key = load4(cell + c);
            const Quad gate = load4(cell + kDim + c);
            const float4 p = __ldg(reinterpret_cast<const float4*>(pos + i * kDim + c));
            const float pe[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                // running softmax over the slots: logit = gate + slot embedding
                const float z = gate.v[e] + pe[e];
                if (z > m[e]) {
                    const float r = expf(m[e] - z);              // 0 for the first slot
                    den[e] = den[e] * r + 1.f;
                    num[e] = num[e] * r + key.v[e];
                    m[e] = z;
                } else if (z != -INFINITY) {                 // a masked slot weighs 0
                    const float w = expf(z - m[e]);
                    den[e] += w;
                    num[e] += w * key.v[e];
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) out.v[e] = den[e] > 0.f ? num[e] / den[e] : 0.f;
    }
    store4(pool_keys + (k0 + j) * kDim + c, out);
}

}  // namespace

cudaError_t launch_pool_compress(const Shape& sh, const BatchDev& b, const void* cells,
                                 const float* pos, void* pool_keys, int32_t* err,
                                 cudaStream_t st) {
    if (b.n_seq == 0 || b.max_q_len == 0) return cudaSuccess;
    // new pools of a sequence: at most ceil(q_len / kpool)
    const int64_t max_new = ((int64_t)b.max_q_len + sh.kpool - 1) / sh.kpool;
    const int64_t gx = (max_new + kWarpsPerCta - 1) / kWarpsPerCta;
    if (gx > 0x7fffffff || b.n_seq > 65535) return cudaErrorInvalidConfiguration;
    const dim3 grid((unsigned)(gx > 0 ? gx : 1), (unsigned)b.n_seq);
    const bool four = sh.kpool == 4;
    if (sh.dtype == DSA_BF16) {
        auto k = four ? pool_compress_kernel<__nv_bfloat16, 4> : pool_compress_kernel<__nv_bfloat16, 0>;
        return launch_plain(k, grid, dim3(32 * kWarpsPerCta), 0, st, b,
                            static_cast<const __nv_bfloat16*>(cells), pos,
                            static_cast<__nv_bfloat16*>(pool_keys), err);
    } else {
        auto k = four ? pool_compress_kernel<float, 4> : pool_compress_kernel<float, 0>;
        return launch_plain(k, grid, dim3(32 * kWarpsPerCta), 0, st, b,
                            static_cast<const float*>(cells), pos, static_cast<float*>(pool_keys),
                            err);
    }
}

}  // namespace dsa
