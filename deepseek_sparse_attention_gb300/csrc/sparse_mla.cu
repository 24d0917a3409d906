// sparse_mla.cu -- absorbed-MLA attention over the selected cache rows,
// CUDA-core path.
//
// For one query with absorbed query q_abs[h, :] (latent part, then rope part)
// and selected rows J:  z[h,j] = scale * q_abs[h,:] . row_j  over the full row,
// p = softmax_j(z),  out[h, c] = sum_j p[h,j] * row_j[c]  for the 512 latent
// columns only ("GLM 5.2 in one C file", "Attention: Multi head Latent
// Attention With a Tiny KV Cache": absorbed score against the latent plus the
// rope dot, softmax, pooled latent; "GLM-5.x (glm-dsa, glm5next)", "The
// block": 64 heads, one 576-wide row, scale 1/16; "Add GLM-5.3-Flash
// support": a NoPE row is the 512-wide latent, key and value alike).
//
// A CTA handles a range of one query's selected rows ("split"), 16 rows at a
// time: the rows are gathered into shared memory, the 64 x 16 logits are
// formed against the staged query, and an online softmax (running max and
// rescaled accumulator) folds them into a 64 x 512 float accumulator held in
// registers.  Splits of one query are combined by a log-sum-exp merge.
#include <math.h>

#include "dsa_kernels.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kHeads = 64;
constexpr int kTile = 16;        // rows per tile
constexpr int kLatent = 512;     // value width
constexpr int kSsStride = kTile + 1;

// Shared-memory row stride in elements: the row width plus 16 bytes, so that
// 16-byte reads of eight consecutive rows land in distinct banks.
template <typename T, int W>
struct Smem {
    static constexpr int kStride = W + 16 / (int)sizeof(T);
    static constexpr size_t kQ = (size_t)kHeads * kStride * sizeof(T);
    static constexpr size_t kR = (size_t)kTile * kStride * sizeof(T);
    static constexpr size_t kS = (size_t)kHeads * kSsStride * sizeof(float);
    static constexpr size_t kStats = 3 * kHeads * sizeof(float) + kTile * sizeof(int32_t);
    static constexpr size_t kTotal = kQ + kR + kS + kStats;
};

__device__ __forceinline__ void acc_dot16(const float* a, const float* b, int n, float& acc) {
    for (int i = 0; i < n; ++i) acc = fmaf(a[i], b[i], acc);
}

// 16 bytes of T widened to float.
__device__ __forceinline__ int widen16(const float* p, float* f) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    return 4;
}
__device__ __forceinline__ int widen16(const __nv_bfloat16* p, float* f) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t wds[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 g = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wds[j]));
        f[2 * j] = g.x;
        f[2 * j + 1] = g.y;
    }
    return 8;
}

__device__ __forceinline__ float4 widen4(const float* p) {
    return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 widen4(const __nv_bfloat16* p) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
    const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
    return make_float4(a.x, a.y, c.x, c.y);
}

template <typename T, int W>
__global__ void __launch_bounds__(kThreads)
sparse_mla_simt(BatchDev b, float scale, const T* __restrict__ q_abs, const T* __restrict__ cache,
                const int32_t* __restrict__ idx, const int32_t* __restrict__ n_sel,
                int64_t idx_width, int32_t rows_per_split, int32_t n_split,
                float* __restrict__ out, float* __restrict__ lse,
                float* __restrict__ part_o, float* __restrict__ part_ml, int32_t* err) {
    using S = Smem<T, W>;
    constexpr int kVec = 16 / (int)sizeof(T);          // elements per 16-byte vector
    constexpr int kRowVecs = W / kVec;
    extern __shared__ __align__(16) unsigned char smem[];
    T* Qs = reinterpret_cast<T*>(smem);
    T* Rs = reinterpret_cast<T*>(smem + S::kQ);
    float* Ss = reinterpret_cast<float*>(smem + S::kQ + S::kR);
    float* m_s = reinterpret_cast<float*>(smem + S::kQ + S::kR + S::kS);
    float* l_s = m_s + kHeads;
    float* alpha_s = l_s + kHeads;
    int32_t* row_ids = reinterpret_cast<int32_t*>(alpha_s + kHeads);

    const int tid = threadIdx.x;
    const int64_t q = blockIdx.y;
    const int split = blockIdx.x;
    QueryInfo qi;
    if (!query_info(b, q, qi, err, /*where=*/3)) return;
    // no selection (idx == nullptr): every visible row, row j being row j
    int64_t ns = idx == nullptr ? qi.L : n_sel[q];
    if (idx != nullptr) ns = ns < 0 ? 0 : (ns > idx_width ? idx_width : ns);
    const int64_t j_begin = (int64_t)split * rows_per_split;
    const int64_t j_end = j_begin + rows_per_split < ns ? j_begin + rows_per_split : ns;

    // stage the query (64 heads x W)
    const T* qsrc = q_abs + q * (int64_t)kHeads * W;
    for (int v = tid; v < kHeads * kRowVecs; v += kThreads) {
        const int h = v / kRowVecs, c = (v % kRowVecs) * kVec;
        *reinterpret_cast<uint4*>(Qs + h * S::kStride + c) =
            __ldg(reinterpret_cast<const uint4*>(qsrc + (int64_t)h * W + c));
    }
    if (tid < kHeads) { m_s[tid] = -INFINITY; l_s[tid] = 0.f; }

    const int oh = tid >> 2, ocg = tid & 3;     // accumulator owner: head, column group
    float o[kLatent / 4];
#pragma unroll
    for (int i = 0; i < kLatent / 4; ++i) o[i] = 0.f;

    for (int64_t j0 = j_begin; j0 < j_end; j0 += kTile) {
        const int nrows = (int)(j_end - j0 < kTile ? j_end - j0 : kTile);
        if (tid < kTile) {
            int32_t r = -1;
            if (tid < nrows) {
                r = idx == nullptr ? (int32_t)(j0 + tid) : idx[q * idx_width + j0 + tid];
                if (r < 0 || r >= qi.L) {
                    record_error(err, kDevBadIndex, (int32_t)q, /*where=*/3);
                    r = -1;
                }
            }
            row_ids[tid] = r;
        }
        __syncthreads();
        // gather the tile's rows
        for (int v = tid; v < kTile * kRowVecs; v += kThreads) {
            const int j = v / kRowVecs, c = (v % kRowVecs) * kVec;
            const int32_t r = row_ids[j];
            uint4 val = make_uint4(0, 0, 0, 0);
            if (r >= 0) val = __ldg(reinterpret_cast<const uint4*>(cache + (qi.row0 + r) * W + c));
            *reinterpret_cast<uint4*>(Rs + j * S::kStride + c) = val;
        }
        __syncthreads();
        // logits: thread -> row j, heads h0 + 16 i
        {
            const int j = tid & (kTile - 1), h0 = tid >> 4;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c = 0; c < W; c += kVec) {
                float rf[kVec];
                widen16(Rs + j * S::kStride + c, rf);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float qf[kVec];
                    widen16(Qs + (h0 + 16 * i) * S::kStride + c, qf);
                    acc_dot16(qf, rf, kVec, acc[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
                Ss[(h0 + 16 * i) * kSsStride + j] = row_ids[j] >= 0 ? acc[i] * scale : -INFINITY;
        }
        __syncthreads();
        // online softmax, one thread per head
        if (tid < kHeads) {
            float* srow = Ss + tid * kSsStride;
            const float m_old = m_s[tid];
            float mx = -INFINITY;
            for (int j = 0; j < kTile; ++j) mx = fmaxf(mx, srow[j]);
            const float m_new = fmaxf(m_old, mx);
            float alpha = 1.f, psum = 0.f;
            if (m_new == -INFINITY) {
                for (int j = 0; j < kTile; ++j) srow[j] = 0.f;
            } else {
                alpha = expf(m_old - m_new);
                for (int j = 0; j < kTile; ++j) {
                    const float p = expf(srow[j] - m_new);
                    srow[j] = p;
                    psum += p;
                }
            }
            l_s[tid] = l_s[tid] * alpha + psum;
            m_s[tid] = m_new;
            alpha_s[tid] = alpha;
        }
        __syncthreads();
        // rescale and accumulate P . R_latent
        {
            const float a = alpha_s[oh];
#pragma unroll
            for (int i = 0; i < kLatent / 4; ++i) o[i] *= a;
            for (int j = 0; j < kTile; ++j) {
                const float p = Ss[oh * kSsStride + j];
                const T* rrow = Rs + j * S::kStride + 4 * ocg;
#pragma unroll
                for (int i = 0; i < kLatent / 16; ++i) {
                    const float4 r4 = widen4(rrow + 16 * i);
                    o[4 * i + 0] = fmaf(p, r4.x, o[4 * i + 0]);
                    o[4 * i + 1] = fmaf(p, r4.y, o[4 * i + 1]);
                    o[4 * i + 2] = fmaf(p, r4.z, o[4 * i + 2]);
                    o[4 * i + 3] = fmaf(p, r4.w, o[4 * i + 3]);
                }
            }
        }
        __syncthreads();
    }
    __syncthreads();

    const float m = m_s[oh], l = l_s[oh];
    if (n_split == 1) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float* dst = out + (q * kHeads + oh) * (int64_t)kLatent + 4 * ocg;
#pragma unroll
        for (int i = 0; i < kLatent / 16; ++i)
            *reinterpret_cast<float4*>(dst + 16 * i) =
                make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
        if (lse != nullptr && ocg == 0) lse[q * kHeads + oh] = l > 0.f ? m + logf(l) : -INFINITY;
    } else {
        const int64_t part = q * n_split + split;
        float* dst = part_o + (part * kHeads + oh) * (int64_t)kLatent + 4 * ocg;
#pragma unroll
        for (int i = 0; i < kLatent / 16; ++i)
            *reinterpret_cast<float4*>(dst + 16 * i) =
                make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        if (ocg == 0) {
            part_ml[(part * kHeads + oh) * 2 + 0] = m;
            part_ml[(part * kHeads + oh) * 2 + 1] = l;
        }
    }
}

// Log-sum-exp merge of the splits of one query: one CTA per (query, head, a
// quarter of the latent columns): 256 CTAs for one query, spread over the
// SMs.  Its 128 threads are four groups of 32, each group a quarter of the
// splits (every split's loads of a group issued at once, eight at a time),
// four latent columns per thread; each group keeps a running maximum, and the
// four groups' (maximum, sum, accumulator) are combined in shared memory.  An
// empty split has m = -inf: weight 0, and its output (never written) is not
// used.
__global__ void __launch_bounds__(128)
merge_splits(int32_t n_split, const float* __restrict__ part_o, const float* __restrict__ part_ml,
             float* __restrict__ out, float* __restrict__ lse) {
    asm volatile("griddepcontrol.wait;" ::: "memory");      // the partials must be complete
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    constexpr int kB = 8;
    constexpr int kGroups = 4;
    __shared__ float4 s_acc[kGroups][32];
    __shared__ float s_m[kGroups][32], s_l[kGroups][32];
    const int h = blockIdx.x >> 2;
    const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
    const int c4 = (blockIdx.x & 3) * 32 + lane;            // columns 4 c4 .. 4 c4 + 3
    const int64_t q = blockIdx.y;
    const int s_lo = (int)((int64_t)n_split * grp / kGroups);
    const int s_hi = (int)((int64_t)n_split * (grp + 1) / kGroups);
    const float2* ml = reinterpret_cast<const float2*>(part_ml) + q * n_split * kHeads + h;
    const float4* po = reinterpret_cast<const float4*>(part_o) +
                       (q * n_split * kHeads + h) * (int64_t)(kLatent / 4) + c4;
    const int64_t o_stride = (int64_t)kHeads * (kLatent / 4);   // float4s between splits
    float M = -INFINITY, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s0 = s_lo; s0 < s_hi; s0 += kB) {
        float2 v[kB];
        float4 o[kB];
#pragma unroll
        for (int k = 0; k < kB; ++k) {
            const bool in = s0 + k < s_hi;
            v[k] = in ? __ldg(ml + (int64_t)(s0 + k) * kHeads) : make_float2(-INFINITY, 0.f);
            o[k] = in ? __ldg(po + (int64_t)(s0 + k) * o_stride) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float Mb = M;
#pragma unroll
        for (int k = 0; k < kB; ++k) Mb = fmaxf(Mb, v[k].x);
        if (Mb == -INFINITY) continue;                      // no weight yet
        const float r = expf(M - Mb);                       // 0 while M is -inf
        L *= r;
        acc.x *= r; acc.y *= r; acc.z *= r; acc.w *= r;
#pragma unroll
        for (int k = 0; k < kB; ++k) {
            if (v[k].x == -INFINITY) continue;              // empty split: its output is never read
            const float f = expf(v[k].x - Mb);
            L = fmaf(v[k].y, f, L);
            acc.x = fmaf(o[k].x, f, acc.x);
            acc.y = fmaf(o[k].y, f, acc.y);
            acc.z = fmaf(o[k].z, f, acc.z);
            acc.w = fmaf(o[k].w, f, acc.w);
        }
        M = Mb;
    }
    s_acc[grp][lane] = acc;
    s_m[grp][lane] = M;
    s_l[grp][lane] = L;
    __syncthreads();
    if (grp != 0) return;
    float Mt = -INFINITY;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) Mt = fmaxf(Mt, s_m[g][lane]);
    float Lt = 0.f;
    float4 at = make_float4(0.f, 0.f, 0.f, 0.f);
    if (Mt != -INFINITY) {
#pragma unroll
        for (int g = 0; g < kGroups; ++g) {
            if (s_m[g][lane] == -INFINITY) continue;        // a group without weight
            const float f = expf(s_m[g][lane] - Mt);
            const float4 a = s_acc[g][lane];
            Lt = fmaf(s_l[g][lane], f, Lt);
            at.x = fmaf(a.x, f, at.x);
            at.y = fmaf(a.y, f, at.y);
            at.z = fmaf(a.z, f, at.z);
            at.w = fmaf(a.w, f, at.w);
        }
    }
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    reinterpret_cast<float4*>(out)[(q * kHeads + h) * (int64_t)(kLatent / 4) + c4] =
        make_float4(at.x * inv, at.y * inv, at.z * inv, at.w * inv);
    if (lse != nullptr && c4 == 0) lse[q * kHeads + h] = Lt > 0.f ? Mt + logf(Lt) : -INFINITY;
}

// Rows per split: enough CTAs to fill the GPU about twice, at least one
// 16-row tile each (a CTA's time is its tile loop: a short query is spread
// over as many CTAs as it has tiles).
void plan_splits_simt(int32_t n_q, int64_t max_rows, int32_t* rows_per_split, int32_t* n_split) {
    if (max_rows < 1) max_rows = 1;
    const int64_t target_ctas = 2 * (int64_t)sm_count();
    int64_t splits = (target_ctas + n_q - 1) / n_q;
    const int64_t max_splits = (max_rows + kTile - 1) / kTile;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    int64_t rps = (max_rows + splits - 1) / splits;
    rps = (rps + kTile - 1) / kTile * kTile;
    splits = (max_rows + rps - 1) / rps;
    *rows_per_split = (int32_t)rps;
    *n_split = (int32_t)splits;
}

template <typename T, int W>
cudaError_t launch_typed(const Shape& sh, const BatchDev& b, const void* q_abs, const void* cache,
                         const int32_t* idx, const int32_t* n_sel, float* out, float* lse,
                         float* part_o, float* part_ml, int32_t rps, int32_t n_split, int32_t* err,
                         cudaStream_t st) {
    using S = Smem<T, W>;
    auto kern = sparse_mla_simt<T, W>;
    cudaError_t e = ensure_dyn_smem((const void*)kern, (int)S::kTotal);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)n_split, (unsigned)b.n_q);
    e = launch_plain(kern, grid, dim3(kThreads), S::kTotal, st, b, sh.scale,
                     static_cast<const T*>(q_abs), static_cast<const T*>(cache), idx, n_sel,
                     sh.index_row_width(), rps, n_split, out, lse, part_o, part_ml, err);
    if (e != cudaSuccess || n_split == 1) return e;
    return launch_merge_splits(b.n_q, n_split, part_o, part_ml, out, lse, st);
}

}  // namespace

cudaError_t launch_merge_splits(int32_t n_q, int32_t n_split, const float* part_o,
                                const float* part_ml, float* out, float* lse, cudaStream_t st) {
    return launch_pdl(merge_splits, dim3(kHeads * 4, (unsigned)n_q), dim3(128), 0, st,
                      n_split, part_o, part_ml, out, lse);
}

void plan_attention_splits(const Shape& sh, const BatchDev& b, int32_t* rows_per_split,
                           int32_t* n_split) {
    const int32_t n_q = b.n_q > 0 ? b.n_q : 1;
    // rows a query attends over at most: its selection, or every visible row
    int64_t max_rows = b.max_kv_len, main_rows = max_rows;
    if (!(b.flags & DSA_FLAG_DENSE) && sh.index_row_width() < max_rows) {
        max_rows = sh.index_row_width();
        // the k-pool tail (fewer than kpool rows past the selected pools'
        // top_k rows) sizes no split: it spills into one more, short split
        main_rows = sh.top_k;
    }
    if (sparse_mla_tc_eligible(sh, b))
        plan_attention_splits_tc(n_q, main_rows, max_rows, rows_per_split, n_split);
    else
        plan_splits_simt(n_q, max_rows, rows_per_split, n_split);
}

size_t sparse_mla_scratch_bytes(const Shape& sh, const BatchDev& b) {
    int32_t rps, n_split;
    plan_attention_splits(sh, b, &rps, &n_split);
    if (n_split == 1) return 0;
    const size_t parts = (size_t)b.n_q * n_split * kHeads;
    return parts * kLatent * sizeof(float) + parts * 2 * sizeof(float);
}

cudaError_t launch_sparse_mla(const Shape& sh, const BatchDev& b, const void* q_abs,
                              const void* cache, const int32_t* idx, const int32_t* n_sel,
                              float* out, float* lse, void* scratch, size_t scratch_bytes,
                              int32_t* err, bool q_early, cudaStream_t st) {
    if (b.n_q == 0) return cudaSuccess;
    int32_t rps, n_split;
    plan_attention_splits(sh, b, &rps, &n_split);
    float* part_o = nullptr;
    float* part_ml = nullptr;
    if (n_split > 1) {
        const size_t parts = (size_t)b.n_q * n_split * kHeads;
        if (scratch == nullptr || scratch_bytes < parts * (kLatent + 2) * sizeof(float))
            return cudaErrorInvalidValue;
        part_o = static_cast<float*>(scratch);
        part_ml = part_o + parts * kLatent;
    }
    if (sparse_mla_tc_eligible(sh, b))
        return launch_sparse_mla_tc(sh, b, q_abs, cache, idx, n_sel, out, lse, part_o, part_ml,
                                    rps, n_split, err, q_early, st);
    const bool f32 = sh.dtype == DSA_F32;
    if (sh.width() == 576) {
        return f32 ? launch_typed<float, 576>(sh, b, q_abs, cache, idx, n_sel, out, lse, part_o,
                                              part_ml, rps, n_split, err, st)
                   : launch_typed<__nv_bfloat16, 576>(sh, b, q_abs, cache, idx, n_sel, out, lse,
                                                      part_o, part_ml, rps, n_split, err, st);
    }
    return f32 ? launch_typed<float, 512>(sh, b, q_abs, cache, idx, n_sel, out, lse, part_o,
                                          part_ml, rps, n_split, err, st)
               : launch_typed<__nv_bfloat16, 512>(sh, b, q_abs, cache, idx, n_sel, out, lse,
                                                  part_o, part_ml, rps, n_split, err, st);
}

}  // namespace dsa
