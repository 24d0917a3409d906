// proj.cu -- the two projections around the absorbed attention: query
// absorption and the output up-projection.
//
// "GLM-5.x (glm-dsa, glm5next)", "The block": the per-head key and value
// decompressions of MLA are folded into the query (attn_k_b) and into the
// output (attn_v_b); "GLM 5.2 in one C file", "Attention: Multi head Latent
// Attention With a Tiny KV Cache": the key up-projection is absorbed into the
// query, which then scores the cached latents directly, and the pooled latent
// is projected to the head's value space once, at the end.
//
//   absorb  q_abs[q,h,i] = sum_{d < nope} q[q,h,d] * w_uk[h,d,i]   (i < kv_lora)
//           q_abs[q,h,kv_lora + r] = q[q,h,nope + r]               (the rope part)
//   up      out[q,h,v]   = sum_{i < kv_lora} w_uv[h,v,i] * o[q,h,i]
//
// Per head both are a weight matrix times the queries' vectors.  On the
// tensor cores the weights are M (128 output features per tile) and the
// queries N (up to 256 per tile, a decode batch padded to 16): the weights --
// 12.6 MB for absorb, 16.8 MB for up at 64 heads -- stream once per query
// tile, which for decode is once.  One CTA per (head, 128-feature block, query
// tile); K in blocks of 64 (one 128-byte swizzle row) through a ring of
// shared-memory stages:
//   warp 0     TMA: the weight block -- absorb: w_uk rows d (K) of 64 features
//              each (MN-major A, two boxes for 128 features); up: w_uv rows v
//              (K-major A) -- and, for absorb, the queries' k-block (a 3-D box
//              of 64 dims x 1 head x N queries, K-major B);
//   warps 2-7  (up) the attention output o is float32: each k-block is split
//              into bf16 hi and lo = o - hi, written in the 128-byte swizzle
//              layout; both are multiplied into the one accumulator, carrying
//              o to about 2^-16 relative (bf16 alone: 2^-9);
//   warp 1     one thread issues the MMAs into a TMEM accumulator [128 x N];
//   warps 4-7  epilogue, one TMEM lane (output feature) per thread: the N query
//              columns read back and stored (absorb: rounded to bf16); warps
//              2-3 of absorb copy the rope part.
// Float32 inputs take a CUDA-core kernel.  All waits are bounded: a timeout
// records the error word and the CTA winds down.
#include "dsa_kernels.cuh"
#include "sm100.cuh"

namespace dsa {
namespace {

using namespace sm100;

constexpr int kThreads = 384;
constexpr int kM = 128;                      // output features per tile (MMA M)
constexpr uint32_t kABytes = kM * 128;       // one k-block of weights: 16 KB
constexpr int kConv = 320;                   // up: threads splitting o (warps 2-11)
constexpr int kMaxStages = 8;
constexpr int kMaxN = 256;
constexpr int kConvIters = (kMaxN * 8 + kConv - 1) / kConv;   // 16-byte chunks per thread
constexpr int kSmallKb = 8;                  // k-blocks held at once for a small query tile
constexpr uint32_t kSmemBudget = 200u * 1024u;
constexpr uint64_t kWaitNs = 2000000000ull;

// Shared memory per stage: the weight k-block, then the queries' k-block
// (up: its hi and lo parts).
__host__ __device__ constexpr uint32_t stage_bytes(int mode, int n) {
    return kABytes + (uint32_t)n * 128u * (mode == 0 ? 1u : 2u);
}

__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1)
proj_tc(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_q,
        const __nv_bfloat16* __restrict__ q_src, const float* __restrict__ o, void* __restrict__ out,
        int32_t n_q, int32_t heads, int32_t N, int32_t n_mblk, int32_t nope, int32_t rope,
        int32_t kv_lora, int32_t v_dim, int32_t stages, int32_t* err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sbytes = stage_bytes(MODE, N);
    // barriers after the stages, or after the output staging if that is larger
    uint32_t pipe = (uint32_t)stages * sbytes;
    if (pipe < (uint32_t)N * kM * (MODE == 0 ? 2u : 4u)) pipe = (uint32_t)N * kM * (MODE == 0 ? 2u : 4u);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pipe);
    uint64_t* full = bars;
    uint64_t* empty = bars + kMaxStages;
    uint64_t* acc_full = bars + 2 * kMaxStages;
    uint64_t* drain = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kMaxStages + 2);
    volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x / n_mblk, mb = blockIdx.x % n_mblk;
    const int64_t q0 = (int64_t)blockIdx.y * N;
    const int n_kb = (MODE == 0 ? nope : kv_lora) / 64;
    uint32_t tmem_cols = 32;
    while (tmem_cols < (uint32_t)N) tmem_cols <<= 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            mbar_init(&full[s], MODE == 0 ? 1 : 1 + kConv);
            mbar_init(&empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, tmem_cols);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        prefetch_tensormap(&tm_w);
        if (MODE == 0) prefetch_tensormap(&tm_q);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the inputs may come from the previous kernel in the stream
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        if (lane == 0) {                                           // ---- TMA producer
            int8_t issued_par[kMaxStages];
            for (int s = 0; s < kMaxStages; ++s) issued_par[s] = -1;
            bool ok = true;
            for (int kb = 0; kb < n_kb && ok; ++kb) {
                const int s = kb % stages;
                const uint32_t ph = (uint32_t)(kb / stages) & 1u;
                if (*abort_flag) { ok = false; break; }
                ok = mbar_wait(&empty[s], ph ^ 1u, kWaitNs);
                if (!ok) break;
                uint8_t* st = smem + s * sbytes;
                mbar_arrive_expect_tx(&full[s], kABytes + (MODE == 0 ? (uint32_t)N * 128u : 0u));
                if (MODE == 0) {
                    const int32_t y = h * nope + kb * 64;
                    tma_load_2d(st, &tm_w, &full[s], mb * kM, y);
                    tma_load_2d(st + kABytes / 2, &tm_w, &full[s], mb * kM + 64, y);
                    tma_load_3d(st + kABytes, &tm_q, &full[s], kb * 64, h, (int32_t)q0);
                } else {
                    tma_load_2d(st, &tm_w, &full[s], kb * 64, h * v_dim + mb * kM);
                }
                issued_par[s] = (int8_t)ph;
            }
            if (!ok) {
                record_error(err, kDevTimeout, blockIdx.x, /*where=*/30);
                *abort_flag = 1;
                for (int s = 0; s < kMaxStages; ++s)       // copies in flight land first
                    if (issued_par[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_par[s], 50000000ull);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {                                           // ---- MMA issuer
            const uint32_t idesc = MODE == 0 ? idesc_bf16_f32_major(kM, N, 1, 0)
                                             : idesc_bf16_f32(kM, N);
            bool ok = true;
            for (int kb = 0; kb < n_kb; ++kb) {
                const int s = kb % stages;
                const uint32_t ph = (uint32_t)(kb / stages) & 1u;
                if (*abort_flag || !mbar_wait(&full[s], ph, kWaitNs)) { ok = false; break; }
                tc_fence_after();
                const uint32_t a = smem_u32(smem + s * sbytes);
                const uint32_t b = a + kABytes;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    if (MODE == 0) {
                        // A: [64 rows d][64 features] blocks, the two feature
                        // halves 8 KB apart (LBO), 8-row groups 1 KB apart (SBO)
                        mma_bf16_ss(tmem_base, sdesc_sw128(a + kk * 2048, kABytes / 2, 1024),
                                    sdesc_kmajor_sw128(b + kk * 32), idesc, (kb | kk) != 0);
                    } else {
                        const uint64_t ad = sdesc_kmajor_sw128(a + kk * 32);
                        mma_bf16_ss(tmem_base, ad, sdesc_kmajor_sw128(b + kk * 32), idesc,
                                    (kb | kk) != 0);
                        mma_bf16_ss(tmem_base, ad, sdesc_kmajor_sw128(b + N * 128 + kk * 32),
                                    idesc, 1u);
                    }
                }
                mma_commit(&empty[s]);
            }
            if (!ok) {
                record_error(err, kDevTimeout, blockIdx.x, /*where=*/31);
                *abort_flag = 1;
            } else {
                mma_commit(acc_full);
            }
            mma_commit(drain);                                     // every issued MMA retired
            mbar_wait(drain, 0, 50000000ull);
        }
    } else if (MODE == 1) {                                        // ---- o -> bf16 hi, lo
        const int tc = threadIdx.x - 64;                           // 0 .. kConv-1
        // One 16-byte chunk c of a k-block: query row c / 8, dims 8 (c % 8) .. + 7,
        // split into bf16 hi and lo in the k-block's stage.
        auto convert = [&](int kb, int c, const float4& a, const float4& bq) {
            uint8_t* hi = smem + (kb % stages) * sbytes + kABytes;
            uint8_t* lo = hi + N * 128;
            const int n = c >> 3, k8 = c & 7;
            const float f[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
            uint32_t vh[4], vl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 hv = __floats2bfloat162_rn(f[2 * e], f[2 * e + 1]);
                const float2 hf = __bfloat1622float2(hv);
                vh[e] = *reinterpret_cast<const uint32_t*>(&hv);
                vl[e] = bf16x2_bits(f[2 * e] - hf.x, f[2 * e + 1] - hf.y);
            }
            const uint32_t off = (uint32_t)n * 128u + ((uint32_t)(k8 ^ (n & 7)) << 4);
            *reinterpret_cast<uint4*>(hi + off) = make_uint4(vh[0], vh[1], vh[2], vh[3]);
            *reinterpret_cast<uint4*>(lo + off) = make_uint4(vl[0], vl[1], vl[2], vl[3]);
        };
        auto chunk_src = [&](int kb, int c) {
            const int64_t q = q0 + (c >> 3);
            return reinterpret_cast<const float4*>(o + (q * heads + h) * (int64_t)kv_lora +
                                                   kb * 64 + (c & 7) * 8);
        };
        if (N * 8 <= kConv && n_kb <= kSmallKb) {
            // A small query tile (a decode batch): at most one chunk of each
            // k-block per thread, and the loads of every k-block in flight at
            // once -- not one k-block's round trip after another.
            const bool has = tc < N * 8 && q0 + (tc >> 3) < n_q;
            float4 xa[kSmallKb], xb[kSmallKb];
#pragma unroll
            for (int kb = 0; kb < kSmallKb; ++kb) {
                xa[kb] = xb[kb] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (kb < n_kb && has) {
                    const float4* src = chunk_src(kb, tc);
                    xa[kb] = __ldg(src);
                    xb[kb] = __ldg(src + 1);
                }
            }
#pragma unroll
            for (int kb = 0; kb < kSmallKb; ++kb) {
                if (kb >= n_kb) break;
                const int s = kb % stages;
                const uint32_t ph = (uint32_t)(kb / stages) & 1u;
                if (*abort_flag || !mbar_wait(&empty[s], ph ^ 1u, kWaitNs)) {
                    record_error(err, kDevTimeout, blockIdx.x, /*where=*/32);
                    *abort_flag = 1;
                    break;
                }
                if (tc < N * 8) convert(kb, tc, xa[kb], xb[kb]);
                fence_proxy_async_smem();                          // generic writes -> MMA reads
                mbar_arrive(&full[s]);
            }
        } else {
            // This thread's chunks of a k-block: c = tc + j kConv; every load of
            // the k-block is issued before the first conversion.
            for (int kb = 0; kb < n_kb; ++kb) {
                const int s = kb % stages;
                const uint32_t ph = (uint32_t)(kb / stages) & 1u;
                float4 xa[kConvIters], xb[kConvIters];
#pragma unroll
                for (int j = 0; j < kConvIters; ++j) {
                    const int c = tc + j * kConv;
                    xa[j] = xb[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (c < N * 8 && q0 + (c >> 3) < n_q) {
                        const float4* src = chunk_src(kb, c);
                        xa[j] = __ldg(src);
                        xb[j] = __ldg(src + 1);
                    }
                }
                if (*abort_flag || !mbar_wait(&empty[s], ph ^ 1u, kWaitNs)) {
                    record_error(err, kDevTimeout, blockIdx.x, /*where=*/32);
                    *abort_flag = 1;
                    break;
                }
#pragma unroll
                for (int j = 0; j < kConvIters; ++j) {
                    const int c = tc + j * kConv;
                    if (c < N * 8) convert(kb, c, xa[j], xb[j]);
                }
                fence_proxy_async_smem();                          // generic writes -> MMA reads
                mbar_arrive(&full[s]);
            }
        }
    } else if (warp < 4 && mb == 0 && rope > 0) {                  // ---- absorb: the rope part
        // 16-byte chunks: thread t copies chunk t % 8 of queries t / 8 + 8 i,
        // eight loads in flight before their stores
        const int t = threadIdx.x - 64;                            // 0..63
        const int W = kv_lora + rope, Q = nope + rope;
        const int per_row = rope / 8, rows_per_pass = 64 / per_row;
        const int k8 = t % per_row;
        __nv_bfloat16* qa = static_cast<__nv_bfloat16*>(out);
        for (int n0 = t / per_row; n0 < N; n0 += 8 * rows_per_pass) {
            uint4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t q = q0 + n0 + i * rows_per_pass;
                v[i] = make_uint4(0, 0, 0, 0);
                if (n0 + i * rows_per_pass < N && q < n_q)
                    v[i] = __ldg(reinterpret_cast<const uint4*>(q_src + (q * heads + h) * Q + nope) + k8);
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t q = q0 + n0 + i * rows_per_pass;
                if (n0 + i * rows_per_pass < N && q < n_q)
                    reinterpret_cast<uint4*>(qa + (q * heads + h) * W + kv_lora)[k8] = v[i];
            }
        }
    }

    if (warp >= 4 && warp < 8) {                                   // ---- epilogue
        // the four warps agree on whether the accumulator is ready (every one
        // reaches this reduction), so all or none of them take the barrier below
        const uint32_t mine = (!*abort_flag && mbar_wait(acc_full, 0, kWaitNs)) ? 1u : 0u;
        uint32_t all;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
            "bar.red.and.pred q, 2, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(all)
            : "r"(mine)
            : "memory");
        const bool ok = all != 0;
        if (!ok) {
            if (lane == 0) record_error(err, kDevTimeout, blockIdx.x, /*where=*/33);
        } else {
            tc_fence_after();
            // The tile [N queries][128 features] (bf16 for absorb, float32 for
            // up) is staged in the stage memory, free once every MMA is done,
            // then written in 16-byte pieces: each (query, head) owns 128
            // consecutive features of the output row.
            const int m = (warp - 4) * 32 + lane;                  // TMEM lane = output feature
            const uint32_t lane_addr = tmem_base + ((uint32_t)((warp - 4) * 32) << 16);
            constexpr int kEsz = MODE == 0 ? 2 : 4;
            uint8_t* stg = smem;
            for (int c0 = 0; c0 < N; c0 += 32) {
                float v[32];
                if (N - c0 >= 32) {
                    tmem_ld_32cols(lane_addr + c0, v);
                } else {
                    float v16[16];
                    tmem_ld_16cols(lane_addr + c0, v16);
#pragma unroll
                    for (int e = 0; e < 16; ++e) { v[e] = v16[e]; v[e + 16] = 0.f; }
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int n = c0 + e;
                    if (n >= N) continue;
                    if (MODE == 0)
                        reinterpret_cast<__nv_bfloat16*>(stg)[n * kM + m] = __float2bfloat16_rn(v[e]);
                    else
                        reinterpret_cast<float*>(stg)[n * kM + m] = v[e];
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");         // the four epilogue warps
            constexpr int kChunks = kM * kEsz / 16;                 // 16-byte pieces per row
            const int t = threadIdx.x - 128;
            const int64_t w_out = MODE == 0 ? (int64_t)(kv_lora + rope) : (int64_t)v_dim;
            uint8_t* dst0 = static_cast<uint8_t*>(out) + (int64_t)mb * kM * kEsz;
            for (int ch = t; ch < N * kChunks; ch += 128) {
                const int n = ch / kChunks, c = ch % kChunks;
                const int64_t q = q0 + n;
                if (q >= n_q) continue;
                *reinterpret_cast<uint4*>(dst0 + ((q * heads + h) * w_out) * kEsz + c * 16) =
                    *reinterpret_cast<const uint4*>(stg + (n * kM) * kEsz + c * 16);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tmem_cols);
    }
}

// Float32 inputs.  Absorb: a CTA per (query, head, 64 output columns); its
// 256 threads are the 64 columns times four interleaved quarters of the sum
// over the nope dimensions, added in shared memory.  Up: a CTA per (query,
// head, 32 outputs), a warp per output, the lanes' strided partial sums
// added by shuffles.  Enough CTAs for one decode query to keep every SM's
// loads in flight.  Float32 accumulation throughout.
constexpr int kSimtAbsorbCols = 64;
constexpr int kSimtUpRows = 32;

__global__ void __launch_bounds__(256)
absorb_simt(const float* __restrict__ q, const float* __restrict__ w_uk, float* __restrict__ q_abs,
            int32_t heads, int32_t nope, int32_t rope, int32_t kv_lora) {
    __shared__ float part[4][kSimtAbsorbCols];
    const int64_t qh = blockIdx.x;                     // (query, head)
    const int h = (int)(qh % heads);
    const int c = threadIdx.x % kSimtAbsorbCols, quarter = threadIdx.x / kSimtAbsorbCols;
    const int i = (int)blockIdx.y * kSimtAbsorbCols + c;
    const float* qv = q + qh * (nope + rope);
    float* dst = q_abs + qh * (kv_lora + rope);
    float acc = 0.f;
    if (i < kv_lora) {
#pragma unroll 8
        for (int d = quarter; d < nope; d += 4)
            acc = fmaf(qv[d], w_uk[((int64_t)h * nope + d) * kv_lora + i], acc);
    }
    part[quarter][c] = acc;
    __syncthreads();
    if (quarter == 0 && i < kv_lora) dst[i] = (part[0][c] + part[1][c]) + (part[2][c] + part[3][c]);
    if (blockIdx.y == 0)
        for (int r = threadIdx.x; r < rope; r += blockDim.x) dst[kv_lora + r] = qv[nope + r];
}

__global__ void __launch_bounds__(256)
up_simt(const float* __restrict__ o, const float* __restrict__ w_uv, float* __restrict__ out,
        int32_t heads, int32_t kv_lora, int32_t v_dim) {
    const int64_t qh = blockIdx.x;
    const int h = (int)(qh % heads);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float* ov = o + qh * kv_lora;
    const int v0 = (int)blockIdx.y * kSimtUpRows;
    const int v1 = v0 + kSimtUpRows < v_dim ? v0 + kSimtUpRows : v_dim;
    for (int v = v0 + warp; v < v1; v += blockDim.x >> 5) {
        const float* wr = w_uv + ((int64_t)h * v_dim + v) * kv_lora;
        float acc = 0.f;
#pragma unroll 8
        for (int i = lane; i < kv_lora; i += 32) acc = fmaf(wr[i], ov[i], acc);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) out[qh * v_dim + v] = acc;
    }
}

int query_tile(int32_t n_q) {
    int n = (n_q + 15) / 16 * 16;
    return n > 256 ? 256 : (n < 16 ? 16 : n);
}

template <int MODE>
cudaError_t launch_tc(const Shape& sh, int32_t n_q, int32_t nope, int32_t v_dim, const void* q,
                      const void* w, const float* o, void* out, int32_t* err, cudaStream_t st) {
    const int N = query_tile(n_q);
    // as many stages as k-blocks when they fit (a decode batch has every
    // k-block in flight at once), else as many as fit
    const int n_kb = (MODE == 0 ? nope : sh.kv_lora) / 64;
    int stages = (int)(kSmemBudget / stage_bytes(MODE, N));
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages > n_kb) stages = n_kb;
    if (stages < 1) return cudaErrorInvalidConfiguration;
    CUtensorMap tm_w, tm_q;
    if (MODE == 0) {
        const uint64_t wd[2] = {(uint64_t)sh.kv_lora, (uint64_t)sh.heads * nope};
        const uint64_t ws[1] = {(uint64_t)sh.kv_lora * 2};
        const uint32_t wb[2] = {64, 64};
        const int Q = nope + sh.rope;
        const uint64_t qd[3] = {(uint64_t)Q, (uint64_t)sh.heads, (uint64_t)n_q};
        const uint64_t qs[2] = {(uint64_t)Q * 2, (uint64_t)sh.heads * Q * 2};
        const uint32_t qb[3] = {64, 1, (uint32_t)N};
        if (!encode_bf16_map(&tm_w, w, 2, wd, ws, wb) || !encode_bf16_map(&tm_q, q, 3, qd, qs, qb))
            return cudaErrorInvalidValue;
    } else {
        const uint64_t wd[2] = {(uint64_t)sh.kv_lora, (uint64_t)sh.heads * v_dim};
        const uint64_t ws[1] = {(uint64_t)sh.kv_lora * 2};
        const uint32_t wb[2] = {64, (uint32_t)kM};
        if (!encode_bf16_map(&tm_w, w, 2, wd, ws, wb)) return cudaErrorInvalidValue;
        tm_q = tm_w;                                   // unused
    }
    const int n_mblk = (MODE == 0 ? sh.kv_lora : v_dim) / kM;
    // the pipeline's stages, which the epilogue then reuses to stage the output
    size_t pipe = (size_t)stages * stage_bytes(MODE, N);
    const size_t staged = (size_t)N * kM * (MODE == 0 ? 2 : 4);
    if (pipe < staged) pipe = staged;
    const size_t smem = pipe + (2 * kMaxStages + 4) * 8 + 1024;
    auto kern = proj_tc<MODE>;
    cudaError_t e = ensure_dyn_smem((const void*)kern, (int)smem);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(n_mblk * sh.heads), (unsigned)((n_q + N - 1) / N));
    return launch_pdl(kern, grid, dim3(kThreads), smem, st, tm_w, tm_q,
                      static_cast<const __nv_bfloat16*>(q), o, out, n_q, (int32_t)sh.heads,
                      (int32_t)N, (int32_t)n_mblk, nope, (int32_t)sh.rope, (int32_t)sh.kv_lora,
                      v_dim, (int32_t)stages, err);
}

}  // namespace

cudaError_t launch_absorb_q(const Shape& sh, int32_t n_q, int32_t nope, const void* q,
                            const void* w_uk, void* q_abs, int32_t* err, cudaStream_t st) {
    if (n_q == 0) return cudaSuccess;
    if (sh.dtype == DSA_BF16)
        return launch_tc<0>(sh, n_q, nope, 0, q, w_uk, nullptr, q_abs, err, st);
    const dim3 grid((unsigned)((int64_t)n_q * sh.heads),
                    (unsigned)((sh.kv_lora + kSimtAbsorbCols - 1) / kSimtAbsorbCols));
    return launch_plain(absorb_simt, grid, dim3(256), 0, st,
                        static_cast<const float*>(q), static_cast<const float*>(w_uk),
                        static_cast<float*>(q_abs), (int32_t)sh.heads, nope, (int32_t)sh.rope,
                        (int32_t)sh.kv_lora);
}

cudaError_t launch_up_project(const Shape& sh, int32_t n_q, int32_t v_dim, const float* o,
                              const void* w_uv, float* out, int32_t* err, cudaStream_t st) {
    if (n_q == 0) return cudaSuccess;
    if (sh.dtype == DSA_BF16)
        return launch_tc<1>(sh, n_q, 0, v_dim, nullptr, w_uv, o, out, err, st);
    const dim3 grid((unsigned)((int64_t)n_q * sh.heads), (unsigned)((v_dim + kSimtUpRows - 1) / kSimtUpRows));
    return launch_plain(up_simt, grid, dim3(256), 0, st, o,
                        static_cast<const float*>(w_uv), out, (int32_t)sh.heads,
                        (int32_t)sh.kv_lora, v_dim);
}

}  // namespace dsa
