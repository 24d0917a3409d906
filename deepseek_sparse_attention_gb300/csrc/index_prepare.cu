// index_prepare.cu -- indexer query / key preparation: rope, then the
// orthonormal Walsh-Hadamard rotation, rounded to the cache's dtype.
//
// "GLM-5.x (glm-dsa, glm5next)", "The sparse-attention path": past top-k the
// indexer applies rope and a Walsh-Hadamard rotation -- an orthonormal
// involution on both sides of the dot product, which cancels in exact
// arithmetic but spreads the rounding of the 16-bit key cache evenly over the
// 128 dimensions; "The block", row "RoPE": NORM mode (adjacent pairs), base 8e6.
//
// Half a warp per 128-vector, eight dimensions per lane, a persistent grid:
// rope on the lane's four adjacent pairs, then the fast Walsh-Hadamard
// transform -- three butterfly stages inside the lane, four across the 16
// lanes by shuffles (eight independent ones per stage) -- and the 1/sqrt(128)
// scale.  HBM-bound streaming: a warp loads kUnroll vector pairs (and their
// positions) before it transforms the first, to keep enough bytes in flight.
// Positions reach 10^6 radians, so the angle is formed in turns with
// integers: each pair's rate theta_i / 2 pi as a 64-bit binary fraction
// (computed once, on the host, in double precision -- this GPU's double rate
// is too low to spend on it per CTA), times the position, wrapping -- the
// fractional turns exactly, with no double-precision work on the device.
#include <math.h>

#include "dsa_kernels.cuh"

namespace dsa {
namespace {

constexpr int kDim = 128;
constexpr int kWarpsPerCta = 8;
constexpr int kUnroll = 4;                 // vector pairs in flight per warp
constexpr int kCtasPerSm = 3;              // resident CTAs per SM (the register bound below)

// Turns per position of pair i: base^(-2i / rope_dims) / (2 pi) < 1, as a
// 64-bit binary fraction.
struct RopeRates {
    unsigned long long r[kDim / 2];
};

__device__ __forceinline__ void store8(float* p, const float (&e)[8]) {
    reinterpret_cast<float4*>(p)[0] = make_float4(e[0], e[1], e[2], e[3]);
    reinterpret_cast<float4*>(p)[1] = make_float4(e[4], e[5], e[6], e[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&e)[8]) {
    uint4 x;
    uint32_t* w = reinterpret_cast<uint32_t*>(&x);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 v = __floats2bfloat162_rn(e[2 * k], e[2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(p) = x;
}

template <typename T>
__global__ void __launch_bounds__(32 * kWarpsPerCta, kCtasPerSm)
index_prepare_kernel(int64_t n, const float* __restrict__ x, const int64_t* __restrict__ pos,
                     int32_t rope_dims, const __grid_constant__ RopeRates rates,
                     T* __restrict__ out) {
    // into shared memory: lanes read different entries, which the parameter
    // space would serve one address at a time
    __shared__ unsigned long long rate[kDim / 2];
    for (int i = threadIdx.x; i < kDim / 2; i += blockDim.x) rate[i] = rates.r[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane >> 4, hl = lane & 15;      // the pair's vector, the lane in it
    // a warp takes vectors vb + 2 r stride + {0, 1}
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerCta * 2;
    for (int64_t vb = ((int64_t)blockIdx.x * kWarpsPerCta + warp) * 2; vb < n;
         vb += kUnroll * stride) {
        float4 xa[kUnroll], xb[kUnroll];
        unsigned long long ps[kUnroll];
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const int64_t v = vb + r * stride + half;
            xa[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            xb[r] = xa[r];
            ps[r] = 0;
            if (v < n) {
                const float4* src = reinterpret_cast<const float4*>(x + v * kDim) + 2 * hl;
                xa[r] = __ldcs(src);
                xb[r] = __ldcs(src + 1);
                if (rope_dims > 0) ps[r] = (unsigned long long)pos[v];
            }
        }
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const int64_t v0 = vb + r * stride;
            if (v0 >= n) break;                          // both halves out of range
            const int64_t v = v0 + half;
            float e[8] = {xa[r].x, xa[r].y, xa[r].z, xa[r].w, xb[r].x, xb[r].y, xb[r].z, xb[r].w};
            // rope: pairs (8 hl + 2 k, 8 hl + 2 k + 1), k < 4
            if (8 * hl < rope_dims) {
                const unsigned long long p = ps[r];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = 4 * hl + k;
                    if (2 * i >= rope_dims) break;
                    // fractional turns of pos * theta_i / 2 pi (the product wraps
                    // modulo 2^64 = whole turns), as a signed fraction in [-1/2, 1/2),
                    // to radians in [-pi, pi): there the hardware sine and cosine
                    // are within 2^-21.4 absolute, far below the output's rounding
                    const int t32 = (int)(unsigned int)((p * rate[i]) >> 32);
                    float sn, cs;
                    __sincosf((float)t32 * 1.4629180792671596e-09f, &sn, &cs);   // 2 pi / 2^32
                    const float x0 = e[2 * k], x1 = e[2 * k + 1];
                    e[2 * k] = x0 * cs - x1 * sn;
                    e[2 * k + 1] = x0 * sn + x1 * cs;
                }
            }
            // Walsh-Hadamard: dimension d = 8 hl + j; the butterfly of bit b maps
            // the pair (d, d | 2^b) with d's bit clear to (sum, difference).
            // Bits 0..2 inside the lane:
#pragma unroll
            for (int m = 1; m < 8; m <<= 1) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j & m) continue;
                    const float a = e[j], c = e[j | m];
                    e[j] = a + c;
                    e[j | m] = a - c;
                }
            }
            // bits 3..6 across the vector's 16 lanes (xor < 16 stays in the half)
#pragma unroll
            for (int m = 1; m < 16; m <<= 1) {
                const bool upper = (hl & m) != 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float o = __shfl_xor_sync(0xffffffffu, e[j], m);
                    e[j] = upper ? o - e[j] : e[j] + o;
                }
            }
            const float norm = 0.08838834764831845f;         // 1 / sqrt(128)
#pragma unroll
            for (int j = 0; j < 8; ++j) e[j] *= norm;
            if (v < n) store8(out + v * kDim + 8 * hl, e);
        }
    }
}

}  // namespace

cudaError_t launch_index_prepare(const Shape& sh, int64_t n_vec, const float* x,
                                 const int64_t* pos, int32_t rope_dims, double base, void* out,
                                 cudaStream_t st) {
    if (n_vec == 0) return cudaSuccess;
    // a persistent grid: one wave of CTAs (kCtasPerSm resident on each SM),
    // each sets up its rope rates once and walks vectors, two per warp at a time
    int64_t blocks = (n_vec + 2 * kWarpsPerCta - 1) / (2 * kWarpsPerCta);
    if (blocks > (int64_t)sm_count() * kCtasPerSm) blocks = (int64_t)sm_count() * kCtasPerSm;
    // the 64-bit fraction of pos * theta_i / 2 pi per unit position: the
    // double rounded to the nearest integer multiple of 2^-64
    RopeRates rates{};
    for (int i = 0; i < rope_dims / 2; ++i)
        rates.r[i] = (unsigned long long)nearbyint(
            ldexp(pow(base, -2.0 * i / (double)rope_dims) / 6.283185307179586, 64));
    if (sh.dtype == DSA_BF16)
        return launch_plain(index_prepare_kernel<__nv_bfloat16>, dim3((unsigned)blocks),
                            dim3(32 * kWarpsPerCta), 0, st, n_vec, x, pos, rope_dims, rates,
                            static_cast<__nv_bfloat16*>(out));
    else
        return launch_plain(index_prepare_kernel<float>, dim3((unsigned)blocks),
                            dim3(32 * kWarpsPerCta), 0, st, n_vec, x, pos, rope_dims, rates,
                            static_cast<float*>(out));
}

}  // namespace dsa
