// index_prepare.cu -- indexer query / key preparation: rope, then the
// orthonormal Walsh-Hadamard rotation, rounded to the cache's dtype.
//
// "GLM-5.x (glm-dsa, glm5next)", "The sparse-attention path": past top-k the
// indexer applies rope and a Walsh-Hadamard rotation -- an orthonormal
// involution on both sides of the dot product, which cancels in exact
// arithmetic but spreads the rounding of the 16-bit key cache evenly over the
// 128 dimensions; "The block", row "RoPE": NORM mode (adjacent pairs), base 8e6.
//
// One warp per 128-vector, four dimensions per lane, a persistent grid: rope on
// the lane's two adjacent pairs, then the fast Walsh-Hadamard transform -- two
// butterfly stages inside the lane, five across lanes by shuffles -- and the
// 1/sqrt(128) scale.  HBM-bound streaming: a warp loads kUnroll vectors (and
// their positions) before it transforms the first, to keep enough bytes in
// flight.  Positions reach 10^6 radians, so the angle is formed in turns with
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
constexpr int kUnroll = 4;

// Turns per position of pair i: base^(-2i / rope_dims) / (2 pi) < 1, as a
// 64-bit binary fraction.
struct RopeRates {
    unsigned long long r[kDim / 2];
};

__device__ __forceinline__ void store4(float* p, const float (&e)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(e[0], e[1], e[2], e[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, const float (&e)[4]) {
    const __nv_bfloat162 a = __floats2bfloat162_rn(e[0], e[1]);
    const __nv_bfloat162 b = __floats2bfloat162_rn(e[2], e[3]);
    uint2 x;
    x.x = *reinterpret_cast<const uint32_t*>(&a);
    x.y = *reinterpret_cast<const uint32_t*>(&b);
    *reinterpret_cast<uint2*>(p) = x;
}

template <typename T>
__global__ void __launch_bounds__(32 * kWarpsPerCta)
index_prepare_kernel(int64_t n, const float* __restrict__ x, const int64_t* __restrict__ pos,
                     int32_t rope_dims, const __grid_constant__ RopeRates rates,
                     T* __restrict__ out) {
    // into shared memory: lanes read different entries, which the parameter
    // space would serve one address at a time
    __shared__ unsigned long long rate[kDim / 2];
    for (int i = threadIdx.x; i < kDim / 2; i += blockDim.x) rate[i] = rates.r[i];
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerCta;
    for (int64_t vb = (int64_t)blockIdx.x * kWarpsPerCta + warp; vb < n; vb += kUnroll * stride) {
        float4 xs[kUnroll];
        unsigned long long ps[kUnroll];
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const int64_t v = vb + r * stride;
            xs[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            ps[r] = 0;
            if (v < n) {
                xs[r] = __ldcs(reinterpret_cast<const float4*>(x + v * kDim) + lane);
                if (rope_dims > 0) ps[r] = (unsigned long long)pos[v];
            }
        }
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const int64_t v = vb + r * stride;
            if (v >= n) break;
            const float4 xv = xs[r];
            float e[4] = {xv.x, xv.y, xv.z, xv.w};
            // rope: pairs (4 lane, 4 lane + 1) and (4 lane + 2, 4 lane + 3)
            if (4 * lane < rope_dims) {
                const unsigned long long p = ps[r];
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int i = 2 * lane + k;
                    if (2 * i >= rope_dims) break;
                    // fractional turns of pos * theta_i / 2 pi (the product wraps
                    // modulo 2^64 = whole turns), as a signed fraction in [-1/2, 1/2)
                    const int t32 = (int)(unsigned int)((p * rate[i]) >> 32);
                    float s, c;
                    sincospif(2.0f * ((float)t32 * 2.3283064365386963e-10f), &s, &c);
                    const float x0 = e[2 * k], x1 = e[2 * k + 1];
                    e[2 * k] = x0 * c - x1 * s;
                    e[2 * k + 1] = x0 * s + x1 * c;
                }
            }
            // Walsh-Hadamard: dimension d = 4 lane + j; the butterfly of bit b maps
            // the pair (d, d | 2^b) with d's bit clear to (sum, difference)
            {
                const float a0 = e[0] + e[1], a1 = e[0] - e[1], a2 = e[2] + e[3], a3 = e[2] - e[3];
                e[0] = a0 + a2; e[2] = a0 - a2; e[1] = a1 + a3; e[3] = a1 - a3;
            }
#pragma unroll
            for (int m = 1; m < 32; m <<= 1) {
                const bool upper = (lane & m) != 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float o = __shfl_xor_sync(0xffffffffu, e[j], m);
                    e[j] = upper ? o - e[j] : e[j] + o;
                }
            }
            const float norm = 0.08838834764831845f;         // 1 / sqrt(128)
#pragma unroll
            for (int j = 0; j < 4; ++j) e[j] *= norm;
            store4(out + v * kDim + 4 * lane, e);
        }
    }
}

}  // namespace

cudaError_t launch_index_prepare(const Shape& sh, int64_t n_vec, const float* x,
                                 const int64_t* pos, int32_t rope_dims, double base, void* out,
                                 cudaStream_t st) {
    if (n_vec == 0) return cudaSuccess;
    // a persistent grid: enough CTAs to fill the GPU, each sets up its rope
    // rates once and walks vectors
    int64_t blocks = (n_vec + kWarpsPerCta - 1) / kWarpsPerCta;
    if (blocks > (int64_t)sm_count() * 8) blocks = (int64_t)sm_count() * 8;
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
