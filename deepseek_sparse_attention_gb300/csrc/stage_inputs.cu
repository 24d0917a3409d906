// stage_inputs.cu -- the per-query inputs of a host-fed decode step moved into
// the workspace by a kernel (dsa_decode_step_host).
//
// The step's query-side inputs (indexer queries, head weights, absorbed
// queries) arrive in page-locked host memory each step.  A copy-engine copy
// breaks the chain of programmatically dependent launches that the step's
// kernels form (each side waits for the other to drain); this kernel is a
// link of that chain instead: its threads load 16-byte vectors of the two
// large inputs straight from host memory over the chip-to-chip link, several
// in flight per thread, and store them into the workspace, where the step's
// kernels read them as usual.  The head weights, whose size need not be a
// multiple of 16 bytes, move as 4-byte words in CTAs of their own.
//
// The sources are the caller's and the kernel before this one may write them:
// every load follows the wait for that kernel.  The dependents are released
// at once, so that the next kernel's CTAs are resident and through their
// set-up when the copy ends (they wait for its completion before reading).
#include "dsa_kernels.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;
constexpr int kVecs = 4;          // 16-byte vectors in flight per thread

__global__ void __launch_bounds__(kThreads)
stage_inputs(StageSeg a, StageSeg b, const uint32_t* __restrict__ w_src,
             uint32_t* __restrict__ w_dst, int64_t w_n, int32_t vec_ctas) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if ((int32_t)blockIdx.x >= vec_ctas) {                  // the head weights
        const int64_t stride = (int64_t)(gridDim.x - vec_ctas) * kThreads;
        for (int64_t i = (int64_t)(blockIdx.x - vec_ctas) * kThreads + threadIdx.x; i < w_n;
             i += stride)
            w_dst[i] = __ldg(w_src + i);
        return;
    }
    // vectors of a, then of b, as one index space
    const int64_t n = a.n + b.n;
    const int64_t stride = (int64_t)vec_ctas * kThreads;
    for (int64_t base = (int64_t)blockIdx.x * kThreads + threadIdx.x; base < n;
         base += stride * kVecs) {
        uint4 v[kVecs];
#pragma unroll
        for (int k = 0; k < kVecs; ++k) {
            const int64_t i = base + k * stride;
            if (i < n) v[k] = __ldg(i < a.n ? a.src + i : b.src + (i - a.n));
        }
#pragma unroll
        for (int k = 0; k < kVecs; ++k) {
            const int64_t i = base + k * stride;
            if (i < n) *(i < a.n ? a.dst + i : b.dst + (i - a.n)) = v[k];
        }
    }
}

}  // namespace

cudaError_t launch_stage_inputs(StageSeg a, StageSeg b, const uint32_t* w_src, uint32_t* w_dst,
                                int64_t w_n, cudaStream_t st) {
    const int64_t n = a.n + b.n;
    if (n == 0 && w_n == 0) return cudaSuccess;
    const int64_t cap = 4 * (int64_t)sm_count();
    int64_t vec_ctas = (n + (int64_t)kThreads * kVecs - 1) / ((int64_t)kThreads * kVecs);
    if (vec_ctas > cap) vec_ctas = cap;
    int64_t w_ctas = (w_n + kThreads - 1) / kThreads;
    if (w_ctas > cap) w_ctas = cap;
    return launch_pdl(stage_inputs, dim3((unsigned)(vec_ctas + w_ctas)), dim3(kThreads), 0, st, a,
                      b, w_src, w_dst, w_n, (int32_t)vec_ctas);
}

}  // namespace dsa
