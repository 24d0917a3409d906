// dsa_noalloc.cu -- dsa_decode_step_noalloc: the whole hot path without a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// Who needs it: code that may not call cudaMalloc at the point where it runs
// the layer -- for example while a framework is capturing the stream into a
// CUDA graph (allocation is not allowed during capture), inside a host engine
// that hands a plugin only its input and output buffers and no allocator, or in
// a latency-critical loop where cudaMalloc's implicit device synchronisation
// would stall other work.  Such callers pass inputs and outputs only; the
// scratch the step needs (scores, selections, attention partials, the device
// error word) lives in one fixed array compiled into this library.
//
// The array is a file-scope __device__ variable of DSA_NOALLOC_SCRATCH_BYTES
// bytes: every GPU that loads libdsa holds it until the process exits.  Host
// code cannot use the variable's name as a device address, so the first call
// on each device looks the address up with cudaGetSymbolAddress (with that
// device current) and caches it; that first call should therefore come before
// any stream capture.  All calls share the array and it keeps the previous
// call's contents: each call clears the part that must start at zero (the error
// word, the grid barrier and the fused selection histograms) on its stream,
// and two calls whose work overlaps on the GPU -- on different streams, or
// different host threads -- race on the array.  The error word a call's kernels
// record is read (and cleared) by dsa_check_device_error with a NULL workspace.
#include <mutex>

#include "dsa.h"
#include "dsa_kernels.cuh"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_ptr[kMaxDevices] = {};

}  // namespace

namespace dsa {

// Device address of the scratch array on the current device (set up once).
dsa_status noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return DSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
            return DSA_ERR_CUDA;
        g_ptr[dev] = p;
    }
    *out = g_ptr[dev];
    return DSA_OK;
}

}  // namespace dsa

extern "C" dsa_status dsa_decode_step_noalloc(const dsa_shape* shape, const dsa_batch* batch,
                                              const void* q_idx, const float* w,
                                              const void* k_idx, const void* q_abs,
                                              const void* cache, float* out, float* lse,
                                              int32_t* idx_out, int32_t* n_sel_out,
                                              void* stream) {
    // every argument is checked before anything is enqueued
    size_t need = 0;
    int32_t n_q = 0;
    dsa_status s = dsa::decode_step_check(shape, batch, q_idx, w, k_idx, q_abs, cache, out, lse,
                                          idx_out, n_sel_out, &need, &n_q);
    if (s != DSA_OK) return s;
    if (need > (size_t)DSA_NOALLOC_SCRATCH_BYTES) return DSA_ERR_UNSUPPORTED;
    if (n_q == 0) return DSA_OK;
    void* scratch = nullptr;
    if ((s = dsa::noalloc_scratch(&scratch)) != DSA_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, dsa::ws_zero_bytes(), st) != cudaSuccess) return DSA_ERR_CUDA;
    return dsa_decode_step(shape, batch, q_idx, w, k_idx, q_abs, cache, out, lse, idx_out,
                           n_sel_out, scratch, (size_t)DSA_NOALLOC_SCRATCH_BYTES, stream);
}
