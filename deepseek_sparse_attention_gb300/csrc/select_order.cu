// select_order.cu -- selections in descending score order.
//
// The selection kernels emit a query's selected rows in ascending row order.
// "Add GLM-5.3-Flash support" (DSA verification) treats the order of a
// selection list as a separate promise from its set: a list in descending
// score order.  This kernel reorders each row by (score descending, index
// ascending) -- ties to the lower index, the tie rule of the selection itself
// ("Add GLM-5.3-Flash support", the router: ties by ascending index).  In
// k-pool mode ("GLM-5.3-Flash on WASTE", "DeepSeek Sparse Attention, k-pool
// flavour") the unit is a pool: the pools are ordered by their scores, each
// pool's kpool rows stay together in ascending order, and the rows of the
// unfilled tail, which have no score of their own, come last in ascending
// order.  A dense selection (every visible row) is ordered the same way.
//
// One CTA per query: the selection's units as 64-bit keys
//     (order_key(score) << 32) | ~unit
// in shared memory, padded with zeros to a power of two (every real key is
// larger: order_key of a finite score is at least 2^23), a bitonic sort into
// descending order, then the rows written back in place.
#include "dsa_kernels.cuh"
#include "sm100.cuh"

namespace dsa {
namespace {

using namespace sm100;

constexpr int kThreads = 1024;
constexpr int kMaxUnits = 16384;                   // 128 KB of keys

__global__ void __launch_bounds__(kThreads)
select_order_desc(BatchDev b, int32_t kpool, const float* __restrict__ scores, int64_t ld,
                  int32_t* __restrict__ idx, const int32_t* __restrict__ n_sel, int64_t width,
                  int32_t max_units, int32_t* err) {
    extern __shared__ unsigned long long keys[];
    // the selection and the scores come from the previous kernels; release the
    // next kernel only after they are complete
    pdl_wait();
    pdl_trigger();
    const int64_t q = blockIdx.x;
    QueryInfo qi;
    if (!query_info(b, q, qi, err, /*where=*/12)) return;
    int64_t ns = n_sel[q];
    ns = ns < 0 ? 0 : (ns > width ? width : ns);
    // the unfilled tail (k-pool mode) is the last L mod kpool rows of the row
    const int64_t tail = kpool > 1 ? qi.L % kpool : 0;
    const int64_t n_units = ns >= tail ? (ns - tail) / kpool : 0;
    if (n_units > max_units) {                       // the shared memory holds max_units
        record_error(err, kDevBadBatch, (int32_t)q, /*where=*/12);
        return;
    }
    int n_pow = 1;
    while (n_pow < n_units) n_pow <<= 1;
    int32_t* row = idx + q * width;
    const float* sc = scores + q * ld;
    for (int64_t i = threadIdx.x; i < n_pow; i += kThreads) {
        unsigned long long k = 0;
        if (i < n_units) {
            const int32_t r = row[i * kpool];           // the unit's first row
            const int64_t unit = kpool > 1 ? r / kpool : r;
            if (r < 0 || unit >= qi.n_keys) {
                record_error(err, kDevBadIndex, (int32_t)q, /*where=*/12);
            } else {
                k = ((unsigned long long)order_key(sc[unit]) << 32) |
                    (unsigned long long)(~(uint32_t)unit);
            }
        }
        keys[i] = k;
    }
    __syncthreads();
    for (int k = 2; k <= n_pow; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n_pow; i += kThreads) {
                const int p = i ^ j;
                if (p > i) {
                    const unsigned long long a = keys[i], c = keys[p];
                    // descending within blocks whose k bit is clear, ascending
                    // in the others: the last merge leaves the whole list descending
                    const bool desc = (i & k) == 0;
                    if (desc ? a < c : a > c) {
                        keys[i] = c;
                        keys[p] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int64_t e = threadIdx.x; e < n_units * kpool; e += kThreads) {
        const int64_t i = e / kpool;
        const uint32_t unit = ~(uint32_t)(keys[i] & 0xffffffffull);
        row[e] = (int32_t)((int64_t)unit * kpool + e % kpool);
    }
}

}  // namespace

cudaError_t launch_select_order_desc(const Shape& sh, const BatchDev& b, const float* scores,
                                     int64_t ld, int32_t* idx, const int32_t* n_sel, int32_t* err,
                                     cudaStream_t st) {
    if (b.n_q == 0) return cudaSuccess;
    int64_t units = sh.top_k / sh.kpool;              // a sparse selection's units
    const int64_t dense_units = sh.index_row_width() / sh.kpool;
    if (dense_units > units) units = dense_units;      // a dense one's
    if (units > kMaxUnits) return cudaErrorInvalidValue;
    int n_pow = 1;
    while (n_pow < units) n_pow <<= 1;
    const size_t smem = (size_t)n_pow * sizeof(unsigned long long);
    cudaError_t e = ensure_dyn_smem((const void*)select_order_desc, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(select_order_desc, dim3((unsigned)b.n_q), dim3(kThreads), smem, st, b,
                      sh.kpool, scores, ld, idx, n_sel, sh.index_row_width(), n_pow, err);
}

}  // namespace dsa
