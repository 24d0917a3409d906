// dsa_common.cuh -- device helpers shared by the DSA kernels (sm_103a).
//
// Batch decoding (which sequence a query belongs to and how many rows it sees),
// the device error word, element loads for the two input dtypes, and the
// order-preserving float -> uint32 map the radix selection runs on.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dsa.h"

namespace dsa {

// Every workspace starts with this many bytes of header; word 0 is the device
// error code, word 1 the first error's detail, word 2 the kernel that set it.
constexpr size_t kWsHeaderBytes = 256;
// Byte offset in the header of the fused kernel's grid barrier (two words).
constexpr size_t kWsGridBarOffset = 64;
// Byte offset in the header of the budget, in nanoseconds, of every wait of a
// CTA on other CTAs (64 bits; 0 = the default of 2 s).
constexpr size_t kWsWaitBudgetOffset = 128;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
// Byte offset in the header of the count of completed fused selection
// launches (32 bits): its parity picks the half of the double-buffered
// per-query state a launch uses.
constexpr size_t kWsLaunchCountOffset = 192;

enum DeviceError : int32_t {
    kDevOk = 0,
    kDevBadIndex = 1,      // a selected index outside [0, L)
    kDevBadBatch = 2,      // offsets inconsistent with the host bounds
    kDevTimeout = 3,       // a bounded wait gave up
};

__device__ __forceinline__ void record_error(int32_t* err, int32_t code, int32_t detail,
                                             int32_t where) {
    if (err != nullptr && atomicCAS(err, 0, code) == 0) {
        err[1] = detail;
        err[2] = where;
    }
}

// Batch description as the kernels receive it (plain device pointers).
struct BatchDev {
    const int64_t* row_off;
    const int64_t* key_off;
    const int64_t* q_off;
    int32_t n_seq;
    int32_t n_q;
    int32_t max_q_len;
    int64_t max_kv_len;
    int64_t total_rows;
    int64_t total_keys;
    int32_t kpool;
    uint32_t flags;        // DSA_FLAG_* of the call
};

struct QueryInfo {
    int32_t seq;
    int64_t row0;      // first cache row of the sequence
    int64_t key0;      // first indexer / pool key of the sequence
    int64_t L;         // rows this query sees, its own included
    int64_t n_keys;    // keys it scores: floor(L / kpool)
};

// Sequence of query q, then its visible length.  In a decode batch (one
// query per sequence: n_q == n_seq) query q is sequence q: the offsets of that
// guess are all read at once (one round trip) and checked; otherwise, or when
// the check fails, a binary search over q_off finds the sequence.
// Returns false (and records kDevBadBatch) when the offsets contradict the
// host bounds; the caller then skips the query.
// a * b / c for a, b, c >= 0, c > 0, in 32-bit arithmetic when the product
// fits (the common case: tile ranges of one launch), else 64-bit.  A 64-bit
// division is a long dependent instruction sequence on the GPU; on a kernel's
// prologue it costs a visible fraction of a microsecond.
__device__ __forceinline__ int64_t mul_div(int64_t a, int64_t b, int64_t c) {
    const int64_t p = a * b;
    if (p < ((int64_t)1 << 32) && c < ((int64_t)1 << 32))
        return (int64_t)((uint32_t)p / (uint32_t)c);
    return p / c;
}

__device__ __forceinline__ bool query_info(const BatchDev& b, int64_t q, QueryInfo& qi,
                                           int32_t* err, int32_t where) {
    int32_t s = -1;
    int64_t q0 = 0, q1 = 0, r0 = 0, r1 = 0, k0 = 0, k1 = 0;
    if (b.n_q == b.n_seq && q >= 0 && q < b.n_seq) {
        q0 = b.q_off[q];
        q1 = b.q_off[q + 1];
        r0 = b.row_off[q];
        r1 = b.row_off[q + 1];
        k0 = b.key_off[q];
        k1 = b.key_off[q + 1];
        if (q0 <= q && q < q1) s = (int32_t)q;
    }
    if (s < 0) {
        int32_t lo = 0, hi = b.n_seq - 1;
        while (lo < hi) {                   // last s with q_off[s] <= q
            int32_t mid = (lo + hi + 1) >> 1;
            if (b.q_off[mid] <= q) lo = mid; else hi = mid - 1;
        }
        s = lo;
        q0 = b.q_off[s];
        q1 = b.q_off[s + 1];
        r0 = b.row_off[s];
        r1 = b.row_off[s + 1];
        k0 = b.key_off[s];
        k1 = b.key_off[s + 1];
    }
    const int64_t kv_len = r1 - r0, q_len = q1 - q0;
    const int64_t L = kv_len - q_len + 1 + (q - q0);
    if (q < q0 || q >= q1 || q_len > kv_len || kv_len > b.max_kv_len || L < 1 || r0 < 0 ||
        r1 > b.total_rows) {
        record_error(err, kDevBadBatch, (int32_t)q, where);
        return false;
    }
    qi.seq = s;
    qi.row0 = r0;
    qi.key0 = k0;
    qi.L = L;
    // 0 < L <= kv_len <= max_kv_len < 2^31 here: 32-bit divisions
    qi.n_keys = (int64_t)((uint32_t)L / (uint32_t)b.kpool);
    if (k1 - k0 < (int64_t)((uint32_t)kv_len / (uint32_t)b.kpool) || k0 < 0 || k1 > b.total_keys) {
        record_error(err, kDevBadBatch, (int32_t)q, where);
        return false;
    }
    return true;
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }

// Order-preserving map: a > b as floats  <=>  order_key(a) > order_key(b) as
// unsigned integers.  Both zeros map to the key of +0 so that they tie and the
// lower index wins, as for every other tie.  Inputs are finite.
__device__ __forceinline__ uint32_t order_key(float s) {
    const uint32_t u = (s == 0.0f) ? 0u : __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace dsa
