// Candidate keys of the keyed sampler, shared by the sampler kernels and the
// LM head's candidate epilogue: a logit and its token id in one 64-bit word
// whose order is the candidate order (logit descending, then id ascending).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace tfk {

// Order-preserving key: larger float -> larger key; -0 and +0 share a key.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// (key, id) -> one word, larger = earlier candidate; never 0 for id >= 0 and a
// key of a finite value.  (key 0, id -1) gives 0, the "no candidate" word.
__device__ __forceinline__ uint64_t composite(uint32_t key, int32_t id) {
    return (uint64_t(key) << 32) | uint64_t(0xFFFFFFFFu - uint32_t(id));
}
__device__ __forceinline__ int32_t composite_id(uint64_t c) { return int32_t(0xFFFFFFFFu - uint32_t(c)); }

// The warp's 32 values sorted in descending order across the lanes (bitonic
// network over shuffles): lane i returns the (i+1)-th largest.
__device__ __forceinline__ uint64_t warp_sort_desc(uint64_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const uint64_t o = __shfl_xor_sync(0xFFFFFFFFu, v, j);
            const bool lower = (lane & j) == 0;
            const bool keep_max = ((lane & k) == 0) == lower;
            v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
        }
    }
    return v;
}

// Merges n <= 32 distinct words P (any order, all above the zero padding)
// into the list L of 64 words sorted in descending order (0-padded), keeping
// the 64 largest: each word's place in the merged order is its own index
// plus the number of words of the other set above it (a binary search in L
// for the words of P), so every word lands at once.  Call with the whole warp.
__device__ __forceinline__ void warp_merge_rank(uint64_t *L, const uint64_t *P, int n) {
    const int lane = threadIdx.x & 31;
    const uint64_t p = lane < n ? P[lane] : 0ull;
    const uint64_t l0 = L[lane], l1 = L[32 + lane];
    int pos_p = 64;
    if (lane < n) {
        int lo = 0, hi = 64;   // number of list words above p
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (L[mid] > p)
                lo = mid + 1;
            else
                hi = mid;
        }
        int above = 0;
        for (int j = 0; j < n; ++j) above += P[j] > p;
        pos_p = lo + above;
    }
    int c0 = 0, c1 = 0;
    for (int j = 0; j < n; ++j) {
        const uint64_t q = P[j];
        c0 += q > l0;
        c1 += q > l1;
    }
    __syncwarp();
    if (lane + c0 < 64) L[lane + c0] = l0;
    if (32 + lane + c1 < 64) L[32 + lane + c1] = l1;
    if (pos_p < 64) L[pos_p] = p;
    __syncwarp();
}

}  // namespace tfk
