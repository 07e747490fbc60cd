// k-th largest selection on order keys (top-k threshold with ties kept).
//
// Keys are the top KB bits of the order-preserving float key (16 for bf16,
// 32 for f32), so "key >= threshold" is "logit >= k-th largest logit".
#pragma once

#include "common.cuh"

namespace specv {

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// The k-th largest key (1-based, counted with multiplicity) among buf[0..n),
// n >= k, computed by one warp with a bitwise radix descent.  CAP/32 entries
// per lane.
template <int KB, int CAP>
__device__ __forceinline__ uint32_t warp_kth_largest(const uint2 *buf, int n, int k) {
    const int lane = threadIdx.x & 31;
    constexpr int PER = CAP / 32;
    uint32_t key[PER];
    bool val[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int idx = lane + 32 * i;
        val[i] = idx < n;
        key[i] = val[i] ? buf[idx].x : 0u;
    }
    uint32_t prefix = 0u;
    unsigned rem = (unsigned)k;
#pragma unroll 1
    for (int bit = KB - 1; bit >= 0; --bit) {
        const uint32_t cand = prefix | (1u << bit);
        unsigned c = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) c += (val[i] && (key[i] >> bit) == (cand >> bit)) ? 1u : 0u;
        c = __reduce_add_sync(kFull, c);
        if (c >= rem) prefix = cand;
        else rem -= c;
    }
    return prefix;
}

// Block-wide k-th largest over a set of entries that each thread enumerates
// with `each(f)` calling f(key) for its entries.  8-bit digits from the top,
// histograms in shared memory (`hist`: 256 words, `bc`: 2 words).  Every
// thread returns the threshold.  Requires the set to hold >= k keys.
template <int KB, int NT, typename Each>
__device__ uint32_t block_kth_largest(Each &&each, unsigned k, unsigned *hist, unsigned *bc) {
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t prefix = 0u;
    unsigned rem = k;
#pragma unroll 1
    for (int shift = KB - 8; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += NT) hist[i] = 0u;
        __syncthreads();
        const int hs = shift + 8;
        each([&](uint32_t key) {
            const bool match = hs >= KB || (uint64_t(key) >> hs) == (uint64_t(prefix) >> hs);
            if (match) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        });
        __syncthreads();
        if (tid < 32) {
            // lane l owns bins 255-8l .. 248-8l, in descending order
            unsigned b[8], s = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                b[q] = hist[255 - 8 * lane - q];
                s += b[q];
            }
            unsigned incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            const unsigned excl = incl - s;
            const bool here = excl < rem && rem <= incl;
            const unsigned who = __ballot_sync(kFull, here);
            if (who == 0u && lane == 0) {  // fewer than k keys: keep everything
                bc[0] = 0u;
                bc[1] = 1u;
            }
            if (who != 0u && lane == (int)(__ffs(who) - 1)) {
                unsigned above = excl;
                int d = 255 - 8 * lane;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    if (above + b[q] >= rem) { d = 255 - 8 * lane - q; break; }
                    above += b[q];
                }
                bc[0] = (unsigned)d;
                bc[1] = rem - above;
            }
        }
        __syncthreads();
        prefix |= bc[0] << shift;
        rem = bc[1];
        __syncthreads();
    }
    return prefix;
}

}  // namespace specv
