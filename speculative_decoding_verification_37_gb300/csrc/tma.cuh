// Bulk global->shared streaming on sm_103a: cp.async.bulk (the TMA unit's
// 1-D copy) completing on mbarriers, with bounded waits.
//
// A slice of one or two logits rows is split into a scalar head, a
// 16-byte-aligned body and a scalar tail.  The body is streamed through a
// ring of NST stages of CH bytes per row: one thread arms a stage's mbarrier
// with the expected byte count and issues one bulk copy per row; every
// thread waits on the stage, processes it from shared memory, and after a
// block barrier the stage is refilled with the chunk NST further on.  The
// bytes in flight per CTA are NST*CH*rows without costing registers.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace specv {

// Programmatic dependent launch: a primary kernel lets its dependent launch
// at once; the dependent waits for the primary's completion (and its memory)
// only where it reads the primary's results.  Both are no-ops without the
// launch attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// bounded spin on an mbarrier phase; false if it did not complete in time
constexpr long long kSpinLimit = 1ll << 22;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_inval(unsigned long long *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// make barrier initialisation visible to the asynchronous (bulk copy) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, unsigned phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(phase)
        : "memory");
    return ok != 0u;
}

__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar, unsigned phase) {
    for (long long it = 0; it < kSpinLimit; ++it)
        if (mbar_try_wait(bar, phase)) return true;
    return false;
}

// After a wait ran out: waits (bounded, four times the normal limit) for a
// stage whose bulk copy was issued and not yet seen complete, so that no copy
// lands in shared memory after the block has moved on or exited.  False if
// even that ran out; the caller then leaves the barrier as it is.
__device__ __forceinline__ bool mbar_drain(unsigned long long *bar, unsigned phase) {
    for (int rep = 0; rep < 4; ++rep)
        if (mbar_wait_bounded(bar, phase)) return true;
    return false;
}

// bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_g2s(void *sdst, const void *gsrc, uint32_t bytes,
                                         unsigned long long *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 policy for data read once: its lines are the first to go, so a stream
// of logits does not push out the small results written next to it
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// bulk_g2s with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_policy(void *sdst, const void *gsrc, uint32_t bytes,
                                                unsigned long long *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(sdst)),
        "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// bulk copy of `bytes` from shared to global memory (same alignment rules),
// tracked by the issuing thread's bulk async-group
__device__ __forceinline__ void bulk_s2g(void *gdst, const void *ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
                 "r"(smem_u32(ssrc)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// asynchronous prefetch of `bytes` (multiple of 16, address 16-byte aligned)
// into L2; no completion to wait for
__device__ __forceinline__ void bulk_prefetch_l2(const void *gsrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// waits until every committed bulk store of this thread has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// waits until every committed bulk store of this thread has read its shared
// memory source (the writes to global memory may still be in flight; they
// complete before the kernel does)
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Ring of NST stages x ROWS rows x CH bytes.
template <int CH, int NST, int ROWS> struct Ring {
    alignas(128) unsigned char buf[NST][ROWS][CH];
    alignas(8) unsigned long long full[NST];
};

// Streams the 16-byte-aligned bodies of `rows` rows (rows <= ROWS):
// body r starts at `src[r]`, all of `nbytes` bytes.  Calls f(stage, off, bytes)
// in chunk order on every thread, where stage[r] points at row r's bytes
// [off, off + bytes) of the body in shared memory.  Returns false if a stage
// did not arrive within the spin limit (the caller flags the request).
template <int CH, int NST, int ROWS, typename F>
__device__ bool ring_stream(Ring<CH, NST, ROWS> &R, const unsigned char *const *src, int rows,
                            uint32_t nbytes, F &&f) {
    const int nch = (int)((nbytes + CH - 1) / CH);
    auto issue = [&](int chunk, int s) {
        const uint32_t off = (uint32_t)chunk * CH;
        const uint32_t bytes = min((uint32_t)CH, nbytes - off);
        mbar_arrive_expect_tx(&R.full[s], bytes * (uint32_t)rows);
        for (int r = 0; r < rows; ++r) bulk_g2s(R.buf[s][r], src[r] + off, bytes, &R.full[s]);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(&R.full[s], 1);
        fence_barrier_init();
        for (int s = 0; s < NST && s < nch; ++s) issue(s, s);
    }
    __syncthreads();
    for (int i = 0; i < nch; ++i) {
        const int s = i % NST;
        const bool ok = mbar_wait_bounded(&R.full[s], (unsigned)((i / NST) & 1));
        const unsigned char *stage[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) stage[r] = R.buf[s][r];
        const uint32_t off = (uint32_t)i * CH;
        f(stage, off, min((uint32_t)CH, nbytes - off));
        if (__syncthreads_or(!ok)) {
            // a chunk did not arrive in time: issue nothing more, wait for
            // the chunks already issued (i .. i+NST-1) before the ring's
            // memory may be used again, and report the failure
            if (threadIdx.x == 0) {
                bool drained = true;
                for (int q = i; q < nch && q < i + NST; ++q)
                    drained &= mbar_drain(&R.full[q % NST], (unsigned)((q / NST) & 1));
                if (drained)
                    for (int t = 0; t < NST; ++t) mbar_inval(&R.full[t]);
            }
            __syncthreads();
            return false;
        }
        if (threadIdx.x == 0 && i + NST < nch) issue(i + NST, s);
    }
    if (threadIdx.x == 0)
        for (int s = 0; s < NST; ++s) mbar_inval(&R.full[s]);
    __syncthreads();
    return true;
}

// Split of a row slice [lo, hi) into scalar head, 16-byte body, scalar tail.
struct SliceSplit {
    int head0, body0, tail0, hi;  // head [head0, body0), body [body0, tail0), tail [tail0, hi)
};

template <typename T> __device__ __forceinline__ SliceSplit split_slice(const T *row, int lo, int hi) {
    SliceSplit s;
    s.head0 = lo;
    s.hi = hi;
    if (hi <= lo) {
        s.body0 = s.tail0 = lo;
        return s;
    }
    const uintptr_t a = reinterpret_cast<uintptr_t>(row + lo);
    int head = (int)(((16u - (unsigned)(a & 15u)) & 15u) / sizeof(T));
    if (head > hi - lo) head = hi - lo;
    s.body0 = lo + head;
    constexpr int VEC = 16 / (int)sizeof(T);
    s.tail0 = s.body0 + ((hi - s.body0) / VEC) * VEC;
    return s;
}

}  // namespace specv
