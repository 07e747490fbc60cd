// Shared device helpers of the verify-and-commit kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "spec_verify.h"

namespace specv {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------------------
// element types: logits are bf16 or f32; 16-byte vectors hold VEC of them
// ---------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
    static constexpr int VEC = 4;
    static constexpr int KEY_BITS = 32;    // significant high bits of the order key
};
template <> struct Elem<__nv_bfloat16> {
    static constexpr int VEC = 8;
    static constexpr int KEY_BITS = 16;
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// 16-byte read-only load that does not allocate in L1 (rows are streamed).
__device__ __forceinline__ uint4 ld_nc16(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <typename T> __device__ __forceinline__ void unpack(const uint4 &v, float *out);
template <> __device__ __forceinline__ void unpack<float>(const uint4 &v, float *out) {
    out[0] = __uint_as_float(v.x);
    out[1] = __uint_as_float(v.y);
    out[2] = __uint_as_float(v.z);
    out[3] = __uint_as_float(v.w);
}
template <> __device__ __forceinline__ void unpack<__nv_bfloat16>(const uint4 &v, float *out) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        out[2 * i] = __uint_as_float(w[i] << 16);
        out[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

template <typename T> __device__ __forceinline__ float ld_elem(const T *row, int64_t i) {
    return to_f32(row[i]);
}

// Order-preserving map float -> uint32 (larger value <=> larger key); -0 is
// folded onto +0 so the two compare equal, as they do as values.
__device__ __forceinline__ uint32_t fkey(float x) {
    uint32_t u = __float_as_uint(x);
    u = (u << 1) == 0u ? 0u : u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// Row slice traversal.  A slice [lo, hi) of a row is split into a scalar
// head up to the first 16-byte boundary, a 16-byte-vector body and a scalar
// tail, so any row alignment works.  Thread `tid` of `nt` visits its
// elements in increasing index order; f(value, index) is called per element.
// ---------------------------------------------------------------------------
template <typename T, int UNROLL, typename F>
__device__ __forceinline__ void for_slice(const T *row, int lo, int hi, int tid, int nt, F &&f) {
    constexpr int VEC = Elem<T>::VEC;
    if (hi <= lo) return;
    const uintptr_t a = reinterpret_cast<uintptr_t>(row + lo);
    int head = (int)(((16u - (unsigned)(a & 15u)) & 15u) / sizeof(T));
    if (head > hi - lo) head = hi - lo;
    const int body0 = lo + head;
    const int nvec = (hi - body0) / VEC;
    const int tail0 = body0 + nvec * VEC;
    if (tid < head) f(ld_elem(row, lo + tid), lo + tid);
    const uint4 *vp = reinterpret_cast<const uint4 *>(row + body0);
    int v = tid;
    for (; v + (UNROLL - 1) * nt < nvec; v += UNROLL * nt) {
        uint4 raw[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) raw[u] = ld_nc16(vp + v + u * nt);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            float x[VEC];
            unpack<T>(raw[u], x);
            const int base = body0 + (v + u * nt) * VEC;
#pragma unroll
            for (int e = 0; e < VEC; ++e) f(x[e], base + e);
        }
    }
    for (; v < nvec; v += nt) {
        float x[VEC];
        unpack<T>(ld_nc16(vp + v), x);
        const int base = body0 + v * VEC;
#pragma unroll
        for (int e = 0; e < VEC; ++e) f(x[e], base + e);
    }
    if (tid < hi - tail0) f(ld_elem(row, tail0 + tid), tail0 + tid);
}

// Same traversal, but f(x[VEC], base, count) is called once per vector (and
// once per scalar with count 1), so a thread can reduce a vector before
// touching its running state.
template <typename T, int UNROLL, typename F>
__device__ __forceinline__ void for_slice_vec(const T *row, int lo, int hi, int tid, int nt, F &&f) {
    constexpr int VEC = Elem<T>::VEC;
    if (hi <= lo) return;
    const uintptr_t a = reinterpret_cast<uintptr_t>(row + lo);
    int head = (int)(((16u - (unsigned)(a & 15u)) & 15u) / sizeof(T));
    if (head > hi - lo) head = hi - lo;
    const int body0 = lo + head;
    const int nvec = (hi - body0) / VEC;
    const int tail0 = body0 + nvec * VEC;
    if (tid < head) {
        float x[VEC];
        x[0] = ld_elem(row, lo + tid);
        f(x, lo + tid, 1);
    }
    const uint4 *vp = reinterpret_cast<const uint4 *>(row + body0);
    int v = tid;
    for (; v + (UNROLL - 1) * nt < nvec; v += UNROLL * nt) {
        uint4 raw[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) raw[u] = ld_nc16(vp + v + u * nt);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            float x[VEC];
            unpack<T>(raw[u], x);
            f(x, body0 + (v + u * nt) * VEC, VEC);
        }
    }
    for (; v < nvec; v += nt) {
        float x[VEC];
        unpack<T>(ld_nc16(vp + v), x);
        f(x, body0 + v * VEC, VEC);
    }
    if (tid < hi - tail0) {
        float x[VEC];
        x[0] = ld_elem(row, tail0 + tid);
        f(x, tail0 + tid, 1);
    }
}

// ---------------------------------------------------------------------------
// Barriers of the first NT threads of a block (named barrier 1).  In a block
// of exactly NT threads they act as __syncthreads (and its count / or
// forms); in a block that adds a producer warp after the first NT threads,
// they synchronise the other threads only, so the producer never waits.
// ---------------------------------------------------------------------------
template <int NT> __device__ __forceinline__ void sync_nt() {
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}
template <int NT> __device__ __forceinline__ int sync_nt_count(bool pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.popc.u32 %0, 1, %2, p;\n\t}"
        : "=r"(r)
        : "r"((int)pred), "n"(NT)
        : "memory");
    return r;
}
template <int NT> __device__ __forceinline__ bool sync_nt_or(bool pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\tselp.s32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((int)pred), "n"(NT)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------------------------
// reductions (fixed combination order, hence deterministic)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}
__device__ __forceinline__ unsigned warp_sum_u(unsigned v) { return __reduce_add_sync(kFull, v); }

// Block sum; every thread gets the result.  `red` needs nt/32 floats.
template <int NT> __device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum(v);
    sync_nt<NT>();
    if (lane == 0) red[w] = v;
    sync_nt<NT>();
    float t = lane < NT / 32 ? red[lane] : 0.0f;
    return warp_sum(t);
}

template <int NT> __device__ __forceinline__ unsigned block_sum_u(unsigned v, unsigned *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum_u(v);
    sync_nt<NT>();
    if (lane == 0) red[w] = v;
    sync_nt<NT>();
    unsigned t = lane < NT / 32 ? red[lane] : 0u;
    return warp_sum_u(t);
}

// Running (max, sum of 2^(x*c - max*c)) pairs of a softmax over x*c.
struct MaxSum {
    float m;  // max raw logit (-inf if empty)
    float s;  // sum of exp2(x*c2 - m*c2)
};

__device__ __forceinline__ MaxSum ms_combine(MaxSum a, MaxSum b, float c2) {
    const float m = fmaxf(a.m, b.m);
    if (m == -INFINITY) return MaxSum{-INFINITY, 0.0f};
    const float sa = a.m == -INFINITY ? 0.0f : a.s * exp2f((a.m - m) * c2);
    const float sb = b.m == -INFINITY ? 0.0f : b.s * exp2f((b.m - m) * c2);
    return MaxSum{m, sa + sb};
}

__device__ __forceinline__ MaxSum warp_ms(MaxSum v, float c2) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        MaxSum o2{__shfl_xor_sync(kFull, v.m, o), __shfl_xor_sync(kFull, v.s, o)};
        v = ms_combine(v, o2, c2);
    }
    return v;
}

template <int NT> __device__ __forceinline__ MaxSum block_ms(MaxSum v, float c2, float2 *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_ms(v, c2);
    sync_nt<NT>();
    if (lane == 0) red[w] = make_float2(v.m, v.s);
    sync_nt<NT>();
    MaxSum t = lane < NT / 32 ? MaxSum{red[lane].x, red[lane].y} : MaxSum{-INFINITY, 0.0f};
    return warp_ms(t, c2);
}

// Argmax with the lowest index winning ties; idx < 0 means "empty".
struct ArgMax {
    float v;
    int idx;
};

__device__ __forceinline__ bool am_better(float v1, int i1, float v2, int i2) {
    if (i2 < 0) return i1 >= 0;
    if (i1 < 0) return false;
    return v1 > v2 || (v1 == v2 && i1 < i2);
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(kFull, a.v, o);
        const int i2 = __shfl_xor_sync(kFull, a.idx, o);
        if (am_better(v2, i2, a.v, a.idx)) a = ArgMax{v2, i2};
    }
    return a;
}

// 64-bit argmax key: order key of the value, then the complemented index, so
// an unsigned max keeps the largest value and, among equal values, the
// lowest index.  Zero is below every real key.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    return ((unsigned long long)fkey(v) << 32) | (unsigned long long)(~(uint32_t)idx);
}
__device__ __forceinline__ int argmax_key_index(unsigned long long k) {
    return (int)(~(uint32_t)(k & 0xffffffffull));
}

// In-place KV commit of a chain request (one thread): the candidates' K/V
// were written at cache positions len .. len+gamma before the verify, so the
// commit advances the length by n_out (the last emitted token and the
// accepted drafts), the draft cache's length is cut back to the same
// boundary (never raised: with every draft accepted it has not seen the last
// one yet) and the blocks in use follow.  A request that fails the check
// keeps every length.
template <typename IP>
__device__ __forceinline__ int inplace_len0(const IP &ip, int b) {
    return ip.len ? ip.len[b] : 0;
}
template <typename IP>
__device__ __forceinline__ unsigned inplace_bad(const IP &ip, int len0, int gamma) {
    if (!ip.len) return 0u;
    const int64_t end = (int64_t)len0 + gamma + 1;
    return (len0 < 0 || end > 0x7fffffffLL || (ip.capacity > 0 && end > ip.capacity)) ? SPEC_FLAG_BAD_INPUT
                                                                                        : 0u;
}
template <typename IP>
__device__ __forceinline__ void inplace_commit(const IP &ip, int b, int len0, int n_out) {
    if (!ip.len) return;
    const int nl = len0 + n_out;
    ip.len[b] = nl;
    if (ip.draft_len) ip.draft_len[b] = min(ip.draft_len[b], nl);
    if (ip.blocks_in_use) ip.blocks_in_use[b] = (int)(((int64_t)nl + ip.block_size - 1) / ip.block_size);
}

// Early end of a chain round ("KV Cache 优化（四）" §5): the emitted tokens
// are cut right after the first end-of-sequence token, then to the request's
// remaining length.  stop_limit: the limit of request b (INT_MAX if none);
// stop_scan: one 32-position chunk of the round (lane = position q, tok its
// token, positions 0..n emitted before the cuts), updating `cut`, the first
// EOS position seen (INT_MAX if none).
template <typename SR> __device__ __forceinline__ int stop_limit(const SR &st, int b) {
    if (!st.max_new) return 0x7fffffff;
    const int m = st.max_new[b];
    return m > 0 ? m : 0;
}
template <typename SR>
__device__ __forceinline__ int stop_scan(const SR &st, int q0, int q, int n, int tok, int cut) {
    const unsigned hit = __ballot_sync(kFull, st.eos >= 0 && q <= n && tok == st.eos);
    return (cut == 0x7fffffff && hit) ? q0 + __ffs(hit) - 1 : cut;
}
// The round's emitted length after the cuts, and the flags that say which
// cut shortened it (an EOS kept as the last token counts as an EOS end).
__device__ __forceinline__ int stop_length(int n, int cut, int lim, unsigned &flags) {
    const int L0 = cut < n ? cut + 1 : n + 1;  // n + 1 tokens unless an EOS comes first
    const int L = L0 < lim ? L0 : lim;
    if (cut <= n && cut < L) flags |= SPEC_FLAG_EOS;
    if (lim < L0) flags |= SPEC_FLAG_LIMIT;
    return L;
}

// Sets a kernel's dynamic shared-memory limit once per device (the setting
// is per device; doing it once keeps it out of captured launch sequences).
// Devices 0..63 remember that it is done; a higher device id sets it on
// every call.
template <typename K>
inline cudaError_t ensure_smem_attr(K kernel, int bytes, std::atomic<unsigned long long> &done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    const unsigned long long bit = 1ull << dev;
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

}  // namespace specv
