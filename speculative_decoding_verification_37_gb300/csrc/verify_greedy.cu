// Greedy chain verification and greedy tree verification (sm_103a).
//
// "KV Cache 优化（四）：Speculative Decoding 投机解码" §4 and "10.6 投机解码"
// §10.6.1: at temperature 0 the acceptance rule reduces to comparing each
// draft token with the target's argmax and emitting the argmax at the first
// mismatch.  "投机推理：小模型搭树，大模型一次验证" (Validation, 接受过程):
// a tree is verified by one root-to-leaf walk over the parents' argmaxes.
//
// Both share one HBM-bound pass: each block reduces the argmax (lowest index
// on ties) of one slice of one logits row and folds it into the row's 64-bit
// key with one atomicMax.  The block that arrives last for a request (an
// arrival counter per request) then runs that request's decision: the chain
// comparison, or the tree walk plus the tree mask and position ids.  No block
// ever waits on another.
#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace specv {

constexpr int kArgNT = 256;
constexpr int kMaxMaskWords = 32;  // trees of up to 1023 draft nodes

__device__ __forceinline__ unsigned long long ld_volatile_u64(const unsigned long long *p) {
    return *reinterpret_cast<const volatile unsigned long long *>(p);
}

// -- chain decision (one thread) ------------------------------------------------
__device__ void greedy_chain_epilogue(const ArgmaxParams &p, int b) {
    const int g = p.gamma, V = p.V;
    unsigned long long *keys = p.keys + (int64_t)b * (g + 1);
    const int *d = p.tokens + (int64_t)b * g;
    bool bad = false;
    for (int k = 0; k < g; ++k) bad |= (d[k] < 0 || d[k] >= V);
    if (bad) {
        p.n_acc[b] = 0;
        p.n_out[b] = 0;
        if (p.flags) p.flags[b] = SPEC_FLAG_BAD_INPUT;
        atomicOr(p.status, SPEC_FLAG_BAD_INPUT);
    } else {
        int n = g;
        for (int k = 0; k < g; ++k) {
            if (d[k] != argmax_key_index(ld_volatile_u64(keys + k))) {
                n = k;
                break;
            }
        }
        int *out = p.out_tokens + (int64_t)b * (g + 1);
        for (int k = 0; k < n; ++k) out[k] = d[k];
        out[n] = argmax_key_index(ld_volatile_u64(keys + n));
        p.n_acc[b] = n;
        p.n_out[b] = n + 1;
        if (p.flags) p.flags[b] = 0;
    }
    for (int k = 0; k <= g; ++k) keys[k] = 0ull;
}

// -- tree decision (whole block) ------------------------------------------------
__device__ void tree_epilogue(const ArgmaxParams &p, int b) {
    const int N = p.N, R = p.R, V = p.V;
    const int *tok = p.node_token + (int64_t)b * N;
    const int *par = p.node_parent + (int64_t)b * N;
    const int *rown = p.row_of_node + (int64_t)b * (N + 1);
    unsigned long long *keys = p.keys + (int64_t)b * R;

    // validate every node: token in [0,V), parent < own id, row in [-1,R)
    int bad = 0;
    for (int i = threadIdx.x; i <= N; i += blockDim.x) {
        const int r = rown[i];
        bad |= (r < -1 || r >= R);
        if (i > 0) bad |= (tok[i - 1] < 0 || tok[i - 1] >= V || par[i - 1] < 0 || par[i - 1] >= i);
    }
    bad = __syncthreads_or(bad);
    if (bad) {
        if (threadIdx.x == 0) {
            p.n_acc[b] = 0;
            p.n_out[b] = 0;
            if (p.n_commit) p.n_commit[b] = 0;
            if (p.flags) p.flags[b] = SPEC_FLAG_BAD_INPUT;
            atomicOr(p.status, SPEC_FLAG_BAD_INPUT);
        }
    } else {
        if (threadIdx.x < 32) {
            // single-path walk by warp 0: lanes search the current node's children
            const int lane = threadIdx.x;
            int *path = p.path + (int64_t)b * N;
            int *out = p.out_tokens + (int64_t)b * (N + 1);
            int *slots = p.commit_slots ? p.commit_slots + (int64_t)b * (N + 1) : nullptr;
            int v = 0, n = 0, extra = -1;
            for (int step = 0; step <= N; ++step) {
                const int r = rown[v];
                if (r < 0) break;
                const int t = argmax_key_index(ld_volatile_u64(keys + r));
                int child = -1;
                for (int c0 = 1; c0 <= N && child < 0; c0 += 32) {
                    const int c = c0 + lane;
                    const bool hit = c <= N && par[c - 1] == v && tok[c - 1] == t;
                    const unsigned m = __ballot_sync(kFull, hit);
                    if (m) child = c0 + __ffs(m) - 1;
                }
                if (child < 0) {
                    extra = t;
                    break;
                }
                if (lane == 0) {
                    path[n] = child;
                    out[n] = tok[child - 1];
                    if (slots) slots[n + 1] = child;
                }
                ++n;
                v = child;
            }
            if (lane == 0) {
                if (extra >= 0) out[n] = extra;
                if (slots) slots[0] = 0;
                p.n_acc[b] = n;
                p.n_out[b] = n + (extra >= 0 ? 1 : 0);
                if (p.n_commit) p.n_commit[b] = n + 1;
                if (p.flags) p.flags[b] = 0;
            }
        }
        // tree mask and position ids ("10.6 投机解码" §10.6.3, Table 10-17):
        // each thread walks one node's ancestor chain
        if (p.mask || p.pos) {
            const int W = (N + 1 + 31) / 32;
            const int len0 = p.committed_len ? p.committed_len[b] : 0;
            for (int i = threadIdx.x; i <= N; i += blockDim.x) {
                uint32_t words[kMaxMaskWords];
#pragma unroll
                for (int w = 0; w < kMaxMaskWords; ++w) words[w] = 0u;
                int j = i, depth = 0;
                while (j > 0) {
                    words[j >> 5] |= 1u << (j & 31);
                    j = par[j - 1];
                    ++depth;
                }
                words[0] |= 1u;
                if (p.mask) {
                    uint32_t *row = p.mask + ((int64_t)b * (N + 1) + i) * W;
                    for (int w = 0; w < W; ++w) row[w] = words[w];
                }
                if (p.pos) p.pos[(int64_t)b * (N + 1) + i] = len0 + depth;
            }
        }
    }
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) keys[r] = 0ull;
}

// -- the pass ---------------------------------------------------------------------
// The block's slice (<= 64 KiB) is staged in shared memory by bulk copies;
// two shared-memory passes then find the largest value and the lowest index
// holding it.
constexpr int kArgStage = 65536;
using ArgRing = Ring<kArgStage, 1, 1>;

template <typename T>
__global__ void __launch_bounds__(kArgNT) argmax_verify_kernel(ArgmaxParams p) {
    constexpr int VEC = Elem<T>::VEC;
    extern __shared__ __align__(128) unsigned char dsm[];
    ArgRing &R = *reinterpret_cast<ArgRing *>(dsm);
    const int tid = threadIdx.x;
    const int slice = blockIdx.x % p.slices;
    const int row = blockIdx.x / p.slices;
    const int req = row / p.rows_per_req;
    const T *r = reinterpret_cast<const T *>(p.rows) + (int64_t)row * p.stride;
    const int lo = min(p.V, slice * p.slice_len);
    const int hi = min(p.V, lo + p.slice_len);
    const SliceSplit sp = split_slice(r, lo, hi);
    // scalar head and tail elements, one per thread at most
    const int nhead = sp.body0 - sp.head0, ntail = sp.hi - sp.tail0;
    const float xh = tid < nhead ? ld_elem(r, sp.head0 + tid) : -INFINITY;
    const float xt = tid < ntail ? ld_elem(r, sp.tail0 + tid) : -INFINITY;

    __shared__ float s_v[kArgNT / 32];
    __shared__ int s_last;
    __shared__ float s_max;
    __shared__ int s_min;
    const int lane = tid & 31, w = tid >> 5;
    int bestidx = INT_MAX;
    bool has = hi > lo;
    auto passes = [&](const uint4 *v, int nv) {
        // pass 1: the largest value of the slice
        float m = fmaxf(xh, xt);
        for (int q = tid; q < nv; q += kArgNT) {
            float x[VEC];
            unpack<T>(v[q], x);
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = fmaxf(m, x[e]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        if (lane == 0) s_v[w] = m;
        __syncthreads();
        if (tid == 0) {
            float t = s_v[0];
            for (int q = 1; q < kArgNT / 32; ++q) t = fmaxf(t, s_v[q]);
            s_max = t;
            s_min = INT_MAX;
        }
        __syncthreads();
        const float M = s_max;
        // pass 2: the lowest index holding it (-0 and +0 compare equal)
        int mine = INT_MAX;
        if (tid < nhead && xh == M) mine = sp.head0 + tid;
        for (int q = tid; q < nv && mine == INT_MAX; q += kArgNT) {
            float x[VEC];
            unpack<T>(v[q], x);
#pragma unroll
            for (int e = VEC - 1; e >= 0; --e)
                if (x[e] == M) mine = sp.body0 + q * VEC + e;
        }
        if (mine == INT_MAX && tid < ntail && xt == M) mine = sp.tail0 + tid;
        if (mine != INT_MAX) atomicMin(&s_min, mine);
        __syncthreads();
        bestidx = s_min;
    };
    const uint32_t nbytes = (uint32_t)((sp.tail0 - sp.body0) * sizeof(T));
    bool ok = true;
    if (nbytes > 0) {
        // the host keeps every slice within one stage, so this is one chunk
        const unsigned char *src[1] = {reinterpret_cast<const unsigned char *>(r + sp.body0)};
        ok = ring_stream(R, src, 1, nbytes, [&](const unsigned char *const *st, uint32_t, uint32_t bytes) {
            passes(reinterpret_cast<const uint4 *>(st[0]), (int)(bytes / 16));
        });
    } else {
        passes(nullptr, 0);
    }
    if (!ok && tid == 0) atomicOr(p.status, SPEC_FLAG_TIMEOUT);
    if (tid == 0) {
        if (has && bestidx != INT_MAX) atomicMax(p.keys + row, argmax_key(s_max, bestidx));
        __threadfence();
        const unsigned prev = atomicAdd(p.counters + req, 1u);
        s_last = prev == (unsigned)(p.slices * p.rows_per_req - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (p.mode == 0) {
        if (tid == 0) greedy_chain_epilogue(p, req);
    } else {
        tree_epilogue(p, req);
    }
    if (tid == 0) p.counters[req] = 0u;
}

size_t argmax_smem_bytes() { return sizeof(ArgRing); }

cudaError_t launch_argmax_verify(const ArgmaxParams &p, int dtype, int n_rows, cudaStream_t s) {
    const dim3 grid((unsigned)((int64_t)n_rows * p.slices));
    const int smem = (int)sizeof(ArgRing);
    static std::atomic<unsigned long long> done_bf16{0}, done_f32{0};
    cudaError_t e;
    if (dtype == SPEC_DTYPE_BF16) {
        e = ensure_smem_attr(argmax_verify_kernel<__nv_bfloat16>, smem, done_bf16);
        if (e != cudaSuccess) return e;
        argmax_verify_kernel<__nv_bfloat16><<<grid, kArgNT, smem, s>>>(p);
    } else {
        e = ensure_smem_attr(argmax_verify_kernel<float>, smem, done_f32);
        if (e != cudaSuccess) return e;
        argmax_verify_kernel<float><<<grid, kArgNT, smem, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace specv
