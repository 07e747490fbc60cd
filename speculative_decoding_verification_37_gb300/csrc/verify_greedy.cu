// Greedy chain verification and greedy tree verification (sm_103a).
//
// "KV Cache 优化（四）：Speculative Decoding 投机解码" §4 and "10.6 投机解码"
// §10.6.1: at temperature 0 the acceptance rule reduces to comparing each
// draft token with the target's argmax and emitting the argmax at the first
// mismatch.  "投机推理：小模型搭树，大模型一次验证" (Validation, 接受过程):
// a tree is verified by one root-to-leaf walk over the parents' argmaxes.
//
// Both share one HBM-bound pass (argmax_pass_kernel): a persistent grid of
// four blocks per SM takes (row, slice) items round-robin through a
// three-stage bulk-copy ring; a block reduces the argmax (lowest index on
// ties) of the slice and folds it into the row's 64-bit key with one
// fire-and-forget atomicMax.  A second, small kernel (argmax_decide_kernel,
// one block per request) then runs each request's decision: the chain
// comparison, or the tree walk plus the tree mask and position ids; it leaves
// the keys zeroed.  No block ever waits on another.
#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace specv {

constexpr int kArgNT = 256;

// (The decision kernel is a programmatic dependent launch of the pass, see
// tma.cuh: it waits for the pass only where it reads the argmax keys.)
constexpr int kMaxMaskWords = 32;  // trees of up to 1023 draft nodes

// -- chain decision (warp 0; lane k takes position k) ---------------------------
__device__ void greedy_chain_decide(const ArgmaxParams &p, int b) {
    const int g = p.gamma, V = p.V, lane = threadIdx.x & 31;
    unsigned long long *keys = p.keys + (int64_t)b * (g + 1);
    const int *d = p.tokens + (int64_t)b * g;
    int n = g;  // the first mismatch (g: every draft matches)
    const int d0 = lane < g ? d[lane] : 0;  // loaded before the keys are ready
    const int len0 = lane == 0 ? inplace_len0(p.ip, b) : 0;
    bool bad = lane == 0 && inplace_bad(p.ip, len0, g);
    pdl_wait_primary();
    for (int k0 = 0; k0 < g; k0 += 32) {
        const int k = k0 + lane;
        int dk = 0;
        int ak = -1;
        if (k < g) {
            dk = k0 == 0 ? d0 : d[k];
            ak = argmax_key_index(keys[k]);
            bad |= dk < 0 || dk >= V;
        }
        const unsigned mis = __ballot_sync(kFull, k < g && dk != ak);
        if (n == g && mis) n = k0 + __ffs(mis) - 1;
    }
    bad = __any_sync(kFull, bad);
    if (bad) {
        if (lane == 0) {
            p.n_acc[b] = 0;
            p.n_out[b] = 0;
            if (p.flags) p.flags[b] = SPEC_FLAG_BAD_INPUT;
            atomicOr(p.status, SPEC_FLAG_BAD_INPUT);
        }
    } else {
        int *out = p.out_tokens + (int64_t)b * (g + 1);
        const int lim = stop_limit(p.stop, b);
        int cut = 0x7fffffff;  // the first EOS position so far
        for (int k0 = 0; k0 <= n; k0 += 32) {  // (n is warp-uniform)
            const int k = k0 + lane;
            const int tok = k < n ? d[k] : (k == n ? argmax_key_index(keys[n]) : -1);
            cut = stop_scan(p.stop, k0, k, n, tok, cut);
            if (k <= n) out[k] = (k < lim && k <= cut) ? tok : -1;
        }
        if (lane == 0) {
            unsigned f = 0u;
            const int L = stop_length(n, cut, lim, f);
            p.n_acc[b] = n < L ? n : L;
            p.n_out[b] = L;
            if (p.flags) p.flags[b] = f;
            inplace_commit(p.ip, b, len0, L);
        }
    }
    __syncwarp();
    for (int k = lane; k <= g; k += 32) keys[k] = 0ull;
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
    if (!bad && (p.mask || p.pos)) {
        // tree mask and position ids ("10.6 投机解码" §10.6.3, Table 10-17): each
        // thread walks one node's ancestor chain; no argmax needed, so this
        // runs while the pass is still finishing
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
    pdl_wait_primary();
    if (bad) {
        if (threadIdx.x == 0) {
            p.n_acc[b] = 0;
            p.n_out[b] = 0;
            if (p.n_commit) p.n_commit[b] = 0;
            if (p.flags) p.flags[b] = SPEC_FLAG_BAD_INPUT;
            atomicOr(p.status, SPEC_FLAG_BAD_INPUT);
        }
    } else if (threadIdx.x < 32) {
        // single-path walk by warp 0: lanes search the current node's children
        const int lane = threadIdx.x;
        int *path = p.path + (int64_t)b * N;
        int *out = p.out_tokens + (int64_t)b * (N + 1);
        int *slots = p.commit_slots ? p.commit_slots + (int64_t)b * (N + 1) : nullptr;
        int v = 0, n = 0, extra = -1;
        // every row's argmax in one load per lane (rows past 32 read on demand)
        const int kt = lane < R ? argmax_key_index(keys[lane]) : -1;
        for (int step = 0; step <= N; ++step) {
            const int r = rown[v];
            if (r < 0) break;
            const int t = r < 32 ? __shfl_sync(kFull, kt, r) : argmax_key_index(keys[r]);
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
    __syncthreads();
    for (int r = threadIdx.x; r < R; r += blockDim.x) keys[r] = 0ull;
}

// -- the pass ---------------------------------------------------------------------
// Items (row, slice) of at most kArgStage bytes, row-major; block g takes items
// g, g + G, g + 2G, ...  Thread 0 keeps kArgNST items in flight (one
// cp.async.bulk each, evict-first in L2, completing on the stage's mbarrier).
// Per item: every thread takes the maximum of each 16-byte vector it holds
// (packed bf16x2 maxima); the block's maximum M; then only the vectors whose
// maximum is M are searched for the lowest index holding it.  Two block
// barriers per item.
constexpr int kArgStage = 16384;
constexpr int kArgNST = 3;
constexpr int kArgBlocksPerSM = 4;
constexpr int kArgVecPerThr = kArgStage / 16 / kArgNT;
static_assert(kArgVecPerThr * 16 * kArgNT == kArgStage, "a stage is whole vectors per thread");

struct ArgRingN {
    alignas(128) unsigned char buf[kArgNST][kArgStage];
};

int argmax_stage_bytes() { return kArgStage; }

__device__ __forceinline__ __nv_bfloat162 u32_as_bf2(uint32_t w) {
    __nv_bfloat162 r;
    memcpy(&r, &w, 4);
    return r;
}
template <typename T> __device__ __forceinline__ float vmax16(const uint4 &v);
template <> __device__ __forceinline__ float vmax16<float>(const uint4 &v) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}
template <> __device__ __forceinline__ float vmax16<__nv_bfloat16>(const uint4 &v) {
    const __nv_bfloat162 a = __hmax2(__hmax2(u32_as_bf2(v.x), u32_as_bf2(v.y)),
                                     __hmax2(u32_as_bf2(v.z), u32_as_bf2(v.w)));
    return fmaxf(__low2float(a), __high2float(a));
}

struct ArgItem {
    int row, lo, hi;
    SliceSplit sp;
};

template <typename T>
__device__ __forceinline__ ArgItem arg_item(const ArgmaxParams &p, int item) {
    ArgItem it;
    it.row = (int)((unsigned)item / (unsigned)p.slices);
    const int slice = item - it.row * p.slices;
    it.lo = min(p.V, slice * p.slice_len);
    it.hi = min(p.V, it.lo + p.slice_len);
    const T *r = reinterpret_cast<const T *>(p.rows) + (int64_t)it.row * p.stride;
    it.sp = split_slice(r, it.lo, it.hi);
    return it;
}

template <typename T>
__device__ __forceinline__ void arg_issue(const ArgmaxParams &p, ArgRingN &R, unsigned long long *full,
                                          int item, int s) {
    const ArgItem it = arg_item<T>(p, item);
    const uint32_t nb = (uint32_t)((it.sp.tail0 - it.sp.body0) * (int)sizeof(T));
    mbar_arrive_expect_tx(&full[s], nb);
    if (nb) {
        const T *r = reinterpret_cast<const T *>(p.rows) + (int64_t)it.row * p.stride;
        bulk_g2s_policy(R.buf[s], r + it.sp.body0, nb, &full[s], l2_evict_first());
    }
}

template <typename T>
__global__ void __launch_bounds__(kArgNT, kArgBlocksPerSM) argmax_pass_kernel(ArgmaxParams p, int n_items) {
    constexpr int VEC = Elem<T>::VEC;
    extern __shared__ __align__(128) unsigned char dsm[];
    ArgRingN &R = *reinterpret_cast<ArgRingN *>(dsm);
    __shared__ __align__(8) unsigned long long full[kArgNST];
    __shared__ float s_v[kArgNT / 32];
    __shared__ int s_i[kArgNT / 32];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int G = gridDim.x;
    unsigned phase = 0u;
    bool timeout = false;
    pdl_launch_dependents();  // the decision blocks may start their own loads
    if (tid == 0) {
        for (int s = 0; s < kArgNST; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        for (int s = 0; s < kArgNST; ++s)
            if ((int)blockIdx.x + s * G < n_items) arg_issue<T>(p, R, full, blockIdx.x + s * G, s);
    }
    __syncthreads();
    int t = 0;
    for (int item = blockIdx.x; item < n_items; item += G, ++t) {
        const int s = t % kArgNST;
        const ArgItem it = arg_item<T>(p, item);
        const SliceSplit sp = it.sp;
        const T *r = reinterpret_cast<const T *>(p.rows) + (int64_t)it.row * p.stride;
        const int nhead = sp.body0 - sp.head0, ntail = sp.hi - sp.tail0;
        const float xh = tid < nhead ? ld_elem(r, sp.head0 + tid) : -INFINITY;
        const float xt = tid < ntail ? ld_elem(r, sp.tail0 + tid) : -INFINITY;
        const bool ok = mbar_wait_bounded(&full[s], (phase >> s) & 1u);
        phase ^= 1u << s;
        const int nvec = (sp.tail0 - sp.body0) / VEC;
        const uint4 *v = reinterpret_cast<const uint4 *>(R.buf[s]);
        // 1. the slice's largest value
        float vm[kArgVecPerThr];
        float m = fmaxf(xh, xt);
#pragma unroll
        for (int i = 0; i < kArgVecPerThr; ++i) {
            const int q = tid + i * kArgNT;
            vm[i] = q < nvec ? vmax16<T>(v[q]) : -INFINITY;
            m = fmaxf(m, vm[i]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        if (lane == 0) s_v[w] = m;
        __syncthreads();
        float M = s_v[0];
#pragma unroll
        for (int q = 1; q < kArgNT / 32; ++q) M = fmaxf(M, s_v[q]);
        // 2. the lowest index holding it (-0 and +0 compare equal)
        int mine = INT_MAX;
        if (tid < nhead && xh == M) mine = sp.head0 + tid;
#pragma unroll
        for (int i = 0; i < kArgVecPerThr; ++i) {
            const int q = tid + i * kArgNT;
            if (mine == INT_MAX && q < nvec && vm[i] == M) {
                float x[VEC];
                unpack<T>(v[q], x);
#pragma unroll
                for (int e = VEC - 1; e >= 0; --e)
                    if (x[e] == M) mine = sp.body0 + q * VEC + e;
            }
        }
        if (mine == INT_MAX && tid < ntail && xt == M) mine = sp.tail0 + tid;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mine = min(mine, __shfl_xor_sync(kFull, mine, o));
        if (lane == 0) s_i[w] = mine;
        if (__syncthreads_or(!ok)) {  // stage s is consumed; a copy did not arrive in time
            // issue nothing more; wait for the copies already issued (this
            // block's local items t .. t+NST-1) before the block may exit
            if (tid == 0) {
                bool drained = true;
                int u = t;
                for (int nxt = item; nxt < n_items && u < t + kArgNST; nxt += G, ++u)
                    drained &= mbar_drain(&full[u % kArgNST], (unsigned)((u / kArgNST) & 1));
                atomicOr(p.status, SPEC_FLAG_TIMEOUT);
                timeout = !drained;  // true: leave the barriers as they are
            }
            __syncthreads();
            if (tid == 0 && !timeout)
                for (int q = 0; q < kArgNST; ++q) mbar_inval(&full[q]);
            return;
        }
        if (tid == 0) {
            int best = s_i[0];
#pragma unroll
            for (int q = 1; q < kArgNT / 32; ++q) best = min(best, s_i[q]);
            if (best != INT_MAX) atomicMax(p.keys + it.row, argmax_key(M, best));
            if (item + kArgNST * G < n_items) arg_issue<T>(p, R, full, item + kArgNST * G, s);
        }
    }
    __syncthreads();
    if (tid == 0)
        for (int s = 0; s < kArgNST; ++s) mbar_inval(&full[s]);
}

// One block per request: the chain decision or the tree decision.
constexpr int kDecideNT = 128;
__global__ void __launch_bounds__(kDecideNT) argmax_decide_kernel(ArgmaxParams p) {
    const int b = blockIdx.x;
    if (p.mode == 0) {
        if (threadIdx.x < 32) greedy_chain_decide(p, b);
    } else {
        tree_epilogue(p, b);
    }
}

cudaError_t launch_argmax_verify(const ArgmaxParams &p, int dtype, int n_rows, int sms, cudaStream_t s) {
    const int64_t items = (int64_t)n_rows * p.slices;
    const int64_t cap = (int64_t)sms * kArgBlocksPerSM;
    const dim3 grid((unsigned)(items < cap ? items : cap));
    const int smem = (int)sizeof(ArgRingN);
    cudaError_t e;
    if (dtype == SPEC_DTYPE_BF16) {
        static std::atomic<unsigned long long> done{0};
        e = ensure_smem_attr(argmax_pass_kernel<__nv_bfloat16>, smem, done);
        if (e != cudaSuccess) return e;
        argmax_pass_kernel<__nv_bfloat16><<<grid, kArgNT, smem, s>>>(p, (int)items);
    } else {
        static std::atomic<unsigned long long> done{0};
        e = ensure_smem_attr(argmax_pass_kernel<float>, smem, done);
        if (e != cudaSuccess) return e;
        argmax_pass_kernel<float><<<grid, kArgNT, smem, s>>>(p, (int)items);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(n_rows / p.rows_per_req));
    cfg.blockDim = dim3(kDecideNT);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, argmax_decide_kernel, p);
}

}  // namespace specv
