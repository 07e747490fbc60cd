// Sampled chain verification with top-k (k <= 128) on sm_103a, without
// thread-block clusters.
//
// The transform ("KV Cache 优化（四）：Speculative Decoding 投机解码" §4) keeps
// every logit >= the row's k-th largest; everything after that works on the
// few kept tokens.  So each (position, slice) block only has to hand on a
// short candidate list:
//
//  1. stage the slice of target row k and draft row k in shared memory with
//     two bulk copies (<= 32 KiB each);
//  2. every thread takes the largest logit it holds; the k-th largest of
//     these per-thread maxima is a lower bound of the slice's k-th largest
//     (k distinct logits reach it), and for spread-out logits a tight one;
//  3. append every logit >= that bound (order key, token id) to the
//     position's pool in the workspace (one atomicAdd per row per block);
//  4. the block that arrives last for the position (arrival counter) loads
//     the pool, finds the exact threshold, and computes acceptance, residual
//     mass and, where this position decides the token, the double-float
//     draw over the kept sets (compact_position).
//
// If a pool would overflow (a slice with hundreds of tied logits) or the two
// rows' 16-byte phases differ, the last block instead runs the exact masked
// computation over the whole row by itself (slow, exact, rare).  Blocks
// never wait on one another; a block that is not last exits right after its
// append, so no block holds resources while others finish.
#include "sample_common.cuh"

namespace specv {

template <typename T>
__global__ void __launch_bounds__(kNT) chain_topk_kernel(SampleParams p) {
    constexpr int VEC = Elem<T>::VEC;
    constexpr int KB = Elem<T>::KEY_BITS;
    __shared__ SampBase sb;
    __shared__ uint2 s_list[2][kSeg];
    __shared__ int s_n[2], s_base[2], s_last;
    extern __shared__ __align__(128) unsigned char dsm[];
    const int tid = threadIdx.x;
    for (int i = tid; i < 65; i += kNT) sb.tab[i] = p.exptab.tab[i];
    if (tid == 0) {
        sb.ln2 = p.exptab.ln2;
        s_n[0] = s_n[1] = 0;
    }

    const int c = p.c;
    const int j = blockIdx.x % c;
    const int qpos = blockIdx.x / c;
    const int g = p.gamma;
    const int k = qpos / p.B, b = qpos % p.B;  // position-major
    const int pos = b * (g + 1) + k;           // record / pool index
    const bool has_draft = k < g;
    const int rows = has_draft ? 2 : 1;
    const int lo = min(p.V, j * p.Vs), hi = min(p.V, lo + p.Vs);
    const T *trow = reinterpret_cast<const T *>(p.target) + (int64_t)(b * (g + 1) + k) * p.tstride;
    const T *drow = has_draft
        ? reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + k) * p.dstride : nullptr;
    const int K = p.top_k;

    const SliceSplit sp = split_slice(trow, lo, hi);
    const bool same = !has_draft ||
        ((reinterpret_cast<uintptr_t>(trow + lo) ^ reinterpret_cast<uintptr_t>(drow + lo)) & 15u) == 0;
    const int nhead = sp.body0 - sp.head0, ntail = sp.hi - sp.tail0, nbody = sp.tail0 - sp.body0;
    bool ovf = !same || (int64_t)nbody * (int64_t)sizeof(T) > kFastStage;
    __syncthreads();
    if (!ovf) {
        FastRing &FR = *reinterpret_cast<FastRing *>(dsm);
        float xh[2] = {-INFINITY, -INFINITY}, xt[2] = {-INFINITY, -INFINITY};
        for (int r = 0; r < rows; ++r) {
            const T *row = r == 0 ? trow : drow;
            if (tid < nhead) xh[r] = ld_elem(row, sp.head0 + tid);
            if (tid < ntail) xt[r] = ld_elem(row, sp.tail0 + tid);
        }
        if (nbody > 0) {
            const unsigned char *src[2] = {reinterpret_cast<const unsigned char *>(trow + sp.body0),
                                           has_draft ? reinterpret_cast<const unsigned char *>(drow + sp.body0)
                                                     : nullptr};
            const bool okc = ring_stream(FR, src, rows, (uint32_t)(nbody * (int)sizeof(T)),
                                         [](const unsigned char *const *, uint32_t, uint32_t) {});
            if (!okc && tid == 0) atomicOr(p.status, SPEC_FLAG_TIMEOUT);
        }
        const int nvec = nbody / VEC;
        const int total = hi - lo;
        for (int r = 0; r < rows; ++r) {
            const uint4 *v = reinterpret_cast<const uint4 *>(FR.buf[0][r]);
            float m = fmaxf(xh[r], xt[r]);
            const bool holds = tid < nhead || tid < ntail || tid < nvec;
            for (int q = tid; q < nvec; q += kNT) {
                float x[VEC];
                unpack<T>(v[q], x);
#pragma unroll
                for (int e = 0; e < VEC; ++e) m = fmaxf(m, x[e]);
            }
            const unsigned nthr = block_sum_u<kNT>(holds ? 1u : 0u, sb.redu);
            float t0 = -INFINITY;
            if (total > K && nthr >= (unsigned)K) {
                const uint32_t th = block_kth_largest<KB, kNT>(
                    [&](auto &&f) { if (holds) f(kkey<T>(m)); }, (unsigned)K, sb.hist, sb.bc);
                t0 = key_value<T>(th);
            }
            auto put = [&](float x, int idx) {
                const int at = atomicAdd(&s_n[r], 1);
                if (at < kSeg) s_list[r][at] = make_uint2(kkey<T>(x), (uint32_t)idx);
            };
            if (tid < nhead && xh[r] >= t0) put(xh[r], sp.head0 + tid);
            for (int q = tid; q < nvec; q += kNT) {
                float x[VEC];
                unpack<T>(v[q], x);
                float vm = x[0];
#pragma unroll
                for (int e = 1; e < VEC; ++e) vm = fmaxf(vm, x[e]);
                if (vm >= t0) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        if (x[e] >= t0) put(x[e], sp.body0 + q * VEC + e);
                }
            }
            if (tid < ntail && xt[r] >= t0) put(xt[r], sp.tail0 + tid);
        }
    }
    __syncthreads();
    // append to the position's pool (an overflowing slice poisons the count)
    unsigned *cnt = p.poolcnt + (int64_t)pos * 2;
    uint2 *pool = p.pool + (int64_t)pos * 2 * kPool;
    if (tid < rows) {
        const int n = s_n[tid];
        const unsigned add = (ovf || n > kSeg) ? (unsigned)(kPool + 1) : (unsigned)n;
        s_base[tid] = (int)atomicAdd(cnt + tid, add);
    }
    __syncthreads();
    for (int r = 0; r < rows; ++r) {
        const int n = min(s_n[r], kSeg);
        if (!ovf && s_base[r] + n <= kPool)
            for (int x = tid; x < n; x += kNT) pool[(int64_t)r * kPool + s_base[r] + x] = s_list[r][x];
    }
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(p.poscnt + pos, 1u) == (unsigned)(c - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- the last block of the position ----
    int n[2];
    n[0] = (int)__ldcg(cnt);
    n[1] = has_draft ? (int)__ldcg(cnt + 1) : 0;
    __syncthreads();
    if (tid == 0) {
        cnt[0] = 0u;
        cnt[1] = 0u;
        p.poscnt[pos] = 0u;
    }
    SoloEx solo;
    if (n[0] > kPool || n[1] > kPool) {
        masked_position<T, true>(p, sb, dsm, solo, k, b, 0, p.V);
        return;
    }
    uint2 *lists_sm = reinterpret_cast<uint2 *>(dsm);
    for (int r = 0; r < rows; ++r)
        for (int x = tid; x < n[r]; x += kNT)
            lists_sm[r * kPool + x] = __ldcg(&pool[(int64_t)r * kPool + x]);  // L2, not a stale L1 line
    __syncthreads();
    const uint2 *lists[2] = {lists_sm, lists_sm + kPool};
    compact_position<T>(p, sb, lists, n, lists_sm + 2 * kPool, dsm, solo, k, b);
}

static_assert((2 * kPool + 3 * kKeptMax) * sizeof(uint2) <= kSampDyn, "merge area fits");

size_t topk_pool_bytes_per_position() { return 2 * kPool * sizeof(uint2); }

cudaError_t launch_chain_topk(const SampleParams &p, int dtype, cudaStream_t s) {
    const dim3 grid((unsigned)((int64_t)p.B * (p.gamma + 1) * p.c));
    const int smem = (int)kSampDyn;
    cudaError_t e;
    if (dtype == SPEC_DTYPE_BF16) {
        static std::atomic<unsigned long long> done{0};
        e = ensure_smem_attr(chain_topk_kernel<__nv_bfloat16>, smem, done);
        if (e != cudaSuccess) return e;
        chain_topk_kernel<__nv_bfloat16><<<grid, kNT, smem, s>>>(p);
    } else {
        static std::atomic<unsigned long long> done{0};
        e = ensure_smem_attr(chain_topk_kernel<float>, smem, done);
        if (e != cudaSuccess) return e;
        chain_topk_kernel<float><<<grid, kNT, smem, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace specv
