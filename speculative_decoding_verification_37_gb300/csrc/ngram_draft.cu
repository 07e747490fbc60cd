// N-gram (prompt-lookup) drafts on sm_103a.
//
// "10.6 投机解码：为什么“先猜后验”能加速" §10.6.3 (model-free drafts: a segment
// of the prompt or the generated text equal to the trailing n-gram, and the
// tokens after it) and "KV Cache 优化（四）：Speculative Decoding 投机解码"
// §10.2.  For each end position e of an earlier window (e <= L-2), the
// backward match length l(e) = the largest k <= n_max with h[e-k+1..e] ==
// h[L-k..L-1].  The answer is the window with the largest min(l(e), n_max) >=
// n_min and, among those, the largest e: the longest n-gram, its most recent
// occurrence.  The draft is h[e+1 .. e+1+gamma), clipped at L.
//
// One block per request: the trailing n_max tokens go to shared memory, each
// thread scans 16 end positions per step with four 16-byte loads in flight
// (rows on 16-byte boundaries; others one token at a time), almost every
// comparison fails at the first token, and the block takes the largest 64-bit
// key (l << 32 | e).  A row is read once: the kernel is an HBM scan of the
// histories.
#include "common.cuh"
#include "spec_verify.h"

namespace specv {

constexpr int kNgThreads = 256;
constexpr int kNgMaxN = 64;

__global__ void __launch_bounds__(kNgThreads) ngram_draft_kernel(SpecNgramArgs a, bool vec16) {
    __shared__ int32_t suf[kNgMaxN];  // suf[k] = h[L-1-k]
    __shared__ unsigned long long red[kNgThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int32_t *h = a.history + (int64_t)b * a.history_stride;
    const int L = a.hist_len[b];
    if (L < 0 || (int64_t)L > a.history_stride) {  // block-uniform
        for (int t = tid; t < a.gamma; t += kNgThreads) a.draft_tokens[(int64_t)b * a.gamma + t] = -1;
        if (tid == 0) {
            a.n_draft[b] = 0;
            if (a.match_n) a.match_n[b] = 0;
            if (a.match_start) a.match_start[b] = -1;
            if (a.flags) a.flags[b] = SPEC_FLAG_BAD_INPUT;
        }
        return;
    }
    const int ns = min(a.n_max, L);
    for (int k = tid; k < ns; k += kNgThreads) suf[k] = h[L - 1 - k];
    __syncthreads();
    const int nmax = a.n_max, nmin = a.n_min;
    unsigned long long best = 0ull;
    // the backward match at end position e (almost always 0: the first
    // comparison fails); the rest of the match is read from global memory
    auto extend = [&](int e, int32_t he) {
        if (he != suf[0]) return;
        int l = 1;
        while (l < nmax && l <= e && h[e - l] == suf[l]) ++l;
        if (l >= nmin) best = max(best, ((unsigned long long)l << 32) | (unsigned)e);
    };
    if (vec16) {
        // 16 tokens per thread per step, four 16-byte loads in flight (eight
        // measured slower)
        constexpr int U = 4;
        const int4 *h4 = reinterpret_cast<const int4 *>(h);
        const int nv = L / 4;  // whole vectors (the last L % 4 tokens below)
        for (int v0 = 0; v0 < nv; v0 += U * kNgThreads) {
            int4 x[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = v0 + u * kNgThreads + tid;
                x[u] = q < nv ? __ldg(h4 + q) : make_int4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int q = v0 + u * kNgThreads + tid;
                if (q >= nv) continue;  // the partial vector is the scalar tail's
                const int e0 = 4 * q;
                if (e0 + 3 <= L - 2) {
                    extend(e0, x[u].x);
                    extend(e0 + 1, x[u].y);
                    extend(e0 + 2, x[u].z);
                    extend(e0 + 3, x[u].w);
                } else if (e0 <= L - 2) {
                    const int32_t xs[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                    for (int k = 0; k < 4 && e0 + k <= L - 2; ++k) extend(e0 + k, xs[k]);
                }
            }
        }
        for (int e = 4 * nv + tid; e <= L - 2; e += kNgThreads) extend(e, h[e]);
    } else {
        for (int e = tid; e <= L - 2; e += kNgThreads) extend(e, h[e]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(kFull, best, o));
    if (lane == 0) red[wid] = best;
    __syncthreads();
    if (wid == 0) {
        best = lane < kNgThreads / 32 ? red[lane] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(kFull, best, o));
        if (lane == 0) red[0] = best;
    }
    __syncthreads();
    best = red[0];
    const int n = (int)(best >> 32), e = (int)(best & 0xffffffffull);
    const int first = e + 1;
    const int cnt = best ? min(a.gamma, L - first) : 0;
    for (int t = tid; t < a.gamma; t += kNgThreads)
        a.draft_tokens[(int64_t)b * a.gamma + t] = t < cnt ? h[first + t] : -1;
    if (tid == 0) {
        a.n_draft[b] = cnt;
        if (a.match_n) a.match_n[b] = best ? n : 0;
        if (a.match_start) a.match_start[b] = best ? e - n + 1 : -1;
        if (a.flags) a.flags[b] = 0u;
    }
}

}  // namespace specv

extern "C" int spec_ngram_draft(const SpecNgramArgs *a, void *stream) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->B < 0 || a->gamma < 0 || a->n_min < 1 || a->n_max < a->n_min || a->n_max > specv::kNgMaxN ||
        a->history_stride < 1)
        return SPEC_ERR_INVALID_ARG;
    if (a->B == 0) return SPEC_OK;
    if (!a->history || !a->hist_len || !a->n_draft || (a->gamma > 0 && !a->draft_tokens))
        return SPEC_ERR_INVALID_ARG;
    // rows on 16-byte boundaries take the vector loads
    const bool vec16 = (reinterpret_cast<uintptr_t>(a->history) % 16 == 0) && (a->history_stride % 4 == 0);
    specv::ngram_draft_kernel<<<(unsigned)a->B, specv::kNgThreads, 0, static_cast<cudaStream_t>(stream)>>>(*a, vec16);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}
