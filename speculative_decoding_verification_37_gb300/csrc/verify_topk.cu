// Sampled chain verification with top-k (k <= 128) on sm_103a: one block per
// logits row, in one kernel.
//
// The transform ("KV Cache 优化（四）：Speculative Decoding 投机解码" §4) keeps
// every logit >= the row's k-th largest, so after one pass over a row only a
// handful of its logits matter; the acceptance test, the residual mass and
// the draw ("10.6 投机解码：为什么“先猜后验”能加速" §10.6.1) then work on the
// two kept sets of a position.
//
// chain_topk_row_kernel: a persistent grid of a few blocks per SM; block i
// takes rows i, i + grid, ... (target row (b,k) and draft row (b,k) of each
// position are neighbours, positions in order).  For its row a block
//  1. streams the 16-byte-aligned body through a ring of shared-memory stages
//     (thread 0 issues one cp.async.bulk per 16 KiB chunk with an evict-first
//     L2 policy, completing on the stage's mbarrier, waits bounded); the
//     scalar head and tail come from plain loads;
//  2. keeps theta, a lower bound of the row's k-th largest logit: from the
//     first chunk, the k-th largest of the threads' maxima (each is a logit,
//     so at least k logits reach it); later, the k-th largest of the listed
//     candidates.  Each thread takes the largest element of each of its
//     16-byte vectors (packed bf16x2 maxima); only vectors reaching theta
//     have their elements listed (order key, token id) in a shared-memory
//     candidate buffer.  One block barrier per chunk gives every warp its
//     offset; when the buffer passes a soft limit one warp compacts it to
//     the entries >= its k-th largest (theta rises); if a chunk would not fit,
//     the chunk's own k-th largest (a block radix search over its elements in
//     registers) raises theta first;
//  3. takes the exact threshold (the k-th largest candidate), the kept set in
//     token order, its maximum and double-float normaliser (and the nucleus
//     when top_p is set), and publishes them to the workspace;
//  4. arrives on its position's counter: the block that arrives second (the
//     bonus position has one row) loads the other row's kept set and decides
//     the position with one warp: a_k = min(1, p(d)/q(d)), the residual mass
//     over the target's kept set (q looked up in the draft's), and the draw
//     where this position decides the token, by a double-float warp scan in
//     token order; finish() records it and the last position of a request
//     writes the request's outputs.
// A row whose candidates do not fit (hundreds of logits tied at the
// threshold) sends its position to the exact masked computation over both
// rows in the deciding block, the nucleus included (slow, exact, rare).
#include "sample_common.cuh"

namespace specv {

constexpr int kRkCH = 16384;              // bytes of a row's body per ring stage
constexpr int kRkNST = 3;                 // ring stages
constexpr int kRkCap = 512;               // candidate entries a row can hold
constexpr int kRkSoft = 320;              // more than this after a chunk: compact
constexpr int kRkBlocksPerSM = 4;
constexpr int kRkVec = kRkCH / 16 / kNT;  // 16-byte vectors per thread and chunk
static_assert(kRkVec * 16 * kNT == kRkCH, "a chunk is whole vectors per thread");
static_assert(kRkVec * 8 <= 32, "a thread's hit bits fit one word");

struct RkRing {
    alignas(128) unsigned char buf[kRkNST][kRkCH];
};
using RkFallbackRing = Ring<8192, 2, 2>;  // the exact masked path's ring
constexpr size_t kRkRingBytes = sizeof(RkRing) > sizeof(RkFallbackRing) ? sizeof(RkRing) : sizeof(RkFallbackRing);
constexpr size_t kRkDyn = kRkRingBytes + kRkCap * sizeof(uint2);

// Decision-time arrays, in the ring's memory (no copy is in flight then).
struct RkDecide {
    uint2 kept[2][kKeptMax];     // target / draft kept set, token order
    float2 wp[2][kKeptMax];      // per kept target entry: p (or the bonus term) and residual weight
    uint2 tmp[kKeptMax];         // unsorted kept entries; top-p: entries by rank
    float2 prb[kKeptMax];        // top-p: probabilities by rank
    unsigned kn[2], th[2], flags[2];
    float m[2];
    float2 S[2];
};
static_assert(sizeof(RkDecide) <= sizeof(RkRing), "decision arrays fit the ring");

constexpr unsigned RK_OVERFLOW = 1u;  // the row's candidates or kept set did not fit

int topk_row_bytes() { return kRkCH; }

// largest element of a 16-byte vector (bf16: packed maxima)
template <typename T> __device__ __forceinline__ float vec_max(const uint4 &v);
template <> __device__ __forceinline__ float vec_max<float>(const uint4 &v) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) {
    __nv_bfloat162 r;
    memcpy(&r, &w, 4);
    return r;
}
template <> __device__ __forceinline__ float vec_max<__nv_bfloat16>(const uint4 &v) {
    const __nv_bfloat162 a = __hmax2(__hmax2(as_bf2(v.x), as_bf2(v.y)), __hmax2(as_bf2(v.z), as_bf2(v.w)));
    return fmaxf(__low2float(a), __high2float(a));
}

// bit e set iff element e of the vector is >= t (t a value of type T)
template <typename T> __device__ __forceinline__ uint32_t vec_ge_mask(const uint4 &v, float t);
template <> __device__ __forceinline__ uint32_t vec_ge_mask<float>(const uint4 &v, float t) {
    return (uint32_t)(__uint_as_float(v.x) >= t) | ((uint32_t)(__uint_as_float(v.y) >= t) << 1) |
           ((uint32_t)(__uint_as_float(v.z) >= t) << 2) | ((uint32_t)(__uint_as_float(v.w) >= t) << 3);
}
template <> __device__ __forceinline__ uint32_t vec_ge_mask<__nv_bfloat16>(const uint4 &v, float t) {
    const __nv_bfloat162 t2 = __float2bfloat162_rn(t);  // exact: t is a bf16 value or -inf
    auto two = [](uint32_t m) { return (m & 1u) | ((m >> 15) & 2u); };
    return two(__hge2_mask(as_bf2(v.x), t2)) | (two(__hge2_mask(as_bf2(v.y), t2)) << 2) |
           (two(__hge2_mask(as_bf2(v.z), t2)) << 4) | (two(__hge2_mask(as_bf2(v.w), t2)) << 6);
}


// element e of a 16-byte vector
template <typename T> __device__ __forceinline__ float vec_elem(const uint4 &v, int e);
template <> __device__ __forceinline__ float vec_elem<float>(const uint4 &v, int e) {
    const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    return __uint_as_float(w);
}
template <> __device__ __forceinline__ float vec_elem<__nv_bfloat16>(const uint4 &v, int e) {
    const int q = e >> 1;
    const uint32_t w = q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
}


// warp-level dd exclusive prefix over lanes (lane order)
__device__ __forceinline__ dd warp_dd_excl_scan(dd v) {
    const int lane = threadIdx.x & 31;
    dd incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const dd y{__shfl_up_sync(kFull, incl.hi, o), __shfl_up_sync(kFull, incl.lo, o)};
        if (lane >= o) incl = dd_add(y, incl);
    }
    dd ex{__shfl_up_sync(kFull, incl.hi, 1), __shfl_up_sync(kFull, incl.lo, 1)};
    if (lane == 0) ex = dd{0.0f, 0.0f};
    return ex;
}

// the smallest finite value of the element type (-inf is never listed: its
// probability is 0 whatever the threshold)
template <typename T> __device__ __forceinline__ float lowest_finite();
template <> __device__ __forceinline__ float lowest_finite<float>() { return -3.40282347e38f; }
template <> __device__ __forceinline__ float lowest_finite<__nv_bfloat16>() { return __uint_as_float(0xff7f0000u); }

// The K-th largest order key among the finite elements the block holds in
// registers (each thread: its vectors v[i] whose slot is < nv, and in the
// first chunk its head/tail scalars), by a 2-bit radix descent with block
// counts; 0 if fewer than K.  Every thread gets it.  All threads call it.
template <typename T>
__device__ __forceinline__ uint32_t block_kth_chunk(const uint4 *v, int nv, float xh, float xt, unsigned K,
                                    unsigned (*red)[3][kNW]) {
    constexpr int VEC = Elem<T>::VEC;
    constexpr int KB = Elem<T>::KEY_BITS;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    uint32_t res = 0u;
    auto cnt = [&](float x, uint32_t c) -> unsigned { return (x > -INFINITY && kkey<T>(x) >= c) ? 1u : 0u; };
    int par = 0;
    for (int bit = KB - 2; bit >= 0; bit -= 2, par ^= 1) {
        const uint32_t c1 = res | (1u << bit), c2 = res | (2u << bit), c3 = res | (3u << bit);
        unsigned n1 = cnt(xh, c1) + cnt(xt, c1), n2 = cnt(xh, c2) + cnt(xt, c2), n3 = cnt(xh, c3) + cnt(xt, c3);
#pragma unroll
        for (int i = 0; i < kRkVec; ++i) {
            if (tid + i * kNT >= nv) continue;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const float x = vec_elem<T>(v[i], e);
                n1 += cnt(x, c1);
                n2 += cnt(x, c2);
                n3 += cnt(x, c3);
            }
        }
        n1 = __reduce_add_sync(kFull, n1);
        n2 = __reduce_add_sync(kFull, n2);
        n3 = __reduce_add_sync(kFull, n3);
        if (lane == 0) {
            red[par][0][wid] = n1;
            red[par][1][wid] = n2;
            red[par][2][wid] = n3;
        }
        __syncthreads();
        unsigned t1 = 0, t2 = 0, t3 = 0;
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
            t1 += red[par][0][w];
            t2 += red[par][1][w];
            t3 += red[par][2][w];
        }
        res |= (t3 >= K ? 3u : t2 >= K ? 2u : t1 >= K ? 1u : 0u) << bit;
    }
    return res;
}

// ---------------------------------------------------------------------------
// Block-wide helpers.  Everything after a row's stream runs on the whole
// block: one dependent warp would share its SM sub-partition with the other
// resident blocks' warps and run several times slower.
// ---------------------------------------------------------------------------
struct RkRed {
    unsigned u[2][kNW];
    float2 f[2][kNW];
};

// block max / min of one value per thread (every thread gets it)
__device__ __forceinline__ uint32_t block_max_u(uint32_t v, unsigned *red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    v = __reduce_max_sync(kFull, v);
    if (lane == 0) red[wid] = v;
    __syncthreads();
    uint32_t t = 0u;
#pragma unroll
    for (int w = 0; w < kNW; ++w) t = max(t, red[w]);
    __syncthreads();
    return t;
}
__device__ __forceinline__ uint32_t block_min_u(uint32_t v, unsigned *red) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    v = __reduce_min_sync(kFull, v);
    if (lane == 0) red[wid] = v;
    __syncthreads();
    uint32_t t = 0xffffffffu;
#pragma unroll
    for (int w = 0; w < kNW; ++w) t = min(t, red[w]);
    __syncthreads();
    return t;
}

// The K-th largest of the keys every thread passes (k0, and k1 when TWO;
// key 0 means "no key"): the largest r such that at least K keys are >= r,
// 0 if there are fewer than K keys.  Bits are fixed from the top, below the
// common prefix of the smallest and largest key, with one block count
// (__syncthreads_count) per bit.  Every thread calls it and gets the result.
template <bool TWO>
__device__ uint32_t block_kth(uint32_t k0, uint32_t k1, unsigned K, RkRed &rd) {
    const unsigned have = (unsigned)__syncthreads_count(k0 != 0u) + (TWO ? (unsigned)__syncthreads_count(k1 != 0u) : 0u);
    if (have < K) return 0u;
    const uint32_t hi = block_max_u(TWO ? max(k0, k1) : k0, rd.u[0]);
    const uint32_t lo = block_min_u(TWO ? min(k0 ? k0 : 0xffffffffu, k1 ? k1 : 0xffffffffu)
                                        : (k0 ? k0 : 0xffffffffu), rd.u[1]);
    if (lo >= hi) return hi;
    const int nb = 32 - __clz(lo ^ hi);
    uint32_t res = nb == 32 ? 0u : (hi >> nb) << nb;  // <= lo: every key reaches it
    for (int bit = nb - 1; bit >= 0; --bit) {
        const uint32_t c = res | (1u << bit);
        unsigned n = (unsigned)__syncthreads_count(k0 >= c);
        if (TWO) n += (unsigned)__syncthreads_count(k1 >= c);
        if (n >= K) res = c;
    }
    return res;
}

// Writes the flagged entries (up to two per thread) to dst in thread order,
// keeping at most `cap`; returns how many were flagged.  Every thread calls
// it; the entries must already be in registers (dst may be their source).
__device__ __forceinline__ int block_compact2(uint2 *dst, int cap, uint2 e0, bool f0, uint2 e1, bool f1, RkRed &rd) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const unsigned lt = lanemask_lt();
    const unsigned b0 = __ballot_sync(kFull, f0), b1 = __ballot_sync(kFull, f1);
    if (lane == 0) rd.u[0][wid] = (unsigned)(__popc(b0) + __popc(b1));
    __syncthreads();  // (also: every thread has read its entries)
    unsigned base = 0u, tot = 0u;
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
        const unsigned c = rd.u[0][w];
        base += w < wid ? c : 0u;
        tot += c;
    }
    const unsigned p0 = base + (unsigned)__popc(b0 & lt);
    const unsigned p1 = base + (unsigned)__popc(b0) + (unsigned)__popc(b1 & lt);
    if (f0 && p0 < (unsigned)cap) dst[p0] = e0;
    if (f1 && p1 < (unsigned)cap) dst[p1] = e1;
    __syncthreads();
    return (int)tot;
}

// block dd sum of one term per thread, in a fixed order (every thread gets it)
__device__ __forceinline__ dd block_dd_sum(dd v, RkRed &rd) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    v = warp_dd_sum(v);
    if (lane == 0) rd.f[0][wid] = make_float2(v.hi, v.lo);
    __syncthreads();
    dd t{0.0f, 0.0f};
#pragma unroll
    for (int w = 0; w < kNW; ++w) t = dd_add(t, dd{rd.f[0][w].x, rd.f[0][w].y});
    __syncthreads();
    return t;
}

// block inclusive dd prefix over threads in thread order
__device__ __forceinline__ dd block_dd_incl_scan(dd v, RkRed &rd) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    dd incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const dd y{__shfl_up_sync(kFull, incl.hi, o), __shfl_up_sync(kFull, incl.lo, o)};
        if (lane >= o) incl = dd_add(y, incl);
    }
    if (lane == 31) rd.f[1][wid] = make_float2(incl.hi, incl.lo);
    __syncthreads();
    dd pre{0.0f, 0.0f};
    for (int w = 0; w < wid; ++w) pre = dd_add(pre, dd{rd.f[1][w].x, rd.f[1][w].y});
    __syncthreads();
    return dd_add(pre, incl);
}

// One warp: the nucleus of a row's kept set (token order in `kept`): the
// entries by probability (larger key first, then the lower token), the first
// rank whose cumulative probability reaches top_p, every entry at or above
// that rank's key kept (ties kept), still in token order; the row's sum is
// taken again over them.  Updates kn, th and S.
template <typename T>
__device__ __noinline__ void row_top_p(uint2 *kept, int &kn, uint32_t &th, float m, dd &S, float top_p, uint2 *srt,
                          float2 *prb, const DdExpTables &EK) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = lanemask_lt();
    const dd iS = dd_recip(S);
    for (int x = lane; x < kn; x += 32) {
        const uint2 e = kept[x];
        int rank = 0;
        for (int y = 0; y < kn; ++y) {
            const uint2 f = kept[y];
            rank += f.x > e.x || (f.x == e.x && f.y < e.y);
        }
        srt[rank] = e;
        const dd pe = dd_mul(dd_expw(key_value<T>(e.x), m, EK), iS);
        prb[rank] = make_float2(pe.hi, pe.lo);
    }
    __syncwarp();
    const int E = (kn + 31) / 32, i0 = lane * E, i1 = min(kn, i0 + E);
    dd part{0.0f, 0.0f};
    for (int i = i0; i < i1; ++i) part = dd_add(part, dd{prb[i].x, prb[i].y});
    dd cum = warp_dd_excl_scan(part);
    const dd tp{top_p, 0.0f};
    int cut = INT_MAX;
    for (int i = i0; i < i1; ++i) {
        cum = dd_add(cum, dd{prb[i].x, prb[i].y});
        if (!dd_gt(tp, cum)) {  // cumulative probability >= top_p
            cut = i;
            break;
        }
    }
    cut = (int)__reduce_min_sync(kFull, (unsigned)cut);
    if (cut == INT_MAX) cut = kn - 1;  // rounding left the total below top_p
    const uint32_t kstar = srt[cut].x;
    int nn = 0;
    for (int x0 = 0; x0 < kn; x0 += 32) {
        const int x = x0 + lane;
        const uint2 e = x < kn ? kept[x] : make_uint2(0u, 0u);
        const bool keep = x < kn && e.x >= kstar;
        const unsigned bal = __ballot_sync(kFull, keep);
        __syncwarp();  // every lane has read its entry before any is moved
        if (keep) kept[nn + __popc(bal & lt)] = e;
        nn += __popc(bal);
    }
    __syncwarp();
    kn = nn;
    th = kstar;
    S = dd{0.0f, 0.0f};
#pragma unroll 1
    for (int x = lane; x < kn; x += 32) S = dd_add(S, dd_expw(key_value<T>(kept[x].x), m, EK));
    S = warp_dd_sum(S);
}

// The outcome of position k of request b from the two kept sets (token
// order, one entry per thread) and their row statistics: acceptance, the
// residual mass, and the draw where this position decides the emitted
// token, by a block dd prefix in token order.  Every thread calls it; the
// result is the same in every thread.
template <typename T>
__device__ __noinline__ Outcome block_outcome(const SampleParams &p, int b, int k, RkDecide &D, const DdExpTables &EK,
                                              RkRed &rd, unsigned *s_rej) {
    const int tid = threadIdx.x;
    const int g = p.gamma;
    const bool has_draft = k < g;
    const int pos = b * (g + 1) + k;
    const T *trow = reinterpret_cast<const T *>(p.target) + (int64_t)pos * p.tstride;
    const T *drow = has_draft ? reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + k) * p.dstride : nullptr;
    const int d = has_draft ? p.tokens[(int64_t)b * g + k] : 0;
    const bool bad_tok = has_draft && (d < 0 || d >= p.V);
    const float l_d = (has_draft && !bad_tok) ? ld_elem(trow, d) : 0.0f;
    const float g_d = (has_draft && !bad_tok) ? ld_elem(drow, d) : 0.0f;
    const float u_k = has_draft ? p.unif[(int64_t)b * (g + 1) + k] : 0.0f;
    const float u_f = p.unif[(int64_t)b * (g + 1) + g];
    if (tid == 0) *s_rej = *((volatile unsigned *)&p.rejword[b]);  // one read, shared by the block
    const uint2 *Kp = D.kept[0], *Kq = D.kept[1];
    const int np = (int)D.kn[0], nq = has_draft ? (int)D.kn[1] : 0;
    const float mp = D.m[0], mq = has_draft ? D.m[1] : 0.0f;
    const dd sp{D.S[0].x, D.S[0].y};
    const dd sq = has_draft ? dd{D.S[1].x, D.S[1].y} : dd{0.0f, 0.0f};
    Outcome o{1.0f, 0.0f, -1, 0u};
    const bool bad_row = mp == -INFINITY || (has_draft && mq == -INFINITY);
    o.info = (bad_tok ? REC_BAD_INPUT : 0u) | (bad_row ? REC_BAD_ROW : 0u);
    __syncthreads();
    const unsigned rej = *s_rej;
    if (bad_tok || bad_row) return o;
    const dd isp = dd_recip(sp);
    const dd isq = has_draft ? dd_recip(sq) : dd{0.0f, 0.0f};
    bool accept = false;
    if (has_draft) {
        const dd pd = kkey<T>(l_d) >= D.th[0] ? dd_mul(dd_expw(l_d, mp, EK), isp) : dd{0.0f, 0.0f};
        const dd qd = kkey<T>(g_d) >= D.th[1] ? dd_mul(dd_expw(g_d, mq, EK), isq) : dd{0.0f, 0.0f};
        float a;
        if (dd_pos(qd)) {
            const dd ratio = dd_mul(pd, dd_recip(qd));
            a = dd_gt(ratio, dd{1.0f, 0.0f}) ? 1.0f : dd_to_f(ratio);
        } else {
            a = dd_pos(pd) ? 1.0f : 0.0f;
        }
        o.a = a;
        accept = u_k < a;
        o.info |= accept ? REC_ACCEPT : 0u;
    }
    // thread t: kept target entry t (token order), its p (the unnormalised
    // term for the bonus draw) and residual weight max(0, p - q)
    dd pi{0.0f, 0.0f}, w{0.0f, 0.0f};
    if (tid < np) {
        const dd ex = dd_expw(key_value<T>(Kp[tid].x), mp, EK);
        pi = ex;
        w = ex;
        if (has_draft) {
            pi = dd_mul(ex, isp);
            const uint32_t id = Kp[tid].y;
            int lo = 0, hi = nq;  // first draft kept entry with token >= id
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (Kq[mid].y < id) lo = mid + 1; else hi = mid;
            }
            const dd qi = (lo < nq && Kq[lo].y == id) ? dd_mul(dd_expw(key_value<T>(Kq[lo].x), mq, EK), isq)
                                                     : dd{0.0f, 0.0f};
            w = dd_max0(dd_add(pi, dd_neg(qi)));
        }
    }
    dd zw{0.0f, 0.0f}, zp{0.0f, 0.0f};
    if (has_draft) {
        zw = block_dd_sum(w, rd);
        zp = block_dd_sum(pi, rd);
        o.z = dd_to_f(zw);
    }
    const bool earlier = rej > (unsigned)(g - k + 1);
    if (has_draft && !accept && tid == 0) atomicMax(p.rejword + b, (unsigned)(g - k + 1));
    if ((!has_draft || !accept) && !earlier) {
        // ---- the draw: the first kept token whose running weight passes u * total ----
        const bool fb = has_draft && dd_le(zw, dd{p.eps, 0.0f});
        if (fb) o.info |= REC_FALLBACK;
        const dd wt = (!has_draft || fb) ? pi : w;
        const dd total = !has_draft ? sp : (fb ? zp : zw);
        const dd t = dd_mul_f(total, u_f);
        const dd cum = block_dd_incl_scan(wt, rd);
        const bool pos_w = tid < np && dd_pos(wt);
        const unsigned hit = block_min_u((pos_w && dd_gt(cum, t)) ? (unsigned)tid : 0xffffffffu, rd.u[0]);
        const unsigned lastp = block_max_u(pos_w ? (unsigned)tid + 1u : 0u, rd.u[1]);
        const int sel = hit != 0xffffffffu ? (int)hit : (int)lastp - 1;
        o.token = sel >= 0 ? (int)Kp[sel].y : -1;
    }
    return o;
}

// the exact masked computation of one position over both whole rows (rows
// whose kept set does not fit), out of line
template <typename T>
__device__ __noinline__ void rk_exact_position(const SampleParams &p, SampBase &sb, unsigned char *dsm, int k, int b) {
    SoloEx solo;
    masked_position<T, true, SoloEx, RkFallbackRing>(p, sb, dsm, solo, k, b, 0, p.V);
}

template <typename T>
__global__ void __launch_bounds__(kNT, kRkBlocksPerSM) chain_topk_row_kernel(SampleParams p) {
    constexpr int VEC = Elem<T>::VEC;
    constexpr int ECH = kRkCH / (int)sizeof(T);  // elements per chunk
    __shared__ SampBase sb;
    __shared__ __align__(8) unsigned long long full[kRkNST];
    __shared__ unsigned s_wcnt[3][kNW];
    __shared__ unsigned s_red[2][3][kNW];
    __shared__ RkRed rd;
    __shared__ unsigned s_last, s_rej;
    extern __shared__ __align__(128) unsigned char dsm[];
    RkRing &R = *reinterpret_cast<RkRing *>(dsm);
    RkDecide &D = *reinterpret_cast<RkDecide *>(dsm);
    uint2 *cand = reinterpret_cast<uint2 *>(dsm + kRkRingBytes);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const unsigned lt = lanemask_lt();
    const unsigned K = (unsigned)p.top_k;
    const int g = p.gamma, B = p.B;
    const int nrows = B * (2 * g + 1);
    const bool nucleus = p.top_p > 0.0f && p.top_p < 1.0f;
    load_exp_tables(p, sb);
    if (tid == 0) {
        for (int s = 0; s < kRkNST; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    const DdExpTables &EK = sb.K;
    const uint64_t pol = l2_evict_first();
    unsigned seq = 0;  // chunks this block has consumed: the ring stage and phase of the next

    for (int q = blockIdx.x; q < nrows; q += gridDim.x) {
        // row q: position-major, a position's target row then its draft row
        int k, b, r;
        if (q < 2 * B * g) {
            k = q / (2 * B);
            const int rem = q - k * 2 * B;
            b = rem >> 1;
            r = rem & 1;
        } else {
            k = g;
            b = q - 2 * B * g;
            r = 0;
        }
        const int pos = b * (g + 1) + k;
        const T *row = r == 0 ? reinterpret_cast<const T *>(p.target) + (int64_t)pos * p.tstride
                              : reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + k) * p.dstride;
        const SliceSplit sp = split_slice(row, 0, p.V);
        const uint32_t body = (uint32_t)(sp.tail0 - sp.body0) * (uint32_t)sizeof(T);
        const int nch = (int)((body + kRkCH - 1) / kRkCH);
        const unsigned char *src = reinterpret_cast<const unsigned char *>(row + sp.body0);
        auto issue = [&](int c) {  // thread 0: chunk c of this row into its stage
            const uint32_t off = (uint32_t)c * kRkCH;
            const uint32_t nb = min((uint32_t)kRkCH, body - off);
            const int s = (int)((seq + c) % kRkNST);
            mbar_arrive_expect_tx(&full[s], nb);
            bulk_g2s_policy(R.buf[s], src + off, nb, &full[s], pol);
        };
        int issued = 0;  // thread 0: chunks of this row issued
        if (tid == 0)
            for (; issued < kRkNST && issued < nch; ++issued) issue(issued);
        const int nhead = sp.body0 - sp.head0, ntail = sp.hi - sp.tail0;
        const float xh = tid < nhead ? ld_elem(row, sp.head0 + tid) : -INFINITY;
        const float xt = tid < ntail ? ld_elem(row, sp.tail0 + tid) : -INFINITY;

        uint32_t theta = 0u;  // order key of the running lower bound of the k-th largest
        int count = 0;        // candidates in the buffer
        bool ovf = false, tmo = false;
        int failed_at = -1;
        const int nwin = nch > 0 ? nch : 1;
        for (int w = 0; w < nwin; ++w) {
            const unsigned gq = seq + (unsigned)w;
            const int s = (int)(gq % kRkNST);
            uint4 v[kRkVec];
            int nv = 0;
            if (w < nch) {
                if (!mbar_wait_bounded(&full[s], (gq / kRkNST) & 1u)) tmo = true;
                nv = (int)(min((uint32_t)kRkCH, body - (uint32_t)w * kRkCH) / 16u);
                const uint4 *st = reinterpret_cast<const uint4 *>(R.buf[s]);
#pragma unroll
                for (int i = 0; i < kRkVec; ++i) {
                    const int qv = tid + i * kNT;
                    v[i] = qv < nv ? st[qv] : make_uint4(0u, 0u, 0u, 0u);
                }
            }
            float vm[kRkVec];
            float tm = w == 0 ? fmaxf(xh, xt) : -INFINITY;
#pragma unroll
            for (int i = 0; i < kRkVec; ++i) {
                vm[i] = tid + i * kNT < nv ? vec_max<T>(v[i]) : -INFINITY;
                tm = fmaxf(tm, vm[i]);
            }
            const int vbase = sp.body0 + w * ECH;  // element index of the chunk's first element
            if (w == 0)  // the k-th largest thread maximum: at least k logits reach it
                theta = block_kth<false>(tm > -INFINITY ? kkey<T>(tm) : 0u, 0u, K, rd);
            // the listed elements: hit bits (VEC per vector) and scalar flags
            uint32_t hm = 0u;
            bool hh = false, ht = false;
            auto tally = [&]() -> unsigned {
                hm = 0u;
                hh = ht = false;
                if (ovf) return 0u;
                const float tf = fmaxf(key_value<T>(theta), lowest_finite<T>());
                if (tm >= tf) {
#pragma unroll
                    for (int i = 0; i < kRkVec; ++i)
                        if (vm[i] >= tf) hm |= vec_ge_mask<T>(v[i], tf) << (VEC * i);
                    hh = xh >= tf && w == 0;
                    ht = xt >= tf && w == 0;
                }
                return (unsigned)__popc(hm) + (hh ? 1u : 0u) + (ht ? 1u : 0u);
            };
            unsigned n = tally();
            unsigned wt = __reduce_add_sync(kFull, n);
            if (lane == 0) s_wcnt[w & 1][wid] = wt;
            if (__syncthreads_or(tmo)) {  // block-uniform: a chunk did not arrive
                failed_at = w;
                break;
            }
            // every thread holds its share of the chunk: refill the stage
            if (tid == 0 && issued < nch) issue(issued++);
            unsigned tot = 0u, before = 0u;
#pragma unroll
            for (int x = 0; x < kNW; ++x) {
                const unsigned cw = s_wcnt[w & 1][x];
                tot += cw;
                before += x < wid ? cw : 0u;
            }
            if (count + (int)tot > kRkCap) {
                // the chunk does not fit: raise theta by the chunk's own k-th
                // largest element and the buffer's, compact, count again
                uint32_t th = block_kth_chunk<T>(v, nv, w == 0 ? xh : -INFINITY, w == 0 ? xt : -INFINITY, K, s_red);
                th = max(th, theta);
                const uint2 e0 = tid < count ? cand[tid] : make_uint2(0u, 0u);
                const uint2 e1 = tid + kNT < count ? cand[tid + kNT] : make_uint2(0u, 0u);
                if ((unsigned)count >= K) th = max(th, block_kth<true>(e0.x, e1.x, K, rd));
                count = block_compact2(cand, kRkCap, e0, e0.x != 0u && e0.x >= th, e1, e1.x != 0u && e1.x >= th, rd);
                theta = th;
                n = tally();
                wt = __reduce_add_sync(kFull, n);
                if (lane == 0) s_wcnt[2][wid] = wt;
                __syncthreads();
                tot = before = 0u;
#pragma unroll
                for (int x = 0; x < kNW; ++x) {
                    const unsigned cw = s_wcnt[2][x];
                    tot += cw;
                    before += x < wid ? cw : 0u;
                }
                if (count + (int)tot > kRkCap) ovf = true;  // block-uniform
            }
            if (!ovf && wt > 0u) {
                unsigned incl = n;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                unsigned at = (unsigned)count + before + incl - n;
#pragma unroll
                for (int i = 0; i < kRkVec; ++i) {
                    uint32_t h = (hm >> (VEC * i)) & ((1u << VEC) - 1u);
                    while (h) {
                        const int e = __ffs(h) - 1;
                        h &= h - 1u;
                        cand[at++] = make_uint2(kkey<T>(vec_elem<T>(v[i], e)),
                                                (uint32_t)(vbase + (tid + i * kNT) * VEC + e));
                    }
                }
                if (hh) cand[at++] = make_uint2(kkey<T>(xh), (uint32_t)(sp.head0 + tid));
                if (ht) cand[at++] = make_uint2(kkey<T>(xt), (uint32_t)(sp.tail0 + tid));
            }
            if (!ovf) count += (int)tot;
            if (!ovf && count > kRkSoft) {  // block-uniform
                __syncthreads();  // the chunk's entries are in the buffer
                const uint2 e0 = tid < count ? cand[tid] : make_uint2(0u, 0u);
                const uint2 e1 = tid + kNT < count ? cand[tid + kNT] : make_uint2(0u, 0u);
                const uint32_t th = max(theta, block_kth<true>(e0.x, e1.x, K, rd));
                count = block_compact2(cand, kRkCap, e0, e0.x != 0u && e0.x >= th, e1, e1.x != 0u && e1.x >= th, rd);
                theta = th;
            }
        }
        if (failed_at >= 0) {
            // A bulk copy did not complete in time: issue nothing more, wait
            // (bounded) for the copies already issued so that none lands in
            // shared memory after the block has moved on, flag the call and stop.
            if (tid == 0) {
                for (int c = failed_at; c < issued; ++c) {
                    const unsigned gq = seq + (unsigned)c;
                    for (int rep = 0; rep < 4; ++rep)
                        if (mbar_wait_bounded(&full[gq % kRkNST], (gq / kRkNST) & 1u)) break;
                }
                atomicOr(p.status, SPEC_FLAG_TIMEOUT);
            }
            return;
        }
        seq += (unsigned)nch;
        __syncthreads();  // the last chunk's entries are in the buffer; the ring is idle

        // ---- the row's kept set: the exact threshold, token order, statistics ----
        const int mine = r;
        {
            uint32_t th = 0u;
            int kn = 0;
            if (!ovf) {
                const uint2 e0 = tid < count ? cand[tid] : make_uint2(0u, 0u);
                const uint2 e1 = tid + kNT < count ? cand[tid + kNT] : make_uint2(0u, 0u);
                th = block_kth<true>(e0.x, e1.x, K, rd);  // 0 (keep all) with fewer than K candidates
                kn = block_compact2(D.tmp, kKeptMax, e0, e0.x != 0u && e0.x >= th, e1, e1.x != 0u && e1.x >= th, rd);
                if (kn > kKeptMax) ovf = true;  // block-uniform
            }
            float m = -INFINITY;
            dd S{0.0f, 0.0f};
            if (!ovf) {
                uint2 e = make_uint2(0u, 0u);
                if (tid < kn) {
                    e = D.tmp[tid];
                    int rank = 0;
                    for (int y = 0; y < kn; ++y) rank += D.tmp[y].y < e.y;
                    D.kept[mine][rank] = e;
                }
                const uint32_t mk = block_max_u(e.x, rd.u[0]);
                m = kn > 0 ? key_value<T>(mk) : -INFINITY;
                if (m != -INFINITY) {
                    S = block_dd_sum(tid < kn ? dd_expw(key_value<T>(e.x), m, EK) : dd{0.0f, 0.0f}, rd);
                    if (nucleus) {
                        if (wid == 0) {
                            row_top_p<T>(D.kept[mine], kn, th, m, S, p.top_p, D.tmp, D.prb, EK);
                            if (lane == 0) {
                                D.kn[mine] = (unsigned)kn;
                                D.th[mine] = th;
                                D.S[mine] = make_float2(S.hi, S.lo);
                            }
                        }
                        __syncthreads();
                        kn = (int)D.kn[mine];
                        th = D.th[mine];
                        S = dd{D.S[mine].x, D.S[mine].y};
                    }
                }
            }
            __syncthreads();  // every thread has read D.kn/th/S above
            if (tid == 0) {
                D.kn[mine] = (unsigned)kn;
                D.th[mine] = th;
                D.m[mine] = m;
                D.S[mine] = make_float2(S.hi, S.lo);
                D.flags[mine] = ovf ? RK_OVERFLOW : 0u;
            }
            if (k < g) {  // publish for the position's other block
                const int64_t ri = (int64_t)pos * 2 + r;
                if (tid == 0) {
                    TopkRow h;
                    h.kn = (unsigned)kn;
                    h.th = th;
                    h.m = m;
                    h.s_hi = S.hi;
                    h.s_lo = S.lo;
                    h.flags = ovf ? RK_OVERFLOW : 0u;
                    h.pad[0] = h.pad[1] = 0u;
                    p.rkrow[ri] = h;
                }
                if (!ovf && tid < kn) p.rkent[ri * kKeptMax + tid] = D.kept[mine][tid];
                __threadfence();
            }
        }
        __syncthreads();
        // ---- the position's decision, by the block that arrives last ----
        if (tid == 0) {
            unsigned last = 1u;
            if (k < g) {
                last = atomicAdd(p.rkcnt + pos, 1u) == 1u;
                if (last) {
                    p.rkcnt[pos] = 0u;  // left zeroed for the next call
                    __threadfence();
                }
            }
            s_last = last;
        }
        __syncthreads();
        if (s_last) {
            if (k < g) {
                // the other row's kept set and statistics
                const int64_t ri = (int64_t)pos * 2 + (1 - r);
                const uint4 *hp = reinterpret_cast<const uint4 *>(p.rkrow + ri);
                const uint4 h0 = __ldcg(hp), h1 = __ldcg(hp + 1);
                const unsigned okn = h0.x;
                if (tid == 0) {
                    D.kn[1 - r] = okn;
                    D.th[1 - r] = h0.y;
                    D.m[1 - r] = __uint_as_float(h0.z);
                    D.S[1 - r] = make_float2(__uint_as_float(h0.w), __uint_as_float(h1.x));
                    D.flags[1 - r] = h1.y;
                }
                if (!(h1.y & RK_OVERFLOW) && tid < (int)okn && tid < kKeptMax)
                    D.kept[1 - r][tid] = __ldcg(p.rkent + ri * kKeptMax + tid);
            }
            __syncthreads();
            const bool exact = ((D.flags[0] | (k < g ? D.flags[1] : 0u)) & RK_OVERFLOW) != 0u;  // block-uniform
            if (exact) {
                rk_exact_position<T>(p, sb, dsm, k, b);
            } else {
                const Outcome o = block_outcome<T>(p, b, k, D, EK, rd, &s_rej);
                finish(p, b, k, o, sb);
            }
        }
        __syncthreads();  // the ring's memory is free again for the next row
    }
    if (tid == 0)
        for (int s = 0; s < kRkNST; ++s) mbar_inval(&full[s]);
}

template <typename T>
static cudaError_t launch_rows(const SampleParams &p, int sms, cudaStream_t s) {
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = ensure_smem_attr(chain_topk_row_kernel<T>, (int)kRkDyn, done);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_topk_row_kernel<T>, kNT, kRkDyn);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t rows = (int64_t)p.B * (2 * p.gamma + 1);
    const int64_t cap = (int64_t)sms * per_sm;
    const unsigned grid = (unsigned)(rows < cap ? rows : cap);
    chain_topk_row_kernel<T><<<grid, kNT, kRkDyn, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_chain_topk(const SampleParams &p, int dtype, int sms, cudaStream_t s) {
    return dtype == SPEC_DTYPE_BF16 ? launch_rows<__nv_bfloat16>(p, sms, s) : launch_rows<float>(p, sms, s);
}

}  // namespace specv
