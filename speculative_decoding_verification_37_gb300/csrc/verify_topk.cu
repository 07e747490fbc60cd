// Sampled chain verification with top-k (k <= 128) on sm_103a: a pass over
// the logits, then one decision block per row.
//
// The transform ("KV Cache 优化（四）：Speculative Decoding 投机解码" §4) keeps
// every logit >= the row's k-th largest, so after one pass over a row only a
// handful of its logits matter; the acceptance test, the residual mass and
// the draw ("10.6 投机解码：为什么“先猜后验”能加速" §10.6.1) then work on the
// two kept sets of a position.
//
// chain_topk_pass_kernel: a persistent grid of four blocks per SM; block i
// takes rows i, i + grid, ...  For its row a block streams the 16-byte-aligned
// body through a ring of shared-memory stages (thread 0 issues one
// cp.async.bulk per 16 KiB chunk with an evict-first L2 policy, completing on
// the stage's mbarrier, waits bounded).  Per chunk a thread only takes the
// maximum of its four 16-byte vectors (packed bf16x2 maxima): a "group" is
// (chunk, thread).  It keeps its maximum over the row (the scalar head and
// tail included) and its four largest groups (16-bit key prefix and chunk),
// and writes them to the workspace at the row's end: the pass streams at the
// memory's pace, with nothing else to wait for.
//
// chain_topk_decide_kernel: one block per row, launched as a programmatic
// dependent of the pass (its launch overlaps the pass's tail; it waits for
// the pass's results before reading them).  For its row:
//  1. theta = the k-th largest of the threads' maxima (each is a logit, so at
//     least k logits reach it: a lower bound of the row's k-th largest).
//     Only groups whose maximum reaches theta's prefix can hold a kept
//     logit, and each thread's such groups are among its four largest unless
//     the fourth qualifies too (ties: then the position takes the exact
//     path).  The candidate groups go into a shared list and each thread
//     reloads one (all reloads in flight at once) and lists its elements
//     >= theta, and the head and tail scalars >= theta, (order key, token id)
//     in a shared buffer;
//  2. the kept set: an entry is kept iff fewer than k listed entries are
//     larger, i.e. exactly the logits >= the k-th largest; then token order,
//     the maximum and the double-float normaliser (and the nucleus when
//     top_p is set), published to the workspace;
//  3. the block that arrives second for a position (one counter per
//     position; the bonus position has one row) reads the other row's kept
//     set and decides: a_k = min(1, p(d)/q(d)), the residual mass over the
//     target's kept set (q looked up in the draft's), and the draw where
//     this position decides the token, by a double-float scan in token
//     order; finish() records it and the last position of a request writes
//     the request's outputs.
// A position whose candidates do not fit (many logits tied at the
// threshold) takes the exact masked computation over both rows instead, the
// nucleus included (slow, exact, rare).
#include "sample_common.cuh"

namespace specv {

constexpr int kRkCH = 16384;              // bytes of a row's body per ring stage
constexpr int kRkNST = 3;                 // ring stages
constexpr int kRkCap = 512;               // candidate entries a row can hold
constexpr int kRkBlocksPerSM = 4;         // pass blocks per SM
constexpr int kRkVec = kRkCH / 16 / kNT;  // 16-byte vectors per thread and chunk
static_assert(kRkVec * 16 * kNT == kRkCH, "a chunk is whole vectors per thread");
static_assert(kRkVec * 8 <= 32, "a thread's hit bits fit one word");
static_assert(kKeptMax == kNT, "one kept-set slot per thread");
static_assert(kTopKThreads == kNT && kTopKGroups == 4, "the workspace layout of the pass's results");

struct RkRing {
    alignas(128) unsigned char buf[kRkNST][kRkCH];
};
using RkFallbackRing = Ring<8192, 2, 2>;  // the exact masked path's ring

// The decision's arrays (dynamic shared memory of a decide block).
struct RkDecide {
    uint2 kept[2][kKeptMax];     // target / draft kept set, token order
    float2 wp[2][kKeptMax];      // per kept target entry: p (or the bonus term) and residual weight
    uint2 tmp[kKeptMax];         // unsorted kept entries; top-p: entries by rank
    float2 prb[kKeptMax];        // top-p: probabilities by rank
    unsigned kn[2], th[2], flags[2];
    float m[2];
    float2 S[2];
    float a;        // a_k, written by the thread holding d's kept target entry
    unsigned ahit;  // 1 once it has
};
constexpr size_t cmax(size_t a, size_t b) { return a > b ? a : b; }
// a decide block's dynamic shared memory: the decision arrays and both rows'
// candidate buffers, or the exact path's ring
constexpr size_t kRkCandOff = (sizeof(RkDecide) + 15) / 16 * 16;
constexpr size_t kRkDecideDyn =
    (cmax(sizeof(RkFallbackRing), kRkCandOff + kRkCap * sizeof(uint2)) + 127) / 128 * 128;

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

// a 16-byte vector of -inf
template <typename T> __device__ __forceinline__ uint4 vec_neg_inf();
template <> __device__ __forceinline__ uint4 vec_neg_inf<float>() {
    return make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
}
template <> __device__ __forceinline__ uint4 vec_neg_inf<__nv_bfloat16>() {
    return make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u);
}
// largest element of N vectors (bf16: packed maxima, one conversion)
template <typename T, int N> __device__ __forceinline__ float vecs_max(const uint4 (&v)[N]);
template <> __device__ __forceinline__ float vecs_max<float, kRkVec>(const uint4 (&v)[kRkVec]) {
    float m = vec_max<float>(v[0]);
#pragma unroll
    for (int i = 1; i < kRkVec; ++i) m = fmaxf(m, vec_max<float>(v[i]));
    return m;
}
template <> __device__ __forceinline__ float vecs_max<__nv_bfloat16, kRkVec>(const uint4 (&v)[kRkVec]) {
    __nv_bfloat162 a = __hmax2(__hmax2(as_bf2(v[0].x), as_bf2(v[0].y)), __hmax2(as_bf2(v[0].z), as_bf2(v[0].w)));
#pragma unroll
    for (int i = 1; i < kRkVec; ++i)
        a = __hmax2(a, __hmax2(__hmax2(as_bf2(v[i].x), as_bf2(v[i].y)), __hmax2(as_bf2(v[i].z), as_bf2(v[i].w))));
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

// ---------------------------------------------------------------------------
// Block-wide helpers.  Everything after a row's stream runs on the whole
// block: one dependent warp would share its SM sub-partition with the other
// resident blocks' warps and run several times slower.
// ---------------------------------------------------------------------------
struct RkRed {
    unsigned u[2][kNW];
    float2 f[2][kNW];
};

// Counts exchanged by the block-wide selections below (double-buffered by
// step parity).
struct RkPairRed {
    unsigned c[2][kNW][8];
};

// The K-th largest of the keys every thread passes (0 = no key): the largest
// r such that at least K keys are >= r, 0 if there are fewer than K keys.
// Two bits per step, counted with warp ballots and one block barrier per
// step.  Every thread calls it and gets the result.
template <int KB>
__device__ uint32_t block_kth_one(uint32_t k0, unsigned K, RkPairRed &pr) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned h = (unsigned)__popc(__ballot_sync(kFull, k0 != 0u));
    if (lane == 0) pr.c[1][wid][0] = h;
    __syncthreads();
    h = 0u;
#pragma unroll
    for (int w = 0; w < kNW; ++w) h += pr.c[1][w][0];
    if (h < K) return 0u;
    uint32_t a = 0u;
    int par = 0;
#pragma unroll 1
    for (int bit = KB - 2; bit >= 0; bit -= 2, par ^= 1) {
        unsigned n[3];
#pragma unroll
        for (int d = 1; d <= 3; ++d) n[d - 1] = (unsigned)__popc(__ballot_sync(kFull, k0 != 0u && k0 >= (a | ((uint32_t)d << bit))));
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < 3; ++j) pr.c[par][wid][j] = n[j];
        __syncthreads();
        unsigned mine = 0u;
        if (lane < 3)
#pragma unroll
            for (int w = 0; w < kNW; ++w) mine += pr.c[par][w][lane];
        const unsigned t0 = __shfl_sync(kFull, mine, 0), t1 = __shfl_sync(kFull, mine, 1), t2 = __shfl_sync(kFull, mine, 2);
        a |= (t2 >= K ? 3u : t1 >= K ? 2u : t0 >= K ? 1u : 0u) << bit;
    }
    return a;
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

// A position's inputs the deciding block needs: its draft token, its two
// uniforms and the request's rejection word, read before the decision.
struct RkInputs {
    int d;
    float u_k, u_f;
    unsigned rej;
};

// The outcome of position k of request b from the two kept sets (token
// order, one entry per thread) and their row statistics: acceptance, the
// residual mass, and the draw where this position decides the emitted
// token, by a block dd prefix in token order.  Every thread calls it; the
// result is the same in every thread.
template <typename T>
__device__ __noinline__ Outcome block_outcome(const SampleParams &p, int b, int k, RkDecide &D, const DdExpTables &EK,
                                              RkRed &rd, float4 *red4, const RkInputs &in) {
    const int tid = threadIdx.x;
    const int g = p.gamma;
    const bool has_draft = k < g;
    const int d = in.d;
    const bool bad_tok = has_draft && (d < 0 || d >= p.V);
    const float u_k = in.u_k, u_f = in.u_f;
    const uint2 *Kp = D.kept[0], *Kq = D.kept[1];
    const int np = (int)D.kn[0], nq = has_draft ? (int)D.kn[1] : 0;
    const float mp = D.m[0], mq = has_draft ? D.m[1] : 0.0f;
    const dd sp{D.S[0].x, D.S[0].y};
    const dd sq = has_draft ? dd{D.S[1].x, D.S[1].y} : dd{0.0f, 0.0f};
    Outcome o{1.0f, 0.0f, -1, 0u};
    const bool bad_row = mp == -INFINITY || (has_draft && mq == -INFINITY);
    o.info = (bad_tok ? REC_BAD_INPUT : 0u) | (bad_row ? REC_BAD_ROW : 0u);
    const unsigned rej = in.rej;
    if (bad_tok || bad_row) return o;
    const dd isp = dd_recip(sp);
    const dd isq = has_draft ? dd_recip(sq) : dd{0.0f, 0.0f};
    // thread t: kept target entry t (token order), its p (the unnormalised
    // term for the bonus draw) and residual weight max(0, p - q).  The thread
    // holding d's entry also forms a_k = min(1, p(d)/q(d)); d outside the
    // target's kept set has p(d) = 0, so a_k = 0 (D.ahit stays 0).
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
            if (id == (uint32_t)d) {
                float a;
                if (dd_pos(qi)) {
                    const dd ratio = dd_mul(pi, dd_recip(qi));
                    a = dd_gt(ratio, dd{1.0f, 0.0f}) ? 1.0f : dd_to_f(ratio);
                } else {
                    a = dd_pos(pi) ? 1.0f : 0.0f;
                }
                D.a = a;
                D.ahit = 1u;
            }
            w = dd_max0(dd_add(pi, dd_neg(qi)));
        }
    }
    dd zw{0.0f, 0.0f}, zp{0.0f, 0.0f};
    bool accept = false;
    if (has_draft) {  // both sums in one block reduction (its barriers publish D.a)
        zw = w;
        zp = pi;
        block_dd_sum2<kNT>(zw, zp, red4);
        o.z = dd_to_f(zw);
        const float a = D.ahit ? D.a : 0.0f;
        o.a = a;
        accept = u_k < a;
        o.info |= accept ? REC_ACCEPT : 0u;
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
        // the first entry past t, and the last with weight (when rounding
        // leaves the total short of t), in one exchange
        const int lane = tid & 31, wid = tid >> 5;
        const unsigned hw = __reduce_min_sync(kFull, (pos_w && dd_gt(cum, t)) ? (unsigned)tid : 0xffffffffu);
        const unsigned lw = __reduce_max_sync(kFull, pos_w ? (unsigned)tid + 1u : 0u);
        if (lane == 0) {
            rd.u[0][wid] = hw;
            rd.u[1][wid] = lw;
        }
        __syncthreads();
        unsigned hit = 0xffffffffu, lastp = 0u;
#pragma unroll
        for (int x = 0; x < kNW; ++x) {
            hit = min(hit, rd.u[0][x]);
            lastp = max(lastp, rd.u[1][x]);
        }
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


// The pass: every row's thread maxima and four largest groups.
template <typename T>
__global__ void __launch_bounds__(kNT, kRkBlocksPerSM) chain_topk_pass_kernel(SampleParams p) {
    constexpr int KB = Elem<T>::KEY_BITS;
    __shared__ __align__(8) unsigned long long full[kRkNST];
    extern __shared__ __align__(128) unsigned char dsm[];
    RkRing &R = *reinterpret_cast<RkRing *>(dsm);
    const int tid = threadIdx.x;
    const int g = p.gamma, B = p.B;
    const int nrows = B * (2 * g + 1);
    if (tid == 0) {
        for (int s = 0; s < kRkNST; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();  // the decision blocks may be scheduled; they wait for this grid's end
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
        float tmax = fmaxf(tid < nhead ? ld_elem(row, sp.head0 + tid) : -INFINITY,
                           tid < ntail ? ld_elem(row, sp.tail0 + tid) : -INFINITY);
        // the four largest groups, (key prefix << 16 | chunk), descending; 0 = none
        uint32_t t4[4] = {0u, 0u, 0u, 0u};
        bool tmo = false;
        int failed_at = -1;
        for (int w = 0; w < nch; ++w) {
            const unsigned gq = seq + (unsigned)w;
            const int s = (int)(gq % kRkNST);
            if (!mbar_wait_bounded(&full[s], (gq / kRkNST) & 1u)) tmo = true;
            const int nv = (int)(min((uint32_t)kRkCH, body - (uint32_t)w * kRkCH) / 16u);
            const uint4 *st = reinterpret_cast<const uint4 *>(R.buf[s]);
            uint4 v[kRkVec];
#pragma unroll
            for (int i = 0; i < kRkVec; ++i) {
                const int qv = tid + i * kNT;
                v[i] = qv < nv ? st[qv] : vec_neg_inf<T>();
            }
            const float tm = vecs_max<T, kRkVec>(v);
            tmax = fmaxf(tmax, tm);
            uint32_t x = tm > -INFINITY ? ((kkey<T>(tm) >> (KB - 16)) << 16) | (uint32_t)w : 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t hi = max(t4[j], x);
                x = min(t4[j], x);
                t4[j] = hi;
            }
            if (__syncthreads_or(tmo)) {  // block-uniform: a chunk did not arrive
                failed_at = w;
                break;
            }
            // every thread holds its share of the chunk: refill the stage
            if (tid == 0 && issued < nch) issue(issued++);
        }
        if (failed_at >= 0) {
            // A bulk copy did not complete in time: issue nothing more, wait
            // (bounded) for the copies already issued so that none lands in
            // shared memory after the block has moved on, flag the call and stop.
            if (tid == 0) {
                bool drained = true;
                for (int c = failed_at; c < issued; ++c) {
                    const unsigned gq = seq + (unsigned)c;
                    drained &= mbar_drain(&full[gq % kRkNST], (gq / kRkNST) & 1u);
                }
                atomicOr(p.status, SPEC_FLAG_TIMEOUT);
                if (drained)
                    for (int s = 0; s < kRkNST; ++s) mbar_inval(&full[s]);
            }
            return;
        }
        seq += (unsigned)nch;
        const int64_t slot = (int64_t)pos * 2 + r;
        p.rkmax[slot * kNT + tid] = tmax > -INFINITY ? kkey<T>(tmax) : 0u;
#pragma unroll
        for (int j = 0; j < 4; ++j) p.rkgrp[(slot * 4 + j) * kNT + tid] = t4[j];
    }
    if (tid == 0)
        for (int s = 0; s < kRkNST; ++s) mbar_inval(&full[s]);
}

// One row of a position, as the decide block sees it.
template <typename T>
struct RkRowView {
    const T *row;
    const uint4 *body;  // the 16-byte-aligned body
    uint32_t bytes;     // its length
    int body0, head0, tail0, nhead, ntail;
    __device__ RkRowView(const T *r, int V) : row(r) {
        const SliceSplit sp = split_slice(r, 0, V);
        body = reinterpret_cast<const uint4 *>(r + sp.body0);
        bytes = (uint32_t)(sp.tail0 - sp.body0) * (uint32_t)sizeof(T);
        body0 = sp.body0;
        head0 = sp.head0;
        tail0 = sp.tail0;
        nhead = sp.body0 - sp.head0;
        ntail = sp.hi - sp.tail0;
    }
    // group (chunk c, thread t): its vectors, -inf past the body (a chunk
    // index past the row, from a pass that did not finish, reads nothing)
    __device__ __forceinline__ void load_group_of(int c, int t, uint4 (&v)[kRkVec]) const {
        const uint32_t off = (uint32_t)c * kRkCH;
        const int nv = off < bytes ? (int)(min((uint32_t)kRkCH, bytes - off) / 16u) : 0;
#pragma unroll
        for (int i = 0; i < kRkVec; ++i) {
            const int qv = t + i * kNT;
            v[i] = qv < nv ? __ldg(body + (int64_t)c * (kRkCH / 16) + qv) : vec_neg_inf<T>();
        }
    }
};

// one slot range per warp (a single shared atomic per warp: the threads'
// atomics on one word would serialize); every lane calls it
__device__ __forceinline__ unsigned warp_reserve(unsigned n, int *cnt) {
    const int lane = threadIdx.x & 31;
    unsigned incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    unsigned base = 0u;
    if (lane == 31 && incl) base = (unsigned)atomicAdd(cnt, (int)incl);
    return __shfl_sync(kFull, base, 31) + incl - n;
}

// the elements of group (chunk c, thread t) that reach tf (bits of hm), from `at` on
template <typename T>
__device__ __forceinline__ void write_group_of(uint2 *cand, unsigned &at, int body0, int c, int t, const uint4 (&v)[kRkVec],
                                               uint32_t hm) {
    constexpr int VEC = Elem<T>::VEC;
    constexpr int ECH = kRkCH / (int)sizeof(T);
    const int vbase = body0 + c * ECH;
#pragma unroll
    for (int i = 0; i < kRkVec; ++i) {
        uint32_t h = (hm >> (VEC * i)) & ((1u << VEC) - 1u);
        while (h) {
            const int e = __ffs(h) - 1;
            h &= h - 1u;
            if (at < (unsigned)kRkCap)
                cand[at] = make_uint2(kkey<T>(vec_elem<T>(v[i], e)), (uint32_t)(vbase + (t + i * kNT) * VEC + e));
            ++at;
        }
    }
}
template <typename T>
__device__ __forceinline__ uint32_t group_hits(const uint4 (&v)[kRkVec], float tf) {
    constexpr int VEC = Elem<T>::VEC;
    uint32_t hm = 0u;
#pragma unroll
    for (int i = 0; i < kRkVec; ++i) hm |= vec_ge_mask<T>(v[i], tf) << (VEC * i);
    return hm;
}

// The decision: one block per row.  A row's block takes its row's threshold
// bound, reloads its candidate groups and builds its kept set; for the two
// rows of a position the block that arrives second (one counter per
// position) reads the other row's published kept set and decides.
template <typename T>
__global__ void __launch_bounds__(kNT, kRkBlocksPerSM) chain_topk_decide_kernel(SampleParams p) {
    constexpr int KB = Elem<T>::KEY_BITS;
    __shared__ SampBase sb;
    __shared__ RkRed rd;
    __shared__ RkPairRed pr;
    __shared__ __align__(16) float4 s_red4[kNW];
    __shared__ int s_cnt;    // candidates listed (may pass kRkCap: then some were lost)
    __shared__ int s_ng;     // candidate groups of the row
    __shared__ unsigned s_last;
    __shared__ RkInputs s_in;
    __shared__ uint32_t glist[3 * kNT];  // (chunk << 8 | owner thread); at most three per pass thread
    extern __shared__ __align__(128) unsigned char dsm[];
    RkDecide &D = *reinterpret_cast<RkDecide *>(dsm);
    uint2 *cand = reinterpret_cast<uint2 *>(dsm + kRkCandOff);  // [kRkCap]
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const unsigned K = (unsigned)p.top_k;
    const int g = p.gamma, B = p.B;
    const bool nucleus = p.top_p > 0.0f && p.top_p < 1.0f;
    // row q: position-major, a position's target row then its draft row (as the pass)
    const int q = blockIdx.x;
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
    load_exp_tables(p, sb);
    const DdExpTables &EK = sb.K;
    if (tid == 0) {
        s_cnt = 0;
        s_ng = 0;
        s_in.d = k < g ? p.tokens[(int64_t)b * g + k] : 0;
        s_in.u_k = k < g ? p.unif[(int64_t)b * (g + 1) + k] : 0.0f;
        s_in.u_f = p.unif[(int64_t)b * (g + 1) + g];
    }
    const RkRowView<T> W(r == 0 ? reinterpret_cast<const T *>(p.target) + (int64_t)pos * p.tstride
                                : reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + k) * p.dstride,
                         p.V);
    const float xh = tid < W.nhead ? ld_elem(W.row, W.head0 + tid) : -INFINITY;
    const float xt = tid < W.ntail ? ld_elem(W.row, W.tail0 + tid) : -INFINITY;

    pdl_wait_primary();  // the pass's results from here on
    const int64_t slot = (int64_t)pos * 2 + r;
    const uint32_t km = __ldcg(p.rkmax + slot * kNT + tid);
    uint32_t t4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) t4[j] = __ldcg(p.rkgrp + (slot * 4 + j) * kNT + tid);
    // theta: the K-th largest thread maximum (0 with fewer than K finite
    // ones: every group is listed, the kept set is every finite logit)
    const uint32_t theta = block_kth_one<KB>(km, K, pr);
    const uint32_t th16 = theta >> (KB - 16);
    const float tf = fmaxf(key_value<T>(theta), lowest_finite<T>());
    auto is_cand = [&](uint32_t t) { return t != 0u && (t >> 16) >= th16; };
    // a thread whose fourth group qualifies may have more: the exact path
    bool ovf = __syncthreads_or(is_cand(t4[3]));  // block-uniform
    int count = 0;
    if (!ovf) {
        // ---- the listing: the candidate groups into a shared list, then
        // one group per thread (the reloads all in flight at once); the head
        // and tail scalars by their own threads ----
        unsigned ng = 0u;
#pragma unroll
        for (int j = 0; j < 3; ++j) ng += is_cand(t4[j]) ? 1u : 0u;
        unsigned at = warp_reserve(ng, &s_ng);
#pragma unroll
        for (int j = 0; j < 3; ++j)
            if (is_cand(t4[j])) glist[at++] = ((t4[j] & 0xffffu) << 8) | (uint32_t)tid;
        const bool hh = xh >= tf, ht = xt >= tf;
        unsigned ah = warp_reserve((hh ? 1u : 0u) + (ht ? 1u : 0u), &s_cnt);
        if (hh) {
            if (ah < (unsigned)kRkCap) cand[ah] = make_uint2(kkey<T>(xh), (uint32_t)(W.head0 + tid));
            ++ah;
        }
        if (ht && ah < (unsigned)kRkCap) cand[ah] = make_uint2(kkey<T>(xt), (uint32_t)(W.tail0 + tid));
        __syncthreads();
        const int ngr = s_ng;  // <= 3 * kNT
        for (int g0 = 0; g0 < ngr; g0 += kNT) {  // (block-uniform trip count)
            const int gi = g0 + tid;
            const bool on = gi < ngr;
            const uint32_t ge = on ? glist[gi] : 0u;
            const int c = (int)(ge >> 8), owner = (int)(ge & 0xffu);
            uint4 v[kRkVec];
            if (on) W.load_group_of(c, owner, v);
            const uint32_t hm = on ? group_hits<T>(v, tf) : 0u;
            unsigned a = warp_reserve((unsigned)__popc(hm), &s_cnt);
            if (hm) write_group_of<T>(cand, a, W.body0, c, owner, v, hm);
        }
        __syncthreads();  // every listed entry is in the buffer
        count = s_cnt;
        ovf = count > kRkCap;  // block-uniform: candidates were lost
    }

    // ---- the kept set: an entry is kept iff fewer than K listed entries are
    // larger, i.e. exactly the entries >= the K-th largest (ties included);
    // token order by counting; maximum, threshold, double-float normaliser ----
    int kn = 0;
    uint32_t th = 0u;
    float m = -INFINITY;
    dd S{0.0f, 0.0f};
    if (!ovf) {
        const int n = count;
        const uint2 e0 = tid < n ? cand[tid] : make_uint2(0u, 0u);
        const uint2 e1 = tid + kNT < n ? cand[tid + kNT] : make_uint2(0u, 0u);
        bool f0 = false, f1 = false;
        unsigned nk = 0u;
        uint32_t mx = 0u, lo = 0xffffffffu;
        if (__any_sync(kFull, tid < n)) {
            unsigned g0 = 0u, g1 = 0u;
            if (n <= kNT) {
#pragma unroll 8
                for (int y = 0; y < n; ++y) g0 += cand[y].x > e0.x ? 1u : 0u;
            } else {
                for (int y = 0; y < n; ++y) {
                    const uint32_t ky = cand[y].x;
                    g0 += ky > e0.x ? 1u : 0u;
                    g1 += ky > e1.x ? 1u : 0u;
                }
            }
            f0 = e0.x != 0u && g0 < K;
            f1 = e1.x != 0u && g1 < K;
            nk = (f0 ? 1u : 0u) + (f1 ? 1u : 0u);
            mx = max(e0.x, e1.x);
            if (f0) lo = e0.x;
            if (f1) lo = min(lo, e1.x);
        }
        nk = __reduce_add_sync(kFull, nk);
        mx = __reduce_max_sync(kFull, mx);
        lo = __reduce_min_sync(kFull, lo);
        if (lane == 0) {
            rd.u[0][wid] = nk;
            rd.u[1][wid] = mx;
            pr.c[0][wid][0] = lo;
        }
        unsigned char *kflag = reinterpret_cast<unsigned char *>(D.prb);  // [kRkCap] kept flags (free until top-p)
        static_assert(sizeof(D.prb) >= kRkCap, "kept flags fit");
        if (tid < n) kflag[tid] = f0;
        if (tid + kNT < n) kflag[tid + kNT] = f1;
        __syncthreads();
        unsigned knu = 0u;
        uint32_t mk = 0u, tl = 0xffffffffu;
#pragma unroll
        for (int w = 0; w < kNW; ++w) {
            knu += rd.u[0][w];
            mk = max(mk, rd.u[1][w]);
            tl = min(tl, pr.c[0][w][0]);
        }
        kn = (int)knu;
        th = (unsigned)n >= K ? tl : 0u;
        m = kn > 0 ? key_value<T>(mk) : -INFINITY;
        if (kn > kKeptMax) {
            ovf = true;  // block-uniform: hundreds of ties
        } else {
            dd t{0.0f, 0.0f};
            if (__any_sync(kFull, f0 || f1)) {
                unsigned r0 = 0u, r1 = 0u;
                if (n <= kNT) {
#pragma unroll 8
                    for (int y = 0; y < n; ++y) r0 += (kflag[y] && cand[y].y < e0.y) ? 1u : 0u;
                } else {
                    for (int y = 0; y < n; ++y) {
                        if (!kflag[y]) continue;
                        const uint32_t ty = cand[y].y;
                        r0 += ty < e0.y ? 1u : 0u;
                        r1 += ty < e1.y ? 1u : 0u;
                    }
                }
                if (f0) {
                    D.kept[r][r0] = e0;
                    t = dd_expw(key_value<T>(e0.x), m, EK);
                }
                if (f1) {
                    D.kept[r][r1] = e1;
                    t = dd_add(t, dd_expw(key_value<T>(e1.x), m, EK));
                }
            }
            S = block_dd_sum(t, rd);  // (its barriers also publish D.kept)
            if (nucleus && m != -INFINITY) {
                if (wid == 0) {
                    row_top_p<T>(D.kept[r], kn, th, m, S, p.top_p, D.tmp, D.prb, EK);
                    if (lane == 0) {
                        D.kn[r] = (unsigned)kn;
                        D.th[r] = th;
                        D.S[r] = make_float2(S.hi, S.lo);
                    }
                }
                __syncthreads();
                kn = (int)D.kn[r];
                th = D.th[r];
                S = dd{D.S[r].x, D.S[r].y};
            }
        }
    }
    __syncthreads();  // every thread has read D.kn/th/S above
    if (tid == 0) {
        D.kn[r] = (unsigned)kn;
        D.th[r] = th;
        D.m[r] = m;
        D.S[r] = make_float2(S.hi, S.lo);
        D.flags[r] = ovf ? 1u : 0u;
    }
    if (k < g) {  // publish for the position's other block
        if (tid == 0) {
            TopkRow h;
            h.kn = (unsigned)kn;
            h.th = th;
            h.m = m;
            h.s_hi = S.hi;
            h.s_lo = S.lo;
            h.flags = ovf ? 1u : 0u;
            h.pad[0] = h.pad[1] = 0u;
            p.rkrow[slot] = h;
        }
        if (!ovf && tid < kn) p.rkent[slot * kKeptMax + tid] = D.kept[r][tid];
        if (tid == 0 || (!ovf && tid < kn)) __threadfence();  // the writers' stores before the arrival
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
    if (!s_last) return;
    // one round of reads: the request's rejection word, the other row's
    // header and every slot of its kept set (those past its count unused)
    const unsigned rejw = tid == 0 ? *((volatile unsigned *)&p.rejword[b]) : 0u;
    if (k < g) {
        const int64_t ri = (int64_t)pos * 2 + (1 - r);
        const uint4 *hp = reinterpret_cast<const uint4 *>(p.rkrow + ri);
        const uint4 h0 = __ldcg(hp), h1 = __ldcg(hp + 1);
        const uint2 oe = __ldcg(p.rkent + ri * kKeptMax + tid);
        const unsigned okn = h0.x;
        if (tid == 0) {
            D.kn[1 - r] = okn;
            D.th[1 - r] = h0.y;
            D.m[1 - r] = __uint_as_float(h0.z);
            D.S[1 - r] = make_float2(__uint_as_float(h0.w), __uint_as_float(h1.x));
            D.flags[1 - r] = h1.y;
        }
        if (!(h1.y & 1u) && tid < (int)okn) D.kept[1 - r][tid] = oe;
    }
    if (tid == 0) {
        s_in.rej = rejw;
        D.ahit = 0u;
    }
    __syncthreads();
    const bool exact = ((D.flags[0] | (k < g ? D.flags[1] : 0u)) & 1u) != 0u;  // block-uniform
    if (exact) {  // the decision arrays are free: the exact path's ring
        __syncthreads();
        rk_exact_position<T>(p, sb, dsm, k, b);
    } else {
        const Outcome o = block_outcome<T>(p, b, k, D, EK, rd, s_red4, s_in);
        finish(p, b, k, o, sb);
    }
}

template <typename T>
static cudaError_t launch_topk(const SampleParams &p, int sms, cudaStream_t s) {
    static std::atomic<unsigned long long> done_pass{0}, done_decide{0};
    constexpr size_t pass_dyn = sizeof(RkRing);
    cudaError_t e = ensure_smem_attr(chain_topk_pass_kernel<T>, (int)pass_dyn, done_pass);
    if (e != cudaSuccess) return e;
    e = ensure_smem_attr(chain_topk_decide_kernel<T>, (int)kRkDecideDyn, done_decide);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_topk_pass_kernel<T>, kNT, pass_dyn);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t rows = (int64_t)p.B * (2 * p.gamma + 1);
    const int64_t cap = (int64_t)sms * per_sm;
    const unsigned grid = (unsigned)(rows < cap ? rows : cap);
    chain_topk_pass_kernel<T><<<grid, kNT, pass_dyn, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)rows);  // one block per row
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = kRkDecideDyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chain_topk_decide_kernel<T>, p);
}

cudaError_t launch_chain_topk(const SampleParams &p, int dtype, int sms, cudaStream_t s) {
    return dtype == SPEC_DTYPE_BF16 ? launch_topk<__nv_bfloat16>(p, sms, s) : launch_topk<float>(p, sms, s);
}

}  // namespace specv
