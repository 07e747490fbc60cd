// Sampled chain verification over the whole vocabulary (no top-k) as one
// persistent kernel of independent warps on sm_103a.
//
// The method ("10.6 投机解码：为什么“先猜后验”能加速" §10.6.1; "KV Cache 优化
// （四）：Speculative Decoding 投机解码" §4, §5): softmax every target and
// draft row at temperature T, accept d_k with probability min(1, p_k(d_k) /
// q_k(d_k)) left to right, and at the first rejection draw from
// norm(max(0, p_k - q_k)) (from p_k when that mass is <= eps), or draw the
// bonus token from p_{gamma+1} when every draft is accepted.
//
// GB300 mapping.  A cooperative grid of one block per SM; the block's warps
// are independent workers (no block barrier after the start), each with its
// own two-stage ring of bulk copies (cp.async.bulk on mbarriers).  A warp
// works through:
//  * stream items (position, 4 KiB slice of each row), position-major and
//    statically round-robin over all warps: the slice's (max, sum of
//    2^(x c2 - m c2)) pair per row, from the warp's maximum (no rescaling).
//    The item holding the draft token also stores l(d) and g(d).
//  * the decision of a position, taken by the warp that completes its last
//    slice (an arrival counter): the row normalisers, a_k = min(1, p/q) and
//    u_k < a_k; an atomic OR into the request's state word (a decided bit
//    and a stop bit per position) shows which update first determines the
//    request's first rejection (or that all drafts are accepted), and that
//    update starts the request's draw.
//  * draw items (request, group of slices) from a device-wide queue, taken
//    before further stream items so the rows are re-read while in L2.  A
//    draw runs in rounds; the warp that completes a round combines the
//    slices' results and scans the slice holding the crossing in token order:
//      round 0, fp32 with a certified error bound: each term's error is
//        bounded (hardware ex2 error, argument rounding) and so is every
//        sum's (summation depth); the drawn token is kept only when the
//        uniform lies farther than the bound from both CDF boundaries
//        around it, otherwise
//      round 1, double-float (ddmath.cuh): sums S_p, S_q and, over
//        P = {p_i > q_i} decided from the pass's fp32 ratio estimate outside
//        a 2^-10 band, P_p and P_q; the elements inside the band are listed
//        and evaluated once S_p, S_q are exact;
//      round 2, double-float residual sums with the exact normalisers, only
//        when a slice listed more elements than it holds (rows that are
//        nearly equal).
//  * the request epilogue: the last of the request's decisions and draw
//    writes its outputs.
// Arrivals are fire-and-forget, a follow-up belongs to a fixed warp that
// polls for it, and the queue's words are read one step ahead, so no step
// waits on a round trip.
// Every wait (a stage's bytes, an idle warp) is bounded and ends with
// SPEC_FLAG_TIMEOUT in the status word.
#include "sample_common.cuh"

namespace specv {

constexpr int kFwWarps = 12;           // workers per block (one block per SM)
constexpr int kFwNST = 2;              // ring stages per warp (12 x 16 KiB of rings per SM)
constexpr int kFwSlice = 4096;         // bytes of one row in one item
constexpr int kFwVecs = kFwSlice / 16 / 32;  // 16-byte vectors per lane and row
static_assert(kFwVecs * 16 * 32 == kFwSlice, "a slice is whole vectors per lane");
constexpr int kFwMaxC = 256;           // slices per row (V * element size <= 1 MiB)
constexpr int kFwAmb = kFullAmb;       // in-band residual elements listed per (request, slice)
constexpr int kFwGroup0 = 4;           // slices per queue item, fp32 round
constexpr int kFwGroupDD = 1;          // slices per queue item, double-float rounds
constexpr long long kFwIdleLimit = 1ll << 21;  // idle polls (about 0.5 us each) before giving up
long long full_idle_limit() { return kFwIdleLimit; }

// ---- the certified fp32 round's error model --------------------------------
// A term 2^((x - m) c) is computed with its exponent exact to ~2^-48 (x - m by
// TwoSum, c = log2(e)/T as a double-float pair), the hardware ex2 on the
// exponent's high part and a first-order correction for its low part.  Its
// relative error is below kTermErr: the ex2.approx.ftz.f32 bound (an
// exhaustive comparison with fp64 over every input in [-126, 1] on this GPU
// found at most 1.46e-7; the bound used is 1.5e-7, and a GPU test re-checks
// it), half an ulp for the correction's rounding, and 1e-10 for the
// neglected exponent and second-order terms.
constexpr float kU = 5.9604644775390625e-8f;  // 2^-24
constexpr float kEx2Err = 1.5e-7f;
float full_ex2_bound() { return kEx2Err; }
constexpr float kTermErr = kEx2Err + 0.5f * kU + 1e-10f;
// A slice sum: pairwise within a 16-byte vector (depth <= 3, plain fp32),
// then compensated (TwoSum) across vectors and lanes and kept as a
// double-float pair: relative error below 3u plus second-order terms.
constexpr float kSumErr = 3.5f * kU;
// fp32 prefix depth of the token-order scan: a lane's run (<= 64), the warp's
// inclusive scan (5), the lane's exclusive prefix (1).
constexpr int kScanDepth = 70;

struct FwRing {
    alignas(128) unsigned char buf[kFwNST][2][kFwSlice];
};

int full_row_bytes() { return kFwSlice; }
int full_max_slices() { return kFwMaxC; }

static_assert(sizeof(DrawRec) == 32 && alignof(DrawRec) == 16, "draw record layout");
static_assert(sizeof(DrawPart) == 64 && alignof(DrawPart) == 16, "draw part layout");

// Queue and termination words, in the workspace header (zero between calls).
struct FuCtl {
    unsigned head, tail, nfin, nexit;
};

__device__ __forceinline__ float ex2f(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ FuCtl *fu_ctl(const SampleParams &p) {
    return reinterpret_cast<FuCtl *>(reinterpret_cast<char *>(p.status) + 64);
}

__device__ __forceinline__ unsigned atom_add_release(unsigned *a, unsigned v) {
    unsigned old;
    asm volatile("atom.add.release.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *a) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.u64 %0, [%1];" : "=l"(v) : "l"(a) : "memory");
    return v;
}

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned *a) {
    unsigned v;
    asm volatile("ld.relaxed.gpu.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

// 2^((x - m) (c2 + c2lo)) with the exponent computed exactly (see kTermErr);
// -inf gives 0.  Branch-free, so a lane's terms interleave.
__device__ __forceinline__ float ex2_exact(float x, float m, float c2, float c2lo) {
    const bool fin = x > -INFINITY;
    const dd d = two_sum(fin ? x : m, -m);  // x - m exactly
    const float zh = __fmul_rn(d.hi, c2);
    const float zl = __fadd_rn(__fmaf_rn(d.hi, c2, -zh), __fmaf_rn(d.hi, c2lo, __fmul_rn(d.lo, c2)));
    const float e = ex2f(zh);
    const float r = __fmaf_rn(e, __fmul_rn(zl, 0.6931471805599453f), e);
    return fin ? r : 0.0f;
}

// compensated accumulation (value, correction) of fp32 terms
struct CSum {
    float s, c;
};
__device__ __forceinline__ void csum_add(CSum &a, float v) {
    const dd t = two_sum(a.s, v);
    a.s = t.hi;
    a.c = __fadd_rn(a.c, t.lo);
}
__device__ __forceinline__ CSum warp_csum(CSum a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(kFull, a.s, o), c2 = __shfl_xor_sync(kFull, a.c, o);
        const dd t = two_sum(a.s, s2);
        a.s = t.hi;
        a.c = __fadd_rn(__fadd_rn(a.c, c2), t.lo);
    }
    return a;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

__device__ __forceinline__ dd shfl_dd(dd v, int src) {
    return dd{__shfl_sync(kFull, v.hi, src), __shfl_sync(kFull, v.lo, src)};
}

// inclusive warp prefix of dd values in lane order
__device__ __forceinline__ dd warp_dd_incl(dd v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const dd y{__shfl_up_sync(kFull, v.hi, o), __shfl_up_sync(kFull, v.lo, o)};
        if (lane >= o) v = dd_add(y, v);
    }
    return v;
}

__device__ __forceinline__ void fu_decode(int t, int c, int B, int &k, int &b, int &j) {
    const int qpos = t / c;
    j = t - qpos * c;
    k = qpos / B;
    b = qpos - k * B;
}

template <typename T> __device__ __forceinline__ int fw_slice_elems() { return kFwSlice / (int)sizeof(T); }

// lane 0: arm stage s of this warp's ring for stream item t
template <typename T>
__device__ __forceinline__ void fw_issue(const SampleParams &p, FwRing &R, unsigned long long *full, int t, int s) {
    int k, b, j;
    fu_decode(t, p.c, p.B, k, b, j);
    const int W = fw_slice_elems<T>();
    const int lo = j * W, n = min(W, p.V - lo);
    const uint32_t bytes = (uint32_t)n * (uint32_t)sizeof(T);
    const bool two = k < p.gamma;
    mbar_arrive_expect_tx(&full[s], bytes * (two ? 2u : 1u));
    const T *trow = reinterpret_cast<const T *>(p.target) + (int64_t)(b * (p.gamma + 1) + k) * p.tstride + lo;
    bulk_g2s(R.buf[s][0], trow, bytes, &full[s]);
    if (two) {
        const T *drow = reinterpret_cast<const T *>(p.draft) + (int64_t)(b * p.gamma + k) * p.dstride + lo;
        bulk_g2s(R.buf[s][1], drow, bytes, &full[s]);
    }
}

// ---------------------------------------------------------------------------
// Request bookkeeping.  The request's state word holds a decided bit (2k) and
// a stop bit (2k+1) per position and, in bit 63, "draw done"; the atomic OR
// that completes every decided bit and the draw bit runs the epilogue.
// ---------------------------------------------------------------------------
constexpr unsigned long long kDrawDone = 1ull << 63;  // positions use bits 0..61: gamma <= 30

__device__ __forceinline__ unsigned long long atom_or_acq_rel(unsigned long long *a, unsigned long long v) {
    unsigned long long old;
    asm volatile("atom.acq_rel.gpu.global.or.b64 %0, [%1], %2;" : "=l"(old) : "l"(a), "l"(v) : "memory");
    return old;
}

__device__ __forceinline__ void red_add_release(unsigned *a, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned *a) {
    unsigned v;
    asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
    return v;
}

// First position that stops the request (rejected, bad, or the bonus row)
// with every earlier position decided; -1 while undetermined.
__device__ __forceinline__ int fu_first_stop(unsigned long long w, int g) {
    for (int k = 0; k <= g; ++k) {
        if (!((w >> (2 * k)) & 1ull)) return -1;
        if (k == g || ((w >> (2 * k + 1)) & 1ull)) return k;
    }
    return -1;
}

__device__ __forceinline__ bool fu_complete(unsigned long long w, int g) {
    const unsigned long long dec = 0x5555555555555555ull & ((2ull << (2 * g)) - 1ull);  // bits 0, 2, .., 2g
    return (w & dec) == dec && (w & kDrawDone);
}

// Warp-level: the request epilogue if the update old -> old|mine completed it.
__device__ void fu_maybe_epilogue(const SampleParams &p, int b, unsigned long long old, unsigned long long mine) {
    const int lane = threadIdx.x & 31;
    const bool done = __shfl_sync(kFull, (int)(fu_complete(old | mine, p.gamma) && !fu_complete(old, p.gamma)), 0);
    if (!done) return;
    write_request_warp(p, b);
    if (lane == 0) {
        p.rstate[b] = 0ull;
        __threadfence();
        atomicAdd(&fu_ctl(p)->nfin, 1u);
    }
}

// Warp-level: marks request b's draw done (lane 0's `old` is broadcast).
__device__ void fu_draw_done(const SampleParams &p, int b) {
    unsigned long long old = 0ull;
    if ((threadIdx.x & 31) == 0) old = atom_or_acq_rel(p.rstate + b, kDrawDone);
    old = __shfl_sync(kFull, old, 0);
    fu_maybe_epilogue(p, b, old, kDrawDone);
}

__device__ __forceinline__ int fw_group(int pass) { return pass == 0 ? kFwGroup0 : kFwGroupDD; }

// Enqueues request b's round `pass` (its draw record already written).
__device__ void fw_enqueue(const SampleParams &p, int b, int pass) {
    const int lane = threadIdx.x & 31;
    const int ng = (p.c + fw_group(pass) - 1) / fw_group(pass);
    unsigned base = 0u;
    if (lane == 0) {
        __threadfence();
        base = atomicAdd(&fu_ctl(p)->tail, (unsigned)ng);
    }
    base = __shfl_sync(kFull, base, 0);
    for (int q = lane; q < ng; q += 32)
        p.qitem[base + q] = (1ull << 63) | ((unsigned long long)b << 20) | (unsigned long long)q;
}

// Starts request b's draw at position kstar (info: that position's bits).
__device__ void fu_start_draw(const SampleParams &p, int b, int kstar, unsigned info) {
    const int g = p.gamma;
    if (info & (REC_BAD_INPUT | REC_BAD_ROW)) {  // no draw: the request is flagged
        fu_draw_done(p, b);
        return;
    }
    if ((threadIdx.x & 31) == 0) {
        DrawRec d;
        d.kstar = kstar;
        d.mode = kstar == g ? 1 : 0;
        d.pass = 0;
        d.pad = 0;
        d.inv = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        p.drec[b] = d;
    }
    fw_enqueue(p, b, 0);
}

// The decision of position pos, by the warp that owns it (the one that
// streamed its first slice) once every slice has arrived.
__device__ __noinline__ void fu_decide(const SampleParams &p, int pos) {
    const int lane = threadIdx.x & 31, g = p.gamma, c = p.c;
    const int b = pos / (g + 1), k = pos - b * (g + 1);
    const bool has_draft = k < g;
    const float c2 = p.c2;
    // every load at once: the slices' pairs, the draft token's logits, the
    // token and the uniform
    constexpr int kPer = kFwMaxC / 32;
    float2 a[kPer], q[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int j = lane + 32 * i;
        a[i] = j < c ? __ldcg(p.fpart + ((int64_t)pos * 2 + 0) * c + j) : make_float2(-INFINITY, 0.0f);
        q[i] = (has_draft && j < c) ? __ldcg(p.fpart + ((int64_t)pos * 2 + 1) * c + j) : make_float2(-INFINITY, 0.0f);
    }
    int d = 0;
    float2 xd = make_float2(0.0f, 0.0f);
    float u = 0.0f;
    if (lane == 0 && has_draft) {
        d = __ldcg(p.tokens + (int64_t)b * g + k);
        xd = __ldcg(p.fxd + pos);
        u = __ldcg(p.unif + (int64_t)b * (g + 1) + k);
    }
    MaxSum mp{-INFINITY, 0.0f}, mq{-INFINITY, 0.0f};
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        mp = ms_combine(mp, MaxSum{a[i].x, a[i].y}, c2);
        mq = ms_combine(mq, MaxSum{q[i].x, q[i].y}, c2);
    }
    mp = warp_ms(mp, c2);
    mq = warp_ms(mq, c2);
    int kstar = -1;
    unsigned info = 0u;
    unsigned long long old = 0ull, mine = 0ull;
    if (lane == 0) {
        const bool bad_tok = has_draft && (d < 0 || d >= p.V);
        const bool bad_row = mp.m == -INFINITY || (has_draft && mq.m == -INFINITY);
        const bool bad = bad_tok || bad_row;
        Outcome o{1.0f, 0.0f, -1, (bad_tok ? REC_BAD_INPUT : 0u) | (bad_row ? REC_BAD_ROW : 0u)};
        bool accept = false;
        if (has_draft && !bad) {
            const float pd = exp2f(fmaf(xd.x, c2, -mp.m * c2)) / mp.s;
            const float qd = exp2f(fmaf(xd.y, c2, -mq.m * c2)) / mq.s;
            o.a = qd > 0.0f ? fminf(1.0f, pd / qd) : (pd > 0.0f ? 1.0f : 0.0f);
            accept = u < o.a;
            o.info |= accept ? REC_ACCEPT : 0u;
        }
        p.fstat[pos] = make_float4(mp.m, mp.s, mq.m, mq.s);
        PosRec rec;
        rec.a = o.a;
        rec.z = 0.0f;
        rec.token = -1;
        rec.info = o.info;
        p.recs[pos] = rec;
        p.pcnt[pos] = 0u;
        const bool stop = !has_draft || bad || !accept;
        mine = (1ull << (2 * k)) | (stop ? (1ull << (2 * k + 1)) : 0ull);
        old = atom_or_acq_rel(p.rstate + b, mine);  // releases the record and the statistics
        const int before = fu_first_stop(old, g), now = fu_first_stop(old | mine, g);
        if (now >= 0 && before < 0) {
            kstar = now;
            info = now == k ? o.info : load_rec(p.recs + b * (g + 1) + now).info;
        }
    }
    kstar = __shfl_sync(kFull, kstar, 0);
    info = __shfl_sync(kFull, info, 0);
    old = __shfl_sync(kFull, old, 0);
    mine = __shfl_sync(kFull, mine, 0);
    if (kstar >= 0) fu_start_draw(p, b, kstar, info);
    fu_maybe_epilogue(p, b, old, mine);
}

// ---------------------------------------------------------------------------
// Stream item t (this warp's stage s): the slice's (max, sum) pair per row.
// Returns the position; the caller counts the arrival one step later.
// ---------------------------------------------------------------------------
template <typename T>
__device__ int fw_stream(const SampleParams &p, FwRing &R, unsigned long long *full, int t, int s, int GW,
                         unsigned &phase, bool &timeout, int &slice, int &issued) {
    constexpr int VEC = Elem<T>::VEC;
    const int lane = threadIdx.x & 31;
    const int g = p.gamma, c = p.c;
    int k, b, j;
    fu_decode(t, c, p.B, k, b, j);
    const int pos = b * (g + 1) + k;
    const int rows = k < g ? 2 : 1;
    const int W = fw_slice_elems<T>();
    const int lo = j * W, n = min(W, p.V - lo);
    const int nvec = n / VEC;
    const float c2 = p.c2;
    int d = -1;
    if (k < g && lane == 0) d = p.tokens[(int64_t)b * g + k];
    const bool landed = mbar_wait_bounded(&full[s], (phase >> s) & 1u);
    if (!landed) timeout = true;
    phase ^= 1u << s;
    float2 res[2] = {make_float2(-INFINITY, 0.0f), make_float2(-INFINITY, 0.0f)};
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        if (r < rows) {
            const uint4 *src = reinterpret_cast<const uint4 *>(R.buf[s][r]);
            float x[kFwVecs][VEC];
#pragma unroll
            for (int i = 0; i < kFwVecs; ++i) {
                const int q = lane + 32 * i;
                if (q < nvec) {
                    unpack<T>(src[q], x[i]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) x[i][e] = -INFINITY;
                }
            }
            float m = -INFINITY;
#pragma unroll
            for (int i = 0; i < kFwVecs; ++i)
#pragma unroll
                for (int e = 0; e < VEC; ++e) m = fmaxf(m, x[i][e]);
            m = warp_max_f(m);
            float sum = 0.0f;
            if (m != -INFINITY) {
                const float mc = m * c2;
#pragma unroll
                for (int i = 0; i < kFwVecs; ++i)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) sum += ex2f(fmaf(x[i][e], c2, -mc));
            }
            res[r] = make_float2(m, warp_sum_f(sum));
        }
    }
    float2 xd = make_float2(0.0f, 0.0f);
    const bool stash = lane == 0 && d >= lo && d < lo + n;
    if (stash) {
        xd.x = to_f32(reinterpret_cast<const T *>(R.buf[s][0])[d - lo]);
        xd.y = to_f32(reinterpret_cast<const T *>(R.buf[s][1])[d - lo]);
    }
    __syncwarp();  // every lane is done with stage s
    if (lane == 0) {
        const int nt = t + kFwNST * GW;
        // (after a copy that did not land, nothing more is issued)
        if (nt < p.B * (g + 1) * c && !timeout) {
            fw_issue<T>(p, R, full, nt, s);
            ++issued;
        }
        p.fpart[((int64_t)pos * 2) * c + j] = res[0];
        if (rows > 1) p.fpart[((int64_t)pos * 2 + 1) * c + j] = res[1];
        if (stash) p.fxd[pos] = xd;
    }
    slice = j;
    return pos;
}

// ---------------------------------------------------------------------------
// Draw rounds
// ---------------------------------------------------------------------------
struct DrawCtx {
    int b, kstar, mode, pass, pos;
    const void *trow, *drow;
    float mp, sp, mq, sq;  // pass statistics of the drawn position
};

template <typename T>
__device__ __forceinline__ void fw_draw_ctx(const SampleParams &p, int b, DrawRec &dr, DrawCtx &cx) {
    const int g = p.gamma;
    const int4 *src = reinterpret_cast<const int4 *>(p.drec + b);
    const int4 h = __ldcg(src);
    dr.kstar = h.x;
    dr.mode = h.y;
    dr.pass = h.z;
    dr.pad = 0;
    dr.inv = __ldcg(reinterpret_cast<const float4 *>(src + 1));
    cx.b = b;
    cx.kstar = dr.kstar;
    cx.mode = dr.mode;
    cx.pass = dr.pass;
    cx.pos = b * (g + 1) + dr.kstar;
    cx.trow = reinterpret_cast<const T *>(p.target) + (int64_t)cx.pos * p.tstride;
    cx.drow = cx.mode == 0 ? reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + dr.kstar) * p.dstride
                           : nullptr;
    const float4 st = __ldcg(p.fstat + cx.pos);
    cx.mp = st.x;
    cx.sp = st.y;
    cx.mq = st.z;
    cx.sq = st.w;
}

// Lists the in-band elements flagged in each lane's mask (bit i: vector i/VEC,
// element i%VEC of the lane's strided vectors) into the slice's list; returns
// the slice's count (may exceed the list).
template <typename T>
__device__ __forceinline__ unsigned fw_list(const SampleParams &p, int b, int j, int lo, uint64_t mask) {
    constexpr int VEC = Elem<T>::VEC;
    const int lane = threadIdx.x & 31;
    const unsigned cnt = (unsigned)__popcll(mask);
    unsigned incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    const unsigned tot = __shfl_sync(kFull, incl, 31);
    unsigned at = incl - cnt;
    int *lst = p.amb + ((int64_t)b * p.c + j) * kFwAmb;
    while (mask) {
        const int bit = __ffsll((long long)mask) - 1;
        mask &= mask - 1ull;
        if (at < (unsigned)kFwAmb) lst[at] = lo + (lane + 32 * (bit / VEC)) * VEC + bit % VEC;
        ++at;
    }
    return tot;
}

// Loads this lane's vectors of slice j of both rows (every load at once).
template <typename T>
__device__ __forceinline__ void fw_load_slice(const SampleParams &p, const DrawCtx &cx, int j, uint4 (&va)[kFwVecs],
                                              uint4 (&vb)[kFwVecs]) {
    constexpr int VEC = Elem<T>::VEC;
    const int lane = threadIdx.x & 31;
    const int W = fw_slice_elems<T>(), lo = j * W, n = min(W, p.V - lo), nvec = n / VEC;
    const bool res = cx.mode == 0;
    const uint4 *ta = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(cx.trow) + lo);
    const uint4 *tb = res ? reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(cx.drow) + lo) : nullptr;
#pragma unroll
    for (int i = 0; i < kFwVecs; ++i) {
        const int q = lane + 32 * i;
        va[i] = q < nvec ? __ldcg(ta + q) : make_uint4(0u, 0u, 0u, 0u);
        vb[i] = (res && q < nvec) ? __ldcg(tb + q) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// Round 0 (fp32) sums of slice j from its loaded vectors: S_p, S_q and, over
// the elements classified into P, P_p and P_q, each as a compensated pair.
template <typename T>
__device__ void fw_round0_slice(const SampleParams &p, const DrawCtx &cx, int j, const uint4 (&va)[kFwVecs],
                                const uint4 (&vb)[kFwVecs]) {
    constexpr int VEC = Elem<T>::VEC;
    const int lane = threadIdx.x & 31;
    const int W = fw_slice_elems<T>(), lo = j * W, n = min(W, p.V - lo), nvec = n / VEC;
    const float c2 = p.c2, c2lo = p.c2lo;
    const bool res = cx.mode == 0;
    const float rho = res ? cx.sp / cx.sq : 0.0f;
    const float rhi = rho * (1.0f + kAmbRel), rlo = rho * (1.0f - kAmbRel);
    CSum acc[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};  // Sp Sq Pp Pq
    uint64_t amb = 0ull;
#pragma unroll
    for (int i = 0; i < kFwVecs; ++i) {
        const int q = lane + 32 * i;
        const bool valid = q < nvec;
        float xa[VEC], xb[VEC];
        unpack<T>(va[i], xa);
        unpack<T>(vb[i], xb);
        float vs[4][VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            // a -inf logit or a lane past the slice end is a zero term
            const float ep = valid ? ex2_exact(xa[e], cx.mp, c2, c2lo) : 0.0f;
            const float eq = (valid && res) ? ex2_exact(xb[e], cx.mq, c2, c2lo) : 0.0f;
            const bool inP = res && ep > eq * rhi;
            if (res && !inP && ep > 0.0f && ep >= eq * rlo) amb |= 1ull << (i * VEC + e);
            vs[0][e] = ep;
            vs[1][e] = eq;
            vs[2][e] = inP ? ep : 0.0f;
            vs[3][e] = inP ? eq : 0.0f;
        }
#pragma unroll
        for (int q2 = 0; q2 < 4; ++q2) {
#pragma unroll
            for (int wdt = VEC / 2; wdt > 0; wdt >>= 1)
#pragma unroll
                for (int e = 0; e < wdt; ++e) vs[q2][e] += vs[q2][e + wdt];
            csum_add(acc[q2], vs[q2][0]);
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = warp_csum(acc[q]);
    const unsigned na = res ? fw_list<T>(p, cx.b, j, lo, amb) : 0u;
    if (lane == 0) {
        DrawPart *dst = p.dpart + (int64_t)cx.b * p.c + j;
        float4 *v = reinterpret_cast<float4 *>(dst->v);
        v[0] = make_float4(acc[0].s, acc[0].c, acc[1].s, acc[1].c);
        v[1] = make_float4(acc[2].s, acc[2].c, acc[3].s, acc[3].c);
        v[2] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        dst->namb = na;
    }
}

// A lane's vectors of one slice, streamed two ahead of their use.
struct VecPipe {
    const uint4 *ta, *tb;
    int nvec, lane;
    uint4 a0, b0, a1, b1;
    __device__ __forceinline__ uint4 ld(const uint4 *base, int i) const {
        const int q = lane + 32 * i;
        return (base && q < nvec) ? __ldcg(base + q) : make_uint4(0u, 0u, 0u, 0u);
    }
    __device__ __forceinline__ void start() {
        a0 = ld(ta, 0);
        b0 = ld(tb, 0);
        a1 = ld(ta, 1);
        b1 = ld(tb, 1);
    }
    // vector i into (a, b); issues the load of vector i + 2
    __device__ __forceinline__ void next(int i, uint4 &a, uint4 &b) {
        a = a0;
        b = b0;
        a0 = a1;
        b0 = b1;
        a1 = ld(ta, i + 2);
        b1 = ld(tb, i + 2);
    }
};

template <typename T>
__device__ void fw_round1_slice(const SampleParams &p, const DrawCtx &cx, int j, const DdExpTables &K) {
    constexpr int VEC = Elem<T>::VEC;
    const int lane = threadIdx.x & 31;
    const int W = fw_slice_elems<T>(), lo = j * W, n = min(W, p.V - lo), nvec = n / VEC;
    const bool res = cx.mode == 0;
    const float rho = res ? cx.sp / cx.sq : 0.0f;
    const float rhi = rho * (1.0f + kAmbRel), rlo = rho * (1.0f - kAmbRel);
    const uint4 *ta = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(cx.trow) + lo);
    const uint4 *tb = res ? reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(cx.drow) + lo) : nullptr;
    dd acc[4] = {{0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}, {0.0f, 0.0f}};
    uint64_t amb = 0ull;
    VecPipe vp{ta, tb, nvec, lane};
    vp.start();
#pragma unroll 1
    for (int i = 0; i < kFwVecs; ++i) {
        const int q = lane + 32 * i;
        uint4 va, vb;
        vp.next(i, va, vb);
        if (q >= nvec) break;
        float xa[VEC], xb[VEC];
        unpack<T>(va, xa);
        unpack<T>(vb, xb);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const dd a = dd_expw(xa[e], cx.mp, K);
            acc[0] = dd_acc(acc[0], a);
            if (res) {
                const dd bq = dd_expw(xb[e], cx.mq, K);
                acc[1] = dd_acc(acc[1], bq);
                if (a.hi > bq.hi * rhi) {
                    acc[2] = dd_acc(acc[2], a);
                    acc[3] = dd_acc(acc[3], bq);
                } else if (a.hi > 0.0f && a.hi >= bq.hi * rlo) {
                    amb |= 1ull << (i * VEC + e);
                }
            }
        }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = warp_dd_sum(acc[q]);
    const unsigned na = res ? fw_list<T>(p, cx.b, j, lo, amb) : 0u;
    if (lane == 0) {
        DrawPart *dst = p.dpart + (int64_t)cx.b * p.c + j;
        float4 *v = reinterpret_cast<float4 *>(dst->v);
        v[0] = make_float4(acc[0].hi, acc[0].lo, acc[1].hi, acc[1].lo);
        v[1] = make_float4(acc[2].hi, acc[2].lo, acc[3].hi, acc[3].lo);
        v[2] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        dst->namb = na;
    }
}

// dd residual weight of a pair with the exact inverse normalisers
__device__ __forceinline__ dd fw_wres_dd(float x, float y, const DrawCtx &cx, dd isp, dd isq, const DdExpTables &K) {
    return dd_max0(dd_add(dd_mul(dd_expw(x, cx.mp, K), isp), dd_neg(dd_mul(dd_expw(y, cx.mq, K), isq))));
}

// Round 2 (dd residual) sum of slice j (words 8, 9 of the slice's record).
template <typename T>
__device__ void fw_round2_slice(const SampleParams &p, const DrawCtx &cx, const DrawRec &dr, int j,
                                const DdExpTables &K) {
    constexpr int VEC = Elem<T>::VEC;
    const int lane = threadIdx.x & 31;
    const int W = fw_slice_elems<T>(), lo = j * W, n = min(W, p.V - lo), nvec = n / VEC;
    const dd isp{dr.inv.x, dr.inv.y}, isq{dr.inv.z, dr.inv.w};
    const uint4 *ta = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(cx.trow) + lo);
    const uint4 *tb = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(cx.drow) + lo);
    dd acc{0.0f, 0.0f};
    VecPipe vp{ta, tb, nvec, lane};
    vp.start();
#pragma unroll 1
    for (int i = 0; i < kFwVecs; ++i) {
        const int q = lane + 32 * i;
        uint4 va, vb;
        vp.next(i, va, vb);
        if (q >= nvec) break;
        float xa[VEC], xb[VEC];
        unpack<T>(va, xa);
        unpack<T>(vb, xb);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc = dd_add(acc, fw_wres_dd(xa[e], xb[e], cx, isp, isq, K));
    }
    acc = warp_dd_sum(acc);
    if (lane == 0) {
        DrawPart *dst = p.dpart + (int64_t)cx.b * p.c + j;
        dst->v[8] = acc.hi;
        dst->v[9] = acc.lo;
    }
}

// One draw item: group q of request b's current round.  Returns its slices.
template <typename T>
__device__ __noinline__ int fw_draw_group(const SampleParams &p, unsigned long long item, const DdExpTables &K) {
    const int b = (int)((item >> 20) & 0x7fffffffull), q = (int)(item & 0xfffffull);
    DrawRec dr;
    DrawCtx cx;
    fw_draw_ctx<T>(p, b, dr, cx);
    const int gs = fw_group(cx.pass);
    const int j0 = q * gs, j1 = min(p.c, j0 + gs);
    if ((threadIdx.x & 31) == 0) {
        // the group's slices of both rows into L2 at once: only the first
        // slice's loads wait on HBM
        const int W = fw_slice_elems<T>(), lo = j0 * W, n = min(j1 * W, p.V) - lo;
        const uint32_t bytes = (uint32_t)n * (uint32_t)sizeof(T);
        bulk_prefetch_l2(reinterpret_cast<const T *>(cx.trow) + lo, bytes);
        if (cx.mode == 0) bulk_prefetch_l2(reinterpret_cast<const T *>(cx.drow) + lo, bytes);
    }
    for (int j = j0; j < j1; ++j) {
        if (cx.pass == 0) {
            uint4 va[kFwVecs], vb[kFwVecs];
            fw_load_slice<T>(p, cx, j, va, vb);
            fw_round0_slice<T>(p, cx, j, va, vb);
        } else if (cx.pass == 1) {
            fw_round1_slice<T>(p, cx, j, K);
        } else {
            fw_round2_slice<T>(p, cx, dr, j, K);
        }
    }
    __syncwarp();
    return j1 - j0;
}

// ---------------------------------------------------------------------------
// Phase ii: the warp that completed a round combines its slices and scans the
// slice holding the crossing.
// ---------------------------------------------------------------------------
// Loads EPL contiguous logits of a row starting at element i (16-byte
// aligned), -inf from element `valid` on.
template <typename T, int EPL>
__device__ __forceinline__ void fw_load_chunk(const T *row, int i, int valid, float (&x)[EPL]) {
    constexpr int VEC = Elem<T>::VEC;
#pragma unroll
    for (int v = 0; v < EPL / VEC; ++v) {
        float y[VEC];
        if (v * VEC < valid) {
            unpack<T>(__ldcg(reinterpret_cast<const uint4 *>(row + i) + v), y);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) y[e] = -INFINITY;
        }
#pragma unroll
        for (int e = 0; e < VEC; ++e) x[v * VEC + e] = y[e];
    }
}

struct Fp32Draw {  // globals of a certified round-0 draw
    float isp, isq, sigp, sigq;
    bool res, mode_p;
};

// round-0 weight and error bound of slice j (normalised units; mode_p:
// unnormalised target terms).  Record words: S_p 0-1, S_q 2-3, P_p 4-5,
// P_q 6-7 (compensated pairs).
__device__ __forceinline__ void fw_slice_w0(const Fp32Draw &f, const DrawPart &q, float L, float EL, dd &w,
                                           float &e) {
    if (f.mode_p) {
        w = dd{q.v[0], q.v[1]};
        e = (kTermErr + kSumErr) * q.v[0] * 1.001f;
    } else {
        w = dd_add(dd_add(dd_mul_f(dd{q.v[4], q.v[5]}, f.isp), dd_neg(dd_mul_f(dd{q.v[6], q.v[7]}, f.isq))),
                   dd{L, 0.0f});
        e = ((kTermErr + kSumErr + f.sigp + 3.0f * kU) * f.isp * q.v[4] +
             (kTermErr + kSumErr + f.sigq + 3.0f * kU) * f.isq * q.v[6] + EL) * 1.001f;
    }
}

// round 0: listed (in-band) elements of slice j: their residual sum and bound
template <typename T>
__device__ __forceinline__ void fw_listed0(const SampleParams &p, const DrawCtx &cx, const Fp32Draw &f, int j,
                                          unsigned na, float &L, float &EL) {
    const T *trow = reinterpret_cast<const T *>(cx.trow);
    const T *drow = reinterpret_cast<const T *>(cx.drow);
    const int *lst = p.amb + ((int64_t)cx.b * p.c + j) * kFwAmb;
    L = 0.0f;
    EL = 0.0f;
    for (unsigned x = 0; x < na; ++x) {
        const int i = __ldcg(lst + x);
        const float pp = __fmul_rn(ex2_exact(ld_elem(trow, i), cx.mp, p.c2, p.c2lo), f.isp);
        const float qq = __fmul_rn(ex2_exact(ld_elem(drow, i), cx.mq, p.c2, p.c2lo), f.isq);
        const float w = fmaxf(pp - qq, 0.0f);
        L += w;
        EL += pp * (kTermErr + f.sigp + 3.0f * kU) + qq * (kTermErr + f.sigq + 3.0f * kU) + kFwAmb * kU * w;
    }
    EL *= 1.001f;
}

// Final outcome of the draw: the token, the residual mass, the fallback bit.
__device__ void fw_finish_draw(const SampleParams &p, const DrawCtx &cx, int token, float z, bool fb) {
    if ((threadIdx.x & 31) == 0) {
        PosRec *r = p.recs + cx.pos;
        r->token = token;
        r->z = z;
        if (fb) r->info |= REC_FALLBACK;
        p.dcnt[cx.b] = 0u;
    }
    fu_draw_done(p, cx.b);
}

// Next round of request b: pass `pass` (inverse normalisers for round 2).
__device__ void fw_next_round(const SampleParams &p, const DrawCtx &cx, const DrawRec &dr, int pass, dd isp, dd isq) {
    if ((threadIdx.x & 31) == 0) {
        p.dcnt[cx.b] = 0u;
        DrawRec d = dr;
        d.pass = pass;
        d.inv = make_float4(isp.hi, isp.lo, isq.hi, isq.lo);
        p.drec[cx.b] = d;
    }
    fw_enqueue(p, cx.b, pass);
}

template <typename T>
__device__ __noinline__ void fw_phase2(const SampleParams &p, int b, const DdExpTables &K) {
    constexpr int VEC = Elem<T>::VEC;
    constexpr int EPL = kFwSlice / (int)sizeof(T) / 32;  // a lane's contiguous run in the scan
    const int lane = threadIdx.x & 31, c = p.c, g = p.gamma;
    DrawRec dr;
    DrawCtx cx;
    fw_draw_ctx<T>(p, b, dr, cx);
    const bool res = cx.mode == 0;
    const float c2 = p.c2;
    const float u_f = p.unif[(int64_t)b * (g + 1) + g];
    const T *trow = reinterpret_cast<const T *>(cx.trow);
    const T *drow = reinterpret_cast<const T *>(cx.drow);
    const DrawPart *parts = p.dpart + (int64_t)b * c;
    const int per = (c + 31) / 32, j0 = min(c, lane * per), j1 = min(c, j0 + per);  // this lane's slices
    const int W = fw_slice_elems<T>();
    auto load_part = [&](int j) -> DrawPart {
        DrawPart q;
        const float4 *src = reinterpret_cast<const float4 *>(parts + j);
        float4 *dst = reinterpret_cast<float4 *>(&q);
#pragma unroll
        for (int r = 0; r < 4; ++r) dst[r] = __ldcg(src + r);
        return q;
    };

    if (cx.pass == 0) {
        // ---- certified fp32 round ---------------------------------------
        Fp32Draw f;
        f.res = res;
        f.mode_p = !res;
        dd Sp{0.0f, 0.0f}, Sq{0.0f, 0.0f};
        unsigned ovf = 0u;
        for (int j = j0; j < j1; ++j) {
            const DrawPart q = load_part(j);
            Sp = dd_add(Sp, dd{q.v[0], q.v[1]});
            Sq = dd_add(Sq, dd{q.v[2], q.v[3]});
            ovf |= q.namb > (unsigned)kFwAmb ? 1u : 0u;
        }
        Sp = warp_dd_sum(Sp);
        Sq = warp_dd_sum(Sq);
        ovf = __reduce_or_sync(kFull, ovf);
        // relative error of the normalisers (summed in dd from the slices)
        f.sigp = (kTermErr + kSumErr) * 1.001f;
        f.sigq = res ? f.sigp : 0.0f;
        f.isp = __frcp_rn(dd_to_f(Sp));
        f.isq = res ? __frcp_rn(dd_to_f(Sq)) : 0.0f;
        bool ok = !ovf && Sp.hi > 0.0f;
        if (res) {
            // the classification by the pass's ratio estimate holds if its
            // error plus two terms' errors stays inside the band
            const float rho_t = cx.sp / cx.sq, rho_h = Sp.hi / Sq.hi;
            const float eta = fabsf(rho_t / rho_h - 1.0f) + f.sigp + f.sigq;
            ok = ok && Sq.hi > 0.0f && (eta + 2.0f * kTermErr + 4.0f * kU) * 1.01f < kAmbRel;
        }
        // the residual mass and its bound (the lane's totals are also the
        // owner search's when the draw is from the residual)
        bool fb = false;
        dd Z{0.0f, 0.0f}, zl_lane{0.0f, 0.0f};
        float el_lane = 0.0f;
        if (ok && res) {
            for (int j = j0; j < j1; ++j) {
                const DrawPart q = load_part(j);
                float L, EL, e;
                fw_listed0<T>(p, cx, f, j, q.namb, L, EL);
                dd w;
                fw_slice_w0(f, q, L, EL, w, e);
                zl_lane = dd_add(zl_lane, w);
                el_lane += e;
            }
            Z = warp_dd_sum(zl_lane);
            const float errZ = warp_sum_f(el_lane);
            const float zf = dd_to_f(Z);
            if (zf - errZ > p.eps) fb = false;
            else if (zf + errZ <= p.eps) fb = true;
            else ok = false;
            f.mode_p = fb;
        }
        // the owner slice: per-lane totals, a lane prefix, then the owner
        // lane walks its slices
        int jstar = -1;
        float E = 0.0f, trel = 0.0f;
        if (ok) {
            const dd t = dd_mul_f(f.mode_p ? Sp : Z, u_f);
            dd lw = zl_lane;
            float le = el_lane;
            if (f.mode_p) {
                lw = dd{0.0f, 0.0f};
                le = 0.0f;
                for (int j = j0; j < j1; ++j) {
                    const DrawPart q = load_part(j);
                    dd w;
                    float e;
                    fw_slice_w0(f, q, 0.0f, 0.0f, w, e);
                    lw = dd_add(lw, w);
                    le += e;
                }
            }
            const dd incl = warp_dd_incl(lw);
            const dd excl = dd_add(incl, dd_neg(lw));
            const float etot = warp_sum_f(le);
            const unsigned own = __ballot_sync(kFull, j0 < j1 && dd_gt(incl, t));
            int jl = -1;
            dd cl{0.0f, 0.0f};
            float ej = 0.0f;
            if (own && lane == __ffs(own) - 1) {
                dd cum = excl;
                for (int j = j0; j < j1; ++j) {
                    const DrawPart q = load_part(j);
                    float L = 0.0f, EL = 0.0f, e;
                    if (!f.mode_p) fw_listed0<T>(p, cx, f, j, q.namb, L, EL);
                    dd w;
                    fw_slice_w0(f, q, L, EL, w, e);
                    if (dd_pos(w) && dd_gt(dd_add(cum, w), t)) {
                        jl = j;
                        cl = cum;
                        ej = e;
                        break;
                    }
                    cum = dd_add(cum, w);
                }
            }
            dd carry{0.0f, 0.0f};
            if (own) {
                const int src = __ffs(own) - 1;
                jstar = __shfl_sync(kFull, jl, src);
                carry = shfl_dd(cl, src);
                ej = __shfl_sync(kFull, ej, src);
            }
            const float tt = dd_to_f(t);
            E = (fmaxf(u_f, 1.0f - u_f) * etot + ej + 4.0f * kU * tt) * 1.01f;
            trel = dd_to_f(dd_add(t, dd_neg(carry)));
            if (jstar < 0) ok = false;
        }
        if (ok) {
            // token-order scan of slice j*: lane `lane` owns [lo + lane*EPL, +EPL)
            const int lo = jstar * W, n = min(W, p.V - lo);
            const int i0 = lo + lane * EPL, valid = max(0, min(EPL, n - lane * EPL));
            auto weight = [&](const float *xa, const float *xb, int e) -> float {
                const float ep = ex2_exact(xa[e], cx.mp, c2, p.c2lo);
                if (f.mode_p) return ep;
                const float eq = ex2_exact(xb[e], cx.mq, c2, p.c2lo);
                return fmaxf(__fmul_rn(ep, f.isp) - __fmul_rn(eq, f.isq), 0.0f);
            };
            float run = 0.0f;
            {
                float xa[EPL], xb[EPL];
                fw_load_chunk<T, EPL>(trow, i0, valid, xa);
                if (!f.mode_p) fw_load_chunk<T, EPL>(drow, i0, valid, xb);
#pragma unroll
                for (int e = 0; e < EPL; ++e) run += weight(xa, xb, e);
            }
            float incl = run;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            const float stot = __shfl_sync(kFull, incl, 31);
            float cum = incl - run;
            int hit = INT_MAX;
            float m1 = 0.0f, m2 = 0.0f;
            {
                float xa[EPL], xb[EPL];
                fw_load_chunk<T, EPL>(trow, i0, valid, xa);
                if (!f.mode_p) fw_load_chunk<T, EPL>(drow, i0, valid, xb);
#pragma unroll
                for (int e = 0; e < EPL; ++e) {
                    const float w = weight(xa, xb, e);
                    const float prev = cum;
                    cum += w;
                    if (hit == INT_MAX && w > 0.0f && cum > trel) {
                        hit = i0 + e;
                        m1 = trel - prev;
                        m2 = cum - trel;
                    }
                }
            }
            const unsigned hb = __ballot_sync(kFull, hit != INT_MAX);
            if (hb) {
                const int src = __ffs(hb) - 1;  // lanes are in token order
                const int token = __shfl_sync(kFull, hit, src);
                m1 = __shfl_sync(kFull, m1, src);
                m2 = __shfl_sync(kFull, m2, src);
                const float rscan = kScanDepth * kU * 1.001f * stot + 2.0f * kU * fabsf(trel);
                if (fminf(m1, m2) > E + rscan) {
                    fw_finish_draw(p, cx, token, res ? dd_to_f(Z) : 0.0f, fb);
                    return;
                }
            }
        }
        fw_next_round(p, cx, dr, 1, dd{0.0f, 0.0f}, dd{0.0f, 0.0f});
        return;
    }

    // ---- double-float rounds ----------------------------------------------
    dd Sp{0.0f, 0.0f}, Sq{0.0f, 0.0f};
    unsigned ovf = 0u;
    for (int j = j0; j < j1; ++j) {
        const DrawPart q = load_part(j);
        Sp = dd_add(Sp, dd{q.v[0], q.v[1]});
        Sq = dd_add(Sq, dd{q.v[2], q.v[3]});
        ovf |= q.namb > (unsigned)kFwAmb ? 1u : 0u;
    }
    Sp = warp_dd_sum(Sp);
    Sq = warp_dd_sum(Sq);
    ovf = __reduce_or_sync(kFull, ovf);
    const dd isp = dd_recip(Sp), isq = res ? dd_recip(Sq) : dd{0.0f, 0.0f};
    if (res && cx.pass == 1) {
        // the listing is exact only if the pass's ratio estimate is well
        // inside the band; otherwise (or on overflow) round 2
        const float rho_t = cx.sp / cx.sq, rho_h = Sp.hi / Sq.hi;
        if (ovf || !(fabsf(rho_t / rho_h - 1.0f) < 0.5f * kAmbRel)) {
            fw_next_round(p, cx, dr, 2, isp, isq);
            return;
        }
    }
    auto wres = [&](int j, const DrawPart &q) -> dd {
        if (cx.pass == 2) return dd{q.v[8], q.v[9]};
        dd L{0.0f, 0.0f};
        const int *lst = p.amb + ((int64_t)b * c + j) * kFwAmb;
        for (unsigned x = 0; x < q.namb; ++x) {
            const int i = __ldcg(lst + x);
            L = dd_add(L, fw_wres_dd(ld_elem(trow, i), ld_elem(drow, i), cx, isp, isq, K));
        }
        return dd_add(dd_add(dd_mul(dd{q.v[4], q.v[5]}, isp), dd_neg(dd_mul(dd{q.v[6], q.v[7]}, isq))), L);
    };
    dd Z{0.0f, 0.0f};
    bool fb = false;
    if (res) {
        dd zl{0.0f, 0.0f};
        for (int j = j0; j < j1; ++j) zl = dd_add(zl, wres(j, load_part(j)));
        Z = warp_dd_sum(zl);
        fb = dd_le(Z, dd{p.eps, 0.0f});
    }
    const bool mode_p = !res || fb;
    const dd t = dd_mul_f(mode_p ? Sp : Z, u_f);
    auto wslice = [&](int j) -> dd {
        const DrawPart q = load_part(j);
        return mode_p ? dd{q.v[0], q.v[1]} : wres(j, q);
    };
    dd lw{0.0f, 0.0f};
    int lastj = -1;
    for (int j = j0; j < j1; ++j) {
        const dd w = wslice(j);
        if (dd_pos(w)) lastj = j;
        lw = dd_add(lw, w);
    }
    const dd incl = warp_dd_incl(lw);
    const dd excl = dd_add(incl, dd_neg(lw));
    const unsigned own = __ballot_sync(kFull, j0 < j1 && dd_gt(incl, t));
    // the owner lane (or, if rounding leaves none, the last lane with weight)
    const unsigned haspos = __ballot_sync(kFull, lastj >= 0);
    const int src = own ? __ffs(own) - 1 : (haspos ? 31 - __clz(haspos) : -1);
    int jstar = -1;
    dd carry{0.0f, 0.0f};
    if (src >= 0) {
        int jl = -1;
        dd cl{0.0f, 0.0f};
        if (lane == src) {
            dd cum = excl;
            int lj = -1;
            dd lc{0.0f, 0.0f};
            for (int j = j0; j < j1; ++j) {
                const dd w = wslice(j);
                if (dd_pos(w)) {
                    if (own && dd_gt(dd_add(cum, w), t)) {
                        jl = j;
                        cl = cum;
                        break;
                    }
                    lj = j;
                    lc = cum;
                }
                cum = dd_add(cum, w);
            }
            if (jl < 0) {
                jl = lj;
                cl = lc;
            }
        }
        jstar = __shfl_sync(kFull, jl, src);
        carry = shfl_dd(cl, src);
    }
    int token = -1;
    if (jstar >= 0) {
        const dd trel = dd_add(t, dd_neg(carry));
        const int lo = jstar * W, n = min(W, p.V - lo);
        const int i0 = lo + lane * EPL, valid = max(0, min(EPL, n - lane * EPL));
        auto wdd = [&](float xa, float xb) -> dd {
            const dd a = dd_expw(xa, cx.mp, K);
            return mode_p ? a : dd_max0(dd_add(dd_mul(a, isp), dd_neg(dd_mul(dd_expw(xb, cx.mq, K), isq))));
        };
        dd run{0.0f, 0.0f};
        for (int v = 0; v < EPL / VEC; ++v) {
            if (v * VEC >= valid) break;
            float xa[VEC], xb[VEC];
            unpack<T>(__ldcg(reinterpret_cast<const uint4 *>(trow + i0) + v), xa);
            if (!mode_p) unpack<T>(__ldcg(reinterpret_cast<const uint4 *>(drow + i0) + v), xb);
#pragma unroll
            for (int e = 0; e < VEC; ++e) run = dd_add(run, wdd(xa[e], mode_p ? 0.0f : xb[e]));
        }
        const dd sincl = warp_dd_incl(run);
        dd cum = dd_add(sincl, dd_neg(run));
        int hit = INT_MAX, lastp = -1;
        for (int v = 0; v < EPL / VEC; ++v) {
            if (v * VEC >= valid) break;
            float xa[VEC], xb[VEC];
            unpack<T>(__ldcg(reinterpret_cast<const uint4 *>(trow + i0) + v), xa);
            if (!mode_p) unpack<T>(__ldcg(reinterpret_cast<const uint4 *>(drow + i0) + v), xb);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                const dd w = wdd(xa[e], mode_p ? 0.0f : xb[e]);
                cum = dd_add(cum, w);
                if (dd_pos(w)) {
                    lastp = i0 + v * VEC + e;
                    if (hit == INT_MAX && dd_gt(cum, trel)) hit = lastp;
                }
            }
        }
        const unsigned hb = __ballot_sync(kFull, hit != INT_MAX);
        if (hb) {
            token = __shfl_sync(kFull, hit, __ffs(hb) - 1);
        } else {
            const unsigned lb = __ballot_sync(kFull, lastp >= 0);
            if (lb) token = __shfl_sync(kFull, lastp, 31 - __clz(lb));
        }
    }
    fw_finish_draw(p, cx, token, res ? dd_to_f(Z) : 0.0f, fb);
}

// ---------------------------------------------------------------------------
// The persistent kernel: every warp loops over its own work.  Each step is a
// decision or phase ii this warp owns and whose arrivals are complete, a draw
// item whose queue slot this warp holds, the next stream item, or (nothing
// left) a short sleep until every request is done.
//
// Arrivals are fire-and-forget (red.release), counted one step after the
// results were written.  A follow-up belongs to a fixed warp, never to the
// last arriver (which would make a late warp later still): the warp that
// streamed a position's first slice decides it, the warp that took a round's
// first group runs its phase ii.  It keeps them in a small watch list and
// reads the head's counter one step ahead.
// ---------------------------------------------------------------------------
enum FwCmd { kCmdStream = 0, kCmdDraw = 1, kCmdDecide = 2, kCmdPhase2 = 3, kCmdIdle = 4, kCmdDone = 5 };
constexpr int kWatch = 16;  // watch list entries per warp (a power of two)

template <typename T>
__global__ void __launch_bounds__(kFwWarps * 32, 1) chain_full_kernel(SampleParams p) {
    __shared__ unsigned long long full[kFwWarps][kFwNST];
    __shared__ int2 watch[kFwWarps][kWatch];  // (command, position or request)
    __shared__ DdExpTables K;
    extern __shared__ __align__(128) unsigned char dsm[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    FwRing &R = reinterpret_cast<FwRing *>(dsm)[w];
    unsigned long long *fb = full[w];
    int2 *wl = watch[w];
    const int nitems = p.B * (p.gamma + 1) * p.c;
    const int GW = (int)gridDim.x * kFwWarps;
    FuCtl *ctl = fu_ctl(p);
    {
        constexpr int NW = (int)(sizeof(DdExpTables) / sizeof(uint32_t));
        const uint32_t *src = reinterpret_cast<const uint32_t *>(&p.exptab);
        uint32_t *dst = reinterpret_cast<uint32_t *>(&K);
        for (int i = threadIdx.x; i < NW; i += blockDim.x) dst[i] = src[i];
    }
    int t = (int)blockIdx.x * kFwWarps + w, it = 0;
    int issued = 0;  // lane 0: stream items of this warp whose copies were issued
    if (lane == 0) {
        for (int s = 0; s < kFwNST; ++s) mbar_init(&fb[s], 1);
        fence_barrier_init();
        for (int s = 0; s < kFwNST; ++s) {
            const int ts = t + s * GW;
            if (ts < nitems) {
                fw_issue<T>(p, R, fb, ts, s);
                ++issued;
            }
        }
    }
    __syncthreads();  // the exponential's tables; from here on warps are independent
    unsigned phase = 0u;
    bool timeout = false;
    // lane 0's state: the queue slot it holds and values read ahead, the
    // arrival still to count, the watch list
    unsigned ticket = 0xffffffffu, tail_pf = 0u, head_pf = 0u, nfin_pf = 0u;
    bool ticket_new = false;
    unsigned long long slot_pf = 0ull;
    unsigned *due = nullptr;
    unsigned due_n = 0u;
    int wh = 0, wt = 0;  // watch list head and tail (running counts)
    unsigned watch_pf = 0u;
    bool watch_pf_ok = false;
    long long idle = 0;
    auto watch_counter = [&](int2 e) -> const unsigned * {
        return e.x == kCmdDecide ? p.pcnt + e.y : p.dcnt + e.y;
    };
    for (;;) {
        int cmd = -1, arg = 0;
        unsigned long long item = 0ull;
        if (lane == 0) {
            // count last step's arrival: its writes are done by now
            if (due) {
                red_add_release(due, due_n);
                due = nullptr;
            }
            if (wh < wt && watch_pf_ok && watch_pf >= (unsigned)p.c) {
                const int2 e = wl[wh & (kWatch - 1)];
                cmd = e.x;
                arg = e.y;
                ++wh;
                watch_pf_ok = false;
            }
            // new work only while the watch list has room for its entry
            const bool room = wt - wh <= kWatch - 2;
            if (cmd < 0) {
                if (ticket != 0xffffffffu && slot_pf != 0ull) {
                    item = slot_pf;
                    p.qitem[ticket] = 0ull;
                    ticket = 0xffffffffu;
                    slot_pf = 0ull;
                    cmd = kCmdDraw;
                } else if (room && ticket == 0xffffffffu && tail_pf > head_pf) {
                    // several warps may claim on the same stale view, so a
                    // ticket can pass the tail (its slot is filled later) or
                    // the queue's end (never filled: dropped; no producer
                    // writes past qcap, and once the head is there no view
                    // shows tail > head again)
                    ticket = atomicAdd(&ctl->head, 1u);
                    ticket_new = true;
                    if (ticket >= p.qcap) ticket = 0xffffffffu;
                }
            }
            if (cmd < 0 && room && t < nitems) cmd = kCmdStream;
            if (cmd < 0) {
                if (wh == wt && nfin_pf >= (unsigned)p.B) {
                    cmd = kCmdDone;
                } else if (++idle > p.idle_limit) {
                    timeout = true;
                    cmd = kCmdDone;
                } else {
                    cmd = kCmdIdle;
                }
            }
            // read ahead for the next step
            if (cmd != kCmdDone) {
                tail_pf = ld_relaxed_u32(&ctl->tail);
                head_pf = ld_relaxed_u32(&ctl->head);
                nfin_pf = ld_relaxed_u32(&ctl->nfin);
                if (ticket != 0xffffffffu && !ticket_new) slot_pf = ld_acquire_u64(p.qitem + ticket);
                ticket_new = false;
                if (wh < wt) {
                    watch_pf = ld_acquire_u32(watch_counter(wl[wh & (kWatch - 1)]));
                    watch_pf_ok = true;
                }
            }
        }
        cmd = __shfl_sync(kFull, cmd, 0);
        arg = __shfl_sync(kFull, arg, 0);
        item = __shfl_sync(kFull, item, 0);
        __syncwarp();  // lane 0's acquire orders the whole warp's loads after it
        if (cmd == kCmdDone) break;
        if (cmd == kCmdStream) {
            int j = 0;
            const int pos = fw_stream<T>(p, R, fb, t, it % kFwNST, GW, phase, timeout, j, issued);
            if (__shfl_sync(kFull, timeout ? 1 : 0, 0)) {  // a copy did not land: stop
                ++it;
                break;
            }
            if (lane == 0) {
                due = p.pcnt + pos;
                due_n = 1u;
                if (j == 0) wl[(wt++) & (kWatch - 1)] = make_int2(kCmdDecide, pos);  // owner
            }
            t += GW;
            ++it;
            idle = 0;
        } else if (cmd == kCmdDraw) {
            const int ns = fw_draw_group<T>(p, item, K);
            if (lane == 0) {
                const int b = (int)((item >> 20) & 0x7fffffffull), q = (int)(item & 0xfffffull);
                due = p.dcnt + b;
                due_n = (unsigned)ns;
                if (q == 0) wl[(wt++) & (kWatch - 1)] = make_int2(kCmdPhase2, b);  // owner
            }
            idle = 0;
        } else if (cmd == kCmdDecide) {
            fu_decide(p, arg);
            idle = 0;
        } else if (cmd == kCmdPhase2) {
            fw_phase2<T>(p, arg, K);
            idle = 0;
        } else {
            if (lane == 0) __nanosleep(300);
            __syncwarp();
        }
    }
    __syncwarp();
    if (lane == 0) {
        if (timeout) atomicOr(p.status, SPEC_FLAG_TIMEOUT);
        // copies issued and not consumed (a wait gave up, or the warp left on
        // the idle limit with items ahead): wait for them (bounded) before
        // the block's shared memory may be reused, from the last item whose
        // wait may have failed
        bool drained = true;
        for (int q = timeout ? it - 1 : it; q < issued; ++q)
            if (q >= 0) drained &= mbar_drain(&fb[q % kFwNST], (unsigned)((q / kFwNST) & 1));
        if (drained)
            for (int s = 0; s < kFwNST; ++s) mbar_inval(&fb[s]);
        __threadfence();
        if (atomicAdd(&ctl->nexit, 1u) == (unsigned)(GW - 1)) {
            ctl->head = 0u;
            ctl->tail = 0u;
            ctl->nfin = 0u;
            ctl->nexit = 0u;
        }
    }
}

template <typename T> static cudaError_t launch_full_t(const SampleParams &p, int sms, cudaStream_t s) {
    static std::atomic<unsigned long long> done{0};
    const int dyn = (int)(kFwWarps * sizeof(FwRing));
    cudaError_t e = ensure_smem_attr(chain_full_kernel<T>, dyn, done);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, chain_full_kernel<T>, kFwWarps * 32, dyn);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int64_t nitems = (int64_t)p.B * (p.gamma + 1) * p.c;
    int64_t grid = (int64_t)sms * per_sm;
    const int64_t need = (nitems + kFwWarps - 1) / kFwWarps;
    if (grid > need) grid = need;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kFwWarps * 32);
    cfg.dynamicSmemBytes = (size_t)dyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every block resident: waits on other warps end
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, chain_full_kernel<T>, p);
}

cudaError_t launch_chain_full(const SampleParams &p, int dtype, int sms, cudaStream_t s) {
    return dtype == SPEC_DTYPE_BF16 ? launch_full_t<__nv_bfloat16>(p, sms, s) : launch_full_t<float>(p, sms, s);
}

}  // namespace specv
