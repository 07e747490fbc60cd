// Device pieces shared by the sampled chain-verification kernels.
//
// verify_sample.cu runs one thread-block cluster per (position, request)
// for full-vocabulary rows and for top-k rows whose threshold needs the
// exact cluster-wide search; verify_topk.cu runs cluster-free kernels for
// top-k rows.  Both end each position with finish() (record + request
// epilogue); masked_position() below is the exact computation of one
// position, over a cluster or over whole rows in one block.
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "ddmath.cuh"
#include "kernels.h"
#include "select.cuh"
#include "tma.cuh"

namespace specv {

namespace cg = cooperative_groups;

constexpr int kNT = 256;
constexpr int kNW = kNT / 32;
constexpr int kMaxCluster = 8;
constexpr int kSeg = 256;        // candidates one top-k slice may contribute per row
constexpr int kScanE = 8;        // elements per thread per tile of the token-order scan
constexpr int kKeptMax = kKeptRowMax;  // kept (top-k) entries per row a position can sort
constexpr int kAmbMax = 128;     // residual elements per CTA left to the exact sums (more: a full pass)
// Margin of the residual classification: p_i > q_i is decided from the fp32
// estimate of S_p/S_q (relative error below ~2e-5) only outside this band.
constexpr float kAmbRel = 1.0f / 1024.0f;

// Dynamic shared memory of the masked path: rows stream through a ring.
constexpr int kRingCH = 8192, kRingNST = 4;
using SampRing = Ring<kRingCH, kRingNST, 2>;
constexpr size_t kSampDyn = sizeof(SampRing);

struct SampBase {
    float2 red2[kNW];
    float redf[kNW];
    unsigned redu[kNW];
    float4 redd[kNW];
    float4 ms[kMaxCluster];       // pushed (m_p, s_p, m_q, s_q) per rank
    float4 dsum[kMaxCluster];     // pushed dd pair of sums per rank
    float zdiag[kMaxCluster];     // pushed fp32 residual mass per rank
    unsigned cnt[2][2][kMaxCluster];
    float4 dsum2[kMaxCluster];    // pushed residual mass (dd) per rank
    unsigned ovfr[kMaxCluster];   // pushed list-overflow bit per rank
    int namb;                     // ambiguous residual elements listed by this CTA
    int amb[kAmbMax];             // their indices
    unsigned rej;                 // earliest-rejection word, pushed by rank 0
    int found, lastpos;
    double redD[kNW];             // the nucleus search: warp totals
    double nuc_above;             //   mass above the chosen digit, pushed by rank 0
    unsigned nuc_dig;             //   the chosen digit, pushed by rank 0
    int nuc_found;
    DdExpTables K;                // the double-float exponential's constants
};

// copies the exponential's constants into shared memory (every thread calls;
// a block barrier must follow before use)
__device__ __forceinline__ void load_exp_tables(const SampleParams &p, SampBase &sb) {
    constexpr int W = (int)(sizeof(DdExpTables) / sizeof(uint32_t));
    static_assert(sizeof(DdExpTables) % sizeof(uint32_t) == 0, "word copy");
    const uint32_t *src = reinterpret_cast<const uint32_t *>(&p.exptab);
    uint32_t *dst = reinterpret_cast<uint32_t *>(&sb.K);
    for (int i = threadIdx.x; i < W; i += blockDim.x) dst[i] = src[i];
}

struct Outcome {
    float a, z;
    int token;
    unsigned info;
};

template <typename T> __device__ __forceinline__ uint32_t kkey(float x) {
    return fkey(x) >> (32 - Elem<T>::KEY_BITS);
}
template <typename T> __device__ __forceinline__ float key_value(uint32_t kk) {
    const uint32_t f = kk << (32 - Elem<T>::KEY_BITS);
    const uint32_t u = (f & 0x80000000u) ? (f & 0x7fffffffu) : ~f;
    return __uint_as_float(Elem<T>::KEY_BITS == 16 ? (u & 0xffff0000u) : u);
}

// Two rows traversed together over one slice: f(xa[VEC], xb[VEC], base, cnt).
template <typename T, int UNROLL, typename F>
__device__ __forceinline__ void for_slice2(const T *ra, const T *rb, int lo, int hi, F &&f) {
    constexpr int VEC = Elem<T>::VEC;
    const int tid = threadIdx.x, nt = blockDim.x;
    if (hi <= lo) return;
    const uintptr_t a = reinterpret_cast<uintptr_t>(ra + lo);
    const bool same_phase = ((a ^ reinterpret_cast<uintptr_t>(rb + lo)) & 15u) == 0;
    int head = (int)(((16u - (unsigned)(a & 15u)) & 15u) / sizeof(T));
    if (head > hi - lo) head = hi - lo;
    const int body0 = lo + head;
    const int nvec = (hi - body0) / VEC;
    const int tail0 = body0 + nvec * VEC;
    if (tid < head) {
        float xa[VEC], xb[VEC];
        xa[0] = ld_elem(ra, lo + tid);
        xb[0] = ld_elem(rb, lo + tid);
        f(xa, xb, lo + tid, 1);
    }
    const uint4 *va = reinterpret_cast<const uint4 *>(ra + body0);
    const uint4 *vb = reinterpret_cast<const uint4 *>(rb + body0);
    int v = tid;
    if (same_phase) {
        for (; v + (UNROLL - 1) * nt < nvec; v += UNROLL * nt) {
            uint4 qa[UNROLL], qb[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                qa[u] = ld_nc16(va + v + u * nt);
                qb[u] = ld_nc16(vb + v + u * nt);
            }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                float xa[VEC], xb[VEC];
                unpack<T>(qa[u], xa);
                unpack<T>(qb[u], xb);
                f(xa, xb, body0 + (v + u * nt) * VEC, VEC);
            }
        }
    }
    for (; v < nvec; v += nt) {
        float xa[VEC], xb[VEC];
        unpack<T>(ld_nc16(va + v), xa);
        const int base = body0 + v * VEC;
        if (same_phase) {
            unpack<T>(ld_nc16(vb + v), xb);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) xb[e] = ld_elem(rb, base + e);
        }
        f(xa, xb, base, VEC);
    }
    if (tid < hi - tail0) {
        float xa[VEC], xb[VEC];
        xa[0] = ld_elem(ra, tail0 + tid);
        xb[0] = ld_elem(rb, tail0 + tid);
        f(xa, xb, tail0 + tid, 1);
    }
}

// Streams slice [lo, hi) of one row (drow == nullptr) or two rows: the scalar
// head and tail from global memory, the 16-byte body through the bulk-copy
// ring.  f(xa[VEC], xb[VEC], base, cnt) as in for_slice2.  Rows whose 16-byte
// phases differ take the register path instead.  Returns false on a wait
// timeout.
template <typename T, int CH, int NST, typename F>
__device__ bool stream_rows(Ring<CH, NST, 2> &R, const T *trow, const T *drow, int lo, int hi, F &&f) {
    constexpr int VEC = Elem<T>::VEC;
    const int tid = threadIdx.x;
    const SliceSplit sp = split_slice(trow, lo, hi);
    const bool two = drow != nullptr;
    const bool same = !two ||
        ((reinterpret_cast<uintptr_t>(trow + lo) ^ reinterpret_cast<uintptr_t>(drow + lo)) & 15u) == 0;
    if (!same) {
        for_slice2<T, 2>(trow, drow, lo, hi, f);
        return true;
    }
    const int nhead = sp.body0 - sp.head0, ntail = sp.hi - sp.tail0;
    if (tid < nhead) {
        float xa[VEC], xb[VEC];
        xa[0] = ld_elem(trow, sp.head0 + tid);
        xb[0] = two ? ld_elem(drow, sp.head0 + tid) : 0.0f;
        f(xa, xb, sp.head0 + tid, 1);
    }
    bool ok = true;
    const uint32_t nbytes = (uint32_t)((sp.tail0 - sp.body0) * (int)sizeof(T));
    if (nbytes > 0) {
        const unsigned char *src[2] = {reinterpret_cast<const unsigned char *>(trow + sp.body0),
                                       two ? reinterpret_cast<const unsigned char *>(drow + sp.body0) : nullptr};
        ok = ring_stream(R, src, two ? 2 : 1, nbytes,
                         [&](const unsigned char *const *st, uint32_t off, uint32_t bytes) {
            const uint4 *va = reinterpret_cast<const uint4 *>(st[0]);
            const uint4 *vb = reinterpret_cast<const uint4 *>(st[1]);
            const int nv = (int)(bytes / 16);
            const int base0 = sp.body0 + (int)(off / sizeof(T));
            for (int q = tid; q < nv; q += kNT) {
                float xa[VEC], xb[VEC];
                unpack<T>(va[q], xa);
                if (two) unpack<T>(vb[q], xb);
                f(xa, xb, base0 + q * VEC, VEC);
            }
        });
    }
    if (tid < ntail) {
        float xa[VEC], xb[VEC];
        xa[0] = ld_elem(trow, sp.tail0 + tid);
        xb[0] = two ? ld_elem(drow, sp.tail0 + tid) : 0.0f;
        f(xa, xb, sp.tail0 + tid, 1);
    }
    return ok;
}

// Online (max, sum) update of one row with one vector of values.
template <int VEC, bool MASK>
__device__ __forceinline__ void ms_update(MaxSum &ms, const float *x, int cnt, uint32_t th,
                                          int ks, float c2) {
    float vm = -INFINITY;
#pragma unroll
    for (int e = 0; e < VEC; ++e)
        if (e < cnt && (!MASK || (fkey(x[e]) >> ks) >= th)) vm = fmaxf(vm, x[e]);
    if (vm > ms.m) {
        ms.s = ms.m == -INFINITY ? 0.0f : ms.s * exp2f((ms.m - vm) * c2);
        ms.m = vm;
    }
    if (ms.m != -INFINITY) {
        const float mc = ms.m * c2;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (e < cnt && (!MASK || (fkey(x[e]) >> ks) >= th)) ms.s += exp2f(fmaf(x[e], c2, -mc));
    }
}

// block-wide dd sum of two accumulators (every thread gets both)
template <int NT>
__device__ __forceinline__ void block_dd_sum2(dd &a, dd &b, float4 *red) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    a = warp_dd_sum(a);
    b = warp_dd_sum(b);
    sync_nt<kNT>();
    if (lane == 0) red[w] = make_float4(a.hi, a.lo, b.hi, b.lo);
    sync_nt<kNT>();
    dd ta{0.0f, 0.0f}, tb{0.0f, 0.0f};
    for (int i = 0; i < NT / 32; ++i) {
        ta = dd_add(ta, dd{red[i].x, red[i].y});
        tb = dd_add(tb, dd{red[i].z, red[i].w});
    }
    a = ta;
    b = tb;
}

// ---------------------------------------------------------------------------
// Token-order scan of one slice: the smallest i in [lo, hi) whose running sum
// (starting at `carry`) exceeds t, among positive weights; if rounding leaves
// none, the last positive-weight index.  weight(i) returns a dd.
// ---------------------------------------------------------------------------
template <int NT, typename W>
__device__ int dd_scan_slice(int lo, int hi, dd carry, dd t, W &&weight, SampBase &sb) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) { sb.found = INT_MAX; sb.lastpos = -1; }
    sync_nt<kNT>();
    for (int base = lo; base < hi; base += NT * kScanE) {
        const int i0 = base + tid * kScanE;
        dd w[kScanE];
        dd run{0.0f, 0.0f};
        int lastp = -1;
#pragma unroll
        for (int e = 0; e < kScanE; ++e) {
            const int i = i0 + e;
            w[e] = i < hi ? weight(i) : dd{0.0f, 0.0f};
            run = dd_add(run, w[e]);
            if (dd_pos(w[e])) lastp = i;
        }
        // inclusive warp scan of the thread totals, then warp totals
        dd incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const dd y{__shfl_up_sync(kFull, incl.hi, o), __shfl_up_sync(kFull, incl.lo, o)};
            if (lane >= o) incl = dd_add(y, incl);
        }
        sync_nt<kNT>();
        if (lane == 31) sb.redd[wid] = make_float4(incl.hi, incl.lo, 0.0f, 0.0f);
        sync_nt<kNT>();
        dd wpre{0.0f, 0.0f}, tile{0.0f, 0.0f};
        for (int q = 0; q < NT / 32; ++q) {
            const dd x{sb.redd[q].x, sb.redd[q].y};
            if (q < wid) wpre = dd_add(wpre, x);
            tile = dd_add(tile, x);
        }
        // exclusive prefix of this thread = carry + earlier warps + earlier lanes
        const dd lane_excl{__shfl_up_sync(kFull, incl.hi, 1), __shfl_up_sync(kFull, incl.lo, 1)};
        dd cum = dd_add(carry, wpre);
        if (lane > 0) cum = dd_add(cum, lane_excl);
        int hit = INT_MAX;
#pragma unroll
        for (int e = 0; e < kScanE; ++e) {
            cum = dd_add(cum, w[e]);
            if (hit == INT_MAX && dd_pos(w[e]) && dd_gt(cum, t)) hit = i0 + e;
        }
        if (hit != INT_MAX) atomicMin(&sb.found, hit);
        if (lastp >= 0) atomicMax(&sb.lastpos, lastp);
        sync_nt<kNT>();
        if (sb.found != INT_MAX) break;
        carry = dd_add(carry, tile);
    }
    return sb.found != INT_MAX ? sb.found : sb.lastpos;
}

// ---------------------------------------------------------------------------
// Per-request settings ("10.6 投机解码" §10.6.3: the requests of a batch
// accept different lengths; "KV Cache 优化（四）" §4: each request's own
// processed distributions): the request's gamma, temperature (0: greedy),
// top-k and top-p, from the per-request arrays when given, else the call's
// scalars.  A value out of range sets `bad`.
// ---------------------------------------------------------------------------
struct ReqCfg {
    int gamma;     // rows 0..gamma of the request's target, 0..gamma-1 of its draft
    float c2;      // log2(e) / T
    float2 it;     // 1 / T as a double-float pair
    int K;         // top-k (0: keep all)
    float top_p;   // the nucleus in (0, 1); 0: off
    bool greedy;
    unsigned bad;  // SPEC_FLAG_BAD_INPUT for a setting out of range
};

__device__ __forceinline__ int req_gamma(const SampleParams &p, int b) {
    if (!p.per_request || !p.rq_gamma) return p.gamma;
    const int gb = p.rq_gamma[b];
    return (gb < 0 || gb > p.gamma) ? p.gamma : gb;
}

__device__ __forceinline__ ReqCfg req_cfg(const SampleParams &p, int b) {
    ReqCfg c;
    c.gamma = p.gamma;
    c.c2 = p.c2;
    c.it = p.exptab.it;
    c.K = p.top_k;
    c.top_p = p.top_p;
    c.greedy = false;
    c.bad = 0u;
    if (!p.per_request) return c;
    if (p.rq_gamma) {
        const int gb = p.rq_gamma[b];
        if (gb < 0 || gb > p.gamma) c.bad = SPEC_FLAG_BAD_INPUT;
        else c.gamma = gb;
    }
    if (p.rq_temp) {
        const float T = p.rq_temp[b];
        if (!(T >= 0.0f) || !isfinite(T)) {
            c.bad = SPEC_FLAG_BAD_INPUT;
        } else if (T == 0.0f) {
            c.greedy = true;
        } else {
            c.c2 = (float)(1.4426950408889634074 / (double)T);
            const float hi = __frcp_rn(T);
            c.it = make_float2(hi, __fmul_rn(__fmaf_rn(-hi, T, 1.0f), hi));  // 1/T = hi + lo to ~2^-46
            if (!isfinite(c.c2) || !isfinite(hi)) c.bad = SPEC_FLAG_BAD_INPUT;
        }
    } else if (p.c2 == 0.0f) {
        c.greedy = true;  // the scalar temperature is 0
    }
    if (p.rq_topk) {
        const int k = p.rq_topk[b];
        if (k < 0) c.bad = SPEC_FLAG_BAD_INPUT;
        c.K = (k < 0 || k >= p.V) ? 0 : k;
    }
    if (p.rq_topp) {
        const float tp = p.rq_topp[b];
        if (!(tp >= 0.0f)) c.bad = SPEC_FLAG_BAD_INPUT;
        c.top_p = (tp > 0.0f && tp < 1.0f) ? tp : 0.0f;
    }
    return c;
}

// ---------------------------------------------------------------------------
// The request epilogue: the last position to arrive writes the outputs.  Run
// by one warp: lane q reads position q's record (one L2 load each, all in
// flight together), ballots find the first rejection and any bad input.
// ---------------------------------------------------------------------------
__device__ __forceinline__ PosRec load_rec(const PosRec *r) {
    const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(r));
    PosRec x;
    x.a = __uint_as_float(v.x);
    x.z = __uint_as_float(v.y);
    x.token = (int)v.z;
    x.info = v.w;
    return x;
}

static __device__ void write_request_warp(const SampleParams &p, int b) {
    const int g = p.gamma, lane = threadIdx.x & 31;
    __threadfence();
    const PosRec *R = p.recs + (int64_t)b * (g + 1);
    const int len0 = lane == 0 ? inplace_len0(p.ip, b) : 0;
    unsigned badbits = lane == 0 ? inplace_bad(p.ip, len0, g) : 0u;
    const int gb = req_gamma(p, b);  // the request's own gamma (records past it are placeholders)
    int n = gb;  // the first rejecting position (gb: all accepted)
    PosRec mine{};
    for (int q0 = 0; q0 <= g; q0 += 32) {
        const int q = q0 + lane;
        PosRec r{};
        if (q <= g) r = load_rec(R + q);
        if (q0 == 0) mine = r;
        badbits |= (q <= gb && (r.info & REC_BAD_INPUT)) ? SPEC_FLAG_BAD_INPUT : 0u;
        badbits |= (q <= gb && (r.info & REC_BAD_ROW)) ? SPEC_FLAG_BAD_ROW : 0u;
        const unsigned rej = __ballot_sync(kFull, q < gb && !(r.info & REC_ACCEPT));
        if (n == gb && rej) n = q0 + __ffs(rej) - 1;
    }
    badbits = __reduce_or_sync(kFull, badbits);
    if (badbits) {
        if (lane == 0) {
            p.n_acc[b] = 0;
            p.n_out[b] = 0;
            if (p.flags) p.flags[b] = badbits;
            atomicOr(p.status, badbits);
        }
    } else {
        int *out = p.out_tokens + (int64_t)b * (g + 1);
        const int *dt = p.tokens + (int64_t)b * g;
        const int lim = stop_limit(p.stop, b);
        int cut = 0x7fffffff;  // the first EOS position so far
        unsigned fb = 0u;
        for (int q0 = 0; q0 <= g; q0 += 32) {  // (uniform trip count: q0 <= g for every lane)
            const int q = q0 + lane;
            PosRec r{};
            if (q <= g) r = q0 == 0 ? mine : load_rec(R + q);
            const int tok = q < n ? dt[q] : (q == n ? r.token : -1);
            cut = stop_scan(p.stop, q0, q, n, tok, cut);
            if (q <= n) out[q] = (q < lim && q <= cut) ? tok : -1;
            if (q == n && (r.info & REC_FALLBACK)) fb = SPEC_FLAG_FALLBACK;
            if (q < gb) {
                if (p.accept_prob) p.accept_prob[(int64_t)b * g + q] = r.a;
                if (p.resid) p.resid[(int64_t)b * g + q] = r.z;
            }
        }
        fb = __reduce_or_sync(kFull, fb);
        if (lane == 0) {
            unsigned f = fb;
            const int L = stop_length(n, cut, lim, f);
            p.n_acc[b] = n < L ? n : L;
            p.n_out[b] = L;
            if (p.flags) p.flags[b] = f;
            inplace_commit(p.ip, b, len0, L);
        }
    }
    if (lane == 0) {
        p.rejword[b] = 0u;
        p.counters[b] = 0u;
    }
}

// Records position k's outcome; the position that arrives last for request b
// writes the request's outputs.  Called by every thread of the block (or, in
// a warp-only caller, every lane of warp 0); warp 0 does the work.
static __device__ void finish(const SampleParams &p, int b, int k, const Outcome &o, SampBase &sb) {
    if (threadIdx.x >= 32) return;
    unsigned last = 0u;
    if (threadIdx.x == 0) {
        PosRec rec;
        rec.a = o.a;
        rec.z = o.z;
        rec.token = o.token;
        rec.info = o.info;
        p.recs[(int64_t)b * (p.gamma + 1) + k] = rec;
        __threadfence();
        last = atomicAdd(p.counters + b, 1u) == (unsigned)p.gamma;
    }
    if (__shfl_sync(kFull, last, 0)) write_request_warp(p, b);
    (void)sb;
}

// ---------------------------------------------------------------------------
// Exchange between the CTAs that share one position: a real thread-block
// cluster (DSMEM pushes, cluster barriers) or a single CTA doing the whole row.
// ---------------------------------------------------------------------------
struct ClusterEx {
    cg::cluster_group cl;
    int c, j;
    bool waited;
    __device__ ClusterEx(int c_, int j_) : cl(cg::this_cluster()), c(c_), j(j_), waited(false) {}
    // the kernel arrived on the cluster barrier at its start; wait once
    // before the first remote write so every CTA of the cluster is running
    __device__ void ready() {
        if (!waited) {
            asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
            waited = true;
        }
    }
    template <class P> __device__ P *at(P *local, int r) { return cl.map_shared_rank(local, r); }
    __device__ void sync() { cl.sync(); }
};

struct SoloEx {
    int c = 1, j = 0;
    __device__ void ready() {}
    template <class P> __device__ P *at(P *local, int) { return local; }
    __device__ void sync() { sync_nt<kNT>(); }
};

// ---------------------------------------------------------------------------
// A greedy request's position (temperature 0; "KV Cache 优化（四）" §4): the
// argmax of target row k over the exchange (lowest index on ties), d_k
// accepted iff it is that argmax; the argmax is the token the position
// emits when it ends the round.
// ---------------------------------------------------------------------------
template <typename T, typename Ex>
__device__ void greedy_position(const SampleParams &p, SampBase &sb, Ex &ex, int k, int b, int lo, int hi,
                                int gamma_b) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, c = ex.c, j = ex.j, g = p.gamma;
    const bool has_draft = k < gamma_b;
    const T *trow = reinterpret_cast<const T *>(p.target) + (int64_t)(b * (g + 1) + k) * p.tstride;
    ArgMax am{-INFINITY, -1};
    for_slice<T, 4>(trow, lo, hi, tid, kNT, [&](float x, int i) {
        if (am_better(x, i, am.v, am.idx)) am = ArgMax{x, i};
    });
    am = warp_argmax(am);
    if (lane == 0) sb.redd[wid] = make_float4(am.v, __int_as_float(am.idx), 0.0f, 0.0f);
    sync_nt<kNT>();
    ArgMax t{-INFINITY, -1};
    if (lane < kNW) t = ArgMax{sb.redd[lane].x, __float_as_int(sb.redd[lane].y)};
    t = warp_argmax(t);
    ex.ready();
    if (tid < c) ex.at(&sb.ms[0], tid)[j] = make_float4(t.v, __int_as_float(t.idx), 0.0f, 0.0f);
    ex.sync();
    ArgMax best{-INFINITY, -1};
    for (int r = 0; r < c; ++r) {
        const ArgMax x{sb.ms[r].x, __float_as_int(sb.ms[r].y)};
        if (am_better(x.v, x.idx, best.v, best.idx)) best = x;
    }
    if (j == 0) {
        const int d = has_draft ? p.tokens[(int64_t)b * g + k] : 0;
        const bool bad_tok = has_draft && (d < 0 || d >= p.V);
        const bool accept = has_draft && !bad_tok && d == best.idx;
        Outcome o{accept ? 1.0f : 0.0f, 0.0f, best.idx, (accept ? REC_ACCEPT : 0u) | (bad_tok ? REC_BAD_INPUT : 0u)};
        finish(p, b, k, o, sb);
    }
}

// ---------------------------------------------------------------------------
// The nucleus cut of one row over the exchange: the largest order key tau
// such that the kept logits (key >= th) at or above tau hold at least top_p
// of the kept mass, i.e. the key of the first token, by probability, at
// which the running mass reaches top_p; every token tied with it stays.  A
// radix descent over 8-bit digits of the key: per digit the masses
// exp((x - m)/T) (double-float terms, summed in fp64) of the keys that
// match the prefix so far, gathered in rank 0's shared memory, which picks
// the digit and pushes it to every CTA.  `dsm` is free (the ring is idle).
// ---------------------------------------------------------------------------
template <typename T, typename Ex>
__device__ uint32_t nucleus_key(Ex &ex, SampBase &sb, unsigned char *dsm, const T *row, int lo, int hi,
                                uint32_t th, float m, float top_p) {
    constexpr int KB = Elem<T>::KEY_BITS;
    constexpr int KS = 32 - KB;
    static_assert(kNT == 256, "one digit per thread");
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, c = ex.c, j = ex.j;
    const DdExpTables &EK = sb.K;
    double *hist = reinterpret_cast<double *>(dsm);  // [256] this CTA's masses by digit
    double *all = hist + 256;                        // [kMaxCluster][256], gathered in rank 0
    uint32_t prefix = 0u;
    int nb = KB;
    double above = 0.0, target = 0.0;
    while (nb > 0) {  // identical in every CTA
        const int sh = nb > 8 ? nb - 8 : 0;
        const uint32_t dmask = (1u << (nb - sh)) - 1u;
        hist[tid] = 0.0;
        sync_nt<kNT>();
        for_slice<T, 4>(row, lo, hi, tid, kNT, [&](float x, int) {
            const uint32_t key = fkey(x) >> KS;
            if (x > -INFINITY && key >= th && (nb == KB || (key >> nb) == (prefix >> nb))) {
                const dd e = dd_expw(x, m, EK);
                atomicAdd(&hist[(key >> sh) & dmask], (double)e.hi + (double)e.lo);
            }
        });
        sync_nt<kNT>();
        ex.ready();
        ex.at(all, 0)[j * 256 + tid] = hist[tid];
        ex.sync();
        if (j == 0) {
            // thread t: digit 255 - t, its mass over the ranks in rank order;
            // an inclusive scan over t gives the mass of the digits >= 255 - t
            double v = 0.0;
            for (int r = 0; r < c; ++r) v += all[r * 256 + (255 - tid)];
            double incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) sb.redD[wid] = incl;
            sync_nt<kNT>();
            double pre = 0.0, tot = 0.0;
            for (int w = 0; w < kNW; ++w) {
                pre += w < wid ? sb.redD[w] : 0.0;
                tot += sb.redD[w];
            }
            if (nb == KB) target = (double)top_p * tot;  // the first digit sees every kept logit
            const double cum = above + pre + incl;
            const bool hit = v > 0.0 && cum >= target && cum - v < target;
            if (tid == 0) sb.nuc_found = 0;
            sync_nt<kNT>();
            if (hit) {
                sb.nuc_found = 1;
                for (int r = 0; r < c; ++r) {
                    *ex.at(&sb.nuc_dig, r) = 255u - (unsigned)tid;
                    *ex.at(&sb.nuc_above, r) = cum - v;
                }
            }
            sync_nt<kNT>();
            if (!sb.nuc_found) {
                // rounding left the mass below top_p: the smallest nonempty digit
                unsigned lastd = v > 0.0 ? (unsigned)tid + 1u : 0u;
                lastd = __reduce_max_sync(kFull, lastd);
                if (lane == 0) sb.redD[wid] = (double)lastd;
                sync_nt<kNT>();
                unsigned best = 0u;
                for (int w = 0; w < kNW; ++w) best = max(best, (unsigned)sb.redD[w]);
                if (best > 0u && tid == (int)best - 1)
                    for (int r = 0; r < c; ++r) {
                        *ex.at(&sb.nuc_dig, r) = 255u - (unsigned)tid;
                        *ex.at(&sb.nuc_above, r) = cum - v;
                    }
            }
        }
        ex.sync();
        prefix |= sb.nuc_dig << sh;
        above = sb.nuc_above;
        nb = sh;
    }
    return prefix;
}

// ---------------------------------------------------------------------------
// One position over the exchange `ex`: optional exact top-k threshold by a
// binary search on order keys (MASK), pass 1 (online max/sum, bulk-copy
// ring), acceptance, optional fp32 residual mass, and the double-float draw
// where this position decides the emitted token.  Every CTA of the exchange
// runs it on its slice [lo, hi); the CTA that ends up holding the whole
// outcome calls finish().
// ---------------------------------------------------------------------------
template <typename T, bool MASK, typename Ex, typename RingT = SampRing>
__device__ void masked_position(const SampleParams &p, SampBase &sb, unsigned char *dsm, Ex &ex,
                                int k, int b, int lo, int hi) {
    constexpr int VEC = Elem<T>::VEC;
    constexpr int KB = Elem<T>::KEY_BITS;
    constexpr int KS = 32 - KB;
    const int tid = threadIdx.x, c = ex.c, j = ex.j, g = p.gamma;
    const ReqCfg cfg = req_cfg(p, b);  // identical in every CTA of the exchange
    if (k > cfg.gamma || cfg.bad) {
        // a position past the request's own gamma (a placeholder for the
        // arrival count), or a request whose settings are out of range
        if (j == 0) {
            Outcome o{1.0f, 0.0f, -1, REC_ACCEPT | (cfg.bad ? REC_BAD_INPUT : 0u)};
            finish(p, b, k, o, sb);
        }
        return;
    }
    if (cfg.greedy) {
        greedy_position<T>(p, sb, ex, k, b, lo, hi, cfg.gamma);
        return;
    }
    if (p.per_request) {  // this request's 1/T for the double-float exponential
        if (tid == 0) sb.K.it = cfg.it;
        sync_nt<kNT>();
    }
    const bool has_draft = k < cfg.gamma;
    const T *trow = reinterpret_cast<const T *>(p.target) + (int64_t)(b * (g + 1) + k) * p.tstride;
    const T *drow = has_draft
        ? reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + k) * p.dstride : nullptr;
    const float c2 = cfg.c2;
    const int d = has_draft ? p.tokens[(int64_t)b * g + k] : 0;
    const bool bad_tok = has_draft && (d < 0 || d >= p.V);
    const float l_d = (has_draft && !bad_tok) ? ld_elem(trow, d) : 0.0f;
    const float g_d = (has_draft && !bad_tok) ? ld_elem(drow, d) : 0.0f;
    const float u_k = has_draft ? p.unif[(int64_t)b * (g + 1) + k] : 0.0f;
    const float u_f = p.unif[(int64_t)b * (g + 1) + cfg.gamma];
    Outcome o{1.0f, 0.0f, -1, 0u};

    uint32_t th_p = 0u, th_q = 0u;
    if (MASK && cfg.K > 0) {
        uint32_t lo_p = 0u, hi_p = KB == 32 ? 0xffffffffu : ((1u << KB) - 1u);
        uint32_t lo_q = 0u, hi_q = has_draft ? hi_p : 0u;
        const unsigned K = (unsigned)cfg.K;
        for (int it = 0; it < KB; ++it) {
            const bool act_p = lo_p < hi_p, act_q = lo_q < hi_q;
            if (!act_p && !act_q) break;  // identical in every CTA of the exchange
            const uint32_t mid_p = lo_p + (uint32_t)(((uint64_t)hi_p - lo_p + 1) >> 1);
            const uint32_t mid_q = lo_q + (uint32_t)(((uint64_t)hi_q - lo_q + 1) >> 1);
            unsigned cp = 0, cq = 0;
            if (act_p)
                for_slice<T, 4>(trow, lo, hi, tid, kNT, [&](float x, int) { cp += (fkey(x) >> KS) >= mid_p; });
            if (act_q)
                for_slice<T, 4>(drow, lo, hi, tid, kNT, [&](float x, int) { cq += (fkey(x) >> KS) >= mid_q; });
            cp = block_sum_u<kNT>(cp, sb.redu);
            cq = block_sum_u<kNT>(cq, sb.redu);
            const int par = it & 1;
            ex.ready();
            if (tid < c) {
                unsigned *dst = ex.at(&sb.cnt[par][0][0], tid);
                dst[j] = cp;
                dst[kMaxCluster + j] = cq;
            }
            ex.sync();
            unsigned tp = 0, tq = 0;
            for (int r = 0; r < c; ++r) {
                tp += sb.cnt[par][0][r];
                tq += sb.cnt[par][1][r];
            }
            if (act_p) { if (tp >= K) lo_p = mid_p; else hi_p = mid_p - 1; }
            if (act_q) { if (tq >= K) lo_q = mid_q; else hi_q = mid_q - 1; }
        }
        th_p = lo_p;
        th_q = lo_q;
    }

    // ---- pass 1 (HBM): online max / sum of the kept logits -------------------
    MaxSum Mp{-INFINITY, 0.0f}, Mq{-INFINITY, 0.0f};
    auto pass1 = [&]() {
        MaxSum msp{-INFINITY, 0.0f}, msq{-INFINITY, 0.0f};
        {
            RingT &R = *reinterpret_cast<RingT *>(dsm);
            const bool okc = stream_rows<T>(R, trow, drow, lo, hi, [&](const float *xa, const float *xb, int, int cnt) {
                ms_update<VEC, MASK>(msp, xa, cnt, th_p, KS, c2);
                if (has_draft) ms_update<VEC, MASK>(msq, xb, cnt, th_q, KS, c2);
            });
            if (!okc && tid == 0) atomicOr(p.status, SPEC_FLAG_TIMEOUT);
        }
        msp = block_ms<kNT>(msp, c2, sb.red2);
        msq = block_ms<kNT>(msq, c2, sb.red2);
        unsigned prior = 0u;
        if (j == 0 && tid == 0) prior = *((volatile unsigned *)&p.rejword[b]);
        ex.ready();
        if (tid < c) {
            float4 *dst = ex.at(&sb.ms[0], tid);
            dst[j] = make_float4(msp.m, msp.s, msq.m, msq.s);
        }
        if (j == 0 && tid == 0)
            for (int r = 0; r < c; ++r) *ex.at(&sb.rej, r) = prior;
        ex.sync();
        Mp = MaxSum{-INFINITY, 0.0f};
        Mq = MaxSum{-INFINITY, 0.0f};
        for (int r = 0; r < c; ++r) {
            Mp = ms_combine(Mp, MaxSum{sb.ms[r].x, sb.ms[r].y}, c2);
            Mq = ms_combine(Mq, MaxSum{sb.ms[r].z, sb.ms[r].w}, c2);
        }
    };
    pass1();
    if (MASK && cfg.top_p > 0.0f && Mp.m > -INFINITY && (!has_draft || Mq.m > -INFINITY)) {
        // top-p after temperature and top-k ("KV Cache 优化（四）" §4): each
        // row's threshold becomes its nucleus cut, then pass 1 again
        th_p = nucleus_key<T, Ex>(ex, sb, dsm, trow, lo, hi, th_p, Mp.m, cfg.top_p);
        if (has_draft) th_q = nucleus_key<T, Ex>(ex, sb, dsm, drow, lo, hi, th_q, Mq.m, cfg.top_p);
        pass1();
    }
    const bool bad_row = Mp.m == -INFINITY || (has_draft && Mq.m == -INFINITY);
    const bool bad = bad_tok || bad_row;
    o.info = (bad_tok ? REC_BAD_INPUT : 0u) | (bad_row ? REC_BAD_ROW : 0u);
    bool accept = false;
    if (has_draft && !bad) {
        const float mcp = Mp.m * c2, mcq = Mq.m * c2;
        const float pd = (!MASK || (fkey(l_d) >> KS) >= th_p) ? exp2f(fmaf(l_d, c2, -mcp)) / Mp.s : 0.0f;
        const float qd = (!MASK || (fkey(g_d) >> KS) >= th_q) ? exp2f(fmaf(g_d, c2, -mcq)) / Mq.s : 0.0f;
        o.a = qd > 0.0f ? fminf(1.0f, pd / qd) : (pd > 0.0f ? 1.0f : 0.0f);
        accept = u_k < o.a;
        o.info |= accept ? REC_ACCEPT : 0u;
    }
    const bool earlier = sb.rej > (unsigned)(g - k + 1);
    if (has_draft && !bad && !accept && j == 0 && tid == 0) atomicMax(p.rejword + b, (unsigned)(g - k + 1));
    const bool draw = !bad && (!has_draft || !accept) && !earlier;
    int writer = 0;

    if (!draw && has_draft && !bad && p.resid) {
        // ---- diagnostic residual mass in fp32 (pass 2, L2) ----
        const float mcp = Mp.m * c2, mcq = Mq.m * c2, isp = 1.0f / Mp.s, isq = 1.0f / Mq.s;
        float zw = 0.0f;
        for_slice2<T, 2>(trow, drow, lo, hi, [&](const float *xa, const float *xb, int, int cnt) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                if (e < cnt) {
                    // explicit roundings: no fused multiply-add may turn p_i - q_i for
                    // identical rows into a rounding residue
                    const float pi = (!MASK || (fkey(xa[e]) >> KS) >= th_p) ? __fmul_rn(exp2f(fmaf(xa[e], c2, -mcp)), isp) : 0.0f;
                    const float qi = (!MASK || (fkey(xb[e]) >> KS) >= th_q) ? __fmul_rn(exp2f(fmaf(xb[e], c2, -mcq)), isq) : 0.0f;
                    zw += fmaxf(pi - qi, 0.0f);
                }
            }
        });
        zw = block_sum<kNT>(zw, sb.redf);
        if (tid < c) *ex.at(&sb.zdiag[j], tid) = zw;
        ex.sync();
        float z = 0.0f;
        for (int r = 0; r < c; ++r) z += sb.zdiag[r];
        o.z = z;
    }

    if (draw) {
        // ---- the draw in dd ----
        // Pass A (L2): the CTA's slice sums S_p, S_q of both rows' terms and,
        // over P = {i : p_i > q_i}, the sums P_p, P_q of the terms whose side
        // the fp32 estimate of S_p/S_q decides with margin; the others are
        // listed and resolved once the exact sums are known:
        //   Z_w = P_p/S_p - P_q/S_q + sum over the listed i of max(0, p_i - q_i).
        // If any CTA's list overflows, a full residual pass replaces it.
        const DdExpTables &K = sb.K;
        const float mp = Mp.m, mq = Mq.m;
        auto ep = [&](float x) -> dd {
            return (!MASK || (fkey(x) >> KS) >= th_p) ? dd_expw(x, mp, K) : dd{0.0f, 0.0f};
        };
        auto eq = [&](float y) -> dd {
            return (!MASK || (fkey(y) >> KS) >= th_q) ? dd_expw(y, mq, K) : dd{0.0f, 0.0f};
        };
        if (tid == 0) sb.namb = 0;
        sync_nt<kNT>();
        dd sp{0.0f, 0.0f}, sq{0.0f, 0.0f}, pp{0.0f, 0.0f}, pq{0.0f, 0.0f};
        if (has_draft) {
            const float rho = Mp.s / Mq.s;  // fp32 estimate of S_p / S_q
            const float rhi = rho * (1.0f + kAmbRel), rlo = rho * (1.0f - kAmbRel);
            for_slice2<T, 2>(trow, drow, lo, hi, [&](const float *xa, const float *xb, int base, int cnt) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    if (e < cnt) {
                        const dd a = ep(xa[e]), q = eq(xb[e]);
                        sp = dd_acc(sp, a);
                        sq = dd_acc(sq, q);
                        if (a.hi > q.hi * rhi) {
                            pp = dd_acc(pp, a);
                            pq = dd_acc(pq, q);
                        } else if (a.hi > 0.0f && a.hi >= q.hi * rlo) {
                            const int at = atomicAdd(&sb.namb, 1);
                            if (at < kAmbMax) sb.amb[at] = base + e;
                        }
                    }
                }
            });
        } else {
            for_slice_vec<T, 4>(trow, lo, hi, tid, kNT, [&](const float *x, int, int cnt) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (e < cnt) sp = dd_acc(sp, ep(x[e]));
            });
        }
        block_dd_sum2<kNT>(sp, sq, sb.redd);
        block_dd_sum2<kNT>(pp, pq, sb.redd);
        const unsigned my_ovf = sb.namb > kAmbMax ? 1u : 0u;
        if (tid < c) {
            *ex.at(&sb.dsum[j], tid) = make_float4(sp.hi, sp.lo, sq.hi, sq.lo);
            *ex.at(&sb.ovfr[j], tid) = my_ovf;
        }
        ex.sync();
        dd Sp{0.0f, 0.0f}, Sq{0.0f, 0.0f};
        unsigned any_ovf = 0u;
        for (int r = 0; r < c; ++r) {
            Sp = dd_add(Sp, dd{sb.dsum[r].x, sb.dsum[r].y});
            Sq = dd_add(Sq, dd{sb.dsum[r].z, sb.dsum[r].w});
            any_ovf |= sb.ovfr[r];
        }
        const dd isp = dd_recip(Sp);
        const dd isq = has_draft ? dd_recip(Sq) : dd{0.0f, 0.0f};
        bool use_p = true, fb = false;
        dd total = Sp;  // bonus and fallback: the unnormalised target terms
        if (has_draft) {
            // this CTA's residual mass
            dd zw{0.0f, 0.0f};
            if (!any_ovf) {
                const int na = sb.namb;
                for (int x = tid; x < na; x += kNT) {
                    const int i = sb.amb[x];
                    const dd pi = dd_mul(ep(ld_elem(trow, i)), isp);
                    const dd qi = dd_mul(eq(ld_elem(drow, i)), isq);
                    zw = dd_add(zw, dd_max0(dd_add(pi, dd_neg(qi))));
                }
            } else {
                for_slice2<T, 2>(trow, drow, lo, hi, [&](const float *xa, const float *xb, int, int cnt) {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        if (e < cnt) {
                            const dd pi = dd_mul(ep(xa[e]), isp);
                            const dd qi = dd_mul(eq(xb[e]), isq);
                            zw = dd_add(zw, dd_max0(dd_add(pi, dd_neg(qi))));
                        }
                    }
                });
            }
            dd unused{0.0f, 0.0f};
            block_dd_sum2<kNT>(zw, unused, sb.redd);
            if (!any_ovf) zw = dd_add(zw, dd_add(dd_mul(pp, isp), dd_neg(dd_mul(pq, isq))));
            sync_nt<kNT>();
            if (tid < c) *ex.at(&sb.dsum2[j], tid) = make_float4(zw.hi, zw.lo, 0.0f, 0.0f);
            ex.sync();
            dd Zw{0.0f, 0.0f};
            for (int r = 0; r < c; ++r) Zw = dd_add(Zw, dd{sb.dsum2[r].x, sb.dsum2[r].y});
            o.z = dd_to_f(Zw);
            fb = dd_le(Zw, dd{p.eps, 0.0f});
            use_p = fb;
            if (!fb) total = Zw;
            if (fb) o.info |= REC_FALLBACK;
        }
        const dd t = dd_mul_f(total, u_f);
        // the slice that holds the crossing (identical choice in every CTA)
        int owner = -1, lastpos = -1;
        dd acc{0.0f, 0.0f}, own_prefix{0.0f, 0.0f}, last_prefix{0.0f, 0.0f};
        // per rank: its S_p (bonus, fallback: the unnormalised target terms) or
        // its residual mass
        const float4 *part = use_p ? sb.dsum : sb.dsum2;
        for (int r = 0; r < c; ++r) {
            const dd prt{part[r].x, part[r].y};
            if (dd_pos(prt)) {
                if (owner < 0 && dd_gt(dd_add(acc, prt), t)) { owner = r; own_prefix = acc; }
                lastpos = r;
                last_prefix = acc;
            }
            acc = dd_add(acc, prt);
        }
        if (owner < 0) { owner = lastpos; own_prefix = last_prefix; }
        writer = owner < 0 ? 0 : owner;
        if (j == owner) {
            o.token = dd_scan_slice<kNT>(lo, hi, own_prefix, t, [&](int i) -> dd {
                const dd e = ep(ld_elem(trow, i));
                if (use_p) return e;
                return dd_max0(dd_add(dd_mul(e, isp), dd_neg(dd_mul(eq(ld_elem(drow, i)), isq))));
            }, sb);
        }
    }
    if (j == writer) finish(p, b, k, o, sb);
}

}  // namespace specv
