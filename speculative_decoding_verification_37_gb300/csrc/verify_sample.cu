// Sampled chain verification (temperature > 0) on sm_103a.
//
// One round of speculative sampling ("10.6 投机解码：为什么“先猜后验”能加速"
// §10.6.1; "KV Cache 优化（四）：Speculative Decoding 投机解码" §4, §5):
// transform each target and draft row (temperature, top-k), accept d_k with
// probability min(1, p_k(d_k)/q_k(d_k)) left to right, draw the replacement
// from norm(max(0, p_k - q_k)) at the first rejection (from p_k itself when
// that mass is <= eps: the glossary page's stable fallback), or a bonus token
// from p_{gamma+1} when every draft is accepted.
//
// GB300 mapping.  One thread-block cluster of c CTAs per (position k,
// request b), clusters in position-major order (all requests' position 0
// first).  CTA j owns vocab slice j of target row k and draft row k.
//
//  * Acceptance.  Full-vocab rows: each CTA streams its slices once from HBM
//    (16-byte loads, both rows interleaved) with an online (max, sum of
//    2^(x log2e / T - m)) pair; the c pairs are pushed over DSMEM into every
//    CTA and combined in rank order, so all CTAs hold identical normalisers
//    and the same a_k.  Top-k rows (k <= 128): each warp keeps the candidates
//    above a rising threshold in shared memory, each CTA reduces its slice to
//    the exact slice top-k (ties kept) and pushes it to rank 0, which merges
//    the c lists into the exact kept set; everything after that is computed
//    from at most a few hundred entries.  If a list overflows (massive ties)
//    or k is large, the exact threshold is found instead by a cluster-wide
//    binary search over order keys and the row is treated as masked.
//  * The draw.  Only the first rejecting position (or the bonus position)
//    decides the emitted token.  Each request keeps the earliest rejection
//    seen so far in a workspace word; position-major order makes earlier
//    positions finish first, so a position that already sees an earlier
//    rejection skips its draw.  The draw is taken in double-float arithmetic
//    (ddmath.cuh), close to float64, because at V ~ 1e5 the CDF boundaries
//    lie ~1e-5 apart and an fp32 CDF would pick a neighbouring token far too
//    often.  Full-vocab draws re-read the slices (from L2: the same CTA read
//    them microseconds earlier), exchange dd slice totals over DSMEM, and the
//    CTA whose slice holds the crossing scans it in token order.
//  * Each position writes one 16-byte record; the position that arrives
//    last for its request (arrival counter) writes the request's outputs.
// No block waits on another except through cluster barriers between
// co-scheduled CTAs of one cluster.
#include <cooperative_groups.h>

#include <type_traits>

#include "common.cuh"
#include "ddmath.cuh"
#include "kernels.h"
#include "select.cuh"

namespace cg = cooperative_groups;

namespace specv {

constexpr int kNT = 256;
constexpr int kNW = kNT / 32;
constexpr int kMaxCluster = 8;
constexpr int kWCap = 256;   // candidate slots per warp per row
constexpr int kSeg = 256;    // entries one slice may send to rank 0 per row
constexpr int kScanE = 8;    // elements per thread per tile of the token-order scan
constexpr int kKeptMax = 1024;  // kept-set entries rank 0 can sort for a draw
static_assert(kNW == kMaxCluster && kWCap == kSeg, "rank 0 receives into its warp buffers");

enum : int { MODE_FULL = 0, MODE_SEARCH = 1, MODE_FAST = 2 };

struct SampBase {
    float2 red2[kNW];
    float redf[kNW];
    unsigned redu[kNW];
    float4 redd[kNW];
    float4 ms[kMaxCluster];       // pushed (m_p, s_p, m_q, s_q) per rank
    float4 dsum[kMaxCluster];     // pushed dd pair of sums per rank
    float zdiag[kMaxCluster];     // pushed fp32 residual mass per rank
    unsigned cnt[2][2][kMaxCluster];
    unsigned rej;                 // earliest-rejection word, pushed by rank 0
    unsigned ovf;                 // candidate-list overflow, OR-ed by every rank
    int found, lastpos, arrive_last;
    unsigned hist[256];
    unsigned bc[2];
    unsigned tau[2];
    float2 tab[65];
    float2 ln2;
};

struct SampFast {
    uint2 cand[2][kNW][kWCap];     // per-warp candidates; rank 0 reuses it as [row][rank][kSeg]
    int cand_n[2][kNW];
    int recv_n[2][kMaxCluster];
    uint2 stage[2][kSeg];          // rank 0's own slice list while others push
    int stage_n[2];
    int kn[2];
};

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
    __syncthreads();
    if (lane == 0) red[w] = make_float4(a.hi, a.lo, b.hi, b.lo);
    __syncthreads();
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
    __syncthreads();
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
        __syncthreads();
        if (lane == 31) sb.redd[wid] = make_float4(incl.hi, incl.lo, 0.0f, 0.0f);
        __syncthreads();
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
        __syncthreads();
        if (sb.found != INT_MAX) break;
        carry = dd_add(carry, tile);
    }
    return sb.found != INT_MAX ? sb.found : sb.lastpos;
}

// ---------------------------------------------------------------------------
// The request epilogue: the last position to arrive writes the outputs.
// ---------------------------------------------------------------------------
__device__ void write_request(const SampleParams &p, int b) {
    const int g = p.gamma;
    __threadfence();
    const volatile PosRec *R = p.recs + (int64_t)b * (g + 1);
    unsigned badbits = 0;
    for (int q = 0; q <= g; ++q) {
        const unsigned info = R[q].info;
        badbits |= (info & REC_BAD_INPUT) ? SPEC_FLAG_BAD_INPUT : 0u;
        badbits |= (info & REC_BAD_ROW) ? SPEC_FLAG_BAD_ROW : 0u;
    }
    if (badbits) {
        p.n_acc[b] = 0;
        p.n_out[b] = 0;
        if (p.flags) p.flags[b] = badbits;
        atomicOr(p.status, badbits);
    } else {
        int n = g;
        for (int q = 0; q < g; ++q)
            if (!(R[q].info & REC_ACCEPT)) { n = q; break; }
        int *out = p.out_tokens + (int64_t)b * (g + 1);
        const int *dt = p.tokens + (int64_t)b * g;
        for (int q = 0; q < n; ++q) out[q] = dt[q];
        out[n] = R[n].token;
        p.n_acc[b] = n;
        p.n_out[b] = n + 1;
        if (p.accept_prob)
            for (int q = 0; q < g; ++q) p.accept_prob[(int64_t)b * g + q] = R[q].a;
        if (p.resid)
            for (int q = 0; q < g; ++q) p.resid[(int64_t)b * g + q] = R[q].z;
        if (p.flags) p.flags[b] = (R[n].info & REC_FALLBACK) ? SPEC_FLAG_FALLBACK : 0u;
    }
    p.rejword[b] = 0u;
    p.counters[b] = 0u;
}

__device__ void finish(const SampleParams &p, int b, int k, const Outcome &o, SampBase &sb) {
    if (threadIdx.x == 0) {
        PosRec rec;
        rec.a = o.a;
        rec.z = o.z;
        rec.token = o.token;
        rec.info = o.info;
        p.recs[(int64_t)b * (p.gamma + 1) + k] = rec;
        __threadfence();
        sb.arrive_last = atomicAdd(p.counters + b, 1u) == (unsigned)p.gamma;
        if (sb.arrive_last) write_request(p, b);
    }
}

// ---------------------------------------------------------------------------
// Top-k candidate collection (MODE_FAST): per-warp candidate buffers with a
// rising threshold, then the exact slice top-k, sent to rank 0.
// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ void warp_insert(SampFast &sf, SampBase &sb, int row, int w, int &n,
                                            uint32_t &tau, int K, uint32_t key, bool pred, int idx,
                                            bool &ovf) {
    constexpr int KB = Elem<T>::KEY_BITS;
    const unsigned bal = __ballot_sync(kFull, pred);
    if (!bal) return;
    const int pos = n + __popc(bal & lanemask_lt());
    if (pred && pos < kWCap) sf.cand[row][w][pos] = make_uint2(key, (uint32_t)idx);
    n += __popc(bal);
    if (n > kWCap - 32) {
        __syncwarp();
        uint2 *buf = sf.cand[row][w];
        const int nn = min(n, kWCap);
        const uint32_t thr = warp_kth_largest<KB, kWCap>(buf, nn, K);
        const uint32_t t = max(thr, *((volatile unsigned *)&sb.tau[row]));
        const int lane = threadIdx.x & 31;
        uint2 e[kWCap / 32];
#pragma unroll
        for (int i = 0; i < kWCap / 32; ++i) {
            const int x = lane + 32 * i;
            e[i] = x < nn ? buf[x] : make_uint2(0u, 0u);
        }
        __syncwarp();
        int m = 0;
#pragma unroll
        for (int i = 0; i < kWCap / 32; ++i) {
            const bool keep = (lane + 32 * i) < nn && e[i].x >= t;
            const unsigned kb = __ballot_sync(kFull, keep);
            if (keep) buf[m + __popc(kb & lanemask_lt())] = e[i];
            m += __popc(kb);
        }
        __syncwarp();
        n = m;
        tau = t;
        if (lane == 0) atomicMax(&sb.tau[row], thr);
        if (n > kWCap - 32) ovf = true;
    }
}

// Streams the slices of one or both rows keeping candidates in per-warp
// buffers.  All warps stay converged inside the loops (ballots).
template <typename T>
__device__ void collect_candidates(const T *trow, const T *drow, int lo, int hi, int K,
                                   SampFast &sf, SampBase &sb, bool &ovf) {
    constexpr int VEC = Elem<T>::VEC;
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int rows = drow ? 2 : 1;
    int n0 = 0, n1 = 0;
    uint32_t tau0 = 0u, tau1 = 0u;
    if (hi > lo) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(trow + lo);
        const bool same_phase = !drow || ((a ^ reinterpret_cast<uintptr_t>(drow + lo)) & 15u) == 0;
        int head = (int)(((16u - (unsigned)(a & 15u)) & 15u) / sizeof(T));
        if (head > hi - lo) head = hi - lo;
        const int body0 = lo + head;
        const int nvec = (hi - body0) / VEC;
        const int tail0 = body0 + nvec * VEC;
        const uint4 *va = reinterpret_cast<const uint4 *>(trow + body0);
        const uint4 *vb = drow ? reinterpret_cast<const uint4 *>(drow + body0) : nullptr;
        // scalar head and tail: warp 0, one element per lane
        if (w == 0) {
            for (int part = 0; part < 2; ++part) {
                const int s0 = part == 0 ? lo : tail0;
                const int cnt = part == 0 ? head : hi - tail0;
                const bool val = lane < cnt;
                const int i = s0 + lane;
                const float x0 = val ? ld_elem(trow, i) : 0.0f;
                const uint32_t k0 = kkey<T>(x0);
                warp_insert<T>(sf, sb, 0, w, n0, tau0, K, k0, val && k0 >= tau0, i, ovf);
                if (rows == 2) {
                    const float x1 = val ? ld_elem(drow, i) : 0.0f;
                    const uint32_t k1 = kkey<T>(x1);
                    warp_insert<T>(sf, sb, 1, w, n1, tau1, K, k1, val && k1 >= tau1, i, ovf);
                }
            }
        }
        // body: warp-uniform trip count, lanes past the end contribute nothing
        for (int vb0 = w * 32; vb0 < nvec; vb0 += kNT * 2) {
            uint4 qa[2], qb[2];
            bool val[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int v = vb0 + lane + u * kNT;
                val[u] = v < nvec;
                qa[u] = val[u] ? ld_nc16(va + v) : make_uint4(0u, 0u, 0u, 0u);
                if (rows == 2) {
                    if (!val[u]) qb[u] = make_uint4(0u, 0u, 0u, 0u);
                    else if (same_phase) qb[u] = ld_nc16(vb + v);
                    else {
                        // gather the draft vector element by element (other 16-byte phase)
                        float y[VEC];
#pragma unroll
                        for (int e = 0; e < VEC; ++e) y[e] = ld_elem(drow, body0 + v * VEC + e);
                        if (sizeof(T) == 4) {
                            qb[u] = make_uint4(__float_as_uint(y[0]), __float_as_uint(y[1]),
                                               __float_as_uint(y[2]), __float_as_uint(y[3]));
                        } else {
                            uint32_t wv[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                wv[e] = (__float_as_uint(y[2 * e]) >> 16) |
                                        (__float_as_uint(y[2 * e + 1]) & 0xffff0000u);
                            qb[u] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                        }
                    }
                }
            }
            const uint32_t blk0 = *((volatile unsigned *)&sb.tau[0]);
            const uint32_t blk1 = *((volatile unsigned *)&sb.tau[1]);
            tau0 = max(tau0, blk0);
            tau1 = max(tau1, blk1);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int base = body0 + (vb0 + lane + u * kNT) * VEC;
                for (int r = 0; r < rows; ++r) {
                    float x[VEC];
                    unpack<T>(r == 0 ? qa[u] : qb[u], x);
                    uint32_t kk[VEC], kmax = 0u;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        kk[e] = kkey<T>(x[e]);
                        kmax = max(kmax, kk[e]);
                    }
                    int &n = r == 0 ? n0 : n1;
                    uint32_t &tau = r == 0 ? tau0 : tau1;
                    if (!__any_sync(kFull, val[u] && kmax >= tau)) continue;
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        warp_insert<T>(sf, sb, r, w, n, tau, K, kk[e], val[u] && kk[e] >= tau, base + e, ovf);
                }
            }
        }
    }
    if (lane == 0) {
        sf.cand_n[0][w] = min(n0, kWCap);
        sf.cand_n[1][w] = min(n1, kWCap);
    }
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <typename T, int MODE>
__global__ void __launch_bounds__(kNT) chain_sample_kernel(SampleParams p) {
    constexpr int VEC = Elem<T>::VEC;
    constexpr int KB = Elem<T>::KEY_BITS;
    constexpr int KS = 32 - KB;
    __shared__ SampBase sb;
    __shared__ std::conditional_t<MODE == MODE_FAST, SampFast, int> sf_storage;
    cg::cluster_group cluster = cg::this_cluster();
    const int tid = threadIdx.x;
    for (int i = tid; i < 65; i += kNT) sb.tab[i] = p.exptab.tab[i];
    if (tid == 0) {
        sb.ln2 = p.exptab.ln2;
        sb.tau[0] = sb.tau[1] = 0u;
        sb.ovf = 0u;
    }
    __syncthreads();
    // Every CTA of the cluster must have started (and initialised the shared
    // words others write into) before any remote access: arrive (release)
    // now, wait just before the first remote write.
    asm volatile("barrier.cluster.arrive.aligned;\n" ::: "memory");
    bool waited = false;
    auto cluster_ready = [&]() {
        if (!waited) {
            asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
            waited = true;
        }
    };

    const int c = p.c;
    const int j = (int)cluster.block_rank();
    const int qpos = blockIdx.x / c;
    const int g = p.gamma;
    const int k = qpos / p.B, b = qpos % p.B;   // position-major
    const bool has_draft = k < g;
    const int lo = min(p.V, j * p.Vs), hi = min(p.V, lo + p.Vs);
    const T *trow = reinterpret_cast<const T *>(p.target) + (int64_t)(b * (g + 1) + k) * p.tstride;
    const T *drow = has_draft
        ? reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + k) * p.dstride : nullptr;
    const float c2 = p.c2;
    const dd c2d{p.c2_hi, p.c2_lo};
    const int d = has_draft ? p.tokens[(int64_t)b * g + k] : 0;
    const bool bad_tok = has_draft && (d < 0 || d >= p.V);
    const float l_d = (has_draft && !bad_tok) ? ld_elem(trow, d) : 0.0f;
    const float g_d = (has_draft && !bad_tok) ? ld_elem(drow, d) : 0.0f;
    const float u_k = has_draft ? p.unif[(int64_t)b * (g + 1) + k] : 0.0f;
    const float u_f = p.unif[(int64_t)b * (g + 1) + g];

    // ======================= top-k candidate path ==========================
    bool fast = false;
    if constexpr (MODE == MODE_FAST) {
        SampFast &sf = sf_storage;
        bool ovf = false;
        collect_candidates<T>(trow, drow, lo, hi, p.top_k, sf, sb, ovf);
        __syncthreads();
        const int rows = has_draft ? 2 : 1;
        const uint32_t floor0 = sb.tau[0], floor1 = sb.tau[1];
        uint32_t thj[2] = {0u, 0u};
        int nsel[2] = {0, 0};
        for (int r = 0; r < rows; ++r) {
            const uint32_t fl = r == 0 ? floor0 : floor1;
            // entries of this slice at or above the block floor
            unsigned cnt = 0;
            const int lane = tid & 31, w = tid >> 5;
            for (int x = lane; x < sf.cand_n[r][w]; x += 32) cnt += sf.cand[r][w][x].x >= fl;
            cnt = block_sum_u<kNT>(cnt, sb.redu);
            uint32_t th = fl;
            if (cnt > (unsigned)p.top_k) {
                th = block_kth_largest<KB, kNT>(
                    [&](auto &&f) {
                        for (int x = lane; x < sf.cand_n[r][w]; x += 32) {
                            const uint32_t kk = sf.cand[r][w][x].x;
                            if (kk >= fl) f(kk);
                        }
                    },
                    (unsigned)p.top_k, sb.hist, sb.bc);
            }
            thj[r] = max(th, fl);
            unsigned cs = 0;
            for (int x = lane; x < sf.cand_n[r][w]; x += 32) cs += sf.cand[r][w][x].x >= thj[r];
            nsel[r] = (int)block_sum_u<kNT>(cs, sb.redu);
            if (nsel[r] > min(kSeg, kKeptMax / c)) ovf = true;
        }
        const bool any_local = __syncthreads_or(ovf);
        // rank 0 stages its own list before the others write into its buffers
        if (j == 0 && !any_local) {
            if (tid < 2) sf.stage_n[tid] = 0;
            __syncthreads();
            const int lane = tid & 31, w = tid >> 5;
            for (int r = 0; r < rows; ++r)
                for (int x = lane; x < sf.cand_n[r][w]; x += 32) {
                    const uint2 e = sf.cand[r][w][x];
                    if (e.x >= thj[r]) sf.stage[r][atomicAdd(&sf.stage_n[r], 1)] = e;
                }
        }
        cluster_ready();
        if (tid == 0 && any_local) {
            for (int r = 0; r < c; ++r) atomicOr(cluster.map_shared_rank(&sb.ovf, r), 1u);
        }
        cluster.sync();  // (A) every CTA is done with its own buffers
        if (sb.ovf == 0u) {
            // push this slice's list into rank 0's segment j
            SampFast *dst = cluster.map_shared_rank(&sf, 0);
            const int lane = tid & 31, w = tid >> 5;
            for (int r = 0; r < rows; ++r) {
                if (j == 0) {
                    for (int x = tid; x < sf.stage_n[r]; x += kNT) dst->cand[r][0][x] = sf.stage[r][x];
                    if (tid == 0) dst->recv_n[r][0] = sf.stage_n[r];
                } else {
                    // compact per warp with a ballot, offsets from a warp scan of counts
                    __shared__ int s_woff[kNW];
                    int mycnt = 0;
                    for (int x = lane; x < sf.cand_n[r][w]; x += 32) mycnt += sf.cand[r][w][x].x >= thj[r];
                    mycnt = __reduce_add_sync(kFull, mycnt);
                    if (lane == 0) s_woff[w] = mycnt;
                    __syncthreads();
                    int off = 0;
                    for (int q = 0; q < w; ++q) off += s_woff[q];
                    for (int x0 = 0; x0 < sf.cand_n[r][w]; x0 += 32) {
                        const int x = x0 + lane;
                        const bool keep = x < sf.cand_n[r][w] && sf.cand[r][w][x].x >= thj[r];
                        const unsigned kb = __ballot_sync(kFull, keep);
                        if (keep) dst->cand[r][j][off + __popc(kb & lanemask_lt())] = sf.cand[r][w][x];
                        off += __popc(kb);
                    }
                    if (tid == 0) {
                        int tot = 0;
                        for (int q = 0; q < kNW; ++q) tot += s_woff[q];
                        dst->recv_n[r][j] = tot;
                    }
                    __syncthreads();
                }
            }
        }
        cluster.sync();  // (B) rank 0 holds every slice's list
        fast = sb.ovf == 0u;
        if (fast && j != 0) return;
    }

    Outcome o{1.0f, 0.0f, -1, 0u};
    if (fast) {
        // ==================== rank 0: compact computation ====================
        if constexpr (MODE == MODE_FAST) {
            SampFast &sf = sf_storage;
            const int rows = has_draft ? 2 : 1;
            uint32_t th[2] = {0u, 0u};
            for (int r = 0; r < rows; ++r) {
                unsigned tot = 0;
                for (int s = 0; s < c; ++s) tot += (unsigned)sf.recv_n[r][s];
                th[r] = block_kth_largest<KB, kNT>(
                    [&](auto &&f) {
                        for (int s = 0; s < c; ++s)
                            for (int x = tid; x < sf.recv_n[r][s]; x += kNT) f(sf.cand[r][s][x].x);
                    },
                    (unsigned)min((unsigned)p.top_k, tot), sb.hist, sb.bc);
                // compact the kept set to the front of row r's receive area
                uint2 tmp[kMaxCluster];
                int nt = 0;
                for (int s = 0; s < c; ++s)
                    for (int x = tid; x < sf.recv_n[r][s]; x += kNT)
                        if (sf.cand[r][s][x].x >= th[r] && nt < kMaxCluster) tmp[nt++] = sf.cand[r][s][x];
                if (tid == 0) sf.kn[r] = 0;
                __syncthreads();
                uint2 *flat = &sf.cand[r][0][0];
                for (int i = 0; i < nt; ++i) flat[atomicAdd(&sf.kn[r], 1)] = tmp[i];
                __syncthreads();
            }
            // row statistics in dd over the kept sets (fixed order per thread)
            const float2 *tab = sb.tab;
            const float2 ln2 = sb.ln2;
            const uint2 *Kp = &sf.cand[0][0][0];
            const uint2 *Kq = &sf.cand[1][0][0];
            const int np = sf.kn[0], nq = rows == 2 ? sf.kn[1] : 0;
            float mp = -INFINITY, mq = -INFINITY;
            for (int i = tid; i < np; i += kNT) mp = fmaxf(mp, key_value<T>(Kp[i].x));
            for (int i = tid; i < nq; i += kNT) mq = fmaxf(mq, key_value<T>(Kq[i].x));
            mp = block_ms<kNT>(MaxSum{mp, 0.0f}, 1.0f, sb.red2).m;
            mq = block_ms<kNT>(MaxSum{mq, 0.0f}, 1.0f, sb.red2).m;
            const bool bad_row = mp == -INFINITY || (has_draft && mq == -INFINITY);
            dd sp{0.0f, 0.0f}, sq{0.0f, 0.0f};
            if (!bad_row) {
                for (int i = tid; i < np; i += kNT) sp = dd_add(sp, dd_expw(key_value<T>(Kp[i].x), mp, c2d, tab, ln2));
                for (int i = tid; i < nq; i += kNT) sq = dd_add(sq, dd_expw(key_value<T>(Kq[i].x), mq, c2d, tab, ln2));
            }
            block_dd_sum2<kNT>(sp, sq, sb.redd);
            const bool bad = bad_tok || bad_row;
            o.info = (bad_tok ? REC_BAD_INPUT : 0u) | (bad_row ? REC_BAD_ROW : 0u);
            if (!bad) {
                const dd isp = dd_recip(sp);
                const dd isq = has_draft ? dd_recip(sq) : dd{0.0f, 0.0f};
                bool accept = false;
                if (has_draft) {
                    const dd pd = kkey<T>(l_d) >= th[0] ? dd_mul(dd_expw(l_d, mp, c2d, tab, ln2), isp) : dd{0.0f, 0.0f};
                    const dd qd = kkey<T>(g_d) >= th[1] ? dd_mul(dd_expw(g_d, mq, c2d, tab, ln2), isq) : dd{0.0f, 0.0f};
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
                // residual weights over the target's kept set (q gathered from the draft row)
                auto qprob = [&](int idx) -> dd {
                    const float y = ld_elem(drow, idx);
                    return kkey<T>(y) >= th[1] ? dd_mul(dd_expw(y, mq, c2d, tab, ln2), isq) : dd{0.0f, 0.0f};
                };
                dd zw{0.0f, 0.0f}, zp{0.0f, 0.0f};
                if (has_draft) {
                    for (int i = tid; i < np; i += kNT) {
                        const dd pi = dd_mul(dd_expw(key_value<T>(Kp[i].x), mp, c2d, tab, ln2), isp);
                        zw = dd_add(zw, dd_max0(dd_add(pi, dd_neg(qprob((int)Kp[i].y)))));
                        zp = dd_add(zp, pi);
                    }
                    block_dd_sum2<kNT>(zw, zp, sb.redd);
                    o.z = dd_to_f(zw);
                }
                if (tid == 0) sb.rej = *((volatile unsigned *)&p.rejword[b]);
                __syncthreads();
                const bool earlier = sb.rej > (unsigned)(g - k + 1);
                if (has_draft && !accept && tid == 0) atomicMax(p.rejword + b, (unsigned)(g - k + 1));
                if ((!has_draft || !accept) && !earlier) {
                    // ---- the draw, in token order over the kept set ----
                    const bool fb = has_draft && dd_le(zw, dd{p.eps, 0.0f});
                    if (fb) o.info |= REC_FALLBACK;
                    const bool use_p = !has_draft || fb;
                    const dd total = !has_draft ? sp : (fb ? zp : zw);
                    const dd t = dd_mul_f(total, u_f);
                    // sort the kept entries by token id (rank = number of smaller ids)
                    float2 *ws = reinterpret_cast<float2 *>(&sf.cand[1][0][0]);
                    int *wi = reinterpret_cast<int *>(&sf.stage[0][0]);
                    __syncthreads();
                    for (int i = tid; i < np; i += kNT) {
                        const uint32_t id = Kp[i].y;
                        int rank = 0;
                        for (int q = 0; q < np; ++q) rank += Kp[q].y < id;
                        dd wgt = dd_expw(key_value<T>(Kp[i].x), mp, c2d, tab, ln2);
                        if (has_draft) {
                            wgt = dd_mul(wgt, isp);
                            if (!use_p) wgt = dd_max0(dd_add(wgt, dd_neg(qprob((int)id))));
                        }
                        ws[rank] = make_float2(wgt.hi, wgt.lo);
                        wi[rank] = (int)id;
                    }
                    __syncthreads();
                    o.token = dd_scan_slice<kNT>(0, np, dd{0.0f, 0.0f}, t,
                                                 [&](int i) { return dd{ws[i].x, ws[i].y}; }, sb);
                    if (o.token >= 0) o.token = wi[o.token];
                }
            }
            finish(p, b, k, o, sb);
            return;
        }
    }

    // ===================== cluster path (full vocab / masked) =================
    uint32_t th_p = 0u, th_q = 0u;
    constexpr bool MASK = MODE != MODE_FULL;
    if (MASK) {
        uint32_t lo_p = 0u, hi_p = KB == 32 ? 0xffffffffu : ((1u << KB) - 1u);
        uint32_t lo_q = 0u, hi_q = has_draft ? hi_p : 0u;
        const unsigned K = (unsigned)p.top_k;
        for (int it = 0; it < KB; ++it) {
            const bool act_p = lo_p < hi_p, act_q = lo_q < hi_q;
            if (!act_p && !act_q) break;  // identical in every CTA of the cluster
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
            cluster_ready();
            if (tid < c) {
                unsigned *dst = cluster.map_shared_rank(&sb.cnt[par][0][0], tid);
                dst[j] = cp;
                dst[kMaxCluster + j] = cq;
            }
            cluster.sync();
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
    MaxSum msp{-INFINITY, 0.0f}, msq{-INFINITY, 0.0f};
    if (has_draft) {
        for_slice2<T, 2>(trow, drow, lo, hi, [&](const float *xa, const float *xb, int, int cnt) {
            ms_update<VEC, MASK>(msp, xa, cnt, th_p, KS, c2);
            ms_update<VEC, MASK>(msq, xb, cnt, th_q, KS, c2);
        });
    } else {
        for_slice_vec<T, 4>(trow, lo, hi, tid, kNT, [&](const float *x, int, int cnt) {
            ms_update<VEC, MASK>(msp, x, cnt, th_p, KS, c2);
        });
    }
    msp = block_ms<kNT>(msp, c2, sb.red2);
    msq = block_ms<kNT>(msq, c2, sb.red2);
    unsigned prior = 0u;
    if (j == 0 && tid == 0) prior = *((volatile unsigned *)&p.rejword[b]);
    cluster_ready();
    if (tid < c) {
        float4 *dst = cluster.map_shared_rank(&sb.ms[0], tid);
        dst[j] = make_float4(msp.m, msp.s, msq.m, msq.s);
    }
    if (j == 0 && tid == 0)
        for (int r = 0; r < c; ++r) *cluster.map_shared_rank(&sb.rej, r) = prior;
    cluster.sync();
    MaxSum Mp{-INFINITY, 0.0f}, Mq{-INFINITY, 0.0f};
    for (int r = 0; r < c; ++r) {
        Mp = ms_combine(Mp, MaxSum{sb.ms[r].x, sb.ms[r].y}, c2);
        Mq = ms_combine(Mq, MaxSum{sb.ms[r].z, sb.ms[r].w}, c2);
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
        if (tid < c) *cluster.map_shared_rank(&sb.zdiag[j], tid) = zw;
        cluster.sync();
        float z = 0.0f;
        for (int r = 0; r < c; ++r) z += sb.zdiag[r];
        o.z = z;
    }

    if (draw) {
        // ---- the draw in dd: slice sums (pass A), residual (pass B), scan ----
        const float2 *tab = sb.tab;
        const float2 ln2 = sb.ln2;
        const float mp = Mp.m, mq = Mq.m;
        auto ep = [&](float x) -> dd {
            return (!MASK || (fkey(x) >> KS) >= th_p) ? dd_expw(x, mp, c2d, tab, ln2) : dd{0.0f, 0.0f};
        };
        auto eq = [&](float y) -> dd {
            return (!MASK || (fkey(y) >> KS) >= th_q) ? dd_expw(y, mq, c2d, tab, ln2) : dd{0.0f, 0.0f};
        };
        dd sp{0.0f, 0.0f}, sq{0.0f, 0.0f};
        if (has_draft) {
            for_slice2<T, 2>(trow, drow, lo, hi, [&](const float *xa, const float *xb, int, int cnt) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    if (e < cnt) {
                        sp = dd_add(sp, ep(xa[e]));
                        sq = dd_add(sq, eq(xb[e]));
                    }
                }
            });
        } else {
            for_slice_vec<T, 4>(trow, lo, hi, tid, kNT, [&](const float *x, int, int cnt) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (e < cnt) sp = dd_add(sp, ep(x[e]));
            });
        }
        block_dd_sum2<kNT>(sp, sq, sb.redd);
        if (tid < c) *cluster.map_shared_rank(&sb.dsum[j], tid) = make_float4(sp.hi, sp.lo, sq.hi, sq.lo);
        cluster.sync();
        dd Sp{0.0f, 0.0f}, Sq{0.0f, 0.0f};
        float4 part[kMaxCluster];
        for (int r = 0; r < c; ++r) {
            Sp = dd_add(Sp, dd{sb.dsum[r].x, sb.dsum[r].y});
            Sq = dd_add(Sq, dd{sb.dsum[r].z, sb.dsum[r].w});
            part[r] = sb.dsum[r];
        }
        const dd isp = dd_recip(Sp);
        const dd isq = has_draft ? dd_recip(Sq) : dd{0.0f, 0.0f};
        bool use_p = true, fb = false;
        dd total = Sp;  // bonus: weights are the unnormalised target terms
        if (has_draft) {
            dd zw{0.0f, 0.0f}, zp{0.0f, 0.0f};
            for_slice2<T, 2>(trow, drow, lo, hi, [&](const float *xa, const float *xb, int, int cnt) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    if (e < cnt) {
                        const dd pi = dd_mul(ep(xa[e]), isp);
                        const dd qi = dd_mul(eq(xb[e]), isq);
                        zw = dd_add(zw, dd_max0(dd_add(pi, dd_neg(qi))));
                        zp = dd_add(zp, pi);
                    }
                }
            });
            block_dd_sum2<kNT>(zw, zp, sb.redd);
            __syncthreads();
            if (tid < c) *cluster.map_shared_rank(&sb.dsum[j], tid) = make_float4(zw.hi, zw.lo, zp.hi, zp.lo);
            cluster.sync();
            dd Zw{0.0f, 0.0f}, Zp{0.0f, 0.0f};
            for (int r = 0; r < c; ++r) {
                Zw = dd_add(Zw, dd{sb.dsum[r].x, sb.dsum[r].y});
                Zp = dd_add(Zp, dd{sb.dsum[r].z, sb.dsum[r].w});
                part[r] = sb.dsum[r];
            }
            o.z = dd_to_f(Zw);
            fb = dd_le(Zw, dd{p.eps, 0.0f});
            use_p = fb;
            total = fb ? Zp : Zw;
            if (fb) o.info |= REC_FALLBACK;
        }
        const dd t = dd_mul_f(total, u_f);
        // the slice that holds the crossing (identical choice in every CTA)
        int owner = -1, lastpos = -1;
        dd acc{0.0f, 0.0f}, own_prefix{0.0f, 0.0f}, last_prefix{0.0f, 0.0f};
        for (int r = 0; r < c; ++r) {
            const dd prt = !has_draft ? dd{part[r].x, part[r].y}
                                      : (use_p ? dd{part[r].z, part[r].w} : dd{part[r].x, part[r].y});
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
                if (!has_draft) return e;
                const dd pi = dd_mul(e, isp);
                if (use_p) return pi;
                return dd_max0(dd_add(pi, dd_neg(dd_mul(eq(ld_elem(drow, i)), isq))));
            }, sb);
        }
    }
    if (j == writer) finish(p, b, k, o, sb);
}

cudaError_t launch_chain_sample(const SampleParams &p, int dtype, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)p.B * (p.gamma + 1) * p.c));
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int mode = p.top_k == 0 ? MODE_FULL : (p.top_k <= kTopKFastMax ? MODE_FAST : MODE_SEARCH);
    if (dtype == SPEC_DTYPE_BF16) {
        using T = __nv_bfloat16;
        if (mode == MODE_FULL) return cudaLaunchKernelEx(&cfg, chain_sample_kernel<T, MODE_FULL>, p);
        if (mode == MODE_FAST) return cudaLaunchKernelEx(&cfg, chain_sample_kernel<T, MODE_FAST>, p);
        return cudaLaunchKernelEx(&cfg, chain_sample_kernel<T, MODE_SEARCH>, p);
    }
    if (mode == MODE_FULL) return cudaLaunchKernelEx(&cfg, chain_sample_kernel<float, MODE_FULL>, p);
    if (mode == MODE_FAST) return cudaLaunchKernelEx(&cfg, chain_sample_kernel<float, MODE_FAST>, p);
    return cudaLaunchKernelEx(&cfg, chain_sample_kernel<float, MODE_SEARCH>, p);
}

}  // namespace specv
