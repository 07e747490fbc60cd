// Sampled chain verification (temperature > 0) on sm_103a.
//
// One round of speculative sampling ("10.6 投机解码：为什么“先猜后验”能加速"
// §10.6.1; "KV Cache 优化（四）：Speculative Decoding 投机解码" §4, §5):
// transform each target and draft row (temperature, top-k), accept d_k with
// probability min(1, p_k(d_k)/q_k(d_k)) left to right, draw the replacement
// from norm(max(0, p_k - q_k)) at the first rejection (from p_k itself when
// that mass is <= eps, the glossary page's "stable fallback"), or a bonus
// token from p_{gamma+1} when every draft is accepted.
//
// GB300 mapping.  A thread-block cluster of c CTAs handles one (request,
// position k): CTA j owns vocab slice j of target row k and of draft row k
// (the bonus position has only the target row).  Each CTA streams its slices
// once from HBM with 16-byte loads and keeps an online (max, sum of exp2)
// pair per row; the c partial pairs are pushed into every CTA's shared
// memory over DSMEM and combined in rank order, so every CTA holds the same
// softmax normalisers and computes the same a_k and accept bit.  Only a
// position that needs a draw (a rejection, or the bonus row) or the residual
// mass runs a second pass over its slices, which were read by the same CTA
// microseconds earlier and are served from L2; the slice totals of the
// residual are exchanged the same way and the one CTA whose slice holds the
// CDF crossing scans it in token order.  Top-k thresholds are found exactly
// by a cluster-wide binary search over order-preserving keys.  Each position
// writes one record; the last position of a request to arrive (an arrival
// counter) writes the request's outputs.  No block spins on another: the
// only waits are cluster barriers between co-scheduled CTAs.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace specv {

constexpr int kSampNT = 256;
constexpr int kMaxCluster = 8;
constexpr int kScanE = 16;  // elements per thread per tile of the CDF scan

template <typename T> __device__ __forceinline__ uint32_t topkey(float x) {
    return fkey(x) >> (32 - Elem<T>::KEY_BITS);
}

// Two rows traversed together over the same slice: f(xa[VEC], xb[VEC], base, cnt).
// Vector loads are used for both rows when they share their 16-byte phase,
// otherwise row b is read element by element.
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
template <int VEC, bool TOPK>
__device__ __forceinline__ void ms_update(MaxSum &ms, const float *x, int cnt, uint32_t th,
                                          int keyshift, float c2) {
    float vm = -INFINITY;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
        const bool keep = e < cnt && (!TOPK || (fkey(x[e]) >> keyshift) >= th);
        if (keep) vm = fmaxf(vm, x[e]);
    }
    if (vm > ms.m) {
        ms.s = ms.m == -INFINITY ? 0.0f : ms.s * exp2f((ms.m - vm) * c2);
        ms.m = vm;
    }
    if (ms.m != -INFINITY) {
        const float mc = ms.m * c2;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const bool keep = e < cnt && (!TOPK || (fkey(x[e]) >> keyshift) >= th);
            if (keep) ms.s += exp2f(fmaf(x[e], c2, -mc));
        }
    }
}

struct RowStats {
    float mc;    // max * c2
    float invS;  // 1 / sum
    uint32_t th; // top-k threshold on the top key bits (0 keeps all)
};

template <bool TOPK>
__device__ __forceinline__ float prob_of(float x, const RowStats &r, int keyshift, float c2) {
    if (TOPK && (fkey(x) >> keyshift) < r.th) return 0.0f;
    return exp2f(fmaf(x, c2, -r.mc)) * r.invS;
}

template <typename T, bool TOPK>
__global__ void __launch_bounds__(kSampNT) chain_sample_kernel(SampleParams p) {
    constexpr int VEC = Elem<T>::VEC;
    constexpr int KB = Elem<T>::KEY_BITS;
    constexpr int keyshift = 32 - KB;
    cg::cluster_group cluster = cg::this_cluster();
    const int c = p.c;
    const int j = (int)cluster.block_rank();
    const int pos_id = blockIdx.x / c;
    const int g = p.gamma;
    const int b = pos_id / (g + 1), k = pos_id % (g + 1);
    const bool has_draft = k < g;
    const int lo = min(p.V, j * p.Vs), hi = min(p.V, lo + p.Vs);
    const T *trow = reinterpret_cast<const T *>(p.target) + (int64_t)(b * (g + 1) + k) * p.tstride;
    const T *drow = has_draft
        ? reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + k) * p.dstride : nullptr;
    const float c2 = p.c2;

    __shared__ float2 s_red2[kSampNT / 32];
    __shared__ float s_redf[kSampNT / 32];
    __shared__ unsigned s_redu[kSampNT / 32];
    __shared__ float2 s_ms[2][kMaxCluster];          // (max, sum) per row, per rank
    __shared__ float2 s_z[kMaxCluster];              // (residual part, target part) per rank
    __shared__ unsigned s_cnt[2][2][kMaxCluster];    // top-k counts [parity][row][rank]
    __shared__ int s_found, s_lastpos, s_arrive_last;

    // Every CTA of the cluster must be running before any of them writes into
    // another's shared memory: arrive now, wait just before the first push.
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
    bool waited = false;
    auto cluster_ready = [&]() {
        if (!waited) {
            asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
            waited = true;
        }
    };

    const int d = has_draft ? p.tokens[(int64_t)b * g + k] : 0;
    const bool bad_tok = has_draft && (d < 0 || d >= p.V);

    // ---- exact top-k thresholds: cluster-wide binary search on order keys ----
    uint32_t th_p = 0, th_q = 0;
    if (TOPK) {
        uint32_t lo_p = 0, hi_p = KB == 32 ? 0xffffffffu : ((1u << KB) - 1u);
        uint32_t lo_q = 0, hi_q = has_draft ? hi_p : 0u;
        const unsigned K = (unsigned)p.top_k;
        for (int it = 0; it < KB; ++it) {
            const bool act_p = lo_p < hi_p, act_q = lo_q < hi_q;
            if (!act_p && !act_q) break;  // identical in every CTA of the cluster
            const uint32_t mid_p = lo_p + (uint32_t)(((uint64_t)hi_p - lo_p + 1) >> 1);
            const uint32_t mid_q = lo_q + (uint32_t)(((uint64_t)hi_q - lo_q + 1) >> 1);
            unsigned cp = 0, cq = 0;
            if (act_p)
                for_slice<T, 4>(trow, lo, hi, threadIdx.x, kSampNT,
                                [&](float x, int) { cp += (fkey(x) >> keyshift) >= mid_p; });
            if (act_q)
                for_slice<T, 4>(drow, lo, hi, threadIdx.x, kSampNT,
                                [&](float x, int) { cq += (fkey(x) >> keyshift) >= mid_q; });
            cp = block_sum_u<kSampNT>(cp, s_redu);
            cq = block_sum_u<kSampNT>(cq, s_redu);
            const int par = it & 1;
            cluster_ready();
            if (threadIdx.x < c) {
                unsigned *dst = cluster.map_shared_rank(&s_cnt[par][0][0], threadIdx.x);
                dst[j] = cp;
                dst[kMaxCluster + j] = cq;
            }
            cluster.sync();
            unsigned tp = 0, tq = 0;
            for (int r = 0; r < c; ++r) {
                tp += s_cnt[par][0][r];
                tq += s_cnt[par][1][r];
            }
            if (act_p) { if (tp >= K) lo_p = mid_p; else hi_p = mid_p - 1; }
            if (act_q) { if (tq >= K) lo_q = mid_q; else hi_q = mid_q - 1; }
        }
        th_p = lo_p;
        th_q = lo_q;
    }

    // ---- pass 1: online max / sum of each row's kept logits -------------------
    MaxSum msp{-INFINITY, 0.0f}, msq{-INFINITY, 0.0f};
    if (has_draft) {
        for_slice2<T, 2>(trow, drow, lo, hi, [&](const float *xa, const float *xb, int, int cnt) {
            ms_update<VEC, TOPK>(msp, xa, cnt, th_p, keyshift, c2);
            ms_update<VEC, TOPK>(msq, xb, cnt, th_q, keyshift, c2);
        });
    } else {
        for_slice_vec<T, 4>(trow, lo, hi, threadIdx.x, kSampNT, [&](const float *x, int, int cnt) {
            ms_update<VEC, TOPK>(msp, x, cnt, th_p, keyshift, c2);
        });
    }
    msp = block_ms<kSampNT>(msp, c2, s_red2);
    msq = block_ms<kSampNT>(msq, c2, s_red2);
    cluster_ready();
    if (threadIdx.x < c) {
        float2 *dst = cluster.map_shared_rank(&s_ms[0][0], threadIdx.x);
        dst[j] = make_float2(msp.m, msp.s);
        dst[kMaxCluster + j] = make_float2(msq.m, msq.s);
    }
    cluster.sync();
    MaxSum Mp{-INFINITY, 0.0f}, Mq{-INFINITY, 0.0f};
    for (int r = 0; r < c; ++r) {
        Mp = ms_combine(Mp, MaxSum{s_ms[0][r].x, s_ms[0][r].y}, c2);
        Mq = ms_combine(Mq, MaxSum{s_ms[1][r].x, s_ms[1][r].y}, c2);
    }
    const bool bad_row = Mp.m == -INFINITY || (has_draft && Mq.m == -INFINITY);
    const RowStats P{Mp.m * c2, 1.0f / Mp.s, th_p};
    const RowStats Q{Mq.m * c2, 1.0f / Mq.s, th_q};
    const bool bad = bad_tok || bad_row;

    // ---- acceptance test (identical in every CTA) ------------------------------
    float a = 1.0f;
    bool accept = false;
    if (has_draft && !bad) {
        const float pd = prob_of<TOPK>(ld_elem(trow, d), P, keyshift, c2);
        const float qd = prob_of<TOPK>(ld_elem(drow, d), Q, keyshift, c2);
        a = qd > 0.0f ? fminf(1.0f, pd / qd) : (pd > 0.0f ? 1.0f : 0.0f);
        accept = p.unif[(int64_t)b * (g + 1) + k] < a;
    }
    const bool need_sample = !bad && (!has_draft || !accept);
    const bool need_z = !bad && has_draft && (p.resid != nullptr || !accept);

    float Z = 0.0f;
    int token = -1, writer = 0;
    bool fallback = false;
    if (need_sample || need_z) {
        // ---- pass 2 (L2): residual mass and target mass of this slice ---------
        float zw = 0.0f, zp = 0.0f;
        if (has_draft) {
            for_slice2<T, 2>(trow, drow, lo, hi, [&](const float *xa, const float *xb, int, int cnt) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    if (e < cnt) {
                        const float pi = prob_of<TOPK>(xa[e], P, keyshift, c2);
                        const float qi = prob_of<TOPK>(xb[e], Q, keyshift, c2);
                        zw += fmaxf(pi - qi, 0.0f);
                        zp += pi;
                    }
                }
            });
        } else {
            for_slice_vec<T, 4>(trow, lo, hi, threadIdx.x, kSampNT, [&](const float *x, int, int cnt) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (e < cnt) zp += prob_of<TOPK>(x[e], P, keyshift, c2);
            });
            zw = zp;
        }
        zw = block_sum<kSampNT>(zw, s_redf);
        zp = block_sum<kSampNT>(zp, s_redf);
        if (threadIdx.x < c) {
            float2 *dst = cluster.map_shared_rank(&s_z[0], threadIdx.x);
            dst[j] = make_float2(zw, zp);
        }
        cluster.sync();
        float zp_tot = 0.0f;
        for (int r = 0; r < c; ++r) {
            Z += s_z[r].x;
            zp_tot += s_z[r].y;
        }
        if (need_sample) {
            // draw weights: the residual, or p itself (bonus row; fallback)
            fallback = has_draft && Z <= p.eps;
            const bool use_p = !has_draft || fallback;
            const float total = use_p ? zp_tot : Z;
            const float t = p.unif[(int64_t)b * (g + 1) + g] * total;
            int owner = -1, last_pos = -1;
            float acc = 0.0f, own_prefix = 0.0f, last_prefix = 0.0f;
            for (int r = 0; r < c; ++r) {
                const float part = use_p ? s_z[r].y : s_z[r].x;
                if (part > 0.0f) {
                    if (owner < 0 && acc + part > t) { owner = r; own_prefix = acc; }
                    last_pos = r;
                    last_prefix = acc;
                }
                acc += part;
            }
            if (owner < 0) { owner = last_pos; own_prefix = last_prefix; }
            writer = owner < 0 ? 0 : owner;
            if (j == owner) {
                // ---- pass 3 (owner only, L2): scan the slice in token order ----
                if (threadIdx.x == 0) { s_found = INT_MAX; s_lastpos = -1; }
                __syncthreads();
                float carry = own_prefix;
                for (int base = lo; base < hi; base += kSampNT * kScanE) {
                    const int i0 = base + threadIdx.x * kScanE;
                    float w[kScanE];
                    float run = 0.0f;
                    int lastp = -1;
#pragma unroll
                    for (int e = 0; e < kScanE; ++e) {
                        const int i = i0 + e;
                        float we = 0.0f;
                        if (i < hi) {
                            const float pi = prob_of<TOPK>(ld_elem(trow, i), P, keyshift, c2);
                            if (use_p) {
                                we = pi;
                            } else {
                                const float qi = prob_of<TOPK>(ld_elem(drow, i), Q, keyshift, c2);
                                we = fmaxf(pi - qi, 0.0f);
                            }
                        }
                        w[e] = we;
                        run += we;
                        if (we > 0.0f) lastp = i;
                    }
                    // exclusive block scan of the per-thread totals
                    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
                    float incl = run;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float y = __shfl_up_sync(kFull, incl, o);
                        if (lane >= o) incl += y;
                    }
                    __syncthreads();
                    if (lane == 31) s_redf[wid] = incl;
                    __syncthreads();
                    float wpre = 0.0f, tile_tot = 0.0f;
                    for (int q = 0; q < kSampNT / 32; ++q) {
                        if (q < wid) wpre += s_redf[q];
                        tile_tot += s_redf[q];
                    }
                    float cum = carry + wpre + (incl - run);
                    int hit = INT_MAX;
#pragma unroll
                    for (int e = 0; e < kScanE; ++e) {
                        cum += w[e];
                        if (hit == INT_MAX && w[e] > 0.0f && cum > t) hit = i0 + e;
                    }
                    if (hit != INT_MAX) atomicMin(&s_found, hit);
                    if (lastp >= 0) atomicMax(&s_lastpos, lastp);
                    __syncthreads();
                    if (s_found != INT_MAX) break;
                    carry += tile_tot;
                }
                token = s_found != INT_MAX ? s_found : s_lastpos;
            }
        }
    }

    // ---- record + arrival ---------------------------------------------------------
    if (j == writer && threadIdx.x == 0) {
        PosRec rec;
        rec.a = a;
        rec.z = Z;
        rec.token = token;
        rec.info = (accept ? REC_ACCEPT : 0u) | (bad_tok ? REC_BAD_INPUT : 0u) |
                   (bad_row ? REC_BAD_ROW : 0u) | (fallback ? REC_FALLBACK : 0u);
        p.recs[pos_id] = rec;
        __threadfence();
        const unsigned prev = atomicAdd(p.counters + b, 1u);
        s_arrive_last = prev == (unsigned)g;
    }
    __syncthreads();
    if (!(j == writer && s_arrive_last)) return;

    // ---- the request's last position to arrive writes its outputs -------------
    if (threadIdx.x == 0) {
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
            for (int q = 0; q < g; ++q) {
                if (!(R[q].info & REC_ACCEPT)) { n = q; break; }
            }
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
        p.counters[b] = 0u;
    }
}

cudaError_t launch_chain_sample(const SampleParams &p, int dtype, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)p.B * (p.gamma + 1) * p.c));
    cfg.blockDim = dim3(kSampNT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool topk = p.top_k > 0;
    if (dtype == SPEC_DTYPE_BF16) {
        return topk ? cudaLaunchKernelEx(&cfg, chain_sample_kernel<__nv_bfloat16, true>, p)
                    : cudaLaunchKernelEx(&cfg, chain_sample_kernel<__nv_bfloat16, false>, p);
    }
    return topk ? cudaLaunchKernelEx(&cfg, chain_sample_kernel<float, true>, p)
                : cudaLaunchKernelEx(&cfg, chain_sample_kernel<float, false>, p);
}

}  // namespace specv
