// Draft-tree builder, one level per call ("投机推理：小模型搭树，大模型一次验证",
// 树形投机怎么配置 and the three expansion steps): each of the level's parents
// gets the top k_j tokens of its draft logits as children, each child's path
// log-probability is its parent's plus the draft's log-softmax at that token,
// and the n_next children with the highest path log-probability (ties to the
// lower node id) become the next level's parents, in node-id order.
//
// Two launches per level.  The pass (one HBM read of the level's rows): work
// items are (row, 2,048-logit slice); each warp takes one item at a time
// (grid-stride), holds the slice in registers and reduces it to the slice's
// summary: its K largest (value, lowest index) keys, its max and its sum of
// exp(x - max).  The merge, a programmatic dependent of the pass, gives each
// request one warp: it merges the request's rows (top k_j tokens,
// log-sum-exp), writes the new nodes and chooses the next parents.  No
// counters: the workspace holds only the summaries.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"
#include "spec_verify.h"

namespace specv {

namespace {

constexpr int kTlWarps = 8;
constexpr float kL2E = 1.4426950408889634f;

__device__ __forceinline__ float tl_ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// unpack() through opaque register moves: the compiler cannot share the
// unpacked values with an earlier unpack of the same vector, so a pass over a
// register-resident slice does not keep every unpacked element alive
template <typename T> __device__ __forceinline__ void unpack_fresh(const uint4 &v, float *out) {
    uint4 w;
    asm volatile("mov.b32 %0, %1;" : "=r"(w.x) : "r"(v.x));
    asm volatile("mov.b32 %0, %1;" : "=r"(w.y) : "r"(v.y));
    asm volatile("mov.b32 %0, %1;" : "=r"(w.z) : "r"(v.z));
    asm volatile("mov.b32 %0, %1;" : "=r"(w.w) : "r"(v.w));
    unpack<T>(w, out);
}

// Largest element of a 16-byte vector (NaNs are ignored unless all are NaN).
template <typename T> __device__ __forceinline__ float vec_max(const uint4 &v);
template <> __device__ __forceinline__ float vec_max<float>(const uint4 &v) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}
template <> __device__ __forceinline__ float vec_max<__nv_bfloat16>(const uint4 &v) {
    const __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&v.y));
    const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162 *>(&v.z),
                                     *reinterpret_cast<const __nv_bfloat162 *>(&v.w));
    const __nv_bfloat162 c = __hmax2(a, b);
    return fmaxf(__low2float(c), __high2float(c));
}

// the value a key was made from (keys are never 0 here)
__device__ __forceinline__ float key_value(unsigned long long key) {
    const uint32_t u = (uint32_t)(key >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// K largest keys, descending; 0 = empty slot (below every real key)
template <int K> struct TopK {
    unsigned long long k[K];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int i = 0; i < K; ++i) k[i] = 0ull;
    }
    __device__ __forceinline__ void insert(unsigned long long key) {
#pragma unroll
        for (int i = K - 1; i >= 0; --i) {
            const unsigned long long up = i > 0 ? k[i - 1] : ~0ull;
            k[i] = key > up ? up : (key > k[i] ? key : k[i]);
        }
    }
    __device__ __forceinline__ void pop() {
#pragma unroll
        for (int i = 0; i < K - 1; ++i) k[i] = k[i + 1];
        k[K - 1] = 0ull;
    }
};

// K rounds of a warp maximum over the lanes' list heads: lane r returns the
// warp's r-th largest key (keys are distinct: they carry the token index).
template <int K> __device__ __forceinline__ unsigned long long warp_topk(TopK<K> &t, int lane) {
    unsigned long long mine = 0ull;
#pragma unroll 1
    for (int r = 0; r < K; ++r) {
        unsigned long long best = t.k[0];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long other = __shfl_xor_sync(kFull, best, o);
            best = other > best ? other : best;
        }
        if (lane == r) mine = best;
        if (best == 0ull) break;  // every list is empty (the row is shorter than K)
        if (t.k[0] == best) t.pop();
    }
    return mine;
}

// (max, sum of exp(x - max)) pairs; a max of -inf carries no mass
__device__ __forceinline__ void ms_add(float &m, float &s, float m2, float s2) {
    if (!(m2 > -INFINITY)) return;
    if (m2 > m) {
        s = (m > -INFINITY ? s * tl_ex2((m - m2) * kL2E) : 0.f) + s2;
        m = m2;
    } else {
        s += s2 * tl_ex2((m2 - m) * kL2E);
    }
}

__device__ __forceinline__ void warp_ms_combine(float &m, float &s) {
    float mw = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(kFull, mw, o));
    float sl = (m > -INFINITY && mw > -INFINITY) ? s * tl_ex2((m - mw) * kL2E) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sl += __shfl_xor_sync(kFull, sl, o);
    m = mw;
    s = sl;
}

// -- the request's new nodes and the next level's parents (one warp) --------
__device__ void tl_request(const TreeLevelParams &p, int b, int lane, unsigned long long *sk) {
    const int H = p.H, n = p.n_nodes;
    const int64_t nb = (int64_t)b * (p.N + 1);
    unsigned bits = 0;
    for (int j = lane; j < H; j += 32) {
        const int pj = p.root ? 0 : p.parents[(int64_t)b * H + j];
        if (pj < 0 || pj > p.n_before) bits |= SPEC_FLAG_BAD_INPUT;
        if (__ldcg(&p.rowrec[(int64_t)b * H + j].bad)) bits |= SPEC_FLAG_BAD_ROW;
    }
    bits = __reduce_or_sync(kFull, bits);
    if (bits) {
        for (int i = lane; i < p.n_next; i += 32) p.next_parents[(int64_t)b * p.n_next + i] = -1;
        if (lane == 0) {
            if (p.flags) p.flags[b] |= bits;
            atomicOr(p.status, bits);
        }
        return;
    }
    for (int i = lane; i < n; i += 32) {
        const int j = p.head_of[i], r = i - p.koff[j];
        const int pj = p.root ? 0 : p.parents[(int64_t)b * H + j];
        const float plp = p.root ? 0.f : __ldcg(&p.node_logp[nb + pj]);
        const TlRow *rr = p.rowrec + (int64_t)b * H + j;
        const float lp = plp + __ldcg(&rr->lq[r]);
        const int id = p.n_before + 1 + i;
        p.node_token[(int64_t)b * p.N + id - 1] = __ldcg(&rr->tok[r]);
        p.node_parent[(int64_t)b * p.N + id - 1] = pj;
        p.node_logp[nb + id] = lp;
        p.row_of_node[nb + id] = -1;
        sk[i] = argmax_key(lp, id);  // larger log-probability, then the lower id
    }
    if (p.root && lane == 0) {
        p.node_logp[nb] = 0.f;
        p.row_of_node[nb] = 0;
    }
    __syncwarp();
    if (p.n_next > 0) {
        int base = 0;
        for (int c0 = 0; c0 < n; c0 += 32) {
            const int i = c0 + lane;
            bool sel = false;
            if (i < n) {
                const unsigned long long key = sk[i];
                int rank = 0;
                for (int q = 0; q < n; ++q) rank += sk[q] > key;
                sel = rank < p.n_next;
            }
            const unsigned ball = __ballot_sync(kFull, sel);
            if (sel) {
                const int pos = base + __popc(ball & ((1u << lane) - 1u));
                const int id = p.n_before + 1 + i;
                p.next_parents[(int64_t)b * p.n_next + pos] = id;
                p.row_of_node[nb + id] = p.next_row0 + pos;
            }
            base += __popc(ball);
        }
    }
}

// -- merge of one row's slice summaries (one warp) -----------------------------
template <int K>
__device__ void tl_row(const TreeLevelParams &p, int row, int lane) {
    const TlItem *its = p.items + (int64_t)row * p.slices;
    TopK<K> t;
    t.init();
    float m = -INFINITY, s = 0.f;
    unsigned nan = 0;
    for (int q = lane; q < p.slices; q += 32) {
#pragma unroll
        for (int i = 0; i < K; ++i) t.insert(__ldcg(&its[q].key[i]));
        ms_add(m, s, __ldcg(&its[q].m), __ldcg(&its[q].s));
        nan |= __ldcg(&its[q].nan);
    }
    const unsigned long long key = warp_topk<K>(t, lane);
    warp_ms_combine(m, s);
    nan = __reduce_or_sync(kFull, nan);
    const int b = row / p.H, j = row - b * p.H;
    const int kj = p.koff[j + 1] - p.koff[j];
    const bool bad = nan || !(m > -INFINITY && m < INFINITY) || !(s > 0.f && s < INFINITY);
    const float lse = m + logf(s);
    TlRow *rr = p.rowrec + row;
    if (lane < kj) {
        rr->tok[lane] = argmax_key_index(key);
        rr->lq[lane] = key_value(key) - lse;
    }
    if (lane == 0) rr->bad = bad ? 1u : 0u;
}

template <typename T> __host__ __device__ constexpr int tl_slice() { return kTlSliceElems; }
template <typename T> __host__ __device__ constexpr int tl_nv() { return kTlSliceElems / (32 * Elem<T>::VEC); }

// Writes an item's summary (the merge kernel reads it after this grid ends).
template <int K>
__device__ __forceinline__ void tl_publish(const TreeLevelParams &p, int64_t item, int lane,
                                           unsigned long long key, float m, float s, unsigned nan) {
    TlItem *it = p.items + item;
    if (lane < K) it->key[lane] = key;
    if (lane == 0) {
        it->m = m;
        it->s = s;
        it->nan = nan;
    }
}

// Any alignment: each lane streams its elements in index order through a
// sorted register list (every element may be inserted).
template <typename T, int K>
__device__ void tl_item_generic(const TreeLevelParams &p, int64_t item, int lane) {
    const int row = (int)(item / p.slices), sl = (int)(item - (int64_t)row * p.slices);
    const T *r = static_cast<const T *>(p.rows) + (int64_t)row * p.stride;
    const int lo = sl * tl_slice<T>(), hi = min(p.V, lo + tl_slice<T>());
    TopK<K> t;
    t.init();
    float m = -INFINITY, s = 0.f;
    bool nan = false;
    for_slice_vec<T, 4>(r, lo, hi, lane, 32, [&](const float *x, int base, int cnt) {
        constexpr int VEC = Elem<T>::VEC;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            if (e < cnt) {
                nan |= x[e] != x[e];
                ms_add(m, s, x[e], 1.f);
                t.insert(argmax_key(x[e], base + e));
            }
        }
    });
    const unsigned long long key = warp_topk<K>(t, lane);
    warp_ms_combine(m, s);
    tl_publish<K>(p, item, lane, key, m, s, __any_sync(kFull, nan) ? 1u : 0u);
}

// Rows on 16-byte boundaries: the slice is loaded into registers at once;
// the warp max, then the sum of exp(x - max) in one pass; candidates for the
// K largest are the elements at or above the K-th largest lane maximum (at
// least K elements reach it, so nothing below it can be among the K
// largest), gathered in shared memory and sorted by one bitonic network.
constexpr int kCandCap = 32;

__device__ __forceinline__ unsigned long long bitonic_desc(unsigned long long v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const unsigned long long o = __shfl_xor_sync(kFull, v, j);
            // descending overall: the pair's lower lane keeps the larger
            // value in blocks whose bit k is clear, the smaller otherwise
            const bool lower = (lane & j) == 0;
            const bool desc = (lane & k) == 0;
            const bool keep_max = lower == desc;
            v = keep_max ? (o > v ? o : v) : (o < v ? o : v);
        }
    }
    return v;
}

__device__ __forceinline__ float bitonic_desc_f(float v, int lane) {
#pragma unroll
    for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
            const float o = __shfl_xor_sync(kFull, v, j);
            const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
            v = keep_max ? fmaxf(o, v) : fminf(o, v);
        }
    }
    return v;
}

// The K largest keys among a slice's elements at or above theta, streamed
// again from memory (for slices with more candidates than the shared list
// holds: many ties at theta, or few finite values).
template <typename T, int K>
__device__ __noinline__ unsigned long long tl_reread_topk(const TreeLevelParams &p, int row, int lo, int lane,
                                                           float theta) {
    const T *r = static_cast<const T *>(p.rows) + (int64_t)row * p.stride;
    TopK<K> t;
    t.init();
    for_slice_vec<T, 1>(r, lo, min(p.V, lo + tl_slice<T>()), lane, 32, [&](const float *x, int base, int cnt) {
#pragma unroll
        for (int e = 0; e < Elem<T>::VEC; ++e)
            if (e < cnt && x[e] >= theta) t.insert(argmax_key(x[e], base + e));
    });
    return warp_topk<K>(t, lane);
}

template <typename T, int K>
__device__ void tl_item_regs(const TreeLevelParams &p, int row, int sl, int lane, unsigned long long *cand,
                             unsigned *ccnt, const uint4 *stage) {
    constexpr int VEC = Elem<T>::VEC, NV = tl_nv<T>();
    const int64_t item = (int64_t)row * p.slices + sl;
    const T *r = static_cast<const T *>(p.rows) + (int64_t)row * p.stride;
    const int lo = sl * tl_slice<T>();
    const int len = min(p.V - lo, tl_slice<T>());  // valid elements of this slice
    const int nfull = len / VEC;                   // whole vectors
    const uint32_t ninf = sizeof(T) == 4 ? 0xff800000u : 0xff80ff80u;
    uint4 raw[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        const int v = u * 32 + lane;
        raw[u] = v < nfull ? stage[v] : make_uint4(ninf, ninf, ninf, ninf);
    }
    if (nfull * VEC < len && lane == (nfull & 31)) {  // the partial last vector, element-wise
        float x[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) x[e] = nfull * VEC + e < len ? ld_elem(r, lo + nfull * VEC + e) : -INFINITY;
        uint32_t w[4];
        if (sizeof(T) == 4) {
#pragma unroll
            for (int e = 0; e < 4; ++e) w[e] = __float_as_uint(x[e]);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                w[e] = (__float_as_uint(x[2 * e]) >> 16) | (__float_as_uint(x[2 * e + 1]) & 0xffff0000u);
        }
        const uint4 pv = make_uint4(w[0], w[1], w[2], w[3]);
#pragma unroll
        for (int u = 0; u < NV; ++u) raw[u] = (u == (nfull >> 5)) ? pv : raw[u];
    }
    // per-vector maxima (bf16 pairs compared packed), then the lane and warp max
    float vm[NV];
#pragma unroll
    for (int u = 0; u < NV; ++u) vm[u] = vec_max<T>(raw[u]);
    float lm = vm[0];
#pragma unroll
    for (int u = 1; u < NV; ++u) lm = fmaxf(lm, vm[u]);
    float m = lm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    // the K-th largest lane maximum
    const float theta = __shfl_sync(kFull, bitonic_desc_f(lm, lane), K - 1);
    // one pass: the sum of exp(x - m) (per-vector sums, then a pairwise tree
    // over the vectors) and the candidates, the valid elements at or above
    // theta, looked for only in vectors whose maximum reaches it.  The
    // vectors are unpacked afresh here (so the unpacked slice is never held
    // in registers across the warp reductions above).
    float s = 0.f;
    bool nan = false;
    const float mk = m > -INFINITY ? m * kL2E : 0.f;
#pragma unroll
    for (int u = 0; u < NV; ++u) {
        float x[VEC];
        unpack_fresh<T>(raw[u], x);
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) a += tl_ex2(fmaf(x[e], kL2E, -mk));
        if (vm[u] >= theta) {
            const int base = lo + (u * 32 + lane) * VEC;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                if (x[e] >= theta && base + e < p.V) {
                    const unsigned pos = atomicAdd(ccnt, 1u);
                    if (pos < kCandCap) cand[pos] = argmax_key(x[e], base + e);
                }
            }
        }
        vm[u] = a;  // the vector's sum from here on
    }
    if (m > -INFINITY) {
#pragma unroll
        for (int w2 = NV / 2; w2 > 0; w2 >>= 1)
#pragma unroll
            for (int u = 0; u < w2; ++u) vm[u] += vm[u + w2];
        s = vm[0];
        nan = s != s;
    } else {  // no finite maximum (the row is flagged): only look for a NaN
#pragma unroll
        for (int u = 0; u < NV; ++u) {
            float x[VEC];
            unpack_fresh<T>(raw[u], x);
#pragma unroll
            for (int e = 0; e < VEC; ++e) nan |= x[e] != x[e];
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    __syncwarp();
    const unsigned nc = *ccnt;
    unsigned long long key;
    if (nc <= kCandCap) {
        key = bitonic_desc(lane < (int)nc ? cand[lane] : 0ull, lane);
    } else {
        key = tl_reread_topk<T, K>(p, row, lo, lane, theta);
    }
    __syncwarp();
    if (lane == 0) *ccnt = 0u;
    tl_publish<K>(p, item, lane, key, m, s, __any_sync(kFull, nan) ? 1u : 0u);
}

// Bulk-copy ring per warp for the register path: stage t % NST holds the
// whole-vector body of the warp's t-th item, issued NST items ahead.
template <typename T> __host__ __device__ constexpr int tl_nst() { return sizeof(T) == 2 ? 3 : 2; }
template <typename T> __host__ __device__ constexpr int tl_ring_bytes() {
    return kTlWarps * tl_nst<T>() * (kTlSliceElems * (int)sizeof(T) + 16);
}

template <typename T, int K, bool REGS>
__global__ void __launch_bounds__(kTlWarps * 32, 2) tree_level_kernel(const TreeLevelParams p) {
    __shared__ unsigned long long cand_all[kTlWarps][kCandCap];
    __shared__ unsigned ccnt_all[kTlWarps];
    __shared__ unsigned long long bar_all[kTlWarps][tl_nst<T>()];
    extern __shared__ __align__(128) unsigned char ring_all[];
    constexpr int NST = tl_nst<T>(), SB = kTlSliceElems * (int)sizeof(T);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (lane == 0) ccnt_all[w] = 0u;
    const int64_t items = (int64_t)p.B * p.H * p.slices;
    const int64_t first = (int64_t)blockIdx.x * kTlWarps + w, stride = (int64_t)gridDim.x * kTlWarps;
    if (!REGS) {
        __syncwarp();
        for (int64_t item = first; item < items; item += stride) tl_item_generic<T, K>(p, item, lane);
        pdl_launch_dependents();
        return;
    }
    unsigned char *ring = ring_all + (size_t)w * NST * SB;
    unsigned long long *bar = bar_all[w];
    // (row, slice) cursors: the item being read and the item being issued
    // (items fit in 32 bits: the host checks rows * slices)
    const int stride32 = (int)stride, srow = stride32 / p.slices, ssl = stride32 - srow * p.slices;
    const int mine = first < items ? (int)((items - first + stride - 1) / stride) : 0;
    struct Cur {
        int row, sl;
    };
    auto advance = [&](Cur &c) {
        c.row += srow;
        c.sl += ssl;
        if (c.sl >= p.slices) {
            c.sl -= p.slices;
            ++c.row;
        }
    };
    Cur rd{(int)(first / p.slices), (int)(first % p.slices)};
    Cur is = rd;
    // issue the body copy of the item at the issue cursor into stage st (lane 0)
    auto issue = [&](int st) {
        const int lo = is.sl * tl_slice<T>();
        const int nfull = min(p.V - lo, tl_slice<T>()) / Elem<T>::VEC;
        const uint32_t bytes = (uint32_t)nfull * 16u;
        mbar_arrive_expect_tx(&bar[st], bytes);
        if (bytes)
            bulk_g2s(ring + (size_t)st * SB, static_cast<const T *>(p.rows) + (int64_t)is.row * p.stride + lo,
                     bytes, &bar[st]);
        advance(is);
    };
    if (lane == 0) {
        for (int st = 0; st < NST; ++st) mbar_init(&bar[st], 1);
        fence_barrier_init();
        for (int t = 0; t < NST && t < mine; ++t) issue(t);
    }
    __syncwarp();
    int t = 0, st = 0;
    unsigned phase = 0u;
    for (; t < mine; ++t) {
        const bool ok = mbar_wait_bounded(&bar[st], phase);
        if (!__all_sync(kFull, ok)) break;
        tl_item_regs<T, K>(p, rd.row, rd.sl, lane, cand_all[w], &ccnt_all[w],
                           reinterpret_cast<const uint4 *>(ring + (size_t)st * SB));
        __syncwarp();  // every lane has read the stage
        if (lane == 0 && t + NST < mine) issue(st);
        advance(rd);
        if (++st == NST) {
            st = 0;
            phase ^= 1u;
        }
    }
    if (t < mine) {
        // a copy did not land in time: flag it, then wait (bounded) for the
        // copies this warp still has in flight before the block may exit
        if (lane == 0) {
            atomicOr(p.status, SPEC_FLAG_TIMEOUT);
            for (int u = t; u < mine && u < t + NST; ++u) {
                mbar_drain(&bar[st], phase);
                if (++st == NST) {
                    st = 0;
                    phase ^= 1u;
                }
            }
        }
        __syncwarp();
    }
    pdl_launch_dependents();  // the merge blocks may start; they wait for this grid to end
}

// One block per request: its warps merge the request's rows (a warp per
// row), then warp 0 writes the nodes and chooses the next parents.  A
// programmatic dependent of the pass: it waits for the whole pass (and its
// memory) before reading the summaries.
template <int K>
__global__ void __launch_bounds__(kTlWarps * 32) tree_merge_kernel(const TreeLevelParams p) {
    __shared__ unsigned long long sk[kTreeMaxLevelNodes];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int b = blockIdx.x;
    pdl_wait_primary();
    if (*(volatile unsigned *)p.status & SPEC_FLAG_TIMEOUT) {  // the pass gave up: no summaries
        if (w == 0) {
            for (int i = lane; i < p.n_next; i += 32) p.next_parents[(int64_t)b * p.n_next + i] = -1;
            if (lane == 0 && p.flags) p.flags[b] |= SPEC_FLAG_TIMEOUT;
        }
        return;
    }
    for (int j = w; j < p.H; j += kTlWarps) tl_row<K>(p, b * p.H + j, lane);
    __threadfence();
    __syncthreads();
    if (w == 0) tl_request(p, b, lane, sk);
}

template <typename T, int K, bool REGS> cudaError_t launch_r(const TreeLevelParams &p, int sms, cudaStream_t s) {
    const int smem = REGS ? tl_ring_bytes<T>() : 0;
    static std::atomic<unsigned long long> attr_done{0};
    if (REGS) {
        const cudaError_t e = ensure_smem_attr(tree_level_kernel<T, K, REGS>, smem, attr_done);
        if (e != cudaSuccess) return e;
    }
    // grid-stride items: every block must be resident at once, so the grid is
    // the SM count times the blocks an SM holds (queried once per kernel)
    static int per_sm = 0;
    if (per_sm == 0) {
        int n = 0;
        const cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, tree_level_kernel<T, K, REGS>, kTlWarps * 32, smem);
        if (e != cudaSuccess) return e;
        per_sm = n > 0 ? n : 1;
    }
    const int64_t items = (int64_t)p.B * p.H * p.slices;
    const int64_t want = (items + kTlWarps - 1) / kTlWarps;
    const int64_t cap = (int64_t)sms * per_sm;
    const int grid = (int)(want < cap ? want : cap);
    tree_level_kernel<T, K, REGS><<<grid, kTlWarps * 32, smem, s>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.B);
    cfg.blockDim = dim3(kTlWarps * 32);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tree_merge_kernel<K>, p);
}

template <typename T, int K> cudaError_t launch_t(const TreeLevelParams &p, int sms, cudaStream_t s) {
    // the register path needs every row on a 16-byte boundary
    const bool regs = reinterpret_cast<uintptr_t>(p.rows) % 16 == 0 && (p.stride * (int64_t)sizeof(T)) % 16 == 0;
    return regs ? launch_r<T, K, true>(p, sms, s) : launch_r<T, K, false>(p, sms, s);
}

}  // namespace

cudaError_t launch_tree_level(const TreeLevelParams &p, int dtype, int kmax, int sms, cudaStream_t s) {
    const bool bf = dtype == SPEC_DTYPE_BF16;
    if (kmax <= 4) return bf ? launch_t<__nv_bfloat16, 4>(p, sms, s) : launch_t<float, 4>(p, sms, s);
    if (kmax <= 8) return bf ? launch_t<__nv_bfloat16, 8>(p, sms, s) : launch_t<float, 8>(p, sms, s);
    return bf ? launch_t<__nv_bfloat16, 16>(p, sms, s) : launch_t<float, 16>(p, sms, s);
}

}  // namespace specv
