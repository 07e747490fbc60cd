// Sampled chain verification with top-k (k <= 128) on sm_103a, in two
// kernels and without thread-block clusters.
//
// The transform ("KV Cache 优化（四）：Speculative Decoding 投机解码" §4) keeps
// every logit >= the row's k-th largest; everything after that works on the
// few kept tokens.  So the work splits into items (position, vocab slice),
// position-major, and each item only hands on a short candidate list.
//
// chain_topk_kernel (the HBM pass):
//  1. The grid is a few blocks per SM, a multiple of the slice count; each
//     block takes one slice index of positions round-robin.  Thread 0 keeps
//     kTkNST items in flight through a ring of shared-memory stages: one
//     cp.async.bulk per row (target row k and draft row k of the slice),
//     completing on the stage's mbarrier; a stage is refilled as soon as its
//     item is in registers.
//  2. Every thread takes the largest logit of each 16-byte vector it holds
//     (packed bf16x2 maxima).  A value reached by at least K vectors' maxima
//     is a lower bound of the slice's K-th largest (each such vector holds a
//     logit >= it).  The block reuses the bound of its previous item (the
//     same slice of another position, with similar logits) when the vectors
//     reaching it prove it valid for this one, and otherwise searches a new
//     one: the K-th largest of the threads' maxima (warp r, row r, a bitwise
//     search with warp reductions).
//  3. Each warp lists the 16-byte vectors (and head/tail scalars) whose
//     maximum reaches the bound, ranked by ballots.  The entries, (order key
//     of the vector's maximum, element index of its first logit; scalars
//     flagged), go out to the item's own region of the workspace with the
//     count and the bound.  No element of a vector is looked at here, no
//     global atomics, no fences, two block barriers per item (four when the
//     bound is searched again).
//
// chain_topk_merge_kernel, a programmatic dependent launch of the pass (its
// prologue overlaps the pass's tail): one block per position gathers the
// listed entries >= T*, the largest slice bound, into shared memory; per row,
// the K-th largest listed key B is a lower bound of the row's K-th largest
// logit, so only the listed vectors whose maximum reaches B are loaded again
// (a few hundred bytes, from L2 or HBM), split into their logits >= B, and
// the exact K-th largest among those is the threshold.  The kept set in
// token order, the double-float acceptance, residual and draw follow.  A
// slice that overflowed its region, rows whose 16-byte phases differ, or a
// kept set too large for the merge (hundreds of tied logits) send the
// position to the exact masked computation over the whole row in that block
// instead (slow, exact, rare).
#include "sample_common.cuh"

namespace specv {

constexpr int kTkNST = 2;             // ring stages (items in flight per block)
constexpr int kTkRowBytes = 16384;    // one row's slice body per stage
constexpr int kTkBlocksPerSM = 3;
// a region entry for a scalar head or tail logit rather than a 16-byte vector
constexpr uint32_t kScalarEntry = 0x80000000u;

constexpr int kTkVecPerThr = kTkRowBytes / 16 / kNT;  // 16-byte vectors per thread and row
static_assert(kTkVecPerThr * 16 * kNT == kTkRowBytes, "a stage row is whole vectors per thread");

struct TkRing {
    alignas(128) unsigned char buf[kTkNST][2][kTkRowBytes];
};

int topk_row_bytes() { return kTkRowBytes; }

template <typename T> struct TkItem {
    int k, b, j, pos, rows;
    const T *trow, *drow;
    SliceSplit sp;
    bool ok;  // both rows share the 16-byte phase and the body fits one stage
};

template <typename T>
__device__ __forceinline__ TkItem<T> tk_item(const SampleParams &p, int k, int b, int j) {
    TkItem<T> it;
    it.j = j;
    it.k = k;
    it.b = b;
    const int g = p.gamma;
    it.pos = b * (g + 1) + k;  // target row and record index
    const bool has_draft = k < g;
    it.rows = has_draft ? 2 : 1;
    it.trow = reinterpret_cast<const T *>(p.target) + (int64_t)it.pos * p.tstride;
    it.drow = has_draft ? reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + k) * p.dstride : nullptr;
    const int lo = min(p.V, j * p.Vs), hi = min(p.V, lo + p.Vs);
    it.sp = split_slice(it.trow, lo, hi);
    const bool same = !has_draft ||
        ((reinterpret_cast<uintptr_t>(it.trow + lo) ^ reinterpret_cast<uintptr_t>(it.drow + lo)) & 15u) == 0;
    it.ok = same && (int64_t)(it.sp.tail0 - it.sp.body0) * (int64_t)sizeof(T) <= kTkRowBytes;
    return it;
}

// Positions of one block, position-major (qpos = k*B + b), stepping by qstep.
struct TkCursor {
    int qpos, k, b;
    __device__ void init(int q, int B) {
        qpos = q;
        k = (int)((unsigned)q / (unsigned)B);
        b = q - k * B;
    }
    __device__ void step(int qstep, int sk, int sb, int B) {
        qpos += qstep;
        k += sk;
        b += sb;
        if (b >= B) {
            b -= B;
            ++k;
        }
    }
};

// region of (position, row, slice): count index and first entry
__device__ __forceinline__ int64_t tk_region(const SampleParams &p, int pos, int r, int j) {
    return ((int64_t)pos * 2 + r) * p.c + j;
}

// thread 0: arm stage s for `item` and start its bulk copies
template <typename T>
__device__ __forceinline__ void tk_issue(const SampleParams &p, TkRing &R, unsigned long long *full,
                                         const TkCursor &cur, int j, int s) {
    const TkItem<T> it = tk_item<T>(p, cur.k, cur.b, j);
    const uint32_t nb = it.ok ? (uint32_t)((it.sp.tail0 - it.sp.body0) * (int)sizeof(T)) : 0u;
    mbar_arrive_expect_tx(&full[s], nb * (uint32_t)it.rows);
    if (nb) {
        // the logits are read once: evict them first, keeping the candidate
        // regions in L2 for the merge
        const uint64_t pol = l2_evict_first();
        bulk_g2s_policy(R.buf[s][0], it.trow + it.sp.body0, nb, &full[s], pol);
        if (it.rows == 2) bulk_g2s_policy(R.buf[s][1], it.drow + it.sp.body0, nb, &full[s], pol);
    }
}
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

// number of elements of the vector that are >= t (t a value of type T)
template <typename T> __device__ __forceinline__ unsigned vec_ge_count(const uint4 &v, float t);
template <> __device__ __forceinline__ unsigned vec_ge_count<float>(const uint4 &v, float t) {
    return (unsigned)(__uint_as_float(v.x) >= t) + (unsigned)(__uint_as_float(v.y) >= t) +
           (unsigned)(__uint_as_float(v.z) >= t) + (unsigned)(__uint_as_float(v.w) >= t);
}
template <> __device__ __forceinline__ unsigned vec_ge_count<__nv_bfloat16>(const uint4 &v, float t) {
    // 16 mask bits per true half: the caller divides the sum by 16
    const __nv_bfloat162 t2 = __float2bfloat162_rn(t);
    return __popc(__hge2_mask(as_bf2(v.x), t2)) + __popc(__hge2_mask(as_bf2(v.y), t2)) +
           __popc(__hge2_mask(as_bf2(v.z), t2)) + __popc(__hge2_mask(as_bf2(v.w), t2));
}
template <typename T> constexpr unsigned kCountScale = 1u;
template <> constexpr unsigned kCountScale<__nv_bfloat16> = 16u;

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

// bit e set iff element e of a 32-bit word (2 bf16 or 1 f32) is >= t
template <typename T> __device__ __forceinline__ uint32_t word_ge_mask(uint32_t w, float t);
template <> __device__ __forceinline__ uint32_t word_ge_mask<float>(uint32_t w, float t) {
    return __uint_as_float(w) >= t ? 1u : 0u;
}
template <> __device__ __forceinline__ uint32_t word_ge_mask<__nv_bfloat16>(uint32_t w, float t) {
    const uint32_t m = __hge2_mask(as_bf2(w), __float2bfloat162_rn(t));  // exact: t is a bf16 value or -inf
    return (m & 1u) | ((m >> 15) & 2u);
}
// element e of a 32-bit word
template <typename T> __device__ __forceinline__ float word_elem(uint32_t w, int e);
template <> __device__ __forceinline__ float word_elem<float>(uint32_t w, int) { return __uint_as_float(w); }
template <> __device__ __forceinline__ float word_elem<__nv_bfloat16>(uint32_t w, int e) {
    return __uint_as_float(e ? (w & 0xffff0000u) : (w << 16));
}

// The K-th largest of kNT keys (one per thread of the block, in smem) by
// one warp: the largest r with at least K keys >= r, fixed two bits per step
// (three independent counts) and only over the bits in which the smallest
// and largest key differ.  Every lane gets it.
__device__ __forceinline__ uint32_t warp_kth_of_block(const uint32_t *keys, unsigned K) {
    constexpr int PER = kNT / 32;
    const int lane = threadIdx.x & 31;
    uint32_t v[PER];
    uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        v[e] = keys[lane + 32 * e];
        lo = min(lo, v[e]);
        hi = max(hi, v[e]);
    }
    lo = __reduce_min_sync(kFull, lo);
    hi = __reduce_max_sync(kFull, hi);
    if (lo == hi) return lo;
    int nb = 32 - __clz(lo ^ hi);                    // bits below the common prefix
    uint32_t res = nb == 32 ? 0u : (hi >> nb) << nb;  // the prefix: the answer is in [lo, hi]
    auto count_ge = [&](uint32_t cand) {
        unsigned c = 0;
#pragma unroll
        for (int e = 0; e < PER; ++e) c += v[e] >= cand;
        return __reduce_add_sync(kFull, c);
    };
#pragma unroll 1
    while (nb >= 2) {
        nb -= 2;
        const unsigned c1 = count_ge(res | (1u << nb));
        const unsigned c2 = count_ge(res | (2u << nb));
        const unsigned c3 = count_ge(res | (3u << nb));
        res |= (c3 >= K ? 3u : c2 >= K ? 2u : c1 >= K ? 1u : 0u) << nb;
    }
    if (nb == 1 && count_ge(res | 1u) >= K) res |= 1u;
    return res;
}

template <typename T>
__global__ void __launch_bounds__(kNT, kTkBlocksPerSM) chain_topk_kernel(SampleParams p) {
    constexpr int VEC = Elem<T>::VEC;
    constexpr int SLOTS = kTkVecPerThr + 2;  // a thread's vectors, then its head and tail scalar
    __shared__ __align__(8) unsigned long long full[kTkNST];
    __shared__ uint32_t s_max[2][kNT];
    __shared__ uint32_t s_t0[2];
    __shared__ unsigned s_hcnt[2][2][kNW];  // [item parity][row][warp]
    extern __shared__ __align__(128) unsigned char dsm[];
    TkRing &R = *reinterpret_cast<TkRing *>(dsm);
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const unsigned lt = lanemask_lt();
    pdl_launch_dependents();  // the merge may launch and run its prologue

    // gridDim.x is a multiple of c: every item of this block is slice j
    const int c = p.c, B = p.B;
    const int j = (int)(blockIdx.x % (unsigned)c);
    const int qstep = (int)(gridDim.x / (unsigned)c);
    const int sk = qstep / B, sb = qstep - sk * B;
    const int npos = B * (p.gamma + 1);
    const unsigned K = (unsigned)p.top_k;
    unsigned phase = 0u;  // bit s: parity of stage s's next completion
    bool timeout = false;
    uint32_t guess[2] = {0xffffffffu, 0xffffffffu};  // reused bound per row (key); none yet

    TkCursor cur, nxt;
    cur.init((int)(blockIdx.x / (unsigned)c), B);
    nxt = cur;  // thread 0: the next item to load
    if (tid == 0) {
        for (int s = 0; s < kTkNST; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
        for (int s = 0; s < kTkNST; ++s) {
            if (nxt.qpos < npos) tk_issue<T>(p, R, full, nxt, j, s);
            nxt.step(qstep, sk, sb, B);
        }
    }
    __syncthreads();

    for (int t = 0; cur.qpos < npos; cur.step(qstep, sk, sb, B), ++t) {
        const int s = t % kTkNST, par = t & 1;
        const TkItem<T> it = tk_item<T>(p, cur.k, cur.b, j);
        const SliceSplit sp = it.sp;
        const int nhead = sp.body0 - sp.head0, ntail = sp.hi - sp.tail0;
        const bool keep_all = sp.hi - sp.head0 <= (int)K;
        // head and tail scalars (none for 16-byte-aligned slices) from global memory
        float xh[2] = {-INFINITY, -INFINITY}, xt[2] = {-INFINITY, -INFINITY};
        if (it.ok) {
            for (int r = 0; r < it.rows; ++r) {
                const T *row = r == 0 ? it.trow : it.drow;
                if (tid < nhead) xh[r] = ld_elem(row, sp.head0 + tid);
                if (tid < ntail) xt[r] = ld_elem(row, sp.tail0 + tid);
            }
        }
        if (!mbar_wait_bounded(&full[s], (phase >> s) & 1u)) timeout = true;
        phase ^= 1u << s;
        const int nvec = it.ok ? (sp.tail0 - sp.body0) / VEC : 0;

        // 1. largest logit per 16-byte vector and per thread
        float vm[2][kTkVecPerThr], mt[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint4 *src = reinterpret_cast<const uint4 *>(R.buf[s][r]);
            float m = fmaxf(xh[r], xt[r]);
#pragma unroll
            for (int i = 0; i < kTkVecPerThr; ++i) {
                const int q = tid + i * kNT;
                vm[r][i] = (r < it.rows && q < nvec) ? vec_max<T>(src[q]) : -INFINITY;
                m = fmaxf(m, vm[r][i]);
            }
            mt[r] = m;
        }
        // 2. the vectors (and scalars) that reach the row's bound: a bit per
        //    slot and the slot's rank among the warp's hits
        float tf[2];
        uint32_t hits[2] = {0u, 0u}, ranks[2][2] = {{0u, 0u}, {0u, 0u}};  // 8-bit ranks, 4 slots per word
        auto list_hits = [&](int r) {
            unsigned n = 0;
            uint32_t h = 0u, rk0 = 0u, rk1 = 0u;
#pragma unroll
            for (int i = 0; i < SLOTS; ++i) {
                bool hit;
                if (i < kTkVecPerThr) hit = tid + i * kNT < nvec && vm[r][i] >= tf[r];
                else if (i == kTkVecPerThr) hit = tid < nhead && xh[r] >= tf[r];
                else hit = tid < ntail && xt[r] >= tf[r];
                const unsigned bal = __ballot_sync(kFull, hit);
                const uint32_t rk = n + __popc(bal & lt);
                if (i < 4) rk0 |= rk << (8 * i); else rk1 |= rk << (8 * (i - 4));
                h |= (hit ? 1u : 0u) << i;
                n += __popc(bal);
            }
            hits[r] = h;
            ranks[r][0] = rk0;
            ranks[r][1] = rk1;
            if (lane == 0) s_hcnt[par][r][wid] = n;
        };
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            tf[r] = keep_all ? -INFINITY : (guess[r] == 0xffffffffu ? INFINITY : key_value<T>(guess[r]));
            if (r < it.rows && it.ok) list_hits(r);
        }
        __syncthreads();  // hit counts; stage s is consumed (the maxima are in registers)
        if (tid == 0) {
            if (nxt.qpos < npos) tk_issue<T>(p, R, full, nxt, j, s);  // refill stage s
            nxt.step(qstep, sk, sb, B);
        }

        // 3. the reused bound holds for this slice if at least K listed slots
        //    reach it (each holds a logit >= it); otherwise (or if it lets in
        //    too many) search the K-th largest thread maximum again
        bool redo[2] = {false, false};
        if (it.ok && !keep_all) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r >= it.rows) break;
                unsigned tot = 0;
#pragma unroll
                for (int w = 0; w < kNW; ++w) tot += s_hcnt[par][r][w];
                redo[r] = tot < K || tot > (unsigned)(kTopKSlicePool / 2);
            }
        }
        if (redo[0] || redo[1]) {  // block-uniform
            for (int r = 0; r < it.rows; ++r) s_max[r][tid] = kkey<T>(mt[r]);
            __syncthreads();
            if (wid < it.rows && (wid == 0 ? redo[0] : redo[1])) {
                const uint32_t t0 = warp_kth_of_block(s_max[wid], min(K, (unsigned)kNT));
                if (lane == 0) s_t0[wid] = t0;
            }
            __syncthreads();
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r >= it.rows || !redo[r]) continue;
                guess[r] = s_t0[r];
                tf[r] = key_value<T>(guess[r]);
                list_hits(r);
            }
            __syncthreads();
        }

        // 4. the listed slots go out to the item's regions as (order key of the
        //    vector maximum or scalar, element index; scalars flagged); thread 0
        //    stores the count and the bound
        if (it.ok) {
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                if (r >= it.rows) break;
                unsigned base = 0u, total = 0u;
#pragma unroll
                for (int w = 0; w < kNW; ++w) {
                    const unsigned cw = s_hcnt[par][r][w];
                    base += w < wid ? cw : 0u;
                    total += cw;
                }
                const int64_t reg = tk_region(p, it.pos, r, j);
                // total > kTopKSlicePool: overflow, the merge takes the exact path
                if (tid == 0) p.slicecb[reg] = make_uint2(total, keep_all ? 0u : kkey<T>(tf[r]));
                uint2 *dst = p.pool + reg * kTopKSlicePool;
                const uint32_t h = hits[r];
#pragma unroll
                for (int i = 0; i < SLOTS; ++i) {
                    if (!(h & (1u << i))) continue;
                    const uint32_t at = base + ((ranks[r][i >> 2] >> (8 * (i & 3))) & 0xffu);
                    if (at >= (uint32_t)kTopKSlicePool) continue;
                    uint2 e;
                    if (i < kTkVecPerThr) e = make_uint2(kkey<T>(vm[r][i]), (uint32_t)(sp.body0 + (tid + i * kNT) * VEC));
                    else if (i == kTkVecPerThr) e = make_uint2(kkey<T>(xh[r]), (uint32_t)(sp.head0 + tid) | kScalarEntry);
                    else e = make_uint2(kkey<T>(xt[r]), (uint32_t)(sp.tail0 + tid) | kScalarEntry);
                    dst[at] = e;
                }
            }
        } else if (tid < it.rows) {
            // poison: the merge takes the exact path
            p.slicecb[tk_region(p, it.pos, tid, j)] = make_uint2((unsigned)(kTopKSlicePool + 1), 0u);
        }
    }
    if (timeout) atomicOr(p.status, SPEC_FLAG_TIMEOUT);
    __syncthreads();
    if (tid == 0)
        for (int s = 0; s < kTkNST; ++s) mbar_inval(&full[s]);
}

// ---------------------------------------------------------------------------
// The merge: one block per position, position-major.
//
//  1. Warp r scans row r's slice records: offsets of the regions, and T*, the
//     largest of the slices' bounds.  Slice j holds at least K logits >= its
//     bound, so T* is a lower bound of the row's K-th largest: entries below
//     it cannot be kept.
//  2. The block gathers the entries >= T* of both rows into shared memory
//     (all loads in flight at once).
//  3. Warp r finds row r's exact K-th largest key (bitwise search), keeps the
//     entries >= it, sorts them by token id and sums the kept set's
//     exponentials in double-float.
//  4. Warp 0 computes acceptance, the residual mass (q looked up in the
//     draft's sorted kept set) and, where this position decides the token,
//     the draw by a warp scan in token order; lane 0 finishes the position.
// ---------------------------------------------------------------------------
constexpr int kMergeMaxC = 256;  // slices per row the merge can take

// the K-th largest key of n entries (smem), by one warp; every lane gets it.
// Up to 256 keys are held in registers (8 per lane); counts are ballots.
__device__ __forceinline__ uint32_t warp_kth_entries(const uint2 *L, int n, unsigned K) {
    constexpr int PER = 8;
    const int lane = threadIdx.x & 31;
    if (n <= 32 * PER) {
        uint32_t v[PER];
        uint32_t lo = 0xffffffffu, hi = 0u;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            const int x = lane + 32 * e;
            v[e] = x < n ? L[x].x : 0u;
            if (x < n) {
                lo = min(lo, v[e]);
                hi = max(hi, v[e]);
            }
        }
        lo = __reduce_min_sync(kFull, lo);
        hi = __reduce_max_sync(kFull, hi);
        if (lo >= hi) return lo;
        const int rows = (n + 31) / 32;  // warp-uniform
        auto count_ge = [&](uint32_t cand) {
            unsigned c = 0;
#pragma unroll
            for (int e = 0; e < PER; ++e)
                if (e < rows) c += __popc(__ballot_sync(kFull, lane + 32 * e < n && v[e] >= cand));
            return c;
        };
        int nb = 32 - __clz(lo ^ hi);
        uint32_t res = nb == 32 ? 0u : (hi >> nb) << nb;
#pragma unroll 1
        while (nb >= 2) {
            nb -= 2;
            const unsigned c1 = count_ge(res | (1u << nb));
            const unsigned c2 = count_ge(res | (2u << nb));
            const unsigned c3 = count_ge(res | (3u << nb));
            res |= (c3 >= K ? 3u : c2 >= K ? 2u : c1 >= K ? 1u : 0u) << nb;
        }
        if (nb == 1 && count_ge(res | 1u) >= K) res |= 1u;
        return res;
    }
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int x = lane; x < n; x += 32) {
        lo = min(lo, L[x].x);
        hi = max(hi, L[x].x);
    }
    lo = __reduce_min_sync(kFull, lo);
    hi = __reduce_max_sync(kFull, hi);
    if (lo >= hi) return lo;
    int nb = 32 - __clz(lo ^ hi);
    uint32_t res = nb == 32 ? 0u : (hi >> nb) << nb;
    auto count_ge = [&](uint32_t cand) {
        unsigned c = 0;
        for (int x0 = 0; x0 < n; x0 += 32) c += __popc(__ballot_sync(kFull, x0 + lane < n && L[x0 + lane].x >= cand));
        return c;
    };
#pragma unroll 1
    while (nb >= 2) {
        nb -= 2;
        const unsigned c1 = count_ge(res | (1u << nb));
        const unsigned c2 = count_ge(res | (2u << nb));
        const unsigned c3 = count_ge(res | (3u << nb));
        res |= (c3 >= K ? 3u : c2 >= K ? 2u : c1 >= K ? 1u : 0u) << nb;
    }
    if (nb == 1 && count_ge(res | 1u) >= K) res |= 1u;
    return res;
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

template <typename T>
__global__ void __launch_bounds__(kNT, 3) chain_topk_merge_kernel(SampleParams p) {
    __shared__ SampBase sb;
    __shared__ uint2 s_kept[2][kKeptMax];
    __shared__ unsigned s_off[2][kMergeMaxC + 1];
    __shared__ uint32_t s_tstar[2], s_th[2];
    __shared__ int s_n[2], s_kn[2], s_bad;
    __shared__ float s_m[2];
    __shared__ float2 s_S[2];
    extern __shared__ __align__(128) unsigned char dsm[];
    uint2 *lists = reinterpret_cast<uint2 *>(dsm);  // [2][kTopKMerge]: gathered, then unsorted kept
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const DdExpTables &EK = sb.K;
    const unsigned lt = lanemask_lt();
    load_exp_tables(p, sb);
    const int k = blockIdx.x / p.B, b = blockIdx.x % p.B;
    const int g = p.gamma, c = p.c;
    const int pos = b * (g + 1) + k;
    const bool has_draft = k < g;
    const int rows = has_draft ? 2 : 1;
    const unsigned K = (unsigned)p.top_k;
    const T *trow = reinterpret_cast<const T *>(p.target) + (int64_t)pos * p.tstride;
    const T *drow = has_draft ? reinterpret_cast<const T *>(p.draft) + (int64_t)(b * g + k) * p.dstride : nullptr;
    if (tid == 0) s_bad = c > kMergeMaxC;
    __syncthreads();
    pdl_wait_primary();  // the HBM pass's regions and records are complete

    // 1. offsets and T* (warp r, row r)
    if (wid < rows && !s_bad) {
        unsigned carry = 0u, tstar = 0u;
        bool bad = false;
        for (int j0 = 0; j0 < c; j0 += 32) {
            const int j = j0 + lane;
            const uint2 cb = j < c ? __ldcg(&p.slicecb[tk_region(p, pos, wid, j)]) : make_uint2(0u, 0u);
            bad |= cb.x > (unsigned)kTopKSlicePool;
            tstar = max(tstar, cb.y);
            unsigned incl = cb.x;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            if (j < c) s_off[wid][j] = carry + incl - cb.x;
            carry += __shfl_sync(kFull, incl, 31);
        }
        bad = __any_sync(kFull, bad) || carry > (unsigned)kTopKMerge;
        tstar = __reduce_max_sync(kFull, tstar);
        if (lane == 0) {
            s_off[wid][c] = carry;
            s_tstar[wid] = tstar;
            s_n[wid] = 0;
            if (bad) s_bad = 1;
        }
    }
    __syncthreads();
    if (!s_bad) {
        // 2. gather the entries >= T* of both rows (flat index over the rows'
        //    regions, every load of a thread in flight at once)
        const unsigned n0 = s_off[0][c], ntot = n0 + (rows == 2 ? s_off[1][c] : 0u);
        constexpr int BATCH = 16;
        for (unsigned f0 = 0; f0 < ntot; f0 += kNT * BATCH) {
            uint2 e[BATCH];
#pragma unroll
            for (int q = 0; q < BATCH; ++q) {
                const unsigned f = f0 + q * kNT + tid;
                e[q] = make_uint2(0u, 0u);
                if (f < ntot) {
                    const int r = f >= n0;
                    const unsigned fr = f - (r ? n0 : 0u);
                    int lo = 0, hi = c - 1;  // the last slice whose offset is <= fr
                    while (lo < hi) {
                        const int mid = (lo + hi + 1) >> 1;
                        if (s_off[r][mid] <= fr) lo = mid; else hi = mid - 1;
                    }
                    e[q] = __ldcg(&p.pool[tk_region(p, pos, r, lo) * kTopKSlicePool + (fr - s_off[r][lo])]);
                }
            }
            // keep masks per row, then one shared-memory atomic per warp and row
            uint32_t km[2] = {0u, 0u};
#pragma unroll
            for (int q = 0; q < BATCH; ++q) {
                const unsigned f = f0 + q * kNT + tid;
                const int r = f >= n0;
                if (f < ntot && e[q].x >= s_tstar[r]) km[r] |= 1u << q;
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
                const unsigned cnt = __popc(km[rr]);
                unsigned incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                const unsigned wtot = __shfl_sync(kFull, incl, 31);
                if (wtot == 0u) continue;
                unsigned base = 0u;
                if (lane == 31) base = (unsigned)atomicAdd(&s_n[rr], (int)wtot);
                base = __shfl_sync(kFull, base, 31) + incl - cnt;
#pragma unroll
                for (int q = 0; q < BATCH; ++q)
                    if (km[rr] & (1u << q)) lists[rr * kTopKMerge + base++] = e[q];
            }
        }
        __syncthreads();

        // 3. warp r: B, the K-th largest listed key (at least K logits of the
        //    row reach it: every listed vector holds its maximum), the listed
        //    vectors reaching B fetched from the row and split into their
        //    logits >= B, the exact threshold among those, the kept set in
        //    token order, row statistics
        if (wid < rows) {
            const int r = wid;
            const T *row = r == 0 ? trow : drow;
            uint2 *L = lists + r * kTopKMerge;
            const int n = s_n[r];
            const uint32_t bk = warp_kth_entries(L, n, min(K, (unsigned)n));
            // candidates (order key, token id) after the gathered entries
            uint2 *cand = L + n;
            const int cap = kTopKMerge - n;
            int nc = 0;
            for (int x0 = 0; x0 < n; x0 += 32) {
                const int x = x0 + lane;
                uint32_t mk = 0u;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                uint2 e = make_uint2(0u, 0u);
                if (x < n && L[x].x >= bk) {
                    e = L[x];
                    if (e.y & kScalarEntry) {
                        mk = 1u;
                    } else {
                        v = ld_nc16(reinterpret_cast<const uint4 *>(row + e.y));
                        mk = vec_ge_mask<T>(v, key_value<T>(bk));
                    }
                }
                const unsigned cnt = __popc(mk);
                unsigned incl = cnt;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned y = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += y;
                }
                int at = nc + (int)(incl - cnt);
                while (mk) {
                    const int q = __ffs(mk) - 1;
                    mk &= mk - 1u;
                    if (at < cap) {
                        cand[at] = (e.y & kScalarEntry) ? make_uint2(e.x, e.y & ~kScalarEntry)
                                                        : make_uint2(kkey<T>(vec_elem<T>(v, q)), e.y + (uint32_t)q);
                    }
                    ++at;
                }
                nc += (int)__shfl_sync(kFull, incl, 31);
            }
            __syncwarp();
            const int ncu = min(nc, cap);
            // the kept logits: the candidates among the row's K largest
            int kn = 0;
            uint2 *tmp = cand + ncu;
            const int cap2 = cap - ncu;
            uint32_t th = warp_kth_entries(cand, ncu, min(K, (unsigned)ncu));
            for (int x0 = 0; x0 < ncu; x0 += 32) {
                const int x = x0 + lane;
                const bool keep = x < ncu && cand[x].x >= th;
                const unsigned bal = __ballot_sync(kFull, keep);
                const int at = kn + __popc(bal & lt);
                if (keep && at < kKeptMax && at < cap2) tmp[at] = cand[x];
                kn += __popc(bal);
            }
            const bool fits = nc <= cap && kn <= kKeptMax && kn <= cap2;
            if (fits) {
                __syncwarp();
                for (int x = lane; x < kn; x += 32) {
                    const uint2 e = tmp[x];
                    int rank = 0;
                    for (int y = 0; y < kn; ++y) rank += tmp[y].y < e.y;
                    s_kept[r][rank] = e;
                }
                __syncwarp();
                uint32_t mk = 0u;
                for (int x = lane; x < kn; x += 32) mk = max(mk, s_kept[r][x].x);
                mk = __reduce_max_sync(kFull, mk);
                const float m = kn > 0 ? key_value<T>(mk) : -INFINITY;
                dd S{0.0f, 0.0f};
                if (m != -INFINITY) {
#pragma unroll 1
                    for (int x = lane; x < kn; x += 32)
                        S = dd_add(S, dd_expw(key_value<T>(s_kept[r][x].x), m, EK));
                }
                S = warp_dd_sum(S);
                if (p.top_p > 0.0f && p.top_p < 1.0f && m != -INFINITY) {
                    // the nucleus of the kept set: its entries by probability
                    // (larger key first, then the lower token), the first rank
                    // whose cumulative probability reaches top_p, and every
                    // entry at or above that rank's key (ties kept), still in
                    // token order; the row's sum is taken again over them
                    uint2 *srt = L;                                          // [kn] by rank
                    float2 *prb = reinterpret_cast<float2 *>(L + kKeptMax);  // [kn] by rank
                    const dd iS = dd_recip(S);
                    for (int x = lane; x < kn; x += 32) {
                        const uint2 e = s_kept[r][x];
                        int rank = 0;
                        for (int y = 0; y < kn; ++y) {
                            const uint2 f = s_kept[r][y];
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
                    const dd tp{p.top_p, 0.0f};
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
                        const uint2 e = x < kn ? s_kept[r][x] : make_uint2(0u, 0u);
                        const bool keep = x < kn && e.x >= kstar;
                        const unsigned bal = __ballot_sync(kFull, keep);
                        __syncwarp();  // every lane has read its entry before any is moved
                        if (keep) s_kept[r][nn + __popc(bal & lt)] = e;
                        nn += __popc(bal);
                    }
                    __syncwarp();
                    kn = nn;
                    th = kstar;
                    S = dd{0.0f, 0.0f};
#pragma unroll 1
                    for (int x = lane; x < kn; x += 32)
                        S = dd_add(S, dd_expw(key_value<T>(s_kept[r][x].x), m, EK));
                    S = warp_dd_sum(S);
                }
                if (lane == 0) {
                    s_m[r] = m;
                    s_S[r] = make_float2(S.hi, S.lo);
                }
            }
            if (lane == 0) {
                s_th[r] = th;
                s_kn[r] = kn;
                if (!fits) s_bad = 1;
            }
        }
        __syncthreads();
    }
    if (s_bad) {
        if (p.top_p > 0.0f && p.top_p < 1.0f) {
            // the masked path has no nucleus: the position is flagged
            if (wid == 0) {
                Outcome o{1.0f, 0.0f, -1, REC_BAD_ROW};
                finish(p, b, k, o, sb);
            }
            return;
        }
        // an overflowed or poisoned slice, or hundreds of logits tied at the
        // threshold: the exact masked path over the whole rows
        SoloEx solo;
        masked_position<T, true>(p, sb, dsm, solo, k, b, 0, p.V);
        return;
    }
    if (wid != 0) return;

    // 4. warp 0: acceptance, residual mass, the draw
    const int d = has_draft ? p.tokens[(int64_t)b * g + k] : 0;
    const bool bad_tok = has_draft && (d < 0 || d >= p.V);
    const float l_d = (has_draft && !bad_tok) ? ld_elem(trow, d) : 0.0f;
    const float g_d = (has_draft && !bad_tok) ? ld_elem(drow, d) : 0.0f;
    const float u_k = has_draft ? p.unif[(int64_t)b * (g + 1) + k] : 0.0f;
    const float u_f = p.unif[(int64_t)b * (g + 1) + g];
    const unsigned rej = *((volatile unsigned *)&p.rejword[b]);
    const uint2 *Kp = s_kept[0], *Kq = s_kept[1];
    const int np = s_kn[0], nq = has_draft ? s_kn[1] : 0;
    const float mp = s_m[0], mq = has_draft ? s_m[1] : 0.0f;
    const dd sp{s_S[0].x, s_S[0].y};
    const dd sq = has_draft ? dd{s_S[1].x, s_S[1].y} : dd{0.0f, 0.0f};
    Outcome o{1.0f, 0.0f, -1, 0u};
    const bool bad_row = mp == -INFINITY || (has_draft && mq == -INFINITY);
    const bool bad = bad_tok || bad_row;
    o.info = (bad_tok ? REC_BAD_INPUT : 0u) | (bad_row ? REC_BAD_ROW : 0u);
    if (!bad) {
        const dd isp = dd_recip(sp);
        const dd isq = has_draft ? dd_recip(sq) : dd{0.0f, 0.0f};
        bool accept = false;
        if (has_draft) {
            const dd pd = kkey<T>(l_d) >= s_th[0] ? dd_mul(dd_expw(l_d, mp, EK), isp) : dd{0.0f, 0.0f};
            const dd qd = kkey<T>(g_d) >= s_th[1] ? dd_mul(dd_expw(g_d, mq, EK), isq) : dd{0.0f, 0.0f};
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
        // q of a token: its draft probability if it is in the draft's kept set
        auto qprob = [&](uint32_t id) -> dd {
            int lo = 0, hi = nq;  // first kept entry with id >= `id`
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (Kq[mid].y < id) lo = mid + 1; else hi = mid;
            }
            return (lo < nq && Kq[lo].y == id) ? dd_mul(dd_expw(key_value<T>(Kq[lo].x), mq, EK), isq)
                                               : dd{0.0f, 0.0f};
        };
        // lane l holds kept entries [l*E, l*E + E) in token order; their p
        // (normalised, or the unnormalised target terms for the bonus draw)
        // and residual weights go to shared memory
        const int E = (np + 31) / 32;
        const int i0 = lane * E, i1 = min(np, i0 + E);
        // per kept target entry: p (or the bonus term) and the residual weight,
        // in the gathered lists' memory (dead by now)
        float2 (*s_wp)[kKeptMax] = reinterpret_cast<float2 (*)[kKeptMax]>(dsm);
        dd zw{0.0f, 0.0f}, zp{0.0f, 0.0f};
#pragma unroll 1
        for (int i = i0; i < i1; ++i) {
            const dd ex = dd_expw(key_value<T>(Kp[i].x), mp, EK);
            dd pi = ex, w = ex;
            if (has_draft) {
                pi = dd_mul(ex, isp);
                w = dd_max0(dd_add(pi, dd_neg(qprob(Kp[i].y))));
                zw = dd_add(zw, w);
                zp = dd_add(zp, pi);
            }
            s_wp[0][i] = make_float2(pi.hi, pi.lo);
            s_wp[1][i] = make_float2(w.hi, w.lo);
        }
        if (has_draft) {
            zw = warp_dd_sum(zw);
            zp = warp_dd_sum(zp);
            o.z = dd_to_f(zw);
        }
        const bool earlier = rej > (unsigned)(g - k + 1);
        if (has_draft && !accept && lane == 0) atomicMax(p.rejword + b, (unsigned)(g - k + 1));
        if ((!has_draft || !accept) && !earlier) {
            // ---- the draw, in token order over the kept set ----
            const bool fb = has_draft && dd_le(zw, dd{p.eps, 0.0f});
            if (fb) o.info |= REC_FALLBACK;
            const float2 *W = (!has_draft || fb) ? s_wp[0] : s_wp[1];
            const dd total = !has_draft ? sp : (fb ? zp : zw);
            const dd t = dd_mul_f(total, u_f);
            dd mine{0.0f, 0.0f};
            int lastpos = -1;
#pragma unroll 1
            for (int i = i0; i < i1; ++i) {
                const dd w{W[i].x, W[i].y};
                mine = dd_add(mine, w);
                if (dd_pos(w)) lastpos = i;
            }
            dd cum = warp_dd_excl_scan(mine);
            int hit = INT_MAX;
#pragma unroll 1
            for (int i = i0; i < i1; ++i) {
                const dd w{W[i].x, W[i].y};
                cum = dd_add(cum, w);
                if (dd_pos(w) && dd_gt(cum, t)) {
                    hit = i;
                    break;
                }
            }
            hit = (int)__reduce_min_sync(kFull, (unsigned)hit);
            lastpos = (int)__reduce_max_sync(kFull, (unsigned)(lastpos + 1)) - 1;
            const int sel = hit != INT_MAX ? hit : lastpos;
            o.token = sel >= 0 ? (int)Kp[sel].y : -1;
        }
    }
    finish(p, b, k, o, sb);
}

static_assert(2 * kTopKMerge * sizeof(uint2) <= kSampDyn, "the merged lists fit the fallback ring's memory");
static_assert(kKeptMax % 32 == 0, "kept entries split evenly over a warp's lanes");

// launches `k` as a programmatic dependent of the previous kernel in `s`
template <typename K>
static cudaError_t launch_pdl(K k, dim3 grid, int smem, cudaStream_t s, const SampleParams &p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, p);
}

cudaError_t launch_chain_topk(const SampleParams &p, int dtype, int sms, cudaStream_t s) {
    // a multiple of c (each block keeps one slice index), at most a full wave
    const int64_t items = (int64_t)p.B * (p.gamma + 1) * p.c;
    const int64_t cap = (int64_t)sms * kTkBlocksPerSM;
    int64_t g = ((items < cap ? items : cap) / p.c) * p.c;
    if (g < p.c) g = p.c;
    const dim3 grid((unsigned)g);
    const dim3 mgrid((unsigned)((int64_t)p.B * (p.gamma + 1)));
    const int smem = (int)sizeof(TkRing);
    const int msmem = (int)kSampDyn;
    cudaError_t e;
    if (dtype == SPEC_DTYPE_BF16) {
        static std::atomic<unsigned long long> done{0}, mdone{0};
        e = ensure_smem_attr(chain_topk_kernel<__nv_bfloat16>, smem, done);
        if (e == cudaSuccess) e = ensure_smem_attr(chain_topk_merge_kernel<__nv_bfloat16>, msmem, mdone);
        if (e != cudaSuccess) return e;
        chain_topk_kernel<__nv_bfloat16><<<grid, kNT, smem, s>>>(p);
        e = launch_pdl(chain_topk_merge_kernel<__nv_bfloat16>, mgrid, msmem, s, p);
        if (e != cudaSuccess) return e;
    } else {
        static std::atomic<unsigned long long> done{0}, mdone{0};
        e = ensure_smem_attr(chain_topk_kernel<float>, smem, done);
        if (e == cudaSuccess) e = ensure_smem_attr(chain_topk_merge_kernel<float>, msmem, mdone);
        if (e != cudaSuccess) return e;
        chain_topk_kernel<float><<<grid, kNT, smem, s>>>(p);
        e = launch_pdl(chain_topk_merge_kernel<float>, mgrid, msmem, s, p);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace specv
