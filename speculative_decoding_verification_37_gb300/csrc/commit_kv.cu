// KV commit and rollback (sm_103a).
//
// "KV Cache 优化（四）：Speculative Decoding 投机解码" §6 and "10.6 投机解码"
// §10.6.3: the candidates' K/V are held tentatively; after verification the
// accepted slots are committed at one boundary in every layer and the commit
// length advances; rejected slots are dropped by not advancing past them,
// never by copying whole blocks.
//
// One single-warp block per (request b, accepted slot i, group): a group is
// up to kCommitStage bytes of token i's 2*L units (one layer's K or V, H*D
// elements each; units larger than a stage are split into pieces).  Lane 0
// moves the group with the bulk-copy (TMA) engine: one cp.async.bulk per
// unit from the temporary slots into shared memory, completing on one
// mbarrier, then one bulk store per unit into the paged cache.  The bytes in
// flight cost no registers, so many blocks share an SM.
//
// No prefix over the batch is needed: a block whose slot is past n_slots[b]
// exits after one load.  The block's lanes validate the whole request (all
// slots and block-table entries) in parallel, so a bad request is skipped as
// a whole by every block.  The block that arrives last for a request (one
// counter per request in the workspace) advances committed_len[b]; every
// block of the request has read the old length before it arrives.
#include "common.cuh"
#include "kernels.h"
#include "tma.cuh"

namespace specv {

constexpr uint32_t kCommitStage = 16384;  // bytes one block moves

CommitGeom commit_geometry(int L, int64_t unit_bytes) {
    CommitGeom g;
    if (unit_bytes > (int64_t)kCommitStage) {
        g.ppu = (int)((unit_bytes + kCommitStage - 1) / kCommitStage);
        g.upp = 1;
        g.groups = 2 * L * g.ppu;
    } else {
        g.ppu = 1;
        g.upp = (int)(kCommitStage / unit_bytes);
        g.groups = (2 * L + g.upp - 1) / g.upp;
    }
    return g;
}

__global__ void __launch_bounds__(32) commit_kv_kernel(CommitParams p) {
    __shared__ __align__(128) unsigned char stage[kCommitStage];
    __shared__ __align__(8) unsigned long long bar;
    const int lane = threadIdx.x;
    const int G = p.groups, S = p.S;
    const int64_t bi = blockIdx.x / G;
    const int grp = (int)(blockIdx.x - bi * G);
    const int b = (int)(bi / S), i = (int)(bi - (int64_t)b * S);
    const bool head = i == 0 && grp == 0;

    const int n = p.n_slots[b];
    const int len0 = p.len[b];  // loaded with n: one round trip
    if (!head && (unsigned)i >= (unsigned)n) return;  // past n_slots (or n < 0: the head flags it)
    bool good = n >= 0 && n <= S && len0 >= 0 && (int64_t)len0 + n <= (int64_t)p.max_blocks * p.bs;
    bool lane_ok = true;
    int slot_i = 0, blk_i = 0;
    if (good) {
        for (int q = lane; q < n; q += 32) {
            const int s = p.slots ? p.slots[(int64_t)b * p.slots_stride + q] : q;
            const int blk = p.table[(int64_t)b * p.max_blocks + (len0 + q) / p.bs];
            lane_ok = lane_ok && s >= 0 && s < S && blk >= 0 && (int64_t)blk < p.nb;
            if (q == i) {
                slot_i = s;
                blk_i = blk;
            }
        }
    }
    good = __all_sync(kFull, lane_ok) && good;
    slot_i = __shfl_sync(kFull, slot_i, i & 31);
    blk_i = __shfl_sync(kFull, blk_i, i & 31);
    if (lane != 0) return;
    if (!good) {
        if (head) {
            if (p.flags) p.flags[b] |= SPEC_FLAG_BAD_INPUT;
            if (p.blocks_in_use) p.blocks_in_use[b] = (len0 + p.bs - 1) / p.bs;
            atomicOr(p.status, SPEC_FLAG_BAD_INPUT);
        }
        return;
    }
    if (n == 0) {
        if (p.blocks_in_use) p.blocks_in_use[b] = (len0 + p.bs - 1) / p.bs;  // head only
        return;
    }

    // pieces [k0, k1) of the token in (unit, piece) order
    const int two_l = 2 * p.L;
    const int64_t unit = p.unit_bytes;
    const int k0 = grp * p.upp;
    const int k1 = p.ppu > 1 ? k0 + 1 : min(two_l, k0 + p.upp);
    auto piece = [&](int k, int &lk, int64_t &off, uint32_t &bytes) {
        lk = k / p.ppu;
        const int sub = k - lk * p.ppu;
        off = (int64_t)sub * kCommitStage;
        bytes = (uint32_t)min((int64_t)kCommitStage, unit - off);
    };
    const int pos = len0 + i;
    const char *src_tok = p.temp + ((int64_t)b * two_l * S + slot_i) * unit;  // + lk*S*unit
    char *dst_tok = p.cache + ((int64_t)blk_i * p.bs + pos % p.bs) * unit;    // + lk*nb*bs*unit
    const int64_t dst_lk = p.nb * p.bs * unit;

    uint32_t total = 0;
    for (int k = k0; k < k1; ++k) {
        int lk; int64_t off; uint32_t bytes;
        piece(k, lk, off, bytes);
        total += bytes;
    }
    mbar_init(&bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(&bar, total);
    uint32_t so = 0;
    for (int k = k0; k < k1; ++k) {
        int lk; int64_t off; uint32_t bytes;
        piece(k, lk, off, bytes);
        bulk_g2s(stage + so, src_tok + (int64_t)lk * S * unit + off, bytes, &bar);
        so += bytes;
    }
    bool ok = mbar_wait_bounded(&bar, 0u);
    if (ok) {
        so = 0;
        for (int k = k0; k < k1; ++k) {
            int lk; int64_t off; uint32_t bytes;
            piece(k, lk, off, bytes);
            bulk_s2g(dst_tok + lk * dst_lk + off, stage + so, bytes);
            so += bytes;
        }
        bulk_commit();
        bulk_wait_read();  // the stage may go; the writes finish before the kernel does
    } else {
        // the loads are still outstanding: wait for them (bounded) before the
        // block (and its shared memory) goes away
        // (then no arrival: the length does not advance past a group that
        // was not copied)
        if (mbar_drain(&bar, 0u)) mbar_inval(&bar);  // otherwise the barrier stays as it is
        if (p.flags) atomicOr(p.flags + b, SPEC_FLAG_TIMEOUT);
        atomicOr(p.status, SPEC_FLAG_TIMEOUT);
        return;
    }
    mbar_inval(&bar);

    // the last block of the request advances its length (every block of the
    // request read the old length before it arrived; nothing in this kernel
    // reads it after, so the arrival need not wait for the writes)
    if (atomicAdd(p.counters + b, 1u) == (unsigned)(n * G - 1)) {
        __threadfence();
        const int nl = len0 + n;
        p.len[b] = nl;
        if (p.blocks_in_use) p.blocks_in_use[b] = (nl + p.bs - 1) / p.bs;
        p.counters[b] = 0u;
    }
}

cudaError_t launch_commit_kv(const CommitParams &p, cudaStream_t s) {
    const int64_t grid = (int64_t)p.B * p.S * p.groups;
    commit_kv_kernel<<<(unsigned)grid, 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace specv
