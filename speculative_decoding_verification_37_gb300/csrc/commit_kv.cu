// KV commit and rollback (sm_103a).
//
// "KV Cache 优化（四）：Speculative Decoding 投机解码" §6 and "10.6 投机解码"
// §10.6.3: the candidates' K/V are held tentatively; after verification the
// accepted slots are committed at one boundary in every layer and the commit
// length advances; rejected slots are dropped by not advancing past them,
// never by copying whole blocks.
//
// The work is a flat list of 2 KiB-class units (one token's K or V of one
// layer: H*D elements).  Every block validates all requests (so a bad
// request is skipped as a whole), builds the exclusive prefix of the
// accepted token counts in shared memory, and then its warps copy units
// unit = (layer*2 + kv) * tokens + token with 16-byte vector loads/stores.
// Consecutive warps take consecutive tokens of one (layer, K|V), so source
// and destination runs are contiguous within a request.  The last block to
// finish (one arrival counter) advances the lengths; every other block only
// reads them.
#include "common.cuh"
#include "kernels.h"

namespace specv {

constexpr int kCommitNT = 512;
constexpr int kCommitBatch = 4;  // 16-byte chunks in flight per lane

int commit_threads() { return kCommitNT; }
size_t commit_smem_bytes(int B) { return (size_t)(B + 1) * sizeof(int) + (size_t)B; }

__global__ void __launch_bounds__(kCommitNT) commit_kv_kernel(CommitParams p) {
    extern __shared__ int smem[];
    int *prefix = smem;                                          // [B+1]
    unsigned char *ok = reinterpret_cast<unsigned char *>(smem + p.B + 1);  // [B]
    __shared__ int s_chunk[kCommitNT];
    __shared__ int s_last;
    const int B = p.B, tid = threadIdx.x;

    // 1. validate each request; accepted count (0 if bad)
    for (int b = tid; b < B; b += kCommitNT) {
        const int n = p.n_slots[b];
        const int len0 = p.len[b];
        bool good = n >= 0 && n <= p.S && len0 >= 0 &&
                    (int64_t)len0 + n <= (int64_t)p.max_blocks * p.bs;
        for (int i = 0; good && i < n; ++i) {
            const int s = p.slots ? p.slots[(int64_t)b * p.slots_stride + i] : i;
            const int blk = p.table[(int64_t)b * p.max_blocks + (len0 + i) / p.bs];
            good = s >= 0 && s < p.S && blk >= 0 && (int64_t)blk < p.nb;
        }
        ok[b] = good;
    }
    __syncthreads();
    // 2. exclusive prefix of the counts: contiguous chunk per thread, then a block scan
    const int per = (B + kCommitNT - 1) / kCommitNT;
    const int c0 = min(B, tid * per), c1 = min(B, c0 + per);
    int sum = 0;
    for (int b = c0; b < c1; ++b) sum += ok[b] ? p.n_slots[b] : 0;
    s_chunk[tid] = sum;
    __syncthreads();
    if (tid < 32) {
        // warp 0 scans the kCommitNT chunk totals
        int carry = 0;
        for (int base = 0; base < kCommitNT; base += 32) {
            int v = s_chunk[base + tid];
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o);
                if (tid >= o) incl += y;
            }
            s_chunk[base + tid] = carry + incl - v;
            carry += __shfl_sync(kFull, incl, 31);
        }
        if (tid == 0) prefix[B] = carry;
    }
    __syncthreads();
    {
        int run = s_chunk[tid];
        for (int b = c0; b < c1; ++b) {
            prefix[b] = run;
            run += ok[b] ? p.n_slots[b] : 0;
        }
    }
    __syncthreads();

    // 3. copy units
    const int tokens = prefix[B];
    const int64_t units = (int64_t)tokens * p.L * 2;
    const int chunks = p.unit_bytes / 16;
    const int lane = tid & 31;
    const int64_t warp = (int64_t)blockIdx.x * (kCommitNT / 32) + (tid >> 5);
    const int64_t nwarps = (int64_t)gridDim.x * (kCommitNT / 32);
    for (int64_t u = warp; u < units; u += nwarps) {
        const int lk = (int)(u / tokens);
        const int t = (int)(u - (int64_t)lk * tokens);
        // request of token t: the last b with prefix[b] <= t (empty requests skipped)
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int b = lo, i = t - prefix[b];
        const int s = p.slots ? p.slots[(int64_t)b * p.slots_stride + i] : i;
        const int pos = p.len[b] + i;
        const int blk = p.table[(int64_t)b * p.max_blocks + pos / p.bs];
        const int layer = lk >> 1, kv = lk & 1;
        const uint4 *src = reinterpret_cast<const uint4 *>(
            p.temp + ((((int64_t)b * p.L + layer) * 2 + kv) * p.S + s) * p.unit_bytes);
        uint4 *dst = reinterpret_cast<uint4 *>(
            p.cache + ((((int64_t)layer * 2 + kv) * p.nb + blk) * p.bs + pos % p.bs) * p.unit_bytes);
        for (int cb = lane; cb < chunks; cb += 32 * kCommitBatch) {
            uint4 v[kCommitBatch];
#pragma unroll
            for (int q = 0; q < kCommitBatch; ++q)
                if (cb + 32 * q < chunks) v[q] = ld_nc16(src + cb + 32 * q);
#pragma unroll
            for (int q = 0; q < kCommitBatch; ++q)
                if (cb + 32 * q < chunks) dst[cb + 32 * q] = v[q];
        }
    }

    // 4. the last block advances the lengths
    __syncthreads();
    if (tid == 0) {
        __threadfence();
        s_last = atomicAdd(p.counter, 1u) == gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    unsigned any_bad = 0;
    for (int b = tid; b < B; b += kCommitNT) {
        if (ok[b]) {
            const int nl = p.len[b] + p.n_slots[b];
            p.len[b] = nl;
            if (p.blocks_in_use) p.blocks_in_use[b] = (nl + p.bs - 1) / p.bs;
        } else {
            any_bad = 1;
            if (p.flags) p.flags[b] |= SPEC_FLAG_BAD_INPUT;
            if (p.blocks_in_use) p.blocks_in_use[b] = (p.len[b] + p.bs - 1) / p.bs;
        }
    }
    if (__syncthreads_or(any_bad) && tid == 0) atomicOr(p.status, SPEC_FLAG_BAD_INPUT);
    if (tid == 0) *p.counter = 0u;
}

cudaError_t launch_commit_kv(const CommitParams &p, int grid, cudaStream_t s) {
    const size_t smem = commit_smem_bytes(p.B);
    if (smem > 48 * 1024) {
        // the largest B (32768) needs the most; set that once per device
        static std::atomic<unsigned long long> done{0};
        cudaError_t e = ensure_smem_attr(commit_kv_kernel, (int)commit_smem_bytes(32768), done);
        if (e != cudaSuccess) return e;
    }
    commit_kv_kernel<<<grid, kCommitNT, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace specv
