// Sampled chain verification (temperature > 0), full-vocabulary rows and
// top-k rows that need the exact cluster-wide threshold search (sm_103a).
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
//  * Acceptance: each CTA streams its slices once from HBM through a
//    bulk-copy ring (tma.cuh) keeping an online (max, sum of 2^(x log2e/T -
//    m)) pair; the c pairs are pushed over DSMEM into every CTA and combined
//    in rank order, so all CTAs hold identical normalisers and the same a_k.
//  * The draw: only the first rejecting position (or the bonus position)
//    decides the emitted token.  Each request keeps the earliest rejection
//    seen so far in a workspace word; position-major order makes earlier
//    positions finish first, so a position that already sees an earlier
//    rejection skips its draw.  The draw is taken in double-float arithmetic
//    (ddmath.cuh), close to float64: at V ~ 1e5 the CDF boundaries lie ~1e-5
//    apart and an fp32 CDF would often pick a neighbouring token.  The slices
//    are re-read from L2 (the same CTA read them microseconds earlier), dd
//    slice totals are exchanged over DSMEM, and the CTA whose slice holds the
//    crossing scans it in token order.
//  * Each position writes one 16-byte record; the position that arrives
//    last for its request (arrival counter) writes the request's outputs.
// No block waits on another except through cluster barriers between
// co-scheduled CTAs of one cluster.
#include "sample_common.cuh"

namespace specv {

template <typename T, bool MASK>
__global__ void __launch_bounds__(kNT, 3) chain_sample_kernel(SampleParams p) {
    __shared__ SampBase sb;
    extern __shared__ __align__(128) unsigned char dsm[];
    load_exp_tables(p, sb);
    __syncthreads();
    // Every CTA of the cluster must have started (and initialised the shared
    // words others write into) before any remote access: arrive (release)
    // now; the exchange waits just before its first remote write.
    asm volatile("barrier.cluster.arrive.aligned;\n" ::: "memory");
    const int c = p.c;
    ClusterEx ex(c, (int)cg::this_cluster().block_rank());
    const int qpos = blockIdx.x / c;
    const int k = qpos / p.B, b = qpos % p.B;   // position-major
    const int lo = min(p.V, ex.j * p.Vs), hi = min(p.V, lo + p.Vs);
    masked_position<T, MASK>(p, sb, dsm, ex, k, b, lo, hi);
}

template <typename T, bool MASK>
static cudaError_t launch_mask(cudaLaunchConfig_t &cfg, const SampleParams &p) {
    static std::atomic<unsigned long long> done{0};
    cudaError_t e = ensure_smem_attr(chain_sample_kernel<T, MASK>, (int)kSampDyn, done);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, chain_sample_kernel<T, MASK>, p);
}

cudaError_t launch_chain_sample(const SampleParams &p, int dtype, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)p.B * (p.gamma + 1) * p.c));
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = kSampDyn;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool mask = p.top_k > 0 || p.per_request;  // per-request top-k and top-p need the masked path
    if (dtype == SPEC_DTYPE_BF16)
        return mask ? launch_mask<__nv_bfloat16, true>(cfg, p) : launch_mask<__nv_bfloat16, false>(cfg, p);
    return mask ? launch_mask<float, true>(cfg, p) : launch_mask<float, false>(cfg, p);
}

}  // namespace specv
