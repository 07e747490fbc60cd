// C ABI of the verify-and-commit library: argument validation, workspace
// layout, launch configuration.  No allocation, no synchronisation (except
// spec_get_status, which says so), no stream creation.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>

#include "kernels.h"
#include "spec_verify.h"

using namespace specv;

namespace {

thread_local char g_cuda_err[256] = "";
std::atomic<long long> g_idle_limit{0};  // 0: the full-vocabulary path's default

int cuda_fail(cudaError_t e) {
    std::snprintf(g_cuda_err, sizeof g_cuda_err, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return SPEC_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t esize(int dtype) { return dtype == SPEC_DTYPE_BF16 ? 2 : 4; }

// Whether this device's hardware exponential keeps within the error bound
// the full-vocabulary path's certified fp32 draw assumes, measured once per
// device by the exhaustive self-test (synchronous, about a second).  Not
// measured while `s` is being captured: such a call takes another path.
bool ex2_certified(cudaStream_t s) {
    static std::atomic<int> state[64];  // 0 unknown, 1 within the bound, 2 not
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const int st = state[dev].load(std::memory_order_acquire);
    if (st != 0) return st == 1;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) return false;
    float worst = 1.0f;
    const bool ok = spec_selftest_ex2(&worst) == SPEC_OK && worst <= full_ex2_bound();
    state[dev].store(ok ? 1 : 2, std::memory_order_release);
    return ok;
}

int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    if (dev >= 0 && dev < 64 && cached[dev].load() > 0) return cached[dev].load();
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    if (dev >= 0 && dev < 64) cached[dev].store(n);
    return n;
}

// Slices per row: the fewest (at most max_slices) whose 16-byte-rounded length
// keeps one slice within `limit` bytes.
int slices_for(int V, int dtype, int max_slices, int64_t limit = 65536) {
    const int64_t e = (int64_t)esize(dtype);
    int64_t c = ((int64_t)V * e + limit - 1) / limit;
    if (c < 1) c = 1;
    while (c < max_slices && ((((int64_t)V + c - 1) / c + 7) & ~int64_t(7)) * e > limit) ++c;
    if (c > max_slices) c = max_slices;
    return (int)c;
}

int slice_len(int V, int c) {
    int s = (V + c - 1) / c;
    return (s + 7) & ~7;  // whole 16-byte vectors for both element types
}

struct Ws {
    unsigned *status;
    unsigned *counters;  // [B] arrival counters
    unsigned *rejword;   // [B] earliest rejection per request (chain, sampled)
    void *data;          // chain: records or argmax keys; tree: argmax keys
    uint32_t *rkmax;     // chain, top-k: [B*(gamma+1)*2][kTopKThreads] thread maxima
    uint32_t *rkgrp;     // chain, top-k: [B*(gamma+1)*2][kTopKGroups][kTopKThreads] largest groups
    TopkRow *rkrow;      // chain, top-k: [B*(gamma+1)*2] published kept-set headers
    uint2 *rkent;        // chain, top-k: [B*(gamma+1)*2][kKeptRowMax] kept entries
    unsigned *rkcnt;     // chain, top-k: [B*(gamma+1)] position arrival counters (zeroed)
    // chain, full vocabulary: see SampleParams
    float2 *fpart, *fxd;
    float4 *fstat;
    unsigned long long *rstate, *qitem;
    unsigned *pcnt, *dcnt;
    DrawRec *drec;
    DrawPart *dpart;
    int *amb;
};

// Slices per row of the full-vocabulary path (sized for fp32 rows, so one
// size serves both element types).
int full_slices(int V, int dtype) {
    return (int)(((int64_t)V * (int64_t)esize(dtype) + full_row_bytes() - 1) / full_row_bytes());
}

enum WsExtra { kWsPlain = 0, kWsPool = 1, kWsFull = 2 };

// One layout for sizing and for pointers.  `rows` = B*(gamma+1) for a chain
// (0 for other kinds), `data_bytes` the per-row keys or records; `extra`
// adds the top-k candidate regions or the full-vocabulary path's state for
// rows of V logits.
size_t ws_layout_bytes(int B, size_t rows, size_t data_bytes, Ws *w, void *base_ptr, int extra = kWsPlain,
                       int V = 0) {
    char *base = static_cast<char *>(base_ptr);
    size_t off = kWsHeader;
    const size_t per_req = ws_align((size_t)B * sizeof(unsigned));
    if (w) {
        *w = Ws{};
        w->status = reinterpret_cast<unsigned *>(base);
        w->counters = reinterpret_cast<unsigned *>(base + off);
        w->rejword = reinterpret_cast<unsigned *>(base + off + per_req);
    }
    off += 2 * per_req;
    if (w) w->data = base + off;
    off += ws_align(data_bytes);
    auto take = [&](size_t bytes) -> char * {
        char *at = base ? base + off : nullptr;
        off += ws_align(bytes);
        return at;
    };
    if (extra == kWsPool) {
        char *rm = take(rows * 2 * (size_t)kTopKThreads * sizeof(uint32_t));
        char *rg = take(rows * 2 * (size_t)kTopKGroups * kTopKThreads * sizeof(uint32_t));
        char *rh = take(rows * 2 * sizeof(TopkRow));
        char *re = take(rows * 2 * (size_t)kKeptRowMax * sizeof(uint2));
        char *rc = take(rows * sizeof(unsigned));
        if (w) {
            w->rkmax = reinterpret_cast<uint32_t *>(rm);
            w->rkgrp = reinterpret_cast<uint32_t *>(rg);
            w->rkrow = reinterpret_cast<TopkRow *>(rh);
            w->rkent = reinterpret_cast<uint2 *>(re);
            w->rkcnt = reinterpret_cast<unsigned *>(rc);
        }
    } else if (extra == kWsFull) {
        const size_t c = (size_t)full_slices(V, SPEC_DTYPE_F32), nb = (size_t)B;
        char *fp = take(rows * 2 * c * sizeof(float2));
        char *fx = take(rows * sizeof(float2));
        char *fs = take(rows * sizeof(float4));
        char *rs = take(nb * sizeof(unsigned long long));
        char *pc = take(rows * sizeof(unsigned));
        char *dr = take(nb * sizeof(DrawRec));
        char *dp = take(nb * c * sizeof(DrawPart));
        char *dc = take(nb * sizeof(unsigned));
        char *am = take(nb * c * (size_t)kFullAmb * sizeof(int));
        char *qi = take(3 * nb * c * sizeof(unsigned long long));
        if (w) {
            w->fpart = reinterpret_cast<float2 *>(fp);
            w->fxd = reinterpret_cast<float2 *>(fx);
            w->fstat = reinterpret_cast<float4 *>(fs);
            w->rstate = reinterpret_cast<unsigned long long *>(rs);
            w->pcnt = reinterpret_cast<unsigned *>(pc);
            w->drec = reinterpret_cast<DrawRec *>(dr);
            w->dpart = reinterpret_cast<DrawPart *>(dp);
            w->dcnt = reinterpret_cast<unsigned *>(dc);
            w->amb = reinterpret_cast<int *>(am);
            w->qitem = reinterpret_cast<unsigned long long *>(qi);
        }
    }
    return off;
}

size_t chain_data_bytes(size_t rows) {
    const size_t rec = rows * sizeof(PosRec);
    const size_t keys = rows * sizeof(unsigned long long);
    return rec > keys ? rec : keys;
}

// Double-float constants for the on-device exponential: ln2/64 in three
// parts (the first rounded to 11 significant bits) and 2^(j/64), j = 0..63,
// each computed in double on the host and split as hi = (float)v,
// lo = (float)(v - hi).  1/T is filled in per call.
void split(double v, float2 &out) {
    out.x = (float)v;
    out.y = (float)(v - (double)out.x);
}

const DdExpTables &exp_tables() {
    static const DdExpTables t = [] {
        DdExpTables x;
        const long double c = 0.693147180559945309417232121458176568L / 64.0L;
        int ex;
        std::frexp((double)c, &ex);
        const double q = std::ldexp(1.0, ex - 11);  // 11 significant bits
        const double c1 = std::nearbyint((double)c / q) * q;
        x.c1 = (float)c1;
        x.c2 = (float)(c - (long double)x.c1);
        x.c3 = (float)(c - (long double)x.c1 - (long double)x.c2);
        for (int j = 0; j < 64; ++j) split(std::exp2((double)j / 64.0), x.tab[j]);
        x.it = make_float2(1.0f, 0.0f);
        return x;
    }();
    return t;
}

}  // namespace

namespace {

// Tree-level workspace: header (status) | slice summaries [B*H*slices] |
// row results [B*H].
size_t tree_level_layout(int32_t B, int32_t H, int32_t V, void *base, TreeLevelParams *p) {
    const size_t rows = (size_t)B * (size_t)H;
    const size_t slices = ((size_t)V + kTlSliceElems - 1) / kTlSliceElems;
    size_t off = kWsHeader;
    const size_t o_it = off;
    off += ws_align(rows * slices * sizeof(TlItem));
    const size_t o_rr = off;
    off += ws_align(rows * sizeof(TlRow));
    if (p) {
        char *c = static_cast<char *>(base);
        p->status = reinterpret_cast<unsigned *>(c);
        p->items = reinterpret_cast<TlItem *>(c + o_it);
        p->rowrec = reinterpret_cast<TlRow *>(c + o_rr);
    }
    return off;
}

}  // namespace

extern "C" size_t spec_workspace_bytes(int kind, int32_t B, int32_t n, int32_t V) {
    if (B < 0 || n < 0 || V < 0) return 0;
    switch (kind) {
    case SPEC_WS_CHAIN:
    case SPEC_WS_CHAIN_TOPK:
    case SPEC_WS_CHAIN_FULL: {
        const size_t rows = (size_t)B * ((size_t)n + 1);
        const int extra = kind == SPEC_WS_CHAIN_TOPK ? kWsPool : kind == SPEC_WS_CHAIN_FULL ? kWsFull : kWsPlain;
        return ws_layout_bytes(B, rows, chain_data_bytes(rows), nullptr, nullptr, extra, V);
    }
    case SPEC_WS_TREE:
        return ws_layout_bytes(B, 0, (size_t)B * (size_t)n * sizeof(unsigned long long), nullptr, nullptr);
    case SPEC_WS_COMMIT:
        return kWsHeader + ws_align((size_t)B * sizeof(unsigned));
    case SPEC_WS_TREE_LEVEL:
        return tree_level_layout(B, n, V, nullptr, nullptr);
    default:
        return 0;
    }
}

namespace specv {

// Every host-side check of a chain call's arguments except the workspace's:
// SPEC_OK or the code the call returns, before anything is enqueued.
int chain_args_check(const SpecChainArgs *a) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->B < 0 || a->gamma < 0 || a->gamma > 4096 || a->V < 1) return SPEC_ERR_INVALID_ARG;
    if (a->dtype != SPEC_DTYPE_BF16 && a->dtype != SPEC_DTYPE_F32) return SPEC_ERR_INVALID_ARG;
    if (!(a->temperature >= 0.0f) || !std::isfinite(a->temperature)) return SPEC_ERR_INVALID_ARG;
    if (a->top_k < 0 || !(a->fallback_eps >= 0.0f) || !std::isfinite(a->fallback_eps))
        return SPEC_ERR_INVALID_ARG;
    if (!(a->top_p >= 0.0f) || !std::isfinite(a->top_p)) return SPEC_ERR_INVALID_ARG;
    if (a->B == 0) return SPEC_OK;
    const bool per_request = a->gamma_per_request || a->temperature_per_request || a->top_k_per_request ||
                             a->top_p_per_request;
    const bool greedy = a->temperature == 0.0f && !a->temperature_per_request;
    if (!a->target_logits || a->target_row_stride < a->V) return SPEC_ERR_INVALID_ARG;
    if (!a->n_acc || !a->out_tokens || !a->n_out) return SPEC_ERR_INVALID_ARG;
    if (a->gamma > 0 && !a->draft_tokens) return SPEC_ERR_INVALID_ARG;
    if (!greedy) {
        if (!a->uniforms) return SPEC_ERR_INVALID_ARG;
        if (a->gamma > 0 && (!a->draft_logits || a->draft_row_stride < a->V)) return SPEC_ERR_INVALID_ARG;
        if (!a->temperature_per_request && !std::isfinite((float)(1.4426950408889634074 / (double)a->temperature)))
            return SPEC_ERR_INVALID_ARG;
    }
    if (per_request && (a->eos_enabled || a->max_new || a->committed_len))
        return SPEC_ERR_UNSUPPORTED;  // per-request rounds: no early end, no in-place commit
    const size_t es = esize(a->dtype);
    if (!aligned(a->target_logits, es) || (a->draft_logits && !aligned(a->draft_logits, es)))
        return SPEC_ERR_INVALID_ARG;
    if (a->blocks_in_use && (!a->committed_len || a->block_size < 1)) return SPEC_ERR_INVALID_ARG;
    if (a->draft_len && !a->committed_len) return SPEC_ERR_INVALID_ARG;
    if (a->kv_capacity < 0) return SPEC_ERR_INVALID_ARG;
    if (a->eos_enabled && (a->eos_token < 0 || a->eos_token >= a->V)) return SPEC_ERR_INVALID_ARG;
    return SPEC_OK;
}

}  // namespace specv

extern "C" int spec_verify_chain(const SpecChainArgs *a, void *workspace, size_t ws_bytes,
                                 void *stream) {
    const int chk = chain_args_check(a);
    if (chk != SPEC_OK) return chk;
    if (a->B == 0) return SPEC_OK;
    const bool per_request = a->gamma_per_request || a->temperature_per_request || a->top_k_per_request ||
                             a->top_p_per_request;
    const bool greedy = a->temperature == 0.0f && !per_request;
    const size_t es = esize(a->dtype);
    InPlace ip{a->committed_len, a->draft_len, a->blocks_in_use, a->block_size, a->kv_capacity};
    const StopRule stop{a->eos_enabled ? a->eos_token : -1, a->max_new};
    const bool nucleus = a->top_p > 0.0f && a->top_p < 1.0f && !greedy;
    const int64_t rows = (int64_t)a->B * (a->gamma + 1);
    if (!workspace || !aligned(workspace, 256) ||
        ws_bytes < spec_workspace_bytes(SPEC_WS_CHAIN, a->B, a->gamma, a->V))
        return SPEC_ERR_INVALID_ARG;
    // the extra regions a larger workspace holds (the kinds never both fit the
    // same size test by accident: each is checked against its own size)
    const bool sampled_full = !greedy && (a->top_k == 0 || a->top_k >= a->V);
    const bool has_full = sampled_full && ws_bytes >= spec_workspace_bytes(SPEC_WS_CHAIN_FULL, a->B, a->gamma, a->V);
    const bool has_pool = !has_full && ws_bytes >= spec_workspace_bytes(SPEC_WS_CHAIN_TOPK, a->B, a->gamma, a->V);
    Ws w;
    ws_layout_bytes(a->B, (size_t)rows, chain_data_bytes((size_t)rows), &w, workspace,
                    has_full ? kWsFull : has_pool ? kWsPool : kWsPlain, a->V);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (greedy) {
        ArgmaxParams p = {};
        p.rows = a->target_logits;
        p.stride = a->target_row_stride;
        p.V = a->V;
        p.slices = slices_for(a->V, a->dtype, 1 << 20, argmax_stage_bytes());
        p.slice_len = slice_len(a->V, p.slices);
        p.rows_per_req = a->gamma + 1;
        p.keys = static_cast<unsigned long long *>(w.data);
        p.counters = w.counters;
        p.status = w.status;
        p.mode = 0;
        p.gamma = a->gamma;
        p.tokens = a->draft_tokens;
        p.n_acc = a->n_acc;
        p.out_tokens = a->out_tokens;
        p.n_out = a->n_out;
        p.flags = a->flags;
        p.ip = ip;
        p.stop = stop;
        if (rows * p.slices > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
        e = launch_argmax_verify(p, a->dtype, (int)rows, sm_count(), s);
    } else {
        SampleParams p = {};
        p.B = a->B;
        p.gamma = a->gamma;
        p.V = a->V;
        p.c = slices_for(a->V, a->dtype, 8, 32768);
        p.Vs = slice_len(a->V, p.c);
        p.target = a->target_logits;
        p.tstride = a->target_row_stride;
        p.draft = a->draft_logits;
        p.dstride = a->draft_row_stride;
        p.tokens = a->draft_tokens;
        p.unif = a->uniforms;
        const double c2 = 1.4426950408889634074 / (double)a->temperature;
        p.c2 = (float)c2;
        p.c2lo = (float)(c2 - (double)p.c2);
        p.exptab = exp_tables();
        split(1.0 / (double)a->temperature, p.exptab.it);
        p.top_k = (a->top_k >= a->V) ? 0 : a->top_k;
        p.top_p = nucleus ? a->top_p : 0.0f;
        p.eps = a->fallback_eps;
        p.n_acc = a->n_acc;
        p.out_tokens = a->out_tokens;
        p.n_out = a->n_out;
        p.accept_prob = a->accept_prob;
        p.resid = a->residual_mass;
        p.flags = a->flags;
        p.status = w.status;
        p.counters = w.counters;
        p.rejword = w.rejword;
        p.recs = static_cast<PosRec *>(w.data);
        p.rkmax = w.rkmax;
        p.rkgrp = w.rkgrp;
        p.rkrow = w.rkrow;
        p.rkent = w.rkent;
        p.rkcnt = w.rkcnt;
        p.fpart = w.fpart;
        p.fxd = w.fxd;
        p.fstat = w.fstat;
        p.rstate = w.rstate;
        p.pcnt = w.pcnt;
        p.drec = w.drec;
        p.dpart = w.dpart;
        p.dcnt = w.dcnt;
        p.amb = w.amb;
        p.qitem = w.qitem;
        p.qcap = (unsigned)(3 * (int64_t)a->B * full_slices(a->V, SPEC_DTYPE_F32));
        p.ip = ip;
        p.stop = stop;
        {
            const long long lim = g_idle_limit.load(std::memory_order_relaxed);
            p.idle_limit = lim > 0 ? lim : full_idle_limit();
        }
        p.rq_gamma = a->gamma_per_request;
        p.rq_temp = a->temperature_per_request;
        p.rq_topk = a->top_k_per_request;
        p.rq_topp = a->top_p_per_request;
        // the top-k path: top_k <= 128, chunk indices within 16 bits
        const bool topk_fast = has_pool && p.top_k > 0 && p.top_k <= kTopKFastMax &&
                               ((int64_t)a->V * (int64_t)es + topk_row_bytes() - 1) / topk_row_bytes() <= 0xffff;
        if (per_request || (nucleus && !topk_fast)) {
            // the exact path: one cluster per position, each request with its own settings
            // (the scalars stand in for arrays not given)
            p.per_request = 1;
            if (a->temperature == 0.0f) {  // a scalar greedy default: no finite 1/T to precompute
                p.c2 = 0.0f;
                p.c2lo = 0.0f;
            }
            if (rows * p.c > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
            e = launch_chain_sample(p, a->dtype, s);
            return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
        }
        if (!std::isfinite(p.c2)) return SPEC_ERR_INVALID_ARG;
        // full vocabulary: the persistent kernel when the workspace, the
        // rows' alignment and the sizes allow it
        const int64_t rbytes = (int64_t)a->V * (int64_t)es;
        // (small calls stay on the cluster kernel: a whole-GPU cooperative
        // grid only pays off with a few thousand slices of work)
        const bool full = !nucleus && has_full && p.top_k == 0 && !a->residual_mass && a->gamma <= 30 &&
                          rows * full_slices(a->V, a->dtype) >= 1024 &&
                          rbytes % 16 == 0 && rbytes <= (int64_t)full_row_bytes() * full_max_slices() &&
                          aligned(a->target_logits, 16) && (a->target_row_stride * (int64_t)es) % 16 == 0 &&
                          (a->gamma == 0 || (aligned(a->draft_logits, 16) &&
                                             (a->draft_row_stride * (int64_t)es) % 16 == 0));
        if (full && ex2_certified(s)) {
            p.c = full_slices(a->V, a->dtype);
            p.Vs = full_row_bytes() / (int)es;
            if (rows * p.c > 0x7fffffffLL / 3 || 3 * (int64_t)a->B * full_slices(a->V, SPEC_DTYPE_F32) > 0x7fffffffLL)
                return SPEC_ERR_UNSUPPORTED;
            e = launch_chain_full(p, a->dtype, sm_count(), s);
            return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
        }
        // top-k <= 128: one block per row, kept sets published per position;
        // otherwise the cluster kernel with its exact threshold search
        if (topk_fast) {
            if ((int64_t)a->B * (2 * (int64_t)a->gamma + 1) > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
            e = launch_chain_topk(p, a->dtype, sm_count(), s);
        } else {
            if (rows * p.c > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
            e = launch_chain_sample(p, a->dtype, s);
        }
    }
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

extern "C" int spec_verify_tree(const SpecTreeArgs *a, void *workspace, size_t ws_bytes, void *stream) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->B < 0 || a->N < 0 || a->N > 1023 || a->R < 1 || a->V < 1) return SPEC_ERR_INVALID_ARG;
    if (a->dtype != SPEC_DTYPE_BF16 && a->dtype != SPEC_DTYPE_F32) return SPEC_ERR_INVALID_ARG;
    if (a->B == 0) return SPEC_OK;
    if (!a->logits || a->row_stride < a->V || !aligned(a->logits, esize(a->dtype)))
        return SPEC_ERR_INVALID_ARG;
    if ((a->N > 0 && (!a->node_token || !a->node_parent || !a->path)) || !a->row_of_node)
        return SPEC_ERR_INVALID_ARG;
    if (!a->n_acc || !a->out_tokens || !a->n_out) return SPEC_ERR_INVALID_ARG;
    if (a->pos && !a->committed_len) return SPEC_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) ||
        ws_bytes < spec_workspace_bytes(SPEC_WS_TREE, a->B, a->R, a->V))
        return SPEC_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)a->B * a->R;
    Ws w;
    ws_layout_bytes(a->B, 0, (size_t)rows * sizeof(unsigned long long), &w, workspace);
    ArgmaxParams p = {};
    p.rows = a->logits;
    p.stride = a->row_stride;
    p.V = a->V;
    p.slices = slices_for(a->V, a->dtype, 1 << 20, argmax_stage_bytes());
    p.slice_len = slice_len(a->V, p.slices);
    p.rows_per_req = a->R;
    p.keys = static_cast<unsigned long long *>(w.data);
    p.counters = w.counters;
    p.status = w.status;
    p.mode = 1;
    p.N = a->N;
    p.R = a->R;
    p.node_token = a->node_token;
    p.node_parent = a->node_parent;
    p.row_of_node = a->row_of_node;
    p.committed_len = a->committed_len;
    p.path = a->path;
    p.mask = a->tree_mask;
    p.pos = a->pos;
    p.commit_slots = a->commit_slots;
    p.n_commit = a->n_commit;
    p.n_acc = a->n_acc;
    p.out_tokens = a->out_tokens;
    p.n_out = a->n_out;
    p.flags = a->flags;
    if (rows * p.slices > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
    const cudaError_t e = launch_argmax_verify(p, a->dtype, (int)rows, sm_count(), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

extern "C" int spec_commit_kv(const SpecCommitArgs *a, void *workspace, size_t ws_bytes, void *stream) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->B < 0 || a->B > 32768 || a->L < 1 || a->H < 1 || a->D < 1 || a->S < 1 ||
        a->block_size < 1 || a->num_blocks < 1 || a->max_blocks < 1)
        return SPEC_ERR_INVALID_ARG;
    if (a->elem_bytes != 1 && a->elem_bytes != 2 && a->elem_bytes != 4) return SPEC_ERR_INVALID_ARG;
    const int64_t unit = (int64_t)a->H * a->D * a->elem_bytes;
    if (unit % 16 != 0 || unit > (1 << 20)) return SPEC_ERR_UNSUPPORTED;
    if (a->B == 0) return SPEC_OK;
    if (!a->temp_kv || !a->cache || !a->block_table || !a->n_slots || !a->committed_len)
        return SPEC_ERR_INVALID_ARG;
    if (!aligned(a->temp_kv, 16) || !aligned(a->cache, 16)) return SPEC_ERR_INVALID_ARG;
    if (a->slots && a->slots_stride < a->S) return SPEC_ERR_INVALID_ARG;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < spec_workspace_bytes(SPEC_WS_COMMIT, a->B, 0, 0))
        return SPEC_ERR_INVALID_ARG;
    char *base = static_cast<char *>(workspace);
    CommitParams p = {};
    p.B = a->B;
    p.L = a->L;
    p.S = a->S;
    p.bs = a->block_size;
    p.unit_bytes = (int)unit;
    p.max_blocks = a->max_blocks;
    p.slots_stride = a->slots_stride;
    p.temp = static_cast<const char *>(a->temp_kv);
    p.cache = static_cast<char *>(a->cache);
    p.nb = a->num_blocks;
    p.table = a->block_table;
    p.slots = a->slots;
    p.n_slots = a->n_slots;
    p.len = a->committed_len;
    p.blocks_in_use = a->blocks_in_use;
    p.flags = a->flags;
    p.status = reinterpret_cast<unsigned *>(base);
    p.counters = reinterpret_cast<unsigned *>(base + kWsHeader);
    const CommitGeom geo = commit_geometry(a->L, unit);
    p.ppu = geo.ppu;
    p.upp = geo.upp;
    p.groups = geo.groups;
    // one block per (request, slot, group); blocks past n_slots exit at once
    if ((int64_t)a->B * a->S * p.groups > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
    const cudaError_t e = launch_commit_kv(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

extern "C" int spec_tree_level(const SpecTreeLevelArgs *a, void *workspace, size_t ws_bytes, void *stream) {
    if (!a) return SPEC_ERR_INVALID_ARG;
    if (a->B < 0 || a->V < 1 || a->H < 1 || a->H > kTreeMaxHeads) return SPEC_ERR_INVALID_ARG;
    if (a->dtype != SPEC_DTYPE_BF16 && a->dtype != SPEC_DTYPE_F32) return SPEC_ERR_INVALID_ARG;
    TreeLevelParams p = {};
    int kmax = 0;
    p.koff[0] = 0;
    for (int j = 0; j < a->H; ++j) {
        const int k = a->k[j];
        if (k < 1 || k > kTreeMaxK || k > a->V) return SPEC_ERR_INVALID_ARG;
        kmax = k > kmax ? k : kmax;
        p.koff[j + 1] = p.koff[j] + k;
        if (p.koff[j + 1] > kTreeMaxLevelNodes) return SPEC_ERR_INVALID_ARG;
        for (int i = p.koff[j]; i < p.koff[j + 1]; ++i) p.head_of[i] = (unsigned char)j;
    }
    const int n = p.koff[a->H];
    if (a->n_next < 0 || a->n_next > 64 || a->n_next > n) return SPEC_ERR_INVALID_ARG;
    if (a->n_before < 0 || a->N < 1 || (int64_t)a->n_before + n > a->N) return SPEC_ERR_INVALID_ARG;
    if (a->next_row0 < 1 || (int64_t)a->next_row0 + a->n_next > 0x7fffffffLL) return SPEC_ERR_INVALID_ARG;
    if (!a->parents && (a->H != 1 || a->n_before != 0)) return SPEC_ERR_INVALID_ARG;
    if (a->B == 0) return SPEC_OK;
    const size_t es = esize(a->dtype);
    if (!a->logits || !aligned(a->logits, es) || a->row_stride < a->V) return SPEC_ERR_INVALID_ARG;
    if (!a->node_token || !a->node_parent || !a->node_logp || !a->row_of_node) return SPEC_ERR_INVALID_ARG;
    if (a->n_next > 0 && !a->next_parents) return SPEC_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)a->B * a->H;
    const int64_t slices = ((int64_t)a->V + kTlSliceElems - 1) / kTlSliceElems;
    if (rows * slices > 0x7fffffffLL || (int64_t)a->B * (a->N + 1) > (int64_t)1 << 40) return SPEC_ERR_UNSUPPORTED;
    if (!workspace || !aligned(workspace, 256) || ws_bytes < spec_workspace_bytes(SPEC_WS_TREE_LEVEL, a->B, a->H, a->V))
        return SPEC_ERR_INVALID_ARG;
    tree_level_layout(a->B, a->H, a->V, workspace, &p);
    p.rows = a->logits;
    p.stride = a->row_stride;
    p.B = a->B;
    p.V = a->V;
    p.H = a->H;
    p.slices = (int)slices;
    p.n_nodes = n;
    p.n_next = a->n_next;
    p.N = a->N;
    p.n_before = a->n_before;
    p.next_row0 = a->next_row0;
    p.root = a->parents ? 0 : 1;
    p.parents = a->parents;
    p.node_token = a->node_token;
    p.node_parent = a->node_parent;
    p.node_logp = a->node_logp;
    p.row_of_node = a->row_of_node;
    p.next_parents = a->next_parents;
    p.flags = a->flags;
    const cudaError_t e = launch_tree_level(p, a->dtype, kmax, sm_count(), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

extern "C" int spec_get_status(void *workspace, void *stream, uint32_t *host_flags) {
    if (!workspace || !host_flags) return SPEC_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(host_flags, workspace, sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s);
    return e == cudaSuccess ? SPEC_OK : cuda_fail(e);
}

extern "C" const char *spec_error_string(int code) {
    switch (code) {
    case SPEC_OK: return "success";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported configuration";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_TOO_LARGE: return "request needs more scratch than the static workspace holds";
    default: return "unknown error code";
    }
}

extern "C" const char *spec_last_cuda_error(void) { return g_cuda_err; }

extern "C" int spec_set_idle_limit(int64_t polls) {
    g_idle_limit.store(polls > 0 ? (long long)polls : 0, std::memory_order_relaxed);
    return SPEC_OK;
}
