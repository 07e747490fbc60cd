// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ddmath.cuh"

struct SpecChainArgs;

namespace specv {

// Host-side checks of a chain call's arguments (all but the workspace):
// SPEC_OK or the error code the call returns before enqueuing anything.
int chain_args_check(const SpecChainArgs *a);

// Workspace layout shared by every verify kind: a sticky status word, one
// arrival counter per request, then per-row argmax keys or per-position
// records.  All of it starts zeroed and is left zeroed (except the status).
constexpr size_t kWsHeader = 256;
inline size_t ws_align(size_t x) { return (x + 255) & ~size_t(255); }

struct PosRec {      // one chain position's outcome, written by its cluster
    float a;         // acceptance probability a_k
    float z;         // residual mass sum max(0, p_k - q_k)
    int token;       // drawn token if this position rejected (or is the bonus row)
    unsigned info;   // REC_* bits
};
constexpr unsigned REC_ACCEPT = 1u, REC_BAD_INPUT = 2u, REC_BAD_ROW = 4u, REC_FALLBACK = 8u;

// In-place KV commit of a chain request: the length pointer advance done in
// the verify call's request epilogue.
struct InPlace {
    int *len, *draft_len, *blocks_in_use;
    int block_size;
    int64_t capacity;  // 0 = unchecked
};

// Early end of a chain round at an end-of-sequence token or the length limit.
struct StopRule {
    int eos;             // < 0: none
    const int *max_new;  // [B] tokens a request may still emit, or null
};

struct ArgmaxParams {
    const void *rows;
    int64_t stride;
    int V, slices, slice_len, rows_per_req;
    unsigned long long *keys;  // [B*rows_per_req]
    unsigned *counters;        // [B]
    unsigned *status;
    int mode;                  // 0 = greedy chain, 1 = tree
    // chain
    int gamma;
    const int *tokens;
    // tree
    int N, R;
    const int *node_token, *node_parent, *row_of_node, *committed_len;
    int *path, *pos, *commit_slots, *n_commit;
    uint32_t *mask;
    // outputs shared by both
    int *n_acc, *out_tokens, *n_out;
    unsigned *flags;
    InPlace ip;  // chain only
    StopRule stop;
};

constexpr int kTopKFastMax = 128;  // top_k served by the row-per-block path
constexpr int kKeptRowMax = 256;   // kept entries of one row a position can hold
constexpr int kTopKGroups = 4;     // groups per thread the top-k pass hands on
constexpr int kTopKThreads = 256;  // threads of a top-k pass block

// One row's kept set on the top-k path, published for its position's
// deciding block (16-byte words, read with two vector loads).
struct alignas(16) TopkRow {
    unsigned kn;      // kept entries, token order, in the row's entry array
    unsigned th;      // order key of the threshold: every kept logit's key is >= it
    float m;          // largest kept logit (-inf: no finite logit)
    float s_hi, s_lo; // sum over the kept set of exp((l - m)/T), double-float
    unsigned flags;   // 1: the kept set did not fit (the position takes the exact path)
    unsigned pad[2];
};

// Full-vocabulary persistent path (verify_full.cu): a request's draw record
// and one (request, slice) result of a draw round.
struct DrawRec {
    int kstar, mode, pass, pad;  // mode 0: residual of position kstar, 1: bonus row
    float4 inv;                  // round 2: 1/S_p and 1/S_q as dd pairs
};
struct alignas(16) DrawPart {  // copied with 16-byte vector loads and stores
    float v[12];
    unsigned namb, pad[3];
};
constexpr int kFullAmb = 16;  // in-band residual elements listed per (request, slice)

struct SampleParams {
    int B, gamma, V, c, Vs;
    const void *target;
    int64_t tstride;
    const void *draft;
    int64_t dstride;
    const int *tokens;
    const float *unif;
    float c2;      // log2(e) / temperature
    float c2lo;    // its rounding residue: c2 + c2lo = log2(e) / temperature to ~2^-48
    DdExpTables exptab;   // 1/T, ln2/64 in parts, 2^(j/64): the double-float exponential
    int top_k;     // 0 = keep all
    float top_p;   // nucleus after top-k when in (0, 1); otherwise off
    float eps;
    int *n_acc, *out_tokens, *n_out;
    float *accept_prob, *resid;
    unsigned *flags;
    unsigned *status, *counters;
    unsigned *rejword;  // [B] earliest rejection seen: gamma - k + 1, 0 = none
    PosRec *recs;       // [B*(gamma+1)]
    // top-k path: per (position, row) slot pos*2 + r, what the pass hands
    // the decision: each thread's maximum (order key) and its four largest
    // groups (key prefix << 16 | chunk), thread-minor
    uint32_t *rkmax;     // [B*(gamma+1)*2][kTopKThreads]
    uint32_t *rkgrp;     // [B*(gamma+1)*2][kTopKGroups][kTopKThreads]
    // and what a row's decision block hands the position's other block
    TopkRow *rkrow;      // [B*(gamma+1)*2]
    uint2 *rkent;        // [B*(gamma+1)*2][kKeptRowMax] (order key, token id), token order
    unsigned *rkcnt;     // [B*(gamma+1)] arrivals, zero between calls
    // full-vocabulary persistent path, c = slices of full_row_bytes()
    float2 *fpart;               // [B*(gamma+1)][2][c] (max, sum) per slice
    float2 *fxd;                 // [B*(gamma+1)] target and draft logit at the draft token
    float4 *fstat;               // [B*(gamma+1)] (M_p, S_p, M_q, S_q)
    unsigned long long *rstate;  // [B] decided / stop bits per position
    unsigned *pcnt;              // [B*(gamma+1)] slice arrivals
    DrawRec *drec;               // [B]
    DrawPart *dpart;             // [B][c]
    unsigned *dcnt;              // [B] draw-round arrivals
    int *amb;                    // [B][c][kFullAmb]
    unsigned long long *qitem;   // [qcap] queue slots
    unsigned qcap;               // 3*B*(slices the workspace was sized for)
    InPlace ip;
    StopRule stop;
    // per-request settings (device [B] or null: the scalars above); when
    // per_request is set the exact cluster path reads them
    const int *rq_gamma;
    const float *rq_temp;
    const int *rq_topk;
    const float *rq_topp;
    int per_request;
    long long idle_limit;  // full-vocabulary path: idle polls before a warp gives up
};


struct CommitParams {
    int B, L, S, bs, unit_bytes, max_blocks, slots_stride;
    int ppu, upp, groups;  // pieces per unit, units per group, groups per token
    const char *temp;
    char *cache;
    int64_t nb;
    const int *table, *slots, *n_slots;
    int *len, *blocks_in_use;
    unsigned *flags, *status, *counters;  // counters: one per request, zero between calls
};

// ---------------------------------------------------------------------------
// draft-tree builder: one level (the parents' draft rows -> children, path
// log-probabilities, next parents)
// ---------------------------------------------------------------------------
constexpr int kTreeMaxHeads = 64, kTreeMaxK = 16, kTreeMaxLevelNodes = 256;
constexpr int kTlSliceElems = 2048;  // logits of a row one warp item covers

struct TlItem {                    // one (row, slice) item's summary
    unsigned long long key[kTreeMaxK];  // its K largest (value, lowest index) keys, 0 = none
    float m, s;                    // slice max and sum of exp(x - m)
    unsigned nan, pad;
};
struct TlRow {                     // one row's result
    int tok[kTreeMaxK];            // top tokens, larger logit first
    float lq[kTreeMaxK];           // their log-softmax values
    unsigned bad, pad[3];
};

struct TreeLevelParams {
    const void *rows;
    int64_t stride;
    int B, V, H, slices, n_nodes, n_next, N, n_before, next_row0, root;
    int koff[kTreeMaxHeads + 1];                // prefix sums of the children counts
    unsigned char head_of[kTreeMaxLevelNodes];  // parent slot of each new node
    const int *parents;
    int *node_token, *node_parent, *row_of_node, *next_parents;
    float *node_logp;
    unsigned *flags, *status;
    TlItem *items;
    TlRow *rowrec;
};
cudaError_t launch_tree_level(const TreeLevelParams &p, int dtype, int kmax, int sms, cudaStream_t s);

cudaError_t launch_argmax_verify(const ArgmaxParams &p, int dtype, int n_rows, int sms, cudaStream_t s);
int argmax_stage_bytes();  // a greedy slice body must fit this
cudaError_t launch_chain_sample(const SampleParams &p, int dtype, cudaStream_t s);
cudaError_t launch_chain_topk(const SampleParams &p, int dtype, int sms, cudaStream_t s);
cudaError_t launch_chain_full(const SampleParams &p, int dtype, int sms, cudaStream_t s);
long long full_idle_limit();  // the default of SampleParams::idle_limit
float full_ex2_bound();       // the hardware exponential's relative error the certified draw assumes
int full_row_bytes();   // one row's slice of the full-vocabulary path
int full_max_slices();  // slices per row it supports
int topk_row_bytes();   // bytes of a row per streamed chunk on the top-k path
struct CommitGeom {
    int ppu, upp, groups;
};
CommitGeom commit_geometry(int L, int64_t unit_bytes);
cudaError_t launch_commit_kv(const CommitParams &p, cudaStream_t s);

}  // namespace specv
