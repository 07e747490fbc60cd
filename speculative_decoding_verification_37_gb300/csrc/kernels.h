// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ddmath.cuh"

namespace specv {

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
};

constexpr int kTopKFastMax = 128;  // top_k served by the candidate-list path

struct SampleParams {
    int B, gamma, V, c, Vs;
    const void *target;
    int64_t tstride;
    const void *draft;
    int64_t dstride;
    const int *tokens;
    const float *unif;
    float c2;      // log2(e) / temperature
    DdExpTables exptab;   // 1/T, ln2/64 in parts, 2^(j/64): the double-float exponential
    int top_k;     // 0 = keep all
    float eps;
    int *n_acc, *out_tokens, *n_out;
    float *accept_prob, *resid;
    unsigned *flags;
    unsigned *status, *counters;
    unsigned *rejword;  // [B] earliest rejection seen: gamma - k + 1, 0 = none
    PosRec *recs;       // [B*(gamma+1)]
    // top-k path: per (position, row, slice) the candidate count with the
    // bound's order key, and a region of kTopKSlicePool (order key, token id)
    // entries, slice stride c
    uint2 *slicecb;      // [B*(gamma+1)][2][c]
    uint2 *pool;         // [B*(gamma+1)][2][c][kTopKSlicePool]
};

constexpr int kTopKSlicePool = 256;  // candidates one slice of one row may hand on
constexpr int kTopKMerge = 4096;     // candidates per row one position can merge

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

cudaError_t launch_argmax_verify(const ArgmaxParams &p, int dtype, int n_rows, int sms, cudaStream_t s);
int argmax_stage_bytes();  // a greedy slice body must fit this
cudaError_t launch_chain_sample(const SampleParams &p, int dtype, cudaStream_t s);
cudaError_t launch_chain_topk(const SampleParams &p, int dtype, int sms, cudaStream_t s);
int topk_row_bytes();  // a top-k slice body per row must fit this
struct CommitGeom {
    int ppu, upp, groups;
};
CommitGeom commit_geometry(int L, int64_t unit_bytes);
cudaError_t launch_commit_kv(const CommitParams &p, cudaStream_t s);

}  // namespace specv
