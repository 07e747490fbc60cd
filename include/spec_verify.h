/*
 * spec_verify.h — C ABI of the batched target-side verify-and-commit step of
 * speculative decoding, built for one GB300 GPU (sm_103a).
 *
 * The step, as the pages define it:
 *   * "10.6 投机解码：为什么“先猜后验”能加速" §10.6.1 (one round): the target
 *     scores [x, d_1..d_gamma] in one forward, giving p_1..p_{gamma+1}; each
 *     draft token d_k is tested left to right and accepted with probability
 *     min(1, p_k(d_k)/q_k(d_k)); the first rejection draws one replacement
 *     from norm(max(0, p_k - q_k)) and drops the rest; if every draft is
 *     accepted a bonus token is drawn from p_{gamma+1}.
 *   * "KV Cache 优化（四）：Speculative Decoding 投机解码" §4: the temperature /
 *     top-k transform is part of p and q; at temperature 0 the rule becomes an
 *     argmax match that emits the target's choice at the first mismatch.
 *   * "投机推理：小模型搭树，大模型一次验证", Validation / 接受过程: a draft tree
 *     is verified by walking one root-to-leaf path, never summing matches
 *     across branches; §10.6.3 Table 10-17: each node attends to its
 *     ancestors only and its position id is its depth.
 *   * "KV Cache 优化（四）" §6 and §10.6.3: the accepted prefix's temporary
 *     K/V is committed at one boundary in every layer, the commit length
 *     advances, rejected slots are rolled back without copying blocks (or,
 *     with reserved slots, the verify call advances the length in place).
 *   * Options of the chain call: top-p after top-k (§4 names it), the early
 *     end of a round at EOS or the length limit (§5).
 *   * The draft side: one level of a topKSpec/topHead draft tree per
 *     spec_tree_level call ("投机推理" 树形投机怎么配置), and prompt-lookup
 *     drafts from the token history (spec_ngram_draft; §10.6.3 实际部署).
 *
 * Conventions for every entry point
 *   * All pointers named "device" are CUDA device (or managed) pointers; the
 *     argument structs themselves live in host memory and are read during
 *     the call only.
 *   * The caller owns every buffer, including the workspace.  The library
 *     never allocates, never synchronises the stream and never creates
 *     streams; each call enqueues its kernels on `stream` (a cudaStream_t,
 *     NULL = legacy default stream) and returns.
 *   * Host-detectable problems return SPEC_ERR_INVALID_ARG or
 *     SPEC_ERR_UNSUPPORTED before anything is enqueued; a failed launch
 *     returns SPEC_ERR_CUDA.  Problems that only the data shows (a token,
 *     node or block id out of range; a row whose kept logits are all -inf)
 *     are found on the device: the request's flags word and the workspace's
 *     sticky status word get a SPEC_FLAG_* bit, the request's outputs are
 *     not written except n_acc = n_out = 0 (and for a commit, nothing is
 *     copied and its length does not advance).  No kernel traps; every wait
 *     on another block's work or on a bulk copy is bounded, and one that
 *     runs out sets SPEC_FLAG_TIMEOUT in the status word.
 *   * Logits must not contain NaN or +inf (-inf is allowed and means "never").
 *   * The workspace must be at least spec_workspace_bytes(...) bytes, 256-byte
 *     aligned and zero-filled before its first use; every call leaves it
 *     zeroed again (except the sticky status word).  Calls sharing one
 *     workspace must be ordered on one stream.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARG 1
#define SPEC_ERR_UNSUPPORTED 2
#define SPEC_ERR_CUDA 3
#define SPEC_ERR_TOO_LARGE 4 /* spec_verify_chain_static: the call needs more than its fixed scratch */

/* logits element types */
#define SPEC_DTYPE_BF16 0
#define SPEC_DTYPE_F32 1

/* per-request flag bits (flags[b]) and sticky status-word bits */
#define SPEC_FLAG_BAD_INPUT 1u  /* token / node / slot / block id out of range: request skipped */
#define SPEC_FLAG_FALLBACK 2u   /* residual mass <= fallback_eps: the draw used p_k itself */
#define SPEC_FLAG_BAD_ROW 4u    /* every kept logit of a row is -inf: request skipped */
#define SPEC_FLAG_TIMEOUT 8u    /* a bulk copy or a wait on other blocks' work did not complete
                                   within its limit (status word only): outputs of the call are
                                   not valid and the workspace must be zeroed again */
#define SPEC_FLAG_EOS 16u       /* the round's output ends with the end-of-sequence token */
#define SPEC_FLAG_LIMIT 32u     /* the round's output was cut at the request's length limit */

/* workspace kinds for spec_workspace_bytes */
#define SPEC_WS_CHAIN 0 /* n = gamma */
#define SPEC_WS_TREE 1  /* n = R (logits rows per request) */
#define SPEC_WS_COMMIT 2
#define SPEC_WS_CHAIN_TOPK 3 /* n = gamma: SPEC_WS_CHAIN plus what the fast top-k path's pass
                                hands its decision and the published kept sets (about 14 KiB per
                                request position) (0 < top_k <= 128) */
#define SPEC_WS_CHAIN_FULL 4 /* n = gamma: SPEC_WS_CHAIN plus the per-slice statistics, draw
                                state and work queue of the persistent full-vocabulary path
                                (top_k == 0; about 2 KiB per request position at V = 128,256) */
#define SPEC_WS_TREE_LEVEL 5 /* n = H (parents a spec_tree_level call expands): one 144-byte
                                summary per (row, 2048-logit slice) and per row */

/*
 * Chain verification, sampled (temperature > 0) or greedy (temperature == 0).
 *
 * Rows: target row (b, k), k = 0..gamma, holds p_{k+1}'s logits at
 *   target_logits + (b*(gamma+1) + k) * target_row_stride elements;
 *   draft row (b, k), k = 0..gamma-1, holds q_{k+1}'s logits at
 *   draft_logits + (b*gamma + k) * draft_row_stride.  Strides are in
 *   elements and >= V; any alignment of the element type is accepted (16-byte
 *   aligned rows are fastest).
 * Transform ("KV Cache 优化（四）" §4): top-k keeps every token whose raw
 *   logit is >= the k-th largest (ties at the threshold are all kept;
 *   top_k == 0 or >= V keeps all), then p_i = exp((l_i - m)/T) / sum over
 *   the kept set.  The draft rows get the same transform.
 * Acceptance (§10.6.1): d_k is accepted iff uniforms[b][k-1] < a_k with
 *   a_k = min(1, p_k(d_k)/q_k(d_k)) (a_k = 1 if q_k(d_k) = 0 < p_k(d_k), 0 if
 *   both are 0).  At the first rejection k: w = max(0, p_k - q_k); if
 *   sum(w) <= fallback_eps, w = p_k (SPEC_FLAG_FALLBACK); the emitted token
 *   is the smallest i with C_i > uniforms[b][gamma] * C_total, C_i = the
 *   running sum of w in token order.  If all are accepted the same rule
 *   draws from p_{gamma+1}.  Exactly one final uniform is used per round.
 * Greedy (temperature == 0): the argmax of each target row (lowest index on
 *   ties) is compared with d_k; draft_logits and uniforms may be NULL.
 *
 * Outputs (device): n_acc[b] in 0..gamma; out_tokens[b][0..n_out-1] = the
 *   accepted drafts then the drawn token (row stride gamma+1); n_out[b] =
 *   n_acc[b] + 1.  Optional (NULL = not written): accept_prob[b][k] = a_k for
 *   every k (sampled only); residual_mass[b][k] = sum max(0, p_k - q_k) for
 *   every k (sampled only; costs a second pass, served from L2, over every
 *   row pair); flags[b].
 * Workspace: spec_workspace_bytes(SPEC_WS_CHAIN, B, gamma, V) bytes suffice
 *   for every call.  Sampled calls with 0 < top_k <= 128 take a faster path
 *   (a maxima-only pass over the rows, then one decision block per row) when
 *   the workspace holds
 *   spec_workspace_bytes(SPEC_WS_CHAIN_TOPK, B, gamma, V) bytes; with less
 *   they take the exact cluster-wide threshold search instead.  Sampled calls
 *   without top-k (and without residual_mass) take a persistent path (one
 *   cooperative kernel: softmax statistics, decisions and the draw, the draw
 *   first in fp32 with a certified error bound, in double-float where the
 *   uniform falls within that bound of a CDF boundary) when the workspace
 *   holds spec_workspace_bytes(SPEC_WS_CHAIN_FULL, B, gamma, V) bytes, rows
 *   and strides are 16-byte aligned, V * element size is a multiple of 16,
 *   gamma <= 30, V * element size <= 1 MiB and the call has at least 1,024
 *   (row, 4 KiB slice) items; otherwise the cluster kernel.  The first such
 *   call on a device first re-measures the error bound of the hardware
 *   exponential that the certified draw assumes (spec_selftest_ex2;
 *   synchronous, about a second: the one place this call synchronises); a
 *   device outside the bound never takes the persistent path, and a call
 *   made while the stream is being captured before that measurement takes
 *   the cluster kernel.
 *   All paths give identical results up to the stated tolerances.
 */
typedef struct SpecChainArgs {
    int32_t B, gamma, V, dtype;
    const void *target_logits;  /* device, [B*(gamma+1)] rows of V logits */
    int64_t target_row_stride;  /* elements */
    const void *draft_logits;   /* device, [B*gamma] rows; NULL when greedy */
    int64_t draft_row_stride;   /* elements */
    const int32_t *draft_tokens; /* device, int32 [B][gamma] */
    const float *uniforms;      /* device, f32 [B][gamma+1] in [0,1); NULL when greedy */
    float temperature;          /* 0 = greedy; otherwise > 0 and finite */
    int32_t top_k;              /* 0 = off */
    float fallback_eps;         /* >= 0; 1e-6 is the documented default */
    int32_t *n_acc;             /* device out [B] */
    int32_t *out_tokens;        /* device out [B][gamma+1] */
    int32_t *n_out;             /* device out [B] */
    float *accept_prob;         /* device out [B][gamma] or NULL */
    float *residual_mass;       /* device out [B][gamma] or NULL */
    uint32_t *flags;            /* device out [B] or NULL */
    /* In-place KV commit ("KV Cache 优化（四）" §6: reserved slots and a
     * commit-length pointer; "10.6 投机解码" §10.6.3: the gamma+1 positions'
     * K/V are in the cache before the verify, the cache length is cut back
     * past a rejection, the draft model's cache rolls back with it).  When
     * committed_len is given, the target forward has written the K/V of the
     * gamma+1 candidates (the last emitted token, then the drafts) at cache
     * positions committed_len[b] .. committed_len[b]+gamma, and this call
     * commits them itself, with no copy and no extra launch:
     *   committed_len[b] += n_out[b]   (that token and the accepted drafts;
     *                                   the rejected ones lie past the new
     *                                   boundary and are simply not kept)
     *   draft_len[b] = min(draft_len[b], committed_len[b])   (the draft
     *                                   cache's length, cut back to the same
     *                                   boundary, never raised)
     *   blocks_in_use[b] = ceil(committed_len[b] / block_size)
     * A request with committed_len[b] < 0, or whose gamma+1 reserved
     * positions pass kv_capacity (> 0) or 2^31-1, is flagged
     * SPEC_FLAG_BAD_INPUT (n_out 0).  A flagged request keeps all three
     * values as they were. */
    int32_t *committed_len;     /* device in/out [B] or NULL (then the rest is ignored) */
    int32_t *draft_len;         /* device in/out [B] or NULL */
    int32_t *blocks_in_use;     /* device out [B] or NULL (needs block_size >= 1) */
    int32_t block_size;         /* tokens per cache block, for blocks_in_use */
    int64_t kv_capacity;        /* positions a request's block table covers; 0 = unchecked */
    /* Early end of the round ("KV Cache 优化（四）" §5: an EOS or the length
     * limit ends a round before its 1..gamma+1 tokens).  The emitted tokens
     * are cut right after the first eos_token (kept), then to max_new[b]
     * tokens (a value <= 0 emits none); n_out is the cut length, n_acc the
     * accepted drafts still emitted, out_tokens entries past n_out are -1
     * where the round would have written them, and flags[b] gets
     * SPEC_FLAG_EOS (the output ends with the EOS) / SPEC_FLAG_LIMIT (the
     * limit cut it).  The in-place commit advances by the cut n_out. */
    int32_t eos_enabled;        /* nonzero: cut after eos_token */
    int32_t eos_token;          /* >= 0 when eos_enabled */
    const int32_t *max_new;     /* device [B] or NULL */
    /* top-p ("KV Cache 优化（四）" §4 names top-p among the processed
     * distributions that enter the acceptance rule): with 0 < top_p < 1,
     * after temperature and top-k each row keeps the smallest set of its
     * most probable tokens whose probability reaches top_p (tokens tied with
     * the least probable kept one are kept too), renormalised; target and
     * draft alike.  With 1 <= top_k <= 128 and a workspace of
     * SPEC_WS_CHAIN_TOPK size it is cut from the fast path's kept set;
     * otherwise the call takes the exact path (below),
     * where any top_k works, 0 included: the nucleus over the full
     * vocabulary.  0 (the zeroed default) or >= 1: off. */
    float top_p;
    /* Per-request settings ("10.6 投机解码" §10.6.3: the requests of one batch
     * accept different lengths and restart at different points; "KV Cache
     * 优化（四）" §4: each request's own processed distributions enter its
     * rule).  Device arrays [B]; NULL = the scalar above for every request.
     * The row layout stays padded to `gamma`: request b uses target rows
     * 0..gamma_b, draft rows and draft tokens 0..gamma_b-1, uniforms
     * u[b][0..gamma_b-1] for its tests and u[b][gamma_b] for its final draw;
     * out_tokens and accept_prob keep the row stride of `gamma`.  A request
     * with temperature 0 is greedy (argmax match, lowest index on ties; its
     * accept_prob entries are 1 or 0 and its residual_mass entries 0).
     * With any of these arrays given (or top_p set without the top-k fast
     * path) the call takes the exact path: one thread-block cluster per
     * position, each request with its own settings; the plain SPEC_WS_CHAIN
     * workspace suffices.  A value out of range (gamma_b outside [0, gamma],
     * a temperature that is negative or not finite, top_k < 0, top_p < 0 or
     * NaN) flags that request SPEC_FLAG_BAD_INPUT. */
    const int32_t *gamma_per_request;       /* device [B] or NULL */
    const float *temperature_per_request;   /* device [B] or NULL */
    const int32_t *top_k_per_request;       /* device [B] or NULL */
    const float *top_p_per_request;         /* device [B] or NULL */
} SpecChainArgs;

int spec_verify_chain(const SpecChainArgs *args, void *workspace, size_t workspace_bytes,
                      void *stream);

/*
 * Greedy tree verification ("投机推理：小模型搭树，大模型一次验证",
 * Validation and 接受过程：沿一条路径走; mask and positions from §10.6.3
 * Table 10-17).
 *
 * Nodes: node 0 is the root (the last emitted token; its K/V is slot 0);
 *   nodes 1..N are drafts with node_token[b][i-1] and node_parent[b][i-1]
 *   (0 <= parent < i, so ids are in breadth-first or any topological order).
 *   row_of_node[b][i] is the logits row scored at node i (-1 = none); row r
 *   of request b is at logits + (b*R + r) * row_stride.
 * Walk: from the root, while the current node has a row, take that row's
 *   argmax t (lowest index on ties) and move to the lowest-id child of the
 *   current node whose token is t; if none matches, t is emitted and the
 *   walk ends; a node without a row ends the walk with no extra token.
 * Outputs (device): path[b][0..n_acc-1] = accepted node ids (row stride N);
 *   n_acc[b]; out_tokens[b][0..n_out-1] = their tokens then the emitted
 *   token if any (row stride N+1); n_out[b].  Optional: tree_mask[b][i][w]
 *   (row stride W = ceil((N+1)/32) words; bit j of word j/32 set iff node j is
 *   node i or an ancestor of it); pos[b][i] = committed_len[b] + depth(i)
 *   (committed_len is then required); commit_slots[b][0..n_commit-1] = root
 *   then the path (row stride N+1) and n_commit[b] = n_acc[b] + 1, ready for
 *   spec_commit_kv; flags[b].
 */
typedef struct SpecTreeArgs {
    int32_t B, N, R, V, dtype;
    const void *logits;          /* device, [B*R] rows */
    int64_t row_stride;          /* elements, >= V */
    const int32_t *node_token;   /* device, int32 [B][N] */
    const int32_t *node_parent;  /* device, int32 [B][N] */
    const int32_t *row_of_node;  /* device, int32 [B][N+1] */
    const int32_t *committed_len; /* device, int32 [B]; may be NULL if pos == NULL */
    int32_t *path;               /* device out [B][N] */
    int32_t *n_acc;              /* device out [B] */
    int32_t *out_tokens;         /* device out [B][N+1] */
    int32_t *n_out;              /* device out [B] */
    uint32_t *tree_mask;         /* device out [B][N+1][W] or NULL */
    int32_t *pos;                /* device out [B][N+1] or NULL */
    int32_t *commit_slots;       /* device out [B][N+1] or NULL */
    int32_t *n_commit;           /* device out [B] or NULL */
    uint32_t *flags;             /* device out [B] or NULL */
} SpecTreeArgs;

int spec_verify_tree(const SpecTreeArgs *args, void *workspace, size_t workspace_bytes,
                     void *stream);

/*
 * KV commit and rollback ("KV Cache 优化（四）" §6; §10.6.3).
 *
 * temp_kv holds each request's temporary K/V: [B][L][2][S][H][D] elements of
 *   elem_bytes bytes (2 for bf16), K at index 0 and V at 1 of the third
 *   dimension.  cache is the paged cache [L][2][num_blocks][block_size][H][D];
 *   block_table[b][j] (row stride max_blocks) is the cache block holding
 *   request b's positions j*block_size .. j*block_size+block_size-1.
 * For i < n_slots[b], slot slots[b][i] (row stride slots_stride; NULL means
 *   slot i) is copied to position committed_len[b] + i in every layer, K and
 *   V alike; then committed_len[b] += n_slots[b].  Slots past n_slots are
 *   never copied: rolling back a rejected draft is not advancing past it.
 *   blocks_in_use[b] (optional) = ceil(new length / block_size): blocks of
 *   the table past it may be released by the caller.
 * Chain rounds pass slots = NULL and n_slots = n_out from spec_verify_chain
 *   (slot 0 = the last emitted token's K/V, slots 1..n_acc = the accepted
 *   drafts); tree rounds pass commit_slots / n_commit from spec_verify_tree.
 * H*D*elem_bytes must be a multiple of 16.  The whole request is skipped
 *   (SPEC_FLAG_BAD_INPUT) if any slot id is outside [0,S), n_slots outside
 *   [0,S], the new length exceeds max_blocks*block_size or a block id it
 *   needs is outside [0,num_blocks).
 * Workspace: spec_workspace_bytes(SPEC_WS_COMMIT, B, 0, 0) bytes (one
 *   arrival counter per request), zero before the first call; every call
 *   leaves it zero.
 */
typedef struct SpecCommitArgs {
    int32_t B, L, H, D, S, block_size, elem_bytes;
    const void *temp_kv;         /* device, [B][L][2][S][H][D] */
    void *cache;                 /* device, [L][2][num_blocks][block_size][H][D] */
    int64_t num_blocks;
    const int32_t *block_table;  /* device, int32 [B][max_blocks] */
    int32_t max_blocks;
    const int32_t *slots;        /* device, int32 [B][slots_stride] or NULL (identity) */
    int32_t slots_stride;        /* >= S when slots != NULL */
    const int32_t *n_slots;      /* device, int32 [B] */
    int32_t *committed_len;      /* device, int32 [B], in/out */
    int32_t *blocks_in_use;      /* device out [B] or NULL */
    uint32_t *flags;             /* device out [B] or NULL (bits are OR-ed in) */
} SpecCommitArgs;

int spec_commit_kv(const SpecCommitArgs *args, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * spec_verify_chain_static — spec_verify_chain for callers that cannot
 * allocate device memory.  The pages have no counterpart; this is a
 * deployment variant of the same computation.
 *
 * Some callers cannot call cudaMalloc where they verify a round: code
 * running under a memory-pool or arena allocator that owns every device
 * byte, plug-ins whose host framework forbids allocation on its hot path,
 * and callers that must avoid an allocation's implicit synchronisation.
 * This call takes the same arguments as spec_verify_chain minus the
 * workspace: its scratch (arrival counters, rejection words, per-position
 * records) is a fixed array of SPEC_STATIC_WORKSPACE_BYTES compiled into the
 * library, resident on every GPU that loads it until the process exits.
 *
 *   * Inputs and outputs are still the caller's device buffers, exactly as
 *     for spec_verify_chain, and the results are identical to it.
 *   * It allocates nothing (no cudaMalloc, cudaFree or allocating library
 *     routine).  It enqueues one small memset of the zero-initialised part
 *     of the array, then the verify kernel, on `stream`.
 *   * The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   * All calls on one GPU share the array and it keeps the last call's
 *     contents: calls whose kernels could overlap on the GPU race on it, so
 *     order them on one stream.
 *   * A call needing more scratch than the array holds (see
 *     spec_workspace_bytes(SPEC_WS_CHAIN, B, gamma, V)) returns
 *     SPEC_ERR_TOO_LARGE.  1 MiB covers, e.g.,
 *     B = 4096 requests at gamma = 8.
 *   * There is no status word to read back: data errors show in flags[b].
 *   * The array holds the plain chain workspace only, without the top-k
 *     path's candidate regions or the full-vocabulary path's state: sampled
 *     calls take the exact cluster path (top-k by its exact threshold
 *     search, top-p and per-request settings included; same results,
 *     slower).
 *   * Every argument check (SPEC_ERR_TOO_LARGE included) returns before
 *     anything is enqueued.
 */
#define SPEC_STATIC_WORKSPACE_BYTES (1u << 20)
int spec_verify_chain_static(const SpecChainArgs *args, void *stream);

/* Workspace bytes for a call of the given kind (n = gamma for SPEC_WS_CHAIN,
 * R for SPEC_WS_TREE, ignored for SPEC_WS_COMMIT).  Returns 0 for an unknown
 * kind or negative sizes. */
size_t spec_workspace_bytes(int kind, int32_t B, int32_t n, int32_t V);

/* Reads (and clears) the workspace's sticky status word: enqueues a copy on
 * `stream`, synchronises that stream, then enqueues the clear.  This is the
 * one call that synchronises. */
int spec_get_status(void *workspace, void *stream, uint32_t *host_flags);

/* Human-readable text for a return code. */
const char *spec_error_string(int code);

/* Text of the last CUDA error a call of this library saw on this thread. */
const char *spec_last_cuda_error(void);

/* How many idle polls (about 0.5 us each) a warp of the persistent
 * full-vocabulary chain path makes, while none of its work is ready, before
 * it gives up: it leaves once the copies it has in flight have landed, and
 * the call sets SPEC_FLAG_TIMEOUT (its outputs are then not valid and the
 * workspace must be zeroed again).  polls <= 0 restores the default, 2^21
 * (about a second).  Process-wide, read when a call is made; meant for
 * tests of the timeout path.  Always SPEC_OK.  (The pages have no
 * counterpart: this bounds a wait of this implementation.) */
int spec_set_idle_limit(int64_t polls);

/*
 * N-gram (prompt-lookup) drafts, a model-free draft source ("10.6 投机解码"
 * §10.6.3 实际部署; "KV Cache 优化（四）" §10.2 N-gram 或前缀匹配): for each
 * request, the longest n in [n_min, n_max] whose trailing n-gram of the
 * history occurs earlier (an occurrence starting before the trailing n-gram
 * itself), the most recent such occurrence, and the up to gamma tokens that
 * follow it (never past the end of the history).  No occurrence gives an
 * empty draft.
 *
 * history: device int32; request b's tokens start at history + b *
 *   history_stride, hist_len[b] of them (0 <= hist_len[b] <= history_stride).
 * Outputs (device): draft_tokens[b][0..gamma) (row stride gamma; entries past
 *   n_draft[b] are -1), n_draft[b]; optional (NULL = not written): match_n[b]
 *   (the n used, 0 if none), match_start[b] (-1 if none), flags[b].
 * Errors: SPEC_ERR_INVALID_ARG for B < 0, gamma < 0, n_min < 1,
 *   n_max < n_min, n_max > 64, history_stride < 1 or a NULL required pointer
 *   (nothing is launched); a hist_len[b] outside [0, history_stride] gives
 *   n_draft[b] = 0, SPEC_FLAG_BAD_INPUT in flags[b] (if given), and that
 *   request only is skipped.  Asynchronous on `stream`; no workspace.
 */
typedef struct SpecNgramArgs {
    int32_t B, gamma, n_min, n_max;
    const int32_t *history;     /* device, int32 [B][history_stride] */
    int64_t history_stride;     /* elements */
    const int32_t *hist_len;    /* device, int32 [B] */
    int32_t *draft_tokens;      /* device out [B][gamma] */
    int32_t *n_draft;           /* device out [B] */
    int32_t *match_n;           /* device out [B] or NULL */
    int32_t *match_start;       /* device out [B] or NULL */
    uint32_t *flags;            /* device out [B] or NULL */
} SpecNgramArgs;

int spec_ngram_draft(const SpecNgramArgs *args, void *stream);

/*
 * One level of a draft tree ("投机推理：小模型搭树，大模型一次验证",
 * 树形投机怎么配置 and its three expansion steps; the real dump example).  The
 * draft model has run once at each of this level's H parents; for every
 * request b this call
 *   - gives parent j (row b*H + j of `logits`) the k[j] tokens with the
 *     largest logits as children (ties to the lower token id), numbered
 *     n_before+1, n_before+2, ... in parent order, then rank order;
 *   - sets each child's path log-probability to its parent's plus the draft's
 *     log-softmax (temperature 1) at its token;
 *   - picks the n_next children with the highest path log-probability (ties
 *     to the lower node id) as the next level's parents, written in id order
 *     to next_parents[b], and gives them logits rows next_row0, next_row0+1,
 *     ... in row_of_node (every other new node gets -1).
 * The root's level passes parents = NULL and H = 1; it also writes node 0's
 * log-probability (0) and row (0).  A full tree is built by calling this once
 * per level with that level's draft rows, passing the previous call's
 * next_parents as `parents`.
 *
 * Layout: node_token/node_parent [B][N] hold node id i at index i-1;
 *   node_logp/row_of_node [B][N+1] are indexed by node id (the root is 0).
 *   These are in/out: the call reads the parents' log-probabilities and
 *   writes only the new nodes' entries (and the chosen nodes' rows).
 * Limits: 1 <= H <= 64, 1 <= k[j] <= min(16, V), sum(k) <= 256,
 *   0 <= n_next <= min(64, sum(k)), n_before + sum(k) <= N.
 * Errors: SPEC_ERR_INVALID_ARG for arguments outside those limits, a NULL
 *   required pointer, a misaligned row or a short workspace (nothing is
 *   launched).  A parent id outside [0, n_before] flags SPEC_FLAG_BAD_INPUT,
 *   a row holding a NaN or with no finite maximum SPEC_FLAG_BAD_ROW; such a
 *   request writes no nodes, its next_parents are -1 (so the next level
 *   flags it too) and its flags[b] gets the bit.
 * Workspace: spec_workspace_bytes(SPEC_WS_TREE_LEVEL, B, H, V) bytes (no
 *   zeroing needed; calls sharing it must be ordered on one stream).
 *   Asynchronous on `stream` (two launches, the second a programmatic
 *   dependent of the first).
 */
#define SPEC_TREE_MAX_HEADS 64
#define SPEC_TREE_MAX_K 16
#define SPEC_TREE_MAX_LEVEL_NODES 256
typedef struct SpecTreeLevelArgs {
    int32_t B, V, dtype;
    int32_t H;                          /* parents expanded at this level */
    int32_t k[SPEC_TREE_MAX_HEADS];     /* k[j]: children of parent j (j < H) */
    int32_t n_next;                     /* parents the next level expands (0: last level) */
    int32_t N;                          /* nodes the per-request arrays hold */
    int32_t n_before;                   /* nodes already in the tree */
    int32_t next_row0;                  /* logits rows given out so far, this level's included */
    const void *logits;                 /* device [B*H rows][V], bf16 or f32 */
    int64_t row_stride;                 /* elements between rows (>= V) */
    const int32_t *parents;             /* device [B][H], ascending node ids; NULL at the root */
    int32_t *node_token;                /* device in/out [B][N] */
    int32_t *node_parent;               /* device in/out [B][N] */
    float *node_logp;                   /* device in/out [B][N+1] */
    int32_t *row_of_node;               /* device in/out [B][N+1] */
    int32_t *next_parents;              /* device out [B][n_next] (may be NULL if n_next == 0) */
    uint32_t *flags;                    /* device in/out [B] (bits OR'ed in) or NULL */
} SpecTreeLevelArgs;

int spec_tree_level(const SpecTreeLevelArgs *args, void *workspace, size_t ws_bytes, void *stream);

/* Diagnostic: the largest relative error of the GPU's hardware exponential
 * (ex2.approx.ftz.f32) against fp64 over every fp32 input in [-126, 1], on the
 * current device.  The full-vocabulary path's certified fp32 draw assumes
 * 1.5e-7; a larger value means that path's certification is not valid on this
 * device.  Synchronous (about a second of GPU time); SPEC_ERR_CUDA on a CUDA
 * error. */
int spec_selftest_ex2(float *max_rel_err);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
