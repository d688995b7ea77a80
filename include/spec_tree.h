/*
 * spec_tree.h -- C ABI of a GB300 (sm_103a) library for one tree-verification
 * step of Medusa/Hydra speculative decoding: draft heads fill a candidate tree,
 * the tree tokens attend over a KV-cache prefix plus their own ancestors, and
 * acceptance picks the longest accepted path (greedy, or the min(1, p/q) rule
 * with residual resampling).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - The caller owns every buffer, device scratch ("workspace") included; its
 *    size comes from the matching *_workspace_size call.  Apart from
 *    spec_tree_build (which copies a small host table to the device and waits
 *    for it) no call allocates, frees or synchronises; all work is queued on
 *    the given stream in order.  0 selects the legacy default stream.  A
 *    sequence of calls on one stream can therefore be captured into a CUDA
 *    graph (make one call first, outside the capture, so that one-time setup
 *    such as kernel attributes happens there) and replayed: the replay
 *    repeats the same work on the same buffers without the per-call host
 *    work.  spec_read_device_status synchronises and is not capturable.
 *    Some kernels launch as programmatic dependents of the kernel before
 *    them on the stream; they wait for it before reading anything it could
 *    have written.
 *  - "device" pointers must point to memory of the current CUDA device and be
 *    16-byte aligned (SPEC_EALIGN otherwise); "host" pointers are read during
 *    the call only.
 *  - Every call checks its arguments on the host before it queues anything.
 *    On failure it returns a non-zero spec_status, queues nothing, writes no
 *    output, and spec_last_error() describes the problem (per host thread).
 *    CUDA launch errors are reported as SPEC_ECUDA.
 *  - Kernels never trap and never wait without bound.  A failure detected on
 *    the device (a bounded wait that ran out, a token or page index out of
 *    range) is recorded in the first 16 bytes of the call's workspace;
 *    spec_read_device_status() returns it.  Each call clears those bytes
 *    before its kernels can record anything (any prior content, including
 *    garbage in a fresh workspace, is discarded), so a workspace may be reused
 *    by any later call on the same stream.
 *  - Tokens are int32, logits and outputs float32; inputs of the float tensors
 *    of a call share one spec_dtype (float32 or bfloat16 bit patterns).
 *  - Tensor shapes are given outermost first and are densely packed (row-major).
 */
#ifndef SPEC_TREE_H
#define SPEC_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t); declared opaquely so this header needs no CUDA headers. */
typedef struct CUstream_st* spec_stream_t;

typedef enum {
    SPEC_OK = 0,
    SPEC_EINVAL = 1,       /* bad argument: null pointer, size out of range, shape mismatch */
    SPEC_ETREE = 2,        /* malformed tree: parent[0] != -1, parent[i] not in [0, i), duplicate sibling rank */
    SPEC_EALIGN = 3,       /* a device pointer is not 16-byte aligned */
    SPEC_EWORKSPACE = 4,   /* workspace missing or smaller than *_workspace_size */
    SPEC_EUNSUPPORTED = 5, /* a valid combination this build does not implement */
    SPEC_ECUDA = 6,        /* a CUDA runtime call or launch failed */
    SPEC_ETIMEOUT = 7      /* device status only: a bounded wait inside a kernel ran out */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

#define SPEC_MAX_T 1024      /* tree nodes, root included */
#define SPEC_MAX_DEPTH 16    /* deepest node; also the most draft heads */
#define SPEC_MAX_TOPK 16     /* largest top-k per head */

/*
 * Candidate tree, encoded once per topology by spec_tree_build.
 *
 * Hydra Guide: Sequentially-Dependent Speculative AI, sections "Candidate Tree
 * Construction" (the root is the base token x_t; a depth-k node holds a token
 * proposed by head k; rank = which of the parent head's top-k candidates it
 * is) and "Tree Attention Matrix with Topology-Aware Causal Masking" (the tree
 * is flattened into one sequence; node u may attend to node v iff v is an
 * ancestor of u or v = u).
 *
 * Host fields are filled by spec_tree_build; the pointers point into the
 * caller's device buffer and stay valid as long as that buffer does.
 */
typedef struct {
    int32_t T;                                   /* nodes, root (node 0) included */
    int32_t max_depth;                           /* largest depth (root: 0) */
    int32_t words;                               /* ceil(T / 64): 64-bit words per ancestor mask */
    int32_t n_internal;                          /* nodes that have at least one child */
    int32_t n_at_depth[SPEC_MAX_DEPTH + 1];      /* host: nodes of each depth */
    int32_t n_internal_at_depth[SPEC_MAX_DEPTH + 1]; /* host: nodes of each depth that have children */
    int32_t max_rank_at_depth[SPEC_MAX_DEPTH + 1];   /* host: largest rank among nodes of each depth (depth >= 1) */
    const int32_t* parent;        /* device [T]; parent[0] = -1, parent[i] < i */
    const int32_t* depth;         /* device [T] */
    const int32_t* rank;          /* device [T]; 0 for the root */
    const uint64_t* anc;          /* device [T][words]; bit j of row i set iff j is i or an ancestor of i */
    const int32_t* internal;      /* device [n_internal]: nodes with children, by depth then index */
    const int32_t* internal_off;  /* device [SPEC_MAX_DEPTH + 2]: depth d's nodes start at internal[internal_off[d]] */
    const int32_t* row_of;        /* device [T]: position of a node within its depth's internal list, -1 for leaves */
    const int32_t* child_off;     /* device [T + 1]: children of u are child_idx[child_off[u] .. child_off[u+1]) */
    const int32_t* child_idx;     /* device [max(T - 1, 1)], ascending per parent */
} spec_tree;

/* Bytes of device memory spec_tree_build needs for a tree of T nodes (0 if T is out of range). */
size_t spec_tree_device_bytes(int32_t T);

/*
 * Validate a parent-index tree and encode it for the other calls.
 *   parent  host [T]: parent[0] = -1, 0 <= parent[i] < i.
 *   rank    host [T] or NULL: rank[i] >= 0 is node i's slot among its parent
 *           head's top-k (0 = most probable); distinct among siblings.  NULL
 *           numbers each node's children 0, 1, ... in index order.
 *   T       1 .. SPEC_MAX_T; the tree's depth must be <= SPEC_MAX_DEPTH.
 *   d_buf   device buffer of at least spec_tree_device_bytes(T) bytes.
 *   out     host struct filled on success.
 * Copies the encoded tables to d_buf on stream s and waits for that copy.
 */
spec_status spec_tree_build(const int32_t* parent, const int32_t* rank, int32_t T,
                            void* d_buf, size_t d_bytes, spec_tree* out, spec_stream_t s);

/* Workspace bytes hydra_draft needs for these shapes (0 on invalid arguments). */
size_t hydra_draft_workspace_size(const spec_tree* tree, int32_t B, int32_t d, int32_t V, int32_t K,
                                  const int32_t* cond, const int32_t* topk, spec_dtype dt);

/*
 * Draft heads: fill every candidate node of every sequence with a token.
 *
 * Medusa Heads (ultralytics glossary), section "So sagen die Köpfe voraus": a
 * head is one feed-forward layer with SiLU and a residual, then a projection
 * onto the vocabulary.  Hydra Guide, sections "1. Embedding Conditioning
 * Mechanics" and "Candidate Tree Construction": a sequentially dependent head
 * also reads the base-embedding row of its parent node's token, and each
 * node's children are the top-k of the head run on that node.  Per head k
 * (filling depth k + 1) and parent node u of sequence b:
 *     u_in = h_b                     if cond[k] == 0   (W1[k] is [d, d])
 *     u_in = [h_b || emb[tok(u)]]    if cond[k] == 1   (W1[k] is [d, 2d])
 *     u_in = [h_b || emb[tok(a_1)] || ... || emb[tok(a_k)]]   if cond[k] == 2
 *            (a_1 .. a_k = u's path below the root, depth 1 first; W1[k] is
 *            [d, (k+1) d]; Hydra Guide, "2. Generalizing to Arbitrary Tree Depths")
 *     z    = h_b + SiLU(W1[k] u_in + b1[k])   (rounded to bf16 when dt is bf16)
 *     l    = W2[k] z                 ([V] logits, never written to memory)
 * A child of rank r gets the (r+1)-th largest logit (ties: lower token id).
 *
 *   h          device [B, d]                 hidden state of each sequence
 *   emb        device [V, d]                 base token-embedding table
 *   K          number of heads, >= tree->max_depth, <= SPEC_MAX_DEPTH
 *   W1, b1, W2 host arrays [K] of device pointers: W1[k] [d, d_in_k] (out x in),
 *              b1[k] [d] (a NULL entry or a NULL array means no bias), W2[k] [V, d]
 *   cond, topk host [K]: cond[k] in {0, 1, 2}; topk[k] in 1 .. SPEC_MAX_TOPK and
 *              > the largest rank among depth-(k+1) nodes
 *   root_tok   device [B]                     token of node 0 (the base token x_t)
 *   node_tok   device [B, T] out: node 0 = root_tok, others = drafted tokens
 *   node_logit device [B, T] out: the node's logit in its parent's row (root: 0)
 *   node_logprob device [B, T] out or NULL: cumulative log-probability along
 *              the node's path, log-softmax of each row (root: 0)
 * Shapes: 1 <= B, d % 8 == 0, 1 <= d <= 16384, topk[k] <= V <= 2^24.
 */
spec_status hydra_draft(const void* h, const void* emb, int32_t K,
                        const void* const* W1, const void* const* b1, const void* const* W2,
                        const int32_t* cond, const int32_t* topk, const int32_t* root_tok,
                        const spec_tree* tree, int32_t B, int32_t d, int32_t V, spec_dtype dt,
                        int32_t* node_tok, float* node_logit, float* node_logprob,
                        void* ws, size_t ws_bytes, spec_stream_t s);

/* Bytes of one folded embedding table (V * d fp32), 0 on invalid shapes. */
size_t hydra_fold_table_bytes(int32_t d, int32_t V);

/*
 * Fold the embedding half of a cond-1 head's first layer into a per-token
 * table, once per set of weights (not per step).  Hydra Guide, "1. Embedding
 * Conditioning Mechanics": the head reads u_in = [h_b || emb[tok]], so
 *     W1 u_in = W1[:, 0:d] h_b + tab[tok],   tab[v, m] = sum_j W1[m, d + j] emb[v, j]
 * and the second term depends on the token alone.
 *
 *   W1   device [d, 2d] in dt (the head's first layer, out x in)
 *   emb  device [V, d] in dt
 *   tab  device fp32 [V, d] out (hydra_fold_table_bytes bytes, caller-owned)
 * fp32 accumulation in a fixed order per element: bf16 inputs on the tensor
 * cores (256 vocabulary rows per launch), fp32 inputs on the CUDA cores.  All
 * pointers 16-byte aligned (SPEC_EALIGN); SPEC_EINVAL on NULL or out-of-range
 * shapes.  Launched on s, asynchronous.  The call has no workspace, so no
 * device status: its kernels' bounded waits cannot run out unless the GPU
 * stops making progress, and then the table is left undefined.
 */
spec_status hydra_fold_embedding(const void* W1, const void* emb, int32_t d, int32_t V, spec_dtype dt,
                                 float* tab, spec_stream_t s);

/*
 * hydra_draft with folded first layers: tab is a host array [K] (or NULL) of
 * device tables from hydra_fold_embedding(W1[k], emb, ...).  On the bf16
 * tensor-core path a cond-1 head with a table streams only W1[k][:, 0:d] per
 * step: a[b] = W1[k][:, 0:d] h_b, and the kernel that picks a node's token
 * writes that node's head input z = h_b + SiLU(a[b] + tab[k][tok] + b1[k])
 * itself.  NULL entries, other heads and the fp32 path use the whole W1[k].
 * The results equal hydra_draft's up to fp32 rounding order.  Workspace:
 * hydra_draft_workspace_size.  Tables must be 16-byte aligned (SPEC_EALIGN);
 * everything else as hydra_draft.
 */
spec_status hydra_draft_folded(const void* h, const void* emb, int32_t K,
                               const void* const* W1, const void* const* b1, const void* const* W2,
                               const float* const* tab, const int32_t* cond, const int32_t* topk,
                               const int32_t* root_tok, const spec_tree* tree, int32_t B, int32_t d,
                               int32_t V, spec_dtype dt, int32_t* node_tok, float* node_logit,
                               float* node_logprob, void* ws, size_t ws_bytes, spec_stream_t s);

/*
 * One draft head for hydra_draft_heads.  form 0 is hydra_draft's head; form 1
 * is the head form that the Hydra Guide prints as code (fusion MLP
 * Linear -> SiLU -> Linear -> LayerNorm, then a bias-free vocabulary
 * projection; its first head Linear -> SiLU -> LayerNorm, i.e. no W1b):
 *   form 0: z = h_b + SiLU(W1 u_in + b1)                         (hidden == d)
 *   form 1: y = W1b SiLU(W1 u_in + b1) + b1b, or y = SiLU(W1 u_in + b1) when
 *           W1b is NULL (then hidden == d);
 *           z = (y - mean(y)) / sqrt(var(y) + ln_eps) * gamma + beta
 *           (mean and biased variance over the d entries of y)
 * then l = W2 z as in hydra_draft.  u_in follows cond exactly as in
 * hydra_draft; with dt bf16, SiLU(W1 u_in + b1) is rounded to bf16 when it
 * feeds W1b, and z is rounded to bf16.
 */
typedef struct {
    int32_t cond;         /* 0, 1 or 2 (hydra_draft) */
    int32_t topk;         /* 1 .. SPEC_MAX_TOPK (hydra_draft) */
    int32_t form;         /* 0 or 1 */
    int32_t hidden;       /* rows of W1: d for form 0 and for form 1 without W1b */
    const void* W1;       /* device [hidden, d_in] */
    const void* b1;       /* device [hidden] or NULL */
    const void* W1b;      /* form 1: device [d, hidden] or NULL */
    const void* b1b;      /* form 1: device [d] or NULL */
    const void* gamma;    /* form 1: device [d] or NULL (ones) */
    const void* beta;     /* form 1: device [d] or NULL (zeros) */
    const void* W2;       /* device [V, d] (heads may share one) */
} spec_head;

/* Workspace bytes hydra_draft_heads needs (0 on invalid arguments). */
size_t hydra_draft_heads_workspace_size(const spec_tree* tree, int32_t B, int32_t d, int32_t V, int32_t K,
                                        const spec_head* heads, spec_dtype dt);

/*
 * hydra_draft with a per-head description (heads: host array [K]); ln_eps > 0
 * is the LayerNorm epsilon of form-1 heads.  Everything else as hydra_draft.
 */
spec_status hydra_draft_heads(const void* h, const void* emb, int32_t K, const spec_head* heads,
                              const int32_t* root_tok, const spec_tree* tree, int32_t B, int32_t d, int32_t V,
                              float ln_eps, spec_dtype dt, int32_t* node_tok, float* node_logit,
                              float* node_logprob, void* ws, size_t ws_bytes, spec_stream_t s);

/* Workspace bytes tree_attention needs for these shapes on the current device (0 on invalid arguments). */
size_t tree_attention_workspace_size(const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv,
                                     int32_t Lmax, int32_t D, spec_dtype dt);

/*
 * Tree attention of one layer.
 *
 * Hydra Guide, section "Tree Attention Matrix with Topology-Aware Causal
 * Masking": every tree token sees the whole cached prefix and, among the tree
 * tokens, only itself and its ancestors (M_tree = 0 there, -inf elsewhere), so
 * its output equals autoregressive attention over [prompt, ancestors, itself].
 * For query head h (KV head h / (Hq / Hkv)), sequence b and node i:
 *     keys  = k_cache[b, :prefix_len[b]] followed by k_tree[b, a] for a in anc*(i)
 *     out   = softmax(scale * q . keys) . values,  lse = log(sum exp(scale * q . keys))
 *
 *   q                 device [B, Hq, T, D]
 *   k_cache, v_cache  device [B, Hkv, Lmax, D]; rows >= prefix_len[b] do not affect the
 *                     result (the tensor-core path reads, then discards, those inside
 *                     the last 128-key tile of a sequence: they must be readable memory)
 *   prefix_len        device [B], each in 0 .. Lmax (values outside are clamped to it)
 *   k_tree, v_tree    device [B, Hkv, T, D]: keys/values of the tree tokens
 *   scale             > 0, or 0 for the usual 1/sqrt(D)
 *   out               device [B, Hq, T, D] float32
 *   lse               device [B, Hq, T] float32, or NULL
 * Shapes: Hq % Hkv == 0, D in {64, 128}, 1 <= Lmax <= 2^22.
 */
spec_status tree_attention(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* prefix_len, const void* k_tree, const void* v_tree,
                           const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax,
                           int32_t D, float scale, spec_dtype dt, float* out, float* lse,
                           void* ws, size_t ws_bytes, spec_stream_t s);

/*
 * tree_attention without a caller-provided workspace.  The pages have no
 * counterpart to this call: it exists for callers that cannot allocate device
 * memory, such as a plugin running inside a host engine that has already
 * handed out the device memory and forbids further cudaMalloc calls, or a
 * caller whose own interface has no way to pass a workspace pointer through.
 *
 * Arguments, results and errors are those of tree_attention without ws and
 * ws_bytes.  The scratch is a 32 MiB array inside this library's device image
 * (every GPU that loads the library holds it until the process exits); shapes
 * whose tree_attention_workspace_size exceeds 32 MiB are rejected with
 * SPEC_EWORKSPACE before anything is queued.  The call allocates nothing.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array and it keeps the
 * last call's contents (each call clears what must start at zero): calls
 * whose work overlaps on the GPU -- on different streams, or from different
 * host threads -- race on it and must not be issued.  A failure the kernels
 * detect (a bounded wait that ran out) goes to the status word at the start
 * of the built-in array; tree_attention_noalloc_status reads it.
 */
spec_status tree_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* prefix_len, const void* k_tree, const void* v_tree,
                                   const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv, int32_t Lmax,
                                   int32_t D, float scale, spec_dtype dt, float* out, float* lse, spec_stream_t s);

/*
 * Device status of the calls that use the built-in scratch (tree_attention_noalloc):
 * the counterpart of spec_read_device_status for a caller workspace.  Waits on
 * stream s for the calls queued before it, copies the status word of the
 * built-in array to *status (host) and returns SPEC_OK, or an error status
 * when the copy fails.  Like tree_attention_noalloc, it looks up the array's
 * address with the current device and allocates nothing.
 */
spec_status tree_attention_noalloc_status(int32_t* status, spec_stream_t s);

/* Workspace bytes tree_attention_paged needs (0 on invalid arguments). */
size_t tree_attention_paged_workspace_size(const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv,
                                           int32_t max_blocks, int32_t block_size, int32_t D, spec_dtype dt);

/*
 * Tree attention over a paged KV cache -- Hydra Guide, "Hydra Production
 * Engineering Checklist", item 3 (KV-Cache Tree Branch Management: the tree
 * attention KV cache lives in pre-allocated static blocks).  The same result
 * as tree_attention with k_cache[b, :, j] = k_pool[block_table[b, j / block_size],
 * :, j % block_size] (likewise V).
 *
 *   k_pool, v_pool  device [num_blocks, Hkv, block_size, D]
 *   block_table     device [B, max_blocks] int32: pool block of positions
 *                   j*block_size .. (j+1)*block_size - 1 of sequence b; only the
 *                   first ceil(prefix_len[b] / block_size) entries are read
 *   prefix_len      device [B], each in 0 .. max_blocks * block_size (clamped)
 *   block_size      a positive multiple of 64; max_blocks * block_size <= 2^22
 *   the rest as tree_attention.
 * A table entry outside 0 .. num_blocks-1 is reported as SPEC_EINVAL in the
 * status word and its keys read as zeros (no memory outside the pool is read).
 */
spec_status tree_attention_paged(const void* q, const void* k_pool, const void* v_pool, int32_t num_blocks,
                                 const int32_t* block_table, int32_t max_blocks, int32_t block_size,
                                 const int32_t* prefix_len, const void* k_tree, const void* v_tree,
                                 const spec_tree* tree, int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                 float scale, spec_dtype dt, float* out, float* lse, void* ws,
                                 size_t ws_bytes, spec_stream_t s);

/* Workspace bytes tree_accept (mode 0 or 1) or tree_accept_typical (mode 2) needs (0 on invalid arguments). */
size_t tree_accept_workspace_size(int32_t mode, const spec_tree* tree, int32_t B, int32_t V);

/*
 * Acceptance: longest accepted path and the extra token.
 *
 * mode 0, greedy -- Hydra Guide, section "Parallel Verification and Greedy
 *   Acceptance Algorithm": a(u) = argmax logits_p[b, u] (ties: lower id); a
 *   node is accepted when its parent is and its token equals a(parent); the
 *   deepest accepted node u* (lowest index on equal depth) ends the path and
 *   a(u*) is the extra token.  temperature, seed, offset and logits_q unused.
 * mode 1, rejection -- Speculative Decoding (thegustafson.com), sections "The
 *   acceptance criterion", "The correctness guarantee" and "A worked example":
 *   p_u = softmax(logits_p[b, u] / temperature), q_u likewise from logits_q;
 *   the edge into node c with token x is accepted iff u_c < p_par(x) / q_par(x);
 *   u* as above; the extra token is drawn from norm(max(p_u* - q_u*, 0)) when u*
 *   has children (from p_u* if that residual is zero), else from p_u*, by
 *   inverse CDF in ascending token order with uniform u'.  u_c is word 0 and u'
 *   word 1 of Philox4x32-10 (Salmon et al., SC'11) with key (seed low, seed
 *   high) and counter (node, b, offset low, offset high) -- u' from node 0 --
 *   each word w mapped to (w >> 8) * 2^-24.
 *
 *   logits_p     device [B, T, V] float32 target logits (row u predicts the token after u)
 *   logits_q     device [B, T, V] float32 draft logits (rejection; rows of leaves not read) or NULL
 *   node_tok     device [B, T]
 *   accept_len   device [B] out: m, the depth of u*
 *   accept_path  device [B, max_depth + 1] out: node ids root first, -1 padded
 *   next_token   device [B] out: the extra token
 *   margin       device [B] out or NULL: distance of the closest decision to its
 *                threshold (greedy: smallest top-1 minus top-2 logit gap over accepted
 *                nodes; rejection: smallest |u_c - ratio| over decided edges with
 *                ratio < 1, or the sampling draw's distance to a CDF breakpoint over the total)
 * Shapes: 2 <= V <= 2^24; temperature > 0 for mode 1.
 */
spec_status tree_accept(int32_t mode, const float* logits_p, const float* logits_q, const int32_t* node_tok,
                        const spec_tree* tree, int32_t B, int32_t V, float temperature,
                        uint64_t seed, uint64_t offset, int32_t* accept_len, int32_t* accept_path,
                        int32_t* next_token, float* margin, void* ws, size_t ws_bytes, spec_stream_t s);

/*
 * Typical acceptance -- Medusa Heads (ultralytics glossary), section "Tree
 * Attention und Akzeptanz": for sampling, a candidate is kept when its
 * probability under the base model exceeds a threshold tied to the entropy of
 * that distribution (more tokens accepted, the distribution no longer exact;
 * Speculative Decoding, section "Beyond draft models: Medusa").  The pages give
 * neither the formula nor the constants; this call takes
 *     p_u = softmax(logits_p[b, u] / temperature),  H_u = -sum_x p_u(x) ln p_u(x),
 *     the edge into node c with token x is accepted iff p_par(x) > min(epsilon, alpha * exp(-H_par)),
 * u* = the deepest accepted node (lowest index on equal depth), and the extra
 * token drawn from p_u* by inverse CDF in ascending token order with the
 * uniform u' of tree_accept (word 1 of Philox4x32-10, counter (0, b, offset)).
 *
 *   margin  device [B] out or NULL: the smallest |p_par(x) / threshold - 1| over
 *           edges with an accepted parent, or the draw's distance to a CDF
 *           breakpoint over the total, whichever is smaller
 *   the rest as tree_accept; epsilon, alpha >= 0 and finite, temperature > 0;
 *   the workspace is tree_accept_workspace_size(2, ...).
 */
spec_status tree_accept_typical(const float* logits_p, const int32_t* node_tok, const spec_tree* tree,
                                int32_t B, int32_t V, float temperature, float epsilon, float alpha,
                                uint64_t seed, uint64_t offset, int32_t* accept_len, int32_t* accept_path,
                                int32_t* next_token, float* margin, void* ws, size_t ws_bytes, spec_stream_t s);

/*
 * The uniforms tree_accept draws, for inspection: u_accept [B, T] (entry
 * [b, c] = word 0 of counter (c, b, offset)), u_sample [B] (word 1 of counter
 * (0, b, offset)).  Device pointers.  Salmon et al., SC'11, Philox4x32-10.
 */
spec_status spec_philox_uniform(uint64_t seed, uint64_t offset, int32_t B, int32_t T,
                                float* u_accept, float* u_sample, spec_stream_t s);

/* Workspace bytes tree_kv_commit needs (its status word only). */
size_t tree_kv_commit_workspace_size(void);

/*
 * KV commit of the accepted path -- Speculative Decoding (thegustafson.com),
 * section "The acceptance criterion" (the suffix past the rejection point is
 * discarded from the caches; the next round starts from the last accepted
 * token), and Hydra Guide, section "3. Tree KV-Cache Page Sizing" (discarded
 * candidates are rolled back without deallocation).
 *
 * For every sequence b with m = accept_len[b] and L = prefix_len[b]: the K and
 * V rows of the m + 1 nodes accept_path[b, 0..m] (root first) of every KV head
 * are copied from the tree buffers to cache rows L .. L + m, and prefix_len[b]
 * becomes L + m + 1.  No other cache row changes: the rejected nodes are never
 * copied.  The extra token tree_accept emits is not committed (it is the root
 * of the next round's tree).
 *
 *   k_tree, v_tree    device [B, Hkv, T, D] (dt): the tree nodes' keys/values
 *   k_cache, v_cache  device [B, Hkv, Lmax, D] (dt), updated in place
 *   prefix_len        device [B], updated in place
 *   accept_len        device [B]; accept_path device [B, max_depth + 1]: the
 *                     outputs of tree_accept for the same tree
 *   ws                >= tree_kv_commit_workspace_size() bytes, 16-byte aligned
 * Tree, cache and tree buffers 16-byte aligned; D * element size a multiple of
 * 16 bytes.  Host-checked arguments fail with a status before anything is
 * queued.  A sequence whose path is not root-first along tree edges, whose m is
 * outside 0..max_depth, or whose commit would pass Lmax is left unchanged and
 * SPEC_EINVAL goes to the status word (spec_read_device_status).  Caller owns
 * every buffer; the call queues work on s and does not synchronise.
 */
spec_status tree_kv_commit(const void* k_tree, const void* v_tree, void* k_cache, void* v_cache,
                           int32_t* prefix_len, const int32_t* accept_len, const int32_t* accept_path,
                           const spec_tree* tree, int32_t B, int32_t Hkv, int32_t Lmax, int32_t D,
                           spec_dtype dt, void* ws, size_t ws_bytes, spec_stream_t s);

/*
 * KV commit into a paged cache -- the same commit as tree_kv_commit (same
 * sections) with the cache in pre-allocated static blocks (Hydra Guide, "Hydra
 * Production Engineering Checklist", item 3), the layout tree_attention_paged
 * reads: cache position L + i of sequence b is row (L + i) % block_size of pool
 * block block_table[b, (L + i) / block_size] of every KV head.
 *
 *   k_pool, v_pool  device [num_blocks, Hkv, block_size, D] (dt), updated in place
 *   block_table     device [B, max_blocks] int32; only the entries of the blocks
 *                   the commit writes are read
 *   block_size      positive; max_blocks * block_size <= 2^22
 *   the rest as tree_kv_commit (ws >= tree_kv_commit_workspace_size() bytes).
 * Besides tree_kv_commit's checks, a sequence whose commit would pass
 * max_blocks * block_size positions or write a block outside 0 .. num_blocks-1
 * is left unchanged and SPEC_EINVAL goes to the status word.
 */
spec_status tree_kv_commit_paged(const void* k_tree, const void* v_tree, void* k_pool, void* v_pool,
                                 int32_t num_blocks, const int32_t* block_table, int32_t max_blocks,
                                 int32_t block_size, int32_t* prefix_len, const int32_t* accept_len,
                                 const int32_t* accept_path, const spec_tree* tree, int32_t B, int32_t Hkv,
                                 int32_t D, spec_dtype dt, void* ws, size_t ws_bytes, spec_stream_t s);

/* Message of the last failed call on this host thread ("" if none). */
const char* spec_last_error(void);

/* Copy the device status word kept at the start of a workspace to *status and wait for it (SPEC_OK = no failure). */
spec_status spec_read_device_status(const void* ws, int32_t* status, spec_stream_t s);

/*
 * Self-test of the device failure path: queues one kernel that waits on a
 * shared-memory barrier nothing completes, with the bounded wait the
 * tensor-core kernels use; after limit_ns (capped at 1 s) it gives up and
 * records SPEC_ETIMEOUT in the first word of ws (read it back with
 * spec_read_device_status).  ws: device, >= 16 bytes, 16-byte aligned.
 */
spec_status spec_selftest_timeout(void* ws, uint64_t limit_ns, spec_stream_t s);

/*
 * Kernel tracing.  While enabled, every kernel this library launches is
 * bracketed by a pair of CUDA events on its launch stream (at most `capacity`
 * launches are recorded).  spec_trace_end waits for them, totals the time per
 * kernel name into out[0 .. max_entries) and returns the number of entries,
 * or -1 on error.  spec_launch_count counts every kernel launch of this
 * library in this process.  Tracing is process-wide and not thread-safe.
 */
typedef struct {
    char name[48];
    int32_t launches;
    double total_ms;
} spec_trace_entry;

spec_status spec_trace_begin(int32_t capacity);
int32_t spec_trace_end(spec_trace_entry* out, int32_t max_entries);
int64_t spec_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_TREE_H */
