/*
 * libspecverify -- the single-forward-pass verification step of
 * self-speculative decoding, for NVIDIA GB300 (sm_103a).
 *
 * One verification step, as the pages describe it:
 *   1. spec_mask_build   which speculative rows see which block columns
 *   2. spec_verify_attn  masked attention of the speculative rows over
 *                        (committed KV prefix || soft prompt || the block)
 *   3. spec_accept       vocab-wide argmax / log-sum-exp per judged row,
 *                        then the LA threshold longest prefix or the greedy
 *                        tree walk
 *   4. kv_commit         append the accepted rows' K/V to the cache; every
 *                        other speculative K/V row is dropped
 * and, around it: spec_accept_soft (soft matching), spec_draft_tree and
 * spec_prune_tree (the next draft), spec_stream_rotate_values (stream values
 * by rotation), spec_future_gather (ConFu's future token),
 * spec_la_prefill_attn (prefill-form LA).
 *
 * Sources, cited by page title and section / equation:
 *   [LA]  "Lookahead Attention: Self-Speculative Verification via Parallel
 *         Token Proposals": sec. 2.1-2.4, sec. 3.1 (mask M_LA), sec. 3.2
 *         (lookahead KV discarded), sec. 3.3 (batched lookahead, padding).
 *   [CF]  "ConFu: Contemplate the Future for Better Speculative Sampling"
 *         (reading notes): key design 1 (soft prompt seen only by
 *         contemplate tokens, one contemplate token per draft node, 2T
 *         tokens in one verify pass).
 *   [SS]  "Speculative Streaming: Fast LLM Inference without Auxiliary
 *         Models": Eq. 1-2 (multi-stream attention), Eq. 4 and the text
 *         after it (tree attention mask), batching with streams, the
 *         verification step (hard matching, beta + 1 tokens advanced).
 *
 * Conventions for every call:
 *   - All tensor arguments are DEVICE pointers owned by the caller, dense
 *     and row-major in the layout stated; the library never frees them and
 *     keeps no reference after the call returns.
 *   - Calls are asynchronous on the caller's CUDA stream (`stream`, a
 *     cudaStream_t; NULL = legacy default stream) and launch only this
 *     library's kernels.  The library allocates no device memory: scratch
 *     comes from a caller-provided workspace (spec_verify_attn), or, for
 *     spec_verify_attn_noalloc, from one fixed array inside the library.
 *   - Errors visible on the host (bad sizes, NULL pointers, unsupported
 *     dtype/shape, a too-small workspace) are returned before anything is
 *     launched.  Errors only visible on the device (a bad parent pointer, a
 *     page id out of range, a full cache) set bits in a per-device status
 *     word and the kernel skips the offending work; nothing traps, and
 *     every wait inside a kernel is bounded (spec_set_wait_limit; on expiry
 *     SPEC_DEV_TIMEOUT is set and the kernel returns).  spec_get_status()
 *     reads and clears that word.
 *   - The status word is shared by all calls on a device: with concurrent
 *     streams, an error bit cannot be attributed to one call.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPECVERIFY_VERSION 100

typedef int spec_status_t;

/* return codes */
#define SPEC_OK              0
#define SPEC_ERR_INVALID_ARG 1  /* NULL pointer, negative / inconsistent size */
#define SPEC_ERR_UNSUPPORTED 2  /* dtype or shape this build does not handle */
#define SPEC_ERR_BAD_TREE    3  /* reserved: tree errors are device-detected */
#define SPEC_ERR_CAPACITY    4  /* workspace too small */
#define SPEC_ERR_CUDA        5  /* a CUDA runtime call failed */
#define SPEC_ERR_DEVICE      6  /* spec_get_status found device error bits */

/* element types */
#define SPEC_F32  0
#define SPEC_BF16 1

/* KV-cache layouts */
#define SPEC_KV_CONTIGUOUS 0
#define SPEC_KV_PAGED      1

/* acceptance modes */
#define SPEC_ACCEPT_THRESH_CHAIN 0  /* [LA] sec. 2.4 */
#define SPEC_ACCEPT_GREEDY_TREE  1  /* [SS] verification step, [CF] */

/* vparent codes (spec_mask_build) */
#define SPEC_VP_ROOT (-1)   /* row sees the prefix and itself only */
#define SPEC_VP_PAD  (-2)   /* padding row ([LA] sec. 3.3): sees nothing */

/* row_flags bits (spec_mask_build output, spec_verify_attn input) */
#define SPEC_ROW_VALID     1u
#define SPEC_ROW_SEES_SOFT 2u

/* device status bits (spec_get_status) */
#define SPEC_DEV_BAD_TREE     0x01  /* vparent not an earlier valid row */
#define SPEC_DEV_BAD_PAGE     0x02  /* page id outside [0, n_pages) */
#define SPEC_DEV_SEQ_OVERFLOW 0x04  /* seq_len outside [0, cache capacity] */
#define SPEC_DEV_CAPACITY     0x08  /* commit: cache or free list full */
#define SPEC_DEV_BAD_INDEX    0x10  /* path / row_of / acc_len out of range */
#define SPEC_DEV_TIMEOUT      0x20  /* an internal pipeline wait expired */

/* Maximum speculative rows per request (block columns). */
#define SPEC_MAX_ROWS 256

/*
 * The committed KV cache ([LA] sec. 3.2, [SS] "no additional KV caching":
 * only accepted tokens' K/V ever enter it).
 *
 * kind == SPEC_KV_CONTIGUOUS:
 *   k, v : [batch][n_kv_heads][max_seq][head_dim]   (dtype)
 *   request b's token t lives at k[b][h][t][:].
 * kind == SPEC_KV_PAGED:
 *   k, v : [n_pages][n_kv_heads][head_dim / 64][page_size][64] (dtype)
 *   page_table : int32 [batch][max_pages_per_seq]; token t of request b
 *   lives in page page_table[b][t / page_size], slot t % page_size, and its
 *   element j of KV head h is k[page][h][j / 64][t % page_size][j % 64].
 *   Within one (page, head) the head dimension is split into 64-element
 *   blocks, each holding page_size rows: one (page, head) is a single
 *   contiguous 2-D tile, fetched by one tensor copy.  For head_dim = 64
 *   this is [n_pages][n_kv_heads][page_size][64].
 *   Entries past ceil(seq_len[b] / page_size) are unused.
 */
typedef struct spec_kv_desc {
    int kind;
    int dtype;
    int n_kv_heads;
    int head_dim;
    void *k;
    void *v;
    int batch;
    int max_seq;             /* contiguous: token capacity per request */
    int n_pages;             /* paged */
    int page_size;           /* paged: tokens per page (multiple of 16) */
    int max_pages_per_seq;   /* paged: row length of page_table */
    int32_t *page_table;     /* paged */
} spec_kv_desc;

/* Shape of one verify-attention call. */
typedef struct spec_attn_desc {
    int batch;         /* B */
    int n_rows;        /* R: padded speculative rows per request (<= 256) */
    int n_q_heads;     /* Hq (multiple of n_kv_heads) */
    int n_kv_heads;    /* Hkv */
    int head_dim;      /* d: 64 or 128 */
    int dtype;         /* SPEC_BF16 or SPEC_F32, for q, kb, vb, soft, o, cache */
    int n_soft;        /* soft-prompt KV entries (0 = none), <= 64 */
    float scale;       /* softmax scale; 0 -> 1/sqrt(head_dim) ([SS] Eq. 1) */
    int split_tokens;  /* prefix tokens per split; 0 = chosen by the library */
} spec_attn_desc;

/* Shape and rule of one acceptance call. */
typedef struct spec_accept_desc {
    int mode;          /* SPEC_ACCEPT_THRESH_CHAIN or SPEC_ACCEPT_GREEDY_TREE */
    float tau;         /* threshold on the proposal probability (chain mode) */
    int batch;         /* B */
    int n_judge_rows;  /* Rj: logits rows per request */
    int vocab;         /* V */
    int logit_dtype;   /* SPEC_BF16 or SPEC_F32 */
    int max_nodes;     /* N: row length of tokens / tree_parent / row_of */
    int path_cap;      /* row length of path */
} spec_accept_desc;

/* Shape of one prefill-form Lookahead Attention call. */
typedef struct spec_prefill_desc {
    int batch;         /* B */
    int n_orig;        /* n: original positions per request (>= 1) */
    int n_look;        /* k: lookahead positions per request (>= 0) */
    int n_q_heads;     /* Hq (multiple of n_kv_heads) */
    int n_kv_heads;    /* Hkv */
    int head_dim;      /* d: 128 */
    int dtype;         /* SPEC_BF16 */
    float scale;       /* softmax scale; 0 -> 1/sqrt(head_dim) */
} spec_prefill_desc;

/* Shape of one soft-matching acceptance call. */
typedef struct spec_soft_desc {
    int batch;          /* B */
    int n_judge_rows;   /* Rj: target logits rows per request */
    int n_draft_rows;   /* Rd: draft logits rows per request (0 = none) */
    int vocab;          /* V (<= 1,048,576) */
    int logit_dtype;    /* SPEC_BF16 or SPEC_F32, target and draft logits */
    int max_nodes;      /* N: row length of tokens / tree_parent / row_of */
    int path_cap;       /* row length of path */
    float temperature;  /* T > 0: p = softmax(z / T), q = softmax(z_d / T) */
} spec_soft_desc;

/* Shape of one draft-tree construction call. */
typedef struct spec_draft_desc {
    int batch;          /* B */
    int n_stream_rows;  /* rows per request in stream_logits */
    int gamma;          /* speculative streams (tree depth) */
    int k;              /* tokens per stream (1..8) */
    int vocab;          /* V (>= k) */
    int logit_dtype;    /* SPEC_BF16 or SPEC_F32 */
    int max_nodes;      /* row length of tokens / tree_parent (>= 1 + sum k^g) */
    int vparent_rows;   /* row length of vparent (>= nodes * (1 + gamma)) */
} spec_draft_desc;

/* Shape and threshold of one tree-pruning call. */
typedef struct spec_prune_desc {
    int batch;          /* B */
    int max_nodes;      /* N (<= 1024): row length of the tree arrays */
    int vocab;          /* V */
    int logit_dtype;    /* SPEC_BF16 or SPEC_F32 (early-exit logits) */
    float threshold;    /* an edge survives iff its probability >= threshold */
    int gamma;          /* stream rows per node in vparent */
    int vparent_rows;   /* row length of vparent (>= N * (1 + gamma)) */
} spec_prune_desc;

/* Shape of one stream value rotation call. */
typedef struct spec_rotate_desc {
    int batch;          /* B */
    int n_rows;         /* R: rows of the block per (request, KV head) */
    int n_kv_heads;     /* Hkv */
    int head_dim;       /* d (multiple of 8) */
    int dtype;          /* SPEC_BF16 or SPEC_F32 */
    int gamma;          /* streams per node (<= 64) */
    float eps;          /* rotation angle per stream index, radians */
} spec_rotate_desc;

/* Library version (SPECVERIFY_VERSION). */
int spec_version(void);

/* Human-readable name of a return code. */
const char *spec_status_string(spec_status_t status);

/*
 * spec_mask_build -- visibility of the speculative block ([LA] sec. 3.1 in
 * its verify form, [SS] Eq. 2 and Eq. 4 with the following text, [CF] key
 * design 1).
 *
 *   vparent    int32 [batch][n_rows]: SPEC_VP_ROOT (-1): the row sees the
 *              prefix and itself; SPEC_VP_PAD (-2): padding row; p >= 0:
 *              the row sees everything row p sees, plus itself (p must be an
 *              earlier, non-padding row: p < r).
 *   soft_flags uint8 [batch][n_rows] or NULL: nonzero -> the row also sees
 *              the soft-prompt columns (ConFu contemplate tokens).
 *   vis        uint32 [batch][n_rows][ceil(n_rows/32)] out: bit c of word
 *              c/32 of row r is set iff row r sees block column c.
 *   row_flags  uint8 [batch][n_rows] out: SPEC_ROW_VALID | SPEC_ROW_SEES_SOFT.
 *
 * A row whose vparent chain is malformed gets vis = 0 and row_flags = 0
 * and sets SPEC_DEV_BAD_TREE.  n_rows <= SPEC_MAX_ROWS.
 */
spec_status_t spec_mask_build(const int32_t *vparent, const uint8_t *soft_flags,
                              int batch, int n_rows, uint32_t *vis,
                              uint8_t *row_flags, void *stream);

/*
 * Bytes of workspace spec_verify_attn needs for this shape and cache
 * (split partials: per request, KV head and split, the packed rows'
 * running max, sum and unnormalised output in fp32; on the tensor-core
 * paths also the first tile of each CTA's range, which the attention
 * kernel writes and the combine reads, and for the tcgen05 kernel a record
 * per CTA of the split segment its range starts inside of).
 */
spec_status_t spec_verify_attn_workspace_size(const spec_attn_desc *attn,
                                              const spec_kv_desc *cache,
                                              size_t *bytes);

/*
 * spec_verify_attn -- masked attention of the speculative rows
 * ([SS] Eq. 1-2, Eq. 4; [LA] sec. 3.1; [CF] key design 1).
 *
 *   q         [batch][n_rows][n_q_heads][head_dim]
 *   cache     committed prefix (see spec_kv_desc); seq_len int32 [batch]
 *             gives each request's prefix length S_b.
 *   kb, vb    [batch][n_kv_heads][n_rows][head_dim]: the block's own K/V
 *             (never aliases the cache).
 *   soft_k/v  [n_kv_heads][n_soft][head_dim], or NULL when n_soft == 0.
 *   vis, row_flags  from spec_mask_build.
 *   o         out [batch][n_rows][n_q_heads][head_dim] (dtype)
 *   lse       out fp32 [batch][n_q_heads][n_rows]: natural-log
 *             log-sum-exp of the row's scaled scores.
 *   workspace device scratch of >= spec_verify_attn_workspace_size bytes,
 *             256-byte aligned; its contents on entry are ignored.
 *
 * For query head h the K/V head is h / (n_q_heads / n_kv_heads).  A valid
 * row r sees prefix columns 0..S_b-1, the n_soft soft columns iff
 * SPEC_ROW_SEES_SOFT, and block column c iff vis bit c; scores are
 * (q . k) * scale.  Rows without SPEC_ROW_VALID get o = 0, lse = -inf.
 * A seq_len outside [0, capacity] is clamped and sets SPEC_DEV_SEQ_OVERFLOW;
 * a page id outside [0, n_pages) is not read and sets SPEC_DEV_BAD_PAGE (the
 * affected outputs are then unspecified).
 */
spec_status_t spec_verify_attn(const spec_attn_desc *attn, const void *q,
                               const spec_kv_desc *cache, const void *kb,
                               const void *vb, const void *soft_k,
                               const void *soft_v, const int32_t *seq_len,
                               const uint32_t *vis, const uint8_t *row_flags,
                               void *o, float *lse, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * spec_accept_soft -- acceptance by soft matching ([SS] verification step:
 * a drafted token x is accepted with probability min(1, p(x) / q(x)), the
 * rejection sampling of Leviathan et al.; one correction token is sampled
 * at the rejection point).
 *
 *   logits          [batch][n_judge_rows][vocab]: target (main-stream) logits.
 *   draft_logits    [batch][n_draft_rows][vocab]: the draft distributions.
 *   tokens, tree_parent, row_of, n_nodes: the draft tree as in spec_accept
 *                   (tree mode); row_of NULL = identity.
 *   child_draft_row int32 [batch][max_nodes]: the draft row node c's children
 *                   were drafted from, -1 if none.  May be NULL only when
 *                   n_draft_rows == 0 (every q is then 0).
 *   u_accept        fp32 [batch][max_nodes]: uniform in [0, 1) used when node
 *                   c is tested.
 *   u_sample        fp32 [batch]: uniform in [0, 1) for the correction token.
 *   lse_t, lse_d    fp32 out [batch][n_judge_rows], [batch][n_draft_rows]:
 *                   ln sum exp(z / T) of each row (scratch the call fills).
 *   acc_len, path, next_token, last_node: out, as spec_accept (tree mode).
 *
 * From node 0, the children c of the current node are tried in index
 * order: c (token x) is accepted iff u_accept[c] * q(x) < p(x), with p the
 * softmax(z / T) of the current node's judge row and q that of its
 * child_draft_row; the first accepted child becomes the current node.  When
 * none is accepted, next_token is drawn from max(0, p - q) normalised (from
 * p when the node has no draft row or p <= q everywhere): the smallest v
 * whose cumulative mass exceeds u_sample[b] times the total (fp32 sums).
 * max_nodes <= SPEC_MAX_ROWS (else SPEC_ERR_UNSUPPORTED).  A malformed index
 * anywhere in the tree (parent, token, judge or draft row) or a path longer
 * than path_cap sets SPEC_DEV_BAD_INDEX; the malformed node is never
 * accepted.  Three launches: two vocab reductions (target, draft) and one
 * test-walk-draw kernel.
 */
spec_status_t spec_accept_soft(const spec_soft_desc *desc, const void *logits,
                               const void *draft_logits, const int32_t *tokens,
                               const int32_t *tree_parent, const int32_t *row_of,
                               const int32_t *child_draft_row, const int32_t *n_nodes,
                               const float *u_accept, const float *u_sample,
                               float *lse_t, float *lse_d, int32_t *acc_len,
                               int32_t *path, int32_t *next_token, int32_t *last_node,
                               void *stream);

/*
 * spec_draft_tree -- the next step's draft tree ([SS] tree draft
 * construction, batching with streams).
 *
 *   stream_logits [batch][n_stream_rows][vocab]: the speculative streams'
 *                 logits; request b's streams 1..gamma are rows
 *                 stream_row[b] .. stream_row[b] + gamma - 1 (stream_row
 *                 NULL: rows 0..gamma-1).
 *   root_token    int32 [batch]: the root's token (the correction token).
 *   tokens, tree_parent  int32 out [batch][max_nodes]; n_nodes int32 out
 *                 [batch] = 1 + sum_{g=1..gamma} k^g.
 *   vparent       int32 out [batch][vparent_rows] or NULL: the flattened
 *                 block for spec_mask_build (see below).
 *
 * The top-k tokens of stream j (largest logit first, ties to the lower
 * token id) are the candidates at depth j; every depth-(j-1) node gets all
 * k of them as children.  The tree is flattened breadth-first: node 0 is
 * the root, depth g holds k^g nodes, node off(g) + m has parent
 * off(g-1) + m / k and the (m % k)-th token of stream g.  vparent: row j < n
 * is node j (SPEC_VP_ROOT for the root, else its parent), row
 * n + j*gamma + (s-1) is stream s of node j (parent: node j for s = 1, the
 * row of stream s-1 otherwise), later rows SPEC_VP_PAD.  Entries past n are
 * -1.  A stream row outside [0, n_stream_rows) sets SPEC_DEV_BAD_INDEX.
 */
spec_status_t spec_draft_tree(const spec_draft_desc *desc, const void *stream_logits,
                              const int32_t *stream_row, const int32_t *root_token,
                              int32_t *tokens, int32_t *tree_parent, int32_t *n_nodes,
                              int32_t *vparent, void *stream);

/*
 * spec_prune_tree -- subtree pruning by early-exit probability ([SS]
 * parallel tree pruning).
 *
 *   tokens, tree_parent, n_nodes  the tree (parents precede children, node 0
 *                 the root), e.g. from spec_draft_tree.
 *   early_logits  [batch][max_nodes][vocab]: early-exit logits at each node.
 *   keep_map      int32 out [batch][max_nodes]: a node's index in the pruned
 *                 tree, or -1.
 *   tokens_out, parent_out  int32 out [batch][max_nodes]: the pruned tree,
 *                 survivors in their original order, parents renumbered;
 *                 entries past n_out are -1.  Must not alias the inputs.
 *   n_out         int32 out [batch].
 *   vparent       int32 out [batch][vparent_rows] or NULL: the pruned tree's
 *                 flattened block (layout as in spec_draft_tree).
 *
 * The edge from node p to its child c survives iff
 * exp(z_p[token c] - ln sum exp z_p) >= threshold (fp32), z_p the early-exit
 * logits at p; c survives iff its edge and its parent survive.  The root
 * always survives.  A parent index that does not precede its node sets
 * SPEC_DEV_BAD_TREE (that node is dropped); a token outside the vocabulary
 * sets SPEC_DEV_BAD_INDEX.  Two launches.
 */
spec_status_t spec_prune_tree(const spec_prune_desc *desc, const int32_t *tokens,
                              const int32_t *tree_parent, const int32_t *n_nodes,
                              const void *early_logits, int32_t *keep_map,
                              int32_t *tokens_out, int32_t *parent_out, int32_t *n_out,
                              int32_t *vparent, void *stream);

/*
 * spec_stream_rotate_values -- stream values by rotation ([SS] Eq. 7,
 * V_tn = V_t e^{i eps n}, 0 <= eps <= pi / (2N) with N the maximum sequence
 * length plus the number of streams).
 *
 *   n_nodes  int32 [batch]: T_b, the nodes of request b's block.
 *   vb       [batch][n_kv_heads][n_rows][head_dim] (dtype), in place: the
 *            block values in the SS layout (rows 0..T_b-1 the nodes, row
 *            T_b + j*gamma + (s-1) stream s of node j).
 *
 * For every node j and stream s = 1..gamma, the stream row's value vector
 * becomes node j's value vector with each pair (v[2i], v[2i+1]), read as
 * v[2i] + i v[2i+1], multiplied by e^{i eps s} (fp32, then the storage
 * type).  Node rows and rows past T_b (1 + gamma) are not touched; the
 * block keys are the caller's.  A request with T_b (1 + gamma) > n_rows is
 * skipped and sets SPEC_DEV_BAD_INDEX.  vb must be 16-byte aligned.  Run it
 * before spec_verify_attn.
 */
spec_status_t spec_stream_rotate_values(const spec_rotate_desc *desc, const int32_t *n_nodes,
                                        void *vb, void *stream);

/*
 * spec_future_gather -- the future-token hand-off ([CF] key design 1: the
 * future prediction of the contemplate token attached to the last accepted
 * node goes to the next round's draft).
 *
 *   o          [batch][n_rows][row_elems] (dtype): e.g. spec_verify_attn's
 *              output with row_elems = n_q_heads * head_dim.
 *   last_node  int32 [batch]: from spec_accept.
 *   out        [batch][row_elems] (dtype) out: row row_offset + last_node[b]
 *              of request b (row_offset = T for the ConFu layout, whose
 *              contemplate token of node j is row T + j).
 *
 * Rows must be whole multiples of 16 bytes and o, out 16-byte aligned.  A
 * row outside [0, n_rows) writes zeros and sets SPEC_DEV_BAD_INDEX.
 */
spec_status_t spec_future_gather(int batch, int n_rows, int row_elems, int dtype,
                                 const void *o, const int32_t *last_node, int row_offset,
                                 void *out, void *stream);

/*
 * spec_la_prefill_attn -- the prefill form of Lookahead Attention ([LA]
 * sec. 3.1): the n original and k lookahead positions of each request attend
 * in one pass under the full (n + k) x (n + k) mask M_LA.
 *
 *   q, o   [batch][n + k][n_q_heads][head_dim] (bf16); positions 0..n-1 are
 *          the originals, n..n+k-1 the lookahead tokens.
 *   k, v   [batch][n + k][n_kv_heads][head_dim] (bf16)
 *   lse    out fp32 [batch][n_q_heads][n + k]: natural-log log-sum-exp of
 *          each position's scaled scores.
 *
 * Position i < n sees keys 0..i (causal attention over the originals);
 * position i >= n sees keys 0..n-1 and itself.  For query head h the K/V
 * head is h / (n_q_heads / n_kv_heads); scores are (q . k) * scale.  q, k
 * and v must be 16-byte aligned.  No workspace: each query tile is finished
 * by one CTA.  Returns SPEC_ERR_UNSUPPORTED unless dtype is SPEC_BF16 and
 * head_dim is 128.
 */
spec_status_t spec_la_prefill_attn(const spec_prefill_desc *desc, const void *q,
                                   const void *k, const void *v, void *o,
                                   float *lse, void *stream);

/* Bytes of the fixed scratch array behind spec_verify_attn_noalloc. */
#define SPEC_NOALLOC_SCRATCH_BYTES (64u << 20)

/*
 * spec_verify_attn_noalloc -- spec_verify_attn for callers that cannot
 * allocate device memory.  The pages have no counterpart: this is a
 * deployment variant of the same computation.
 *
 * Meant for callers that have no workspace to give: for example an engine
 * that reserved all of the GPU's memory for its own KV-cache pool and allows
 * no later allocation, or a plugin hook whose framework owns the memory and
 * forbids allocating while it runs (cudaMalloc may also synchronise the
 * whole device).  Arguments and results are exactly those of
 * spec_verify_attn without `workspace` / `workspace_bytes`; the split
 * partials go to a fixed array of SPEC_NOALLOC_SCRATCH_BYTES (64 MiB) that
 * is part of the library, held on every GPU that loads the library's kernels
 * until the process exits.
 *
 *   - Returns SPEC_ERR_CAPACITY, before launching anything, when the shape
 *     needs more scratch than that (spec_verify_attn_workspace_size tells);
 *     such shapes must use spec_verify_attn.
 *   - Calls no allocating routine (no cudaMalloc, cudaFree or the like).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; it is looked up again
 *     only when the device's context has changed (e.g. after
 *     cudaDeviceReset).  Under lazy module loading (the CUDA default) that
 *     first lookup loads the library module holding the array, and that
 *     load is when the 64 MiB are taken from the device.  So make the first
 *     call on each device (any arguments: the lookup comes before every
 *     check) before reserving the rest of the device's memory, and before
 *     any stream capture.
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents (nothing needs to start at zero: the kernels write each
 *     partial before reading it).  Calls that can overlap on the GPU (other
 *     streams, other host threads) race on the array and must be serialised
 *     by the caller.
 */
spec_status_t spec_verify_attn_noalloc(const spec_attn_desc *attn, const void *q,
                                       const spec_kv_desc *cache, const void *kb,
                                       const void *vb, const void *soft_k,
                                       const void *soft_v, const int32_t *seq_len,
                                       const uint32_t *vis, const uint8_t *row_flags,
                                       void *o, float *lse, void *stream);

/*
 * spec_vocab_reduce -- per logits row ([LA] sec. 2.4 needs the proposal's
 * probability, [SS] hard matching needs the greedy token):
 *
 *   logits    [n_rows][vocab] (dtype)
 *   proposal  int32 [n_rows] or NULL
 *   argmax    out int32 [n_rows]: index of the maximum, lowest on ties
 *   lse       out fp32 [n_rows]: ln sum_j exp(z_j)
 *   zprop     out fp32 [n_rows] (may be NULL iff proposal is NULL):
 *             z[proposal[i]]; NaN if the proposal is outside [0, vocab).
 */
spec_status_t spec_vocab_reduce(const void *logits, int dtype, int n_rows,
                                int vocab, const int32_t *proposal,
                                int32_t *argmax, float *lse, float *zprop,
                                void *stream);

/*
 * spec_accept -- the acceptance step.
 *
 * If `logits` ([batch][n_judge_rows][vocab]) is non-NULL, spec_vocab_reduce
 * runs first and writes argmax / lse / zprop ([batch][n_judge_rows]); in
 * chain mode the proposal of judge row i is tokens[b][i].  If `logits` is
 * NULL, argmax / lse / zprop are read as inputs.
 *
 *   tokens      int32 [batch][max_nodes]: chain mode: proposal i of request
 *               b; tree mode: draft token of node j (node 0 = root).
 *   tree_parent int32 [batch][max_nodes] (tree mode): parent node, -1 for
 *               the root; parents precede children.  Ignored in chain mode.
 *   row_of      int32 [batch][max_nodes] or NULL (identity): judge row of
 *               node j (tree mode).  Must be NULL in chain mode.
 *   n_nodes     int32 [batch]: proposals (chain: k_b) or tree nodes.
 *
 * Chain mode ([LA] sec. 2.4): L = the largest l <= n_nodes[b] with
 *   zprop_i - lse_i >= ln(tau) for all i < l (fp32, row i judges proposal i).
 *   acc_len = L, path = 0..L-1, next_token = argmax of row L (or -1 when
 *   L == n_nodes[b]), last_node = L - 1.
 * Tree mode ([SS] verification step): from node 0 move to the child whose
 *   token equals the argmax of the current node's judge row (lowest node
 *   index on duplicate sibling tokens) until none matches.
 *   acc_len = nodes on the path including the root (beta + 1),
 *   path = those nodes, next_token = argmax at the last node (the
 *   correction token), last_node = last node on the path.  Tree mode takes
 *   max_nodes <= SPEC_MAX_ROWS (else SPEC_ERR_UNSUPPORTED).
 * path entries past acc_len are set to -1.  A path longer than path_cap or
 * an index out of range stops the walk and sets SPEC_DEV_BAD_INDEX.
 */
spec_status_t spec_accept(const spec_accept_desc *desc, const void *logits,
                          const int32_t *tokens, const int32_t *tree_parent,
                          const int32_t *row_of, const int32_t *n_nodes,
                          int32_t *argmax, float *lse, float *zprop,
                          int32_t *acc_len, int32_t *path, int32_t *next_token,
                          int32_t *last_node, void *stream);

/*
 * kv_commit -- append each request's accepted block rows to the cache and
 * drop the rest ([LA] sec. 3.2, [SS] lazy removal of pruned KV).
 *
 *   kb, vb    [batch][n_kv_heads][n_rows][head_dim], as for spec_verify_attn
 *   path      int32 [batch][path_cap]: block rows to append, in order
 *   acc_len   int32 [batch]: how many entries of path to append
 *   seq_len   int32 [batch], in/out: += appended rows
 *   free_pages int32 [n_free], free_head int32 [1] in/out (paged only;
 *             NULL / 0 for contiguous caches).
 *
 * Row path[b][i] goes to token position seq_len[b] + i.  Paged caches:
 * requests are served in ascending b; each first fills its partly used last
 * page, then takes pages free_pages[*free_head], free_pages[*free_head+1],
 * ... in order, recording them in page_table.
 * A request that would exceed its capacity (max_seq, or max_pages_per_seq)
 * is skipped and sets SPEC_DEV_CAPACITY; if the free list cannot serve all
 * requests, nothing is written and SPEC_DEV_CAPACITY is set.  Out-of-range
 * path entries are not written (SPEC_DEV_BAD_INDEX).
 */
spec_status_t kv_commit(const spec_kv_desc *cache, int batch, int n_rows,
                        const void *kb, const void *vb, int path_cap,
                        const int32_t *path, const int32_t *acc_len,
                        int32_t *seq_len, const int32_t *free_pages,
                        int n_free, int32_t *free_head, void *stream);

/*
 * spec_set_wait_limit -- limit, in SM clock cycles, of the internal pipeline
 * waits of the kernels launched from now on (verify attention, prefill
 * attention, and the bulk row stream of the vocabulary reduction),
 * process-wide.  The pages have no counterpart: this is the
 * library's guard against a hang.  A wait that runs out sets
 * SPEC_DEV_TIMEOUT; the kernel then stops issuing work, waits (with the
 * default limit) for its own copies and tensor-core operations, frees its
 * tensor memory and returns, and the context stays usable.  cycles < 0
 * restores the default (2e9 cycles, about one second); 0 makes any wait
 * whose condition is not already met fail at once, which is how the tests
 * exercise this path.  Returns the previous limit.  Not for use while other
 * threads launch work of this library.
 */
long long spec_set_wait_limit(long long cycles);

/*
 * spec_get_status -- synchronise `stream`, then read and clear the current
 * device's status word.  *out receives the SPEC_DEV_* bits (0 = none).
 * Returns SPEC_OK if no bit was set, SPEC_ERR_DEVICE otherwise.
 */
spec_status_t spec_get_status(void *stream, int32_t *out);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
