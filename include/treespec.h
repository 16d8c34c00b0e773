/*
 * treespec -- tree-attention verification and the accept walk of EAGLE-2-style
 * speculative decoding, for one NVIDIA GB300 (sm_103a).
 *
 * The method (from the pages this library follows):
 *   - "Tech Radar: SGLang EAGLE-2", section 2 (Dynamic Tree-Attention Verification):
 *     each draft node attends only to its tree ancestors and itself, on top of the
 *     cached prefix; section 5 item 1: for trees of at most 64 nodes the ancestor
 *     relation is one 64-bit word per node, tested with a single AND.  Trees of up
 *     to 128 nodes ("EAGLE-2 & Lookahead Decoding", section 6: the tree size follows
 *     the load) use two such words per node.
 *   - "Speculative Decoding in Production: EAGLE-3 Dynamic Trees", section
 *     "Mathematical Proof of Lossless Speedup", steps 1-3: accept a draft token with
 *     probability min(1, p/q), otherwise resample from the normalised max(0, p - q);
 *     section "From Linear Sequences to Dynamic Draft Trees": when branch B1 is
 *     rejected the next sibling B2 is tried.
 *   - "EAGLE-2 & Lookahead Decoding", section 4: greedy verification keeps the longest
 *     path whose tokens the target agrees with.
 *
 * Conventions shared by every entry point
 *   - Every data pointer is a DEVICE pointer owned by the caller; the library never
 *     allocates, frees or retains memory.  Scratch space is the caller's `workspace`
 *     (device memory, 256-byte aligned, at least the size the matching *_workspace_bytes
 *     query returns for the same arguments).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream) and are stream-ordered: inputs may be reused once the stream reaches
 *     the call's end.
 *   - Return value: TREESPEC_OK, or a negative TREESPEC_ERR_* code for an argument the
 *     host can check (nothing is launched in that case).  Index data that lives on the
 *     device (parent arrays, page ids, prefix lengths, tokens) is checked by the kernels:
 *     a bad entry sets a TREESPEC_STATUS_* bit in the workspace status word, the
 *     offending element is skipped (never dereferenced), and the caller reads the word
 *     with treespec_read_status() after the call.
 *   - Tree layout: tree_parents[b][0] = -1 is the root (the last verified token) and
 *     0 <= tree_parents[b][i] < i for i >= 1 (topological order), N <= 128.
 *     Trees of different sizes share a batch ("EAGLE-2 & Lookahead Decoding", section
 *     6, batched dynamic tree slicing): sequence b's tree is the N_b <= N entries
 *     before the first TREESPEC_ABSENT (-2) of its row, and every later entry must be
 *     TREESPEC_ABSENT too (a padding slot).
 */
#ifndef TREESPEC_H
#define TREESPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *treespec_stream_t;   /* a cudaStream_t */

enum treespec_dtype {
    TREESPEC_DTYPE_F32 = 0,    /* IEEE float32 storage and arithmetic */
    TREESPEC_DTYPE_BF16 = 1,   /* bfloat16 storage, float32 accumulation */
};

/* Parent entry of a padding slot after a tree smaller than the batch's N. */
#define TREESPEC_ABSENT (-2)

enum treespec_kernel {
    TREESPEC_KERNEL_AUTO = 0,  /* tensor-core kernel for bf16 with head_dim 128, else CUDA cores */
    TREESPEC_KERNEL_SIMT = 1,  /* CUDA-core split-KV kernel (any dtype) */
    TREESPEC_KERNEL_TC = 2,    /* tcgen05/TMA split-KV kernel (bf16, head_dim 128), one 128-row query tile per CTA */
    TREESPEC_KERNEL_TC_PAIR = 3,  /* the same with two 128-row query tiles per CTA (bf16, head_dim 128, an even
                                     number of 128-row blocks ceil(N*G / 128)) */
    TREESPEC_KERNEL_TC_2SM = 4,   /* tcgen05/TMA split-KV kernel whose MMAs span a pair of CTAs (cta_group::2):
                                     two 128-row blocks per cluster of two SMs, each SM copying half of every K/V
                                     tile (bf16, head_dim 128, an even number of 128-row blocks) */
    TREESPEC_KERNEL_TC_STREAM = 5,  /* the two-tile kernel as one persistent CTA per SM: every SM takes an equal
                                       share of all KV tiles, a kv head's range cut between SMs is merged by the
                                       SM that finishes it last (bf16, head_dim 128, an even number of 128-row
                                       blocks, batch <= 256); num_splits does not apply */
};

enum treespec_accept_mode {
    TREESPEC_ACCEPT_AUTO = 0,       /* path-only */
    TREESPEC_ACCEPT_ALL_ROWS = 1,   /* reduce every (sequence, node) row, then walk */
    TREESPEC_ACCEPT_PATH_ONLY = 2,  /* walk first; reduce only the rows the walk visits */
};

enum treespec_error {
    TREESPEC_OK = 0,
    TREESPEC_ERR_NULL_POINTER = -1,   /* a required pointer is NULL */
    TREESPEC_ERR_SHAPE = -2,          /* a size is out of the supported range */
    TREESPEC_ERR_DTYPE = -3,          /* unknown dtype, or a kernel that does not take it */
    TREESPEC_ERR_WORKSPACE = -4,      /* workspace NULL, misaligned or too small */
    TREESPEC_ERR_SAMPLING = -5,       /* temperature < 0 / NaN, or T > 0 without probs/uniforms */
    TREESPEC_ERR_ALIGNMENT = -6,      /* a tensor is not 16-byte aligned */
    TREESPEC_ERR_DEVICE = -7,         /* no usable CUDA device, or not sm_103 */
    TREESPEC_ERR_LAUNCH = -8,         /* the CUDA runtime refused a launch */
};

enum treespec_status_bits {
    TREESPEC_STATUS_BAD_PARENT = 1u << 0,  /* parents[0] != -1, parents[i] not in [0, i), or a node after padding */
    TREESPEC_STATUS_BAD_PAGE = 1u << 1,    /* a page id outside [0, num_pool_pages) */
    TREESPEC_STATUS_BAD_LENGTH = 1u << 2,  /* prefix_len < 0 or prefix_len + N > pages * page_size */
    TREESPEC_STATUS_BAD_TOKEN = 1u << 3,   /* a draft token outside [0, vocab) */
    TREESPEC_STATUS_TIMEOUT = 1u << 4,     /* a bounded wait inside a kernel ran out */
    TREESPEC_STATUS_INTERNAL = 1u << 5,    /* a launch-configuration invariant failed (work skipped) */
    TREESPEC_STATUS_BAD_PATH = 1u << 6,    /* tree_kv_commit: accept_len or accept_path out of range */
};

/* ------------------------------------------------------------------ tree attention */

typedef struct {
    int32_t batch;              /* B >= 1 */
    int32_t num_nodes;          /* N, tree nodes including the root, 1..128 */
    int32_t num_q_heads;        /* Hq */
    int32_t num_kv_heads;       /* Hkv, Hq % Hkv == 0; G = Hq / Hkv query heads share a kv head */
    int32_t head_dim;           /* D: 64 or 128 */
    int32_t page_size;          /* tokens per KV page: 16 */
    int32_t max_pages_per_seq;  /* row length of page_table */
    int32_t num_pool_pages;     /* P, pages in k_pages / v_pages */
    int32_t dtype;              /* enum treespec_dtype, shared by q, k_pages, v_pages, out */
    int32_t kernel;             /* enum treespec_kernel (0 = automatic) */
    int32_t num_splits;         /* KV splits per (sequence, kv head); 0 = planner's choice */
} treespec_attn_shape;

typedef struct {
    int32_t kernel;             /* the kernel the call will run (SIMT, TC, TC_PAIR or TC_2SM) */
    int32_t num_splits;         /* KV splits per (sequence, kv head, row block or pair of them) */
    int32_t split_tokens;       /* logical tokens per split (a multiple of the tile) */
    int32_t rows_per_block;     /* query rows (node x group) one CTA holds */
    int32_t row_blocks;         /* ceil(N*G / rows_per_block) */
    int32_t merge;              /* 1 if a split-merge kernel runs after the split kernel */
} treespec_attn_plan;

/* Workspace bytes tree_attn_verify needs for `shape` (0 if the shape is invalid). */
size_t treespec_attn_workspace_bytes(const treespec_attn_shape *shape);

/* How tree_attn_verify will execute `shape` on the current device.  Returns an error code. */
int treespec_attn_plan_for(const treespec_attn_shape *shape, treespec_attn_plan *plan);

/*
 * tree_attn_verify -- one tree-attention verification pass (one layer) for a batch.
 *
 * Operation ("Tech Radar: SGLang EAGLE-2", section 2 mask M and section 5 bitmask):
 * for sequence b with prefix length S = prefix_lens[b], the N_b tree tokens occupy
 * logical positions S .. S+N_b-1 in node order (N_b = N unless the row is padded).  Logical token t lives in physical
 * page page_table[b][t / page_size], slot t % page_size.  For node i and query head
 * hq (kv head h = hq / G):
 *     allowed(i) = {0 .. S-1} U {S + j : j is an ancestor of i, or j == i}
 *     out[b][i][hq] = softmax_t( q[b][i][hq] . K[t][h] / sqrt(D) ) over allowed(i),
 *                     applied to V[t][h].
 *
 *   q            [B][N][Hq][D]            dtype
 *   k_pages      [P][page_size][Hkv][D]   dtype  (the tree's own K at positions S..S+N_b-1)
 *   v_pages      [P][page_size][Hkv][D]   dtype
 *   page_table   [B][max_pages_per_seq]   int32, entries >= ceil((S+N_b)/page_size) unused
 *   prefix_lens  [B]                      int32, S >= 0 and S + N_b <= max_pages_per_seq*page_size
 *   tree_parents [B][N]                   int32, see the tree layout above
 *   out          [B][N][Hq][D]            dtype, written in full (zeros for a sequence
 *                                         whose prefix length is invalid and for the
 *                                         rows of padding slots)
 * Slots of a sequence's last page beyond S+N and pages outside the table are never
 * read, so they may hold anything (NaN included).  bf16 outputs are rounded to
 * nearest-even from float32.  All tensors must be 16-byte aligned and contiguous.
 */
int tree_attn_verify(const void *q, const void *k_pages, const void *v_pages,
                     const int32_t *page_table, const int32_t *prefix_lens,
                     const int32_t *tree_parents, void *out,
                     const treespec_attn_shape *shape,
                     void *workspace, size_t workspace_bytes, treespec_stream_t stream);

/*
 * tree_attn_verify_noalloc -- tree_attn_verify without a caller-provided workspace.
 *
 * The method's description has no counterpart to this call; it exists for callers
 * that cannot allocate device memory where they verify a tree (an application that
 * reserves nearly all device memory up front for its own pools, or a decode loop that
 * cannot afford an allocation's implicit synchronisation).  Arguments, layouts and
 * results are those of tree_attn_verify; the scratch space lives in one fixed 32 MiB
 * device array inside the library instead of `workspace`.
 *   - The array is held on every GPU that loads the library until the process exits.
 *   - The first call on a device looks up the array's device address (with that device
 *     current); make that first call before any stream capture.  Nothing is allocated.
 *   - A shape whose treespec_attn_workspace_bytes exceeds 32 MiB is rejected with
 *     TREESPEC_ERR_WORKSPACE (fewer splits via shape->num_splits shrink it); other
 *     argument errors are those of tree_attn_verify.
 *   - All calls on a device share the array: calls whose work overlaps on the GPU race
 *     and corrupt each other; serialise them (one stream).  The device status word of
 *     the last call is read with treespec_noalloc_read_status.
 */
int tree_attn_verify_noalloc(const void *q, const void *k_pages, const void *v_pages,
                             const int32_t *page_table, const int32_t *prefix_lens,
                             const int32_t *tree_parents, void *out,
                             const treespec_attn_shape *shape, treespec_stream_t stream);

/*
 * treespec_noalloc_read_status -- synchronise `stream` and copy the device status word
 * (TREESPEC_STATUS_* bits) of the last tree_attn_verify_noalloc call on the current
 * device into *status.  Like the entry point it serves, the method's description has no
 * counterpart to it: a caller of the no-allocation entry point holds no workspace
 * pointer, so treespec_read_status cannot reach its status word.  Returns an error code.
 */
int treespec_noalloc_read_status(uint32_t *status, treespec_stream_t stream);

/* --------------------------------------------------------------------- accept walk */

/* Workspace bytes tree_accept needs (0 if the sizes are invalid). */
size_t treespec_accept_workspace_bytes(int32_t batch, int32_t num_nodes, int32_t vocab);

/*
 * tree_accept -- walk each sequence's draft tree from the root and decide which
 * draft tokens the target accepts, plus the bonus token that follows them.
 *
 * Children of a node are tried in ascending node index.
 * Greedy (temperature == 0; "EAGLE-2 & Lookahead Decoding", section 4): a child is
 *   accepted iff its token equals the argmax of the current node's target logits
 *   (ties: lowest token id); the bonus token is the argmax at the last accepted node.
 * Stochastic (temperature > 0; rejection rule of "Speculative Decoding in Production:
 *   EAGLE-3 Dynamic Trees", section "Mathematical Proof of Lossless Speedup"): with
 *   p = softmax(target_logits[cur] / T), q = draft_probs[cur] and r = p, child c with
 *   token x is accepted iff r(x) > 0 and uniforms[c] * q(x) <= r(x); on rejection
 *   r <- max(0, r - q) / sum(max(0, r - q)) (left unchanged if that sum is 0) and the
 *   next sibling is tried.  With no child accepted, the bonus token is the smallest v
 *   with sum_{w <= v} r(w) > uniforms[0] * sum_w r(w).
 *
 *   target_logits [B][N][V] float32  row i = target logits after node i's token
 *   draft_tokens  [B][N]    int32    token of node i (entry 0, the root, is unused)
 *   draft_probs   [B][N][V] float32  q_i, the draft distribution i's children were drawn
 *                                    from (used as given); may be NULL when T == 0
 *   tree_parents  [B][N]    int32    may be padded (see the tree layout); a padding
 *                                    slot's rows and entries are never read as a node
 *   uniforms      [B][N]    float32  uniforms[b][c], c >= 1: accept coin of node c;
 *                                    uniforms[b][0]: the bonus-sample coin; NULL when T == 0
 *   temperature   0 for greedy, else > 0
 *   accept_path   [B][N]    int32    out: accepted node indices root-first, root excluded,
 *                                    padded with -1
 *   accept_len    [B]       int32    out: number of accepted draft nodes
 *   bonus_token   [B]       int32    out
 * Limits: N in 1..128, V in 1..2^30.  A draft token outside [0, V) is rejected and
 * flagged with TREESPEC_STATUS_BAD_TOKEN.
 * target_logits and draft_probs may point to device memory or to host memory the device
 * can address (pinned, e.g. from cudaHostAlloc): the kernels then read the rows in place
 * over the CPU-GPU link, and the path-only schedule reads only the rows on each
 * sequence's walk instead of all B*N of them.  The other arrays live on the device.
 */
int tree_accept(const float *target_logits, const int32_t *draft_tokens,
                const float *draft_probs, const int32_t *tree_parents,
                const float *uniforms, float temperature,
                int32_t *accept_path, int32_t *accept_len, int32_t *bonus_token,
                int32_t batch, int32_t num_nodes, int32_t vocab,
                void *workspace, size_t workspace_bytes, treespec_stream_t stream);

/*
 * tree_accept_with_mode -- tree_accept with an explicit schedule (enum treespec_accept_mode).
 * Both schedules return identical results; they differ in which rows they read: all
 * B*N rows up front, or only the rows on each sequence's walk.
 */
int tree_accept_with_mode(const float *target_logits, const int32_t *draft_tokens,
                          const float *draft_probs, const int32_t *tree_parents,
                          const float *uniforms, float temperature,
                          int32_t *accept_path, int32_t *accept_len, int32_t *bonus_token,
                          int32_t batch, int32_t num_nodes, int32_t vocab, int32_t mode,
                          void *workspace, size_t workspace_bytes, treespec_stream_t stream);

/* ----------------------------------------------------------------------- KV commit */

/* Workspace bytes tree_kv_commit needs (its status word). */
size_t treespec_commit_workspace_bytes(void);

/*
 * tree_kv_commit -- keep the accepted path's K/V, drop the rejected branches
 * ("Tech Radar: SGLang EAGLE-2", section 2: after verification the target retains the
 * accepted path's KV and discards the rejected branches; "EAGLE-2 & Lookahead
 * Decoding", section 6, paged tree KV-cache allocation: the positions of rejected
 * candidates go back to the pool).
 *
 * As tree_attn_verify lays a tree out, node n of sequence b sits at logical position
 * S + n (S = prefix_lens[b]) and node 0 is the root.  For k < accept_len[b] the K and V
 * rows (all kv heads) of node accept_path[b][k] are copied to logical position
 * S + 1 + k, in place in the page pool, and new_prefix_lens[b] = S + 1 + accept_len[b]:
 * the sequence then ends with the root and its accepted descendants, and the positions
 * after it are free for the next tree.  Every source row is read before any destination
 * row is written, so overlapping positions are safe.
 *   k_pages, v_pages  [P][16][Hkv][D] in shape->dtype, modified in place
 *   page_table [B][max_pages], prefix_lens [B]   int32, as given to tree_attn_verify
 *   accept_path [B][N], accept_len [B]           int32, as returned by tree_accept
 *   new_prefix_lens [B]                          int32 out (a separate buffer)
 *   shape: batch, num_nodes, num_kv_heads, head_dim, page_size, max_pages_per_seq,
 *          num_pool_pages and dtype are used; num_q_heads, kernel, num_splits are not.
 * The commit touches logical positions S .. S + max(path) only (the root stays at S), so
 * the bound is S + 1 + max(path) <= max_pages_per_seq * page_size (max(path) = 0 for an
 * empty path), whatever N is: a tree padded after its own last node with TREESPEC_ABSENT
 * commits whenever its accepted path fits.
 * A sequence whose prefix length is negative or whose touched positions run past its
 * page table (BAD_LENGTH), whose accept_len is outside [0, N-1] or whose path does not
 * increase strictly within [1, N) (BAD_PATH), or whose pages touched are outside the pool
 * (BAD_PAGE) is left unchanged and gets new_prefix_lens[b] = -1; the bit goes to the
 * workspace status word.
 */
int tree_kv_commit(void *k_pages, void *v_pages, const int32_t *page_table,
                   const int32_t *prefix_lens, const int32_t *accept_path,
                   const int32_t *accept_len, int32_t *new_prefix_lens,
                   const treespec_attn_shape *shape,
                   void *workspace, size_t workspace_bytes, treespec_stream_t stream);

/* ---------------------------------------------------------------- draft-tree build */

/* Workspace bytes tree_draft_step / tree_rerank need (0 if the sizes are invalid). */
size_t treespec_draft_workspace_bytes(int32_t batch, int32_t frontier, int32_t topk);

/*
 * tree_draft_step -- one expansion step of the draft tree ("EAGLE-2 & Lookahead
 * Decoding", section 4: a path's confidence is the product of its conditional
 * probabilities and only the most confident branches keep expanding; "Speculative
 * Decoding" (SGLang), EAGLE decoding: speculative_eagle_topk children per expanded node
 * and step, then a rerank over the candidates).
 *
 * Node arrays [B][max_nodes]: node 0 is the root (score 0).  Step s (0-based) expands a
 * frontier of F nodes -- the root at step 0 (F = 1), else the frontier the previous step
 * returned (F = topk) -- and every one of the F*topk candidates becomes a node:
 * candidate c = f*topk + r (frontier row f, rank r) is node base + c, with base = 1 at
 * step 0 and 1 + topk + (s-1)*topk*topk after that.
 *   logprobs     [B][F][V] float32: the draft model's log-probabilities of the next token
 *                after each frontier node, rows in frontier order (not NaN)
 *   frontier_in  [B][F] int32: the previous step's frontier_out (unused at step 0)
 *   frontier_out [B][topk] int32 out: the topk best candidates of this step, best first
 * A frontier node's children are its topk tokens (ties: lower token id), scored parent
 * score + log-probability in float32; ranking across the step breaks ties by the lower
 * candidate index.  Step 0 also writes the root (parent -1, token -1, score 0).
 * Limits: topk in 1..16, V >= topk, base + F*topk <= max_nodes <= 1024.  A row with
 * fewer than topk non-NaN values sets TREESPEC_STATUS_BAD_TOKEN.
 */
int tree_draft_step(const float *logprobs, int32_t batch, int32_t frontier, int32_t vocab,
                    int32_t topk, int32_t step, const int32_t *frontier_in,
                    int32_t *node_parent, int32_t *node_token, float *node_score,
                    int32_t max_nodes, int32_t *frontier_out,
                    void *workspace, size_t workspace_bytes, treespec_stream_t stream);

/*
 * tree_rerank -- keep the draft tree's best num_nodes nodes (the SGLang page: after the
 * expansion, reranking keeps the top speculative_num_draft_tokens nodes).
 *
 * From node arrays [B][max_nodes] (node 0 the root, every parent index smaller than its
 * node's), keeps the root and the num_nodes - 1 non-root nodes with the highest score
 * (ties: lower node index), numbered in increasing original index, and writes the tree
 * tree_attn_verify and tree_accept take: tree_parents [B][num_nodes] (root -1) and
 * draft_tokens [B][num_nodes].  A parent index that is not smaller than its node's, or
 * a kept node whose parent was dropped (possible only with positive log-probabilities),
 * is attached to the root and sets TREESPEC_STATUS_BAD_PARENT.
 * Limits: 1 <= num_nodes <= min(128, max_nodes), max_nodes <= 1024.
 */
int tree_rerank(const int32_t *node_parent, const int32_t *node_token, const float *node_score,
                int32_t batch, int32_t max_nodes, int32_t num_nodes,
                int32_t *tree_parents, int32_t *draft_tokens,
                void *workspace, size_t workspace_bytes, treespec_stream_t stream);

/*
 * tree_rerank_pool -- tree_rerank among a given set of candidates.  The SGLang page's
 * rerank may be read over all scored candidates (tree_rerank) or over the nodes that
 * entered some step's beam (the reading under which 5 steps of top-4 rerank 20
 * candidates): pass the union of the steps' frontier_out arrays as the pool.
 *   pool [B][pool_size] int32: node ids eligible besides the root; ids outside
 *        1 .. max_nodes-1 are ignored, duplicates count once.  1 <= pool_size <= 1024.
 * Keeps the root and the num_nodes - 1 best pool nodes (ties: lower node index).  With
 * fewer eligible nodes than num_nodes - 1 the tree is smaller: its row is padded after
 * the last kept node with TREESPEC_ABSENT parents and token -1 (the padded layout the
 * verify and accept calls take).  A kept node whose parent is not kept is attached to the
 * root and sets TREESPEC_STATUS_BAD_PARENT.  Other arguments and limits as tree_rerank.
 */
int tree_rerank_pool(const int32_t *node_parent, const int32_t *node_token, const float *node_score,
                     const int32_t *pool, int32_t pool_size,
                     int32_t batch, int32_t max_nodes, int32_t num_nodes,
                     int32_t *tree_parents, int32_t *draft_tokens,
                     void *workspace, size_t workspace_bytes, treespec_stream_t stream);

/* ------------------------------------------------------------------------- helpers */

/* Synchronise `stream` and copy the status word of a workspace used by the last call
 * on it into *status (0 = clean).  Returns an error code. */
int treespec_read_status(const void *workspace, uint32_t *status, treespec_stream_t stream);

/* Static description of an error code. */
const char *treespec_error_string(int code);

/* Library version as major * 10000 + minor * 100 + patch. */
int treespec_version(void);

/* The CUDA runtime's error code (a cudaError_t; 0 if none) behind the most recent
 * TREESPEC_ERR_LAUNCH of tree_attn_verify in this process, and its name in *name when
 * name is not NULL. */
int treespec_last_launch_error(const char **name);

/* Kernels this process has launched through the library so far (all entry points). */
uint64_t treespec_launch_count(void);

/*
 * treespec_set_wait_limit_ns -- for tests of the failure path only.  Every wait inside
 * the tensor-core attention kernels (on a TMA copy, a tensor-core result or another warp)
 * gives up after 2 s by default: the CTA then sets TREESPEC_STATUS_TIMEOUT, waits (with
 * the default bound) for the copies and tensor-core work it has already started, frees
 * its tensor memory and exits, leaving its rows incomplete.  This call sets that bound,
 * in nanoseconds, for the tree_attn_verify calls this process makes afterwards; a bound
 * shorter than the kernels' normal hand-offs (1 ns, say) makes them give up on purpose.
 * 0 restores the default.  Not thread-safe against concurrent calls.
 */
void treespec_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* TREESPEC_H */
