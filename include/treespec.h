/*
 * treespec.h -- C ABI of the GB300 (sm_103a) tree-based speculative
 * verification library (libtreespec.so).
 *
 * One verification step of tree-based speculative inference, as SpecInfer
 * describes it ("SpecInfer: Accelerating Large Language Model Serving with
 * Tree-based Speculative Inference and Verification", arXiv 2305.09781):
 *
 *   tree_build       linearise a token tree in depth-first order (sec. 4.2,
 *                    Fig. 4) from a parent array, an expansion configuration
 *                    <k1..km> (sec. 3, Fig. 3) or merged drafter chains (Def. 3.2)
 *   tree_expand_topk draft an expansion tree <k1..km> from drafter distributions
 *                    (sec. 3, Fig. 3: each node's children are its k most likely
 *                    next tokens)
 *   kv_append        write the tree nodes' K/V after the verified prefix of one
 *                    shared KV cache, in depth-first order (sec. 4.2)
 *   tree_attention   TreeAttention(u) = Attention(S_u) for every node (Def. 4.1)
 *                    in one kernel, topology-aware mask built in registers
 *   verify_greedy    VerifyGreedy (Algorithm 2)
 *   verify_mss       VerifyStochastic: multi-step speculative sampling (Algorithm 2)
 *   verify_naive     naive sampling, the comparison verifier of sec. 4.3 / 6.6
 *   kv_commit        keep only the accepted path's K/V (sec. 4.2, last paragraph)
 *
 * Conventions shared by every call
 *  - All array arguments are DEVICE pointers owned by the caller, unless the
 *    comment says "host". The library allocates no device memory and never
 *    synchronises: every call enqueues its kernels on `stream` and returns.
 *  - Per-node arrays given by the caller (tokens, parent, q, k_new, v_new,
 *    logits rows, uniforms, q_row, p_row) are in the caller's INPUT NODE ORDER,
 *    v = 0..n-1. tree_build returns the depth-first order (perm / dfs_of).
 *  - Host-detectable errors (NULL pointer, bad size, misalignment, unsupported
 *    shape) return TS_ERR_INVALID_ARG before anything is launched; the message
 *    is available from treespec_last_error(). A failed launch returns
 *    TS_ERR_CUDA.
 *  - Device-detected problems are OR-ed into *status (a device uint32, may be
 *    NULL) as TS_STATUS_* bits. An affected request is emptied: tree_build
 *    writes n_nodes[b] = 0, the verifiers write out_count[b] = 0; the other
 *    requests are unaffected. No kernel traps, asserts or waits without bound.
 *  - 16-byte alignment is required of q, out, k_new, v_new and both caches.
 *  - Limits: 1 <= n_max <= TS_MAX_NODES, head_dim in {64, 128}; bf16 or fp32.
 */
#ifndef TREESPEC_H
#define TREESPEC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#ifndef __CUDA_RUNTIME_API_H__
typedef struct CUstream_st *cudaStream_t;
#endif

#define TS_MAX_NODES 256
#define TS_MASK_WORDS(n) (((n) + 31) / 32)

typedef enum { TS_OK = 0, TS_ERR_INVALID_ARG = 1, TS_ERR_CUDA = 2, TS_ERR_UNSUPPORTED = 3 } ts_status;
typedef enum { TS_F32 = 0, TS_BF16 = 1 } ts_dtype;
typedef enum { TS_OP_ATTENTION = 0, TS_OP_VERIFY_GREEDY = 1, TS_OP_VERIFY_MSS = 2 } ts_op;

/* device status bits */
#define TS_STATUS_BAD_TREE 1u    /* no single root, parent out of range, cycle, n > n_max */
#define TS_STATUS_NONFINITE 2u   /* NaN/Inf in a logits or drafter row that was read     */
#define TS_STATUS_ZERO_RESID 4u  /* residual normaliser <= 0; residual kept unchanged    */
#define TS_STATUS_INDEX 8u       /* token >= V, row index out of range, prefix+n > L_max  */
#define TS_STATUS_TIMEOUT 16u    /* a bounded wait inside a kernel gave up               */

/*
 * The linearised tree. The struct itself is a HOST object holding DEVICE
 * pointers to caller-owned arrays; tree_build fills them, the other calls read
 * them. i is a depth-first index, v an input node id.
 *   n_nodes [B]                 node count (0 marks a rejected request)
 *   perm    [B][n_max]          perm[i]   = input id of DFS node i
 *   dfs_of  [B][n_max]          dfs_of[v] = DFS index of input node v
 *   parent  [B][n_max]          DFS index of DFS node i's parent, -1 for the root
 *   token   [B][n_max]          token of DFS node i
 *   depth   [B][n_max]          edges from the root (root 0)
 *   pos     [B][n_max]          position id prefix_len[b] + depth (may be NULL)
 *   sub_end [B][n_max]          one past the last DFS index of node i's subtree
 *   anc     [B][n_max][W]       W = TS_MASK_WORDS(n_max); bit j of row i set iff
 *                               DFS node j is an ancestor of i or i itself
 * Rows i >= n_nodes[b] hold -1 (anc rows 0). Children of DFS node i are
 * i+1, sub_end[i+1], ... while below sub_end[i], in input order.
 */
typedef struct ts_tree {
    int32_t B;
    int32_t n_max;
    int32_t *n_nodes;
    int32_t *perm;
    int32_t *dfs_of;
    int32_t *parent;
    int32_t *token;
    int32_t *depth;
    int32_t *pos;
    int32_t *sub_end;
    uint32_t *anc;
} ts_tree;

/*
 * A paged KV cache: keys (and values) live in pages of TS_PAGE_KEYS rows; page
 * g holds, for every head h, rows [g][h][0..TS_PAGE_KEYS) of d values
 * (layout [num_pages][H][TS_PAGE_KEYS][d], 16-byte aligned). Logical row r of
 * request b is row r % TS_PAGE_KEYS of page block_table[b][r / TS_PAGE_KEYS].
 * The pages of one request need not be contiguous or ordered; every page a
 * request's rows 0 .. P + n - 1 touch must be listed, and distinct requests
 * must not share the pages they write. Device pointers, owned by the caller.
 */
#define TS_PAGE_KEYS 64
typedef struct ts_paged_kv {
    void *k_pages, *v_pages;       /* [num_pages][H][TS_PAGE_KEYS][d] */
    const int32_t *block_table;    /* [B][max_pages] page ids */
    int32_t num_pages, max_pages;
} ts_paged_kv;

/*
 * tree_build -- depth-first linearisation (SpecInfer sec. 4.2 and Fig. 4;
 * expansion configuration of sec. 3 / Fig. 3; position ids = prefix length +
 * depth as on the "Speculative decoding" concept page, Implementation sketch).
 *
 * Parent mode (widths == NULL):
 *   tokens  [B][n_max]  token of every input node (the root's is the committed token)
 *   parent  [B][n_max]  parent input id, -1 for the single root
 *   n_nodes [B]         nodes per request (may alias t->n_nodes)
 * Expansion mode (widths != NULL, host array of m entries, each >= 1):
 *   the tree with root 0 where every node of depth i-1 has widths[i-1]
 *   children, numbered in level order; tokens [B][n_max] in that order;
 *   parent and n_nodes are ignored (n = 1 + sum_l prod_{i<=l} k_i, which
 *   must not exceed n_max).
 * prefix_len [B] (may be NULL) fills t->pos.
 * Children are visited in increasing input id. One CTA per request.
 */
ts_status tree_build(const ts_tree *t, const int32_t *tokens, const int32_t *parent,
                     const int32_t *n_nodes, const int32_t *widths, int m,
                     const int32_t *prefix_len, uint32_t *status, cudaStream_t stream);

/*
 * tree_build_chains -- merge C drafter chains of `len` tokens into one tree
 * (SpecInfer Def. 3.2): one node per distinct token sequence, rooted at
 * root_token[b]; chains[B][C][len]. New nodes are numbered in creation order
 * (chain 0 first, root = input node 0), so children appear in the order their
 * first chain proposed them. Requires 1 + C*len <= n_max.
 * Outputs besides *t (all [B][n_max], input node order):
 *   tokens_out  token of each merged node (may be NULL)
 *   p_row       target-logits row of node v: 0 for the root, 1 + c*len + p for
 *               the node first created by chain c at position p (may be NULL)
 *   q_row       drafter row c*len + p of that chain, the distribution the
 *               node's token was proposed from (root: -1) (may be NULL)
 */
ts_status tree_build_chains(const ts_tree *t, const int32_t *root_token, const int32_t *chains,
                            int C, int len, int32_t *tokens_out, int32_t *p_row, int32_t *q_row,
                            const int32_t *prefix_len, uint32_t *status, cudaStream_t stream);

/*
 * tree_expand_topk -- the drafter's top-k expansion (SpecInfer sec. 3, Fig. 3:
 * every node of depth i-1 gets the k_i most likely next tokens as children).
 * For the expansion tree <widths[0..m-1]> numbered level by level (as
 * tree_build's widths mode numbers it), the children of internal node u take,
 * best first, the widths[depth(u)] most probable tokens of ssm_probs[b][u],
 * ties to the lower token id; tokens[b][0] = root_token[b].
 *   tokens      [B][n_max]  out: the tree's tokens in level order (entries past
 *                           the tree's size are not written)
 *   root_token  [B]
 *   ssm_probs   [B][NQ][V]  fp32, row u = drafter distribution after node u;
 *                           NQ >= the number of internal nodes
 * A non-finite value in a row gives that node's children token -1 and sets
 * TS_STATUS_NONFINITE. The result feeds tree_build(..., widths, m, ...).
 */
ts_status tree_expand_topk(int32_t *tokens, const int32_t *root_token, const float *ssm_probs, int NQ,
                           int B, int n_max, const int32_t *widths, int m, int V, uint32_t *status,
                           cudaStream_t stream);

/*
 * tree_build_append -- tree_build in widths mode (an expansion tree, SpecInfer
 * sec. 3) and kv_append (sec. 4.2) in one launch, for a dense cache: the tree
 * arrays of t and the cache rows P + dfs(v) equal those of the two separate
 * calls. Arguments as for the two calls; prefix_len is required. The copy does
 * not wait for the tree arrays (an expansion tree's depth-first positions are
 * arithmetic), which takes one launch off the step's critical path.
 * A request with prefix_len[b] + n > L_max gets its tree arrays but no rows
 * (TS_STATUS_INDEX).
 */
ts_status tree_build_append(const ts_tree *t, const int32_t *tokens, const int32_t *widths, int m,
                            const int32_t *prefix_len, void *k_cache, void *v_cache, const void *k_new,
                            const void *v_new, int H, int d, int L_max, ts_dtype dtype, uint32_t *status,
                            cudaStream_t stream);

/*
 * kv_append -- place the pass's fresh K/V in the shared cache in depth-first
 * order right after the verified prefix (SpecInfer sec. 4.2):
 *   cache[b][h][prefix_len[b] + dfs_of[v]][:] = new[b][v][h][:]
 * k_new, v_new [B][n_max][H][d]; k_cache, v_cache [B][H][L_max][d]; dtype of both.
 * A request with prefix_len[b] + n_nodes[b] > L_max is skipped (TS_STATUS_INDEX).
 */
ts_status kv_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                    const int32_t *prefix_len, const ts_tree *t, int H, int d, int L_max,
                    ts_dtype dtype, uint32_t *status, cudaStream_t stream);

/*
 * tree_attention -- for every request b, head h and node v:
 *   out[b][v][h][:] = softmax_j(scale * q[b][v][h] . k_j) v_j
 * over the keys j of the verified prefix (cache rows 0..P_b-1) and of the
 * nodes on v's root path (rows P_b + dfs index), i.e. Attention(S_v) of
 * SpecInfer Def. 4.1 with the topology-aware mask of sec. 4.2. The mask is
 * the ancestor-or-self bitmask of *t, tested in registers; no N x N tensor.
 * q, out [B][n_max][H][d]; caches [B][H][L_max][d] as filled by kv_append.
 * scale <= 0 selects 1/sqrt(d). bf16: fp32 accumulation, bf16 output;
 * fp32: fp32 throughout. ws (ws_bytes >= treespec_workspace_size(
 * TS_OP_ATTENTION, ...)) holds what the chosen kernel shares between its CTAs:
 * for the split-KV kernel the partial results of the key splits and the
 * per-(b, h) counters by which the last CTA of each (b, h) finds that it
 * merges them (one launch); for the persistent kernel the queue its CTAs take
 * (request, head) items from. ws must be zero-filled before its first use
 * (treespec_workspace_init); calls leave it so. Calls that share one ws must
 * not overlap on the GPU.
 */
ts_status tree_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *prefix_len, const ts_tree *t, int H, int d, int L_max,
                         ts_dtype dtype, float scale, void *ws, size_t ws_bytes, uint32_t *status,
                         cudaStream_t stream);

/*
 * tree_attention_append -- kv_append and tree_attention in one call (SpecInfer
 * sec. 4.2: the tree's new keys and values join the KV cache in depth-first
 * order, and every node attends to the prefix and its root path): the rows
 * k_new / v_new [B][n_max][H][d] go to cache rows P_b + dfs(v) exactly as
 * kv_append writes them, and out gets exactly what tree_attention computes on
 * the appended cache. Arguments, layouts, workspace and status as for those
 * two calls; the caches are written. For the persistent tcgen05 kernel (bf16,
 * head_dim 128, at most 128 nodes) one launch does both: a tenth warp of each
 * CTA copies an item's rows into the cache an item ahead of the TMA loads
 * that read them back, so the new rows are read from HBM once; otherwise the
 * call makes the two launches of the separate calls.
 */
ts_status tree_attention_append(void *out, const void *q, void *k_cache, void *v_cache, const void *k_new,
                                const void *v_new, const int32_t *prefix_len, const ts_tree *t, int H, int d,
                                int L_max, ts_dtype dtype, float scale, void *ws, size_t ws_bytes,
                                uint32_t *status, cudaStream_t stream);

/*
 * verify_greedy -- VerifyGreedy of SpecInfer Algorithm 2: O(u) = argmax of
 * the target logits at u (ties to the lowest token id); from the root follow
 * the first child whose token equals O(u); at the first node without such a
 * child append O(u) and stop.
 *   logits     [B][n_max][V] fp32, row v = target logits after node v
 *   out_tokens [B][n_max+1]  accepted tokens, then the target's own token
 *   out_path   [B][n_max+1]  input ids of the root and of each accepted node
 *   out_count  [B]           number of tokens (1 .. depth+1); 0 on error
 *   argmax_out [B][n_max]    O(v) per input node (may be NULL)
 * A non-finite value in any node row empties the request (TS_STATUS_NONFINITE).
 * ws: treespec_workspace_size(TS_OP_VERIFY_GREEDY, ...) bytes, zero-filled
 * before first use; calls leave it zeroed.
 */
ts_status verify_greedy(int32_t *out_tokens, int32_t *out_path, int32_t *out_count,
                        int32_t *argmax_out, const float *logits, const ts_tree *t, int V, void *ws,
                        size_t ws_bytes, uint32_t *status, cudaStream_t stream);

/*
 * verify_mss -- VerifyStochastic, multi-step speculative sampling (SpecInfer
 * Algorithm 2; residual norm(max(0, p - q)) of "How Speculative Decoding in
 * LLM Serving Actually Works"): at node u, p = softmax(logits/T); children
 * are tried in input order, child c (token x) accepted iff
 * uniforms[b][0][c] <= min(1, r(x)/q_c(x)) (1 when q_c(x) = 0); a rejection
 * replaces r by norm(max(0, r - q_c)); when no child is accepted (or u is a
 * leaf) the inverse-CDF sample of r with uniforms[b][1][u] is appended and
 * the walk stops.
 *   target_logits [B][NP][V] fp32; node v reads row p_row[b][v] (identity
 *                 when p_row is NULL, then NP >= n_max)
 *   ssm_probs     [B][NQ][V] fp32 drafter probabilities (already tempered);
 *                 child v is tested against row q_row[b][v]
 *   uniforms      [B][2][n_max] fp32 in [0, 1)
 *   temperature   > 0, divides the target logits
 * Outputs as verify_greedy, plus
 *   out_lowmargin [B] (may be NULL) the number of decisions of the request's
 *                 walk whose margin, as computed here, is below 1e-6: an accept
 *                 test with |u - a| < 1e-6, or a final sample whose u * S lies
 *                 within 1e-6 * S of the cumulative sums on either side of the
 *                 drawn token (S the residual's total). Such a decision may
 *                 differ from one taken in exact arithmetic; a request with a
 *                 count of 0 took every decision with at least that margin.
 * Arithmetic: fp32 elementwise, compensated sums combined in fp64. A
 * non-finite value met on the walk empties the request. No workspace.
 */
ts_status verify_mss(int32_t *out_tokens, int32_t *out_path, int32_t *out_count,
                     int32_t *out_lowmargin, const float *target_logits, const int32_t *p_row,
                     int NP, const float *ssm_probs, const int32_t *q_row, int NQ,
                     const float *uniforms, float temperature, const ts_tree *t, int V,
                     uint32_t *status, cudaStream_t stream);

/*
 * verify_naive -- naive sampling (SpecInfer sec. 4.3, the verifier that
 * multi-step speculative sampling is compared with in sec. 6.6 / Table 3):
 * at the visited node u draw x from p = softmax(logits_u / T) by inverse CDF
 * with uniforms[b][1][u] (the first x, by id, with C(x) > u * sum p); if a
 * child of u (in input order) has token x, accept it and continue there,
 * else append x and stop. Arguments as verify_mss without the drafter rows;
 * uniforms[b][0][*] are not read. Same outputs (out_lowmargin counts the
 * samples), status bits and floating-point rules as verify_mss.
 */
ts_status verify_naive(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *out_lowmargin,
                       const float *target_logits, const int32_t *p_row, int NP, const float *uniforms,
                       float temperature, const ts_tree *t, int V, uint32_t *status, cudaStream_t stream);

/*
 * kv_commit -- keep the accepted path's K/V (SpecInfer sec. 4.2: only the
 * accepted tokens keep their cache entries). Path node i (out_path[b][i],
 * i < out_count[b]; the root first) moves from cache row
 * prefix_len[b] + dfs_of[node] to row prefix_len[b] + i, and
 * new_prefix_len[b] = prefix_len[b] + out_count[b]. new_prefix_len must not
 * alias prefix_len.
 */
ts_status kv_commit(void *k_cache, void *v_cache, const int32_t *prefix_len,
                    int32_t *new_prefix_len, const int32_t *out_path, const int32_t *out_count,
                    const ts_tree *t, int H, int d, int L_max, ts_dtype dtype, uint32_t *status,
                    cudaStream_t stream);

/*
 * tree_attention_noalloc -- tree_attention for callers that cannot allocate
 * device memory. The paper has no counterpart: this is a packaging variant of
 * the same computation. Some callers may not call cudaMalloc themselves --
 * plugin or callback code run by a host framework that owns every device
 * allocation and forbids allocating on its execution path, or serving loops
 * that must not allocate once warmed up. They pass inputs and outputs exactly
 * as for tree_attention but no workspace: the split-KV partial results go to
 * a scratch array of TS_NOALLOC_SCRATCH_BYTES compiled into the library, which
 * every GPU that loads the library holds until the process exits.
 *  - Sizes whose workspace (treespec_workspace_size(TS_OP_ATTENTION, ...))
 *    exceeds TS_NOALLOC_SCRATCH_BYTES are rejected with TS_ERR_INVALID_ARG
 *    and a message saying so; nothing is launched.
 *  - The first call on a device looks the scratch address up
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture.
 *  - All calls on a device share the one scratch array, which keeps the last
 *    call's contents; each call clears the part that must start at zero on
 *    its stream (cudaMemsetAsync). Calls whose kernels may overlap on the GPU
 *    (different streams with no ordering) race on the scratch and must not be
 *    issued.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * fp32 inputs need no workspace and behave exactly as tree_attention.
 */
#define TS_NOALLOC_SCRATCH_BYTES (8u << 20)
ts_status tree_attention_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *prefix_len, const ts_tree *t, int H, int d, int L_max,
                                 ts_dtype dtype, float scale, uint32_t *status, cudaStream_t stream);

/*
 * Paged-cache forms of kv_append, tree_attention and kv_commit (the shared
 * tree cache of SpecInfer sec. 4.2 kept in pages, so requests of different
 * lengths need no common L_max): the same operations, arguments and rules as
 * the dense calls, with the cache given as a ts_paged_kv instead of
 * (k_cache, v_cache, L_max). bf16 only (TS_ERR_UNSUPPORTED otherwise) and
 * head_dim 128 or 64. tree_attention_paged runs the kernels tree_attention
 * chooses (one 64-key tile is one page) except the small-tree tcgen05 kernel,
 * whose 128-key tiles span two pages; its workspace is
 * treespec_workspace_size(TS_OP_ATTENTION, B, H, n_max, d,
 * max_pages * TS_PAGE_KEYS, V). A page id outside [0, num_pages) sets
 * TS_STATUS_INDEX: tree_attention_paged reads zeros in its place (the
 * request's outputs are then not meaningful), kv_append_paged and
 * kv_commit_paged leave that request's pages unchanged.
 */
ts_status kv_append_paged(const ts_paged_kv *kv, const void *k_new, const void *v_new, const int32_t *prefix_len,
                          const ts_tree *t, int H, int d, uint32_t *status, cudaStream_t stream);
ts_status tree_attention_paged(void *out, const void *q, const ts_paged_kv *kv, const int32_t *prefix_len,
                               const ts_tree *t, int H, int d, float scale, void *ws, size_t ws_bytes,
                               uint32_t *status, cudaStream_t stream);
ts_status kv_commit_paged(const ts_paged_kv *kv, const int32_t *prefix_len, int32_t *new_prefix_len,
                          const int32_t *out_path, const int32_t *out_count, const ts_tree *t, int H, int d,
                          uint32_t *status, cudaStream_t stream);

/* Bytes of workspace an op needs for these sizes on the current device (0 if none). */
size_t treespec_workspace_size(ts_op op, int B, int H, int n_max, int d, int L_max, int V);

/*
 * Name of the kernel tree_attention launches for these sizes on the current
 * device ("k_attn_f32", "k_attn_bf16<D,NT,NG,KS>" or "k_attn_tq"), as chosen
 * by the same plan the launch uses (including the TREESPEC_ATTN_KERNEL and
 * TREESPEC_ATTN_SPLITS environment overrides). Static string owned by the
 * library; "" for sizes tree_attention would reject. No GPU work.
 */
const char *treespec_attention_kernel(int B, int H, int n_max, int d, int L_max, ts_dtype dtype);

/* Zero-fill a workspace on `stream` (cudaMemsetAsync). */
ts_status treespec_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);

/* Message of the last failed call on this host thread ("" if none). */
const char *treespec_last_error(void);

/* Library version string. */
const char *treespec_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TREESPEC_H */
