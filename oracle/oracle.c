/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY. Not part of the product path.
 *
 * A plain, slow, obviously-correct CPU restatement (C99, fp64) of what one step
 * of tree-based speculative verification computes. Only the tests, the smoke
 * check and the benchmark's CPU-baseline / reference arm may load this library.
 * It shares no source, header, table or helper with the CUDA library; neither
 * includes nor links the other.
 *
 * Sources (page title, then the section / equation / figure followed):
 *   [SI] "SpecInfer: Accelerating Large Language Model Serving with Tree-based
 *        Speculative Inference and Verification" (arXiv 2305.09781):
 *        Def. 3.1 / Fig. 3 (expansion tree, widths <k1..km>), Def. 3.2 (merge),
 *        Eq. 1-4 + Def. 4.1 (tree attention), Fig. 4 + topology-aware causal
 *        mask (sec. 4.2), Algorithm 2 VerifyGreedy and VerifyStochastic
 *        (multi-step speculative sampling, sec. 4.3).
 *   [UI] "How Speculative Decoding in LLM Serving Actually Works": the residual
 *        distribution norm(max(0, P - Q)) and its exactness proof; the 6-node
 *        tree-mask table.
 *   [WK] "Speculative decoding" (wikillm concept page), Implementation sketch:
 *        tree position ids = prefix length + depth, temperature applied to both
 *        distributions, zero-normaliser guard, bonus token at a leaf.
 *
 * Readings taken where the pages are silent (each is listed in the design notes):
 *   - the root is the newest committed token and is node 0 of the tree walk;
 *   - children are visited in input order (DFS pre-order, children by id);
 *   - mask = ancestor-or-self ([SI] sec. 4.2 "or v = u", [UI] table diagonal);
 *   - greedy argmax ties -> lowest token id; duplicate sibling tokens -> first;
 *   - MSS tries children in input order; accept iff u <= a; a = 1 if q(x) = 0;
 *   - residual subtracts the full drafter distribution q of the rejected child;
 *   - zero residual normaliser: keep the residual unchanged, flag the request;
 *   - inverse CDF: first x (ascending id) with C(x) > u * S; if rounding leaves
 *     none, the largest x with positive mass;
 *   - uniforms[b][0][v] = accept test of node v as a child, uniforms[b][1][u] =
 *     final sample at node u.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* OR_MUTANT (default 0) plants one known mistake, for the tests that show the
 * pins catch it; a normal build never defines it. */
#ifndef OR_MUTANT
#define OR_MUTANT 0
#endif

#define OR_OK 0
#define OR_BAD_TREE 1
#define OR_INDEX 2
#define OR_NONFINITE 4
#define OR_ZERO_RESID 8
#define OR_BAD_ARG 16

/* ------------------------------------------------------------------------- */
/* Token tree layout ([SI] Def. 3.1, sec. 4.2 depth-first KV-cache layout).   */
/* ------------------------------------------------------------------------- */

/* Validate a parent array: exactly one root (parent -1), every other parent a
 * node of the tree, and every node reaches the root (no cycle). */
static int check_tree(int n, const int32_t *parent) {
    int roots = 0;
    if (n < 1) return OR_BAD_TREE;
    for (int v = 0; v < n; ++v) {
        if (parent[v] == -1) { roots++; continue; }
        if (parent[v] < 0 || parent[v] >= n || parent[v] == v) return OR_BAD_TREE;
    }
    if (roots != 1) return OR_BAD_TREE;
    for (int v = 0; v < n; ++v) {
        int u = v, steps = 0;
        while (parent[u] != -1) {
            u = parent[u];
            if (++steps > n) return OR_BAD_TREE;
        }
    }
    return OR_OK;
}

static int find_root(int n, const int32_t *parent) {
    for (int v = 0; v < n; ++v)
        if (parent[v] == -1) return v;
    return -1;
}

/* Depth-first pre-order from the root, children in increasing input id.
 * An explicit stack; children pushed in reverse so the smallest id pops first. */
static void dfs_order(int n, const int32_t *parent, int32_t *order) {
    int32_t *stack = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n + 1));
    int sp = 0, k = 0;
    stack[sp++] = find_root(n, parent);
    while (sp > 0) {
        int u = stack[--sp];
        order[k++] = u;
        for (int v = n - 1; v >= 0; --v)
            if (parent[OR_MUTANT == 3 ? n - 1 - v : v] == u) stack[sp++] = OR_MUTANT == 3 ? n - 1 - v : v;
    }
    free(stack);
}

/* One request: linearise the tree.
 *   perm[i]    = input id of the i-th node in DFS pre-order
 *   dfs_of[v]  = DFS index of input node v
 *   dparent[i] = DFS index of the parent of DFS node i (-1 for the root)
 *   dtoken[i]  = token of DFS node i
 *   depth[i]   = number of edges from the root
 *   sub_end[i] = one past the last DFS index inside the subtree of DFS node i
 *   anc[i*n_stride + j] = 1 iff DFS node j is an ancestor of DFS node i or i itself.
 */
int or_tree_build(int n, const int32_t *parent, const int32_t *tokens, int n_stride,
                  int32_t *perm, int32_t *dfs_of, int32_t *dparent, int32_t *dtoken,
                  int32_t *depth, int32_t *sub_end, uint8_t *anc) {
    int rc = check_tree(n, parent);
    if (rc) return rc;
    dfs_order(n, parent, perm);
    for (int i = 0; i < n; ++i) dfs_of[perm[i]] = i;
    for (int i = 0; i < n; ++i) {
        int v = perm[i];
        dparent[i] = parent[v] < 0 ? -1 : dfs_of[parent[v]];
        dtoken[i] = tokens ? tokens[v] : 0;
        int d = 0;
        for (int u = v; parent[u] != -1; u = parent[u]) d++;
        depth[i] = d;
    }
    /* subtree size by counting descendants: j lies in i's subtree iff i is on
     * j's root path */
    for (int i = 0; i < n; ++i) {
        int size = 0;
        for (int j = 0; j < n; ++j) {
            int u = perm[j];
            for (;;) {
                if (u == perm[i]) { size++; break; }
                if (parent[u] == -1) break;
                u = parent[u];
            }
        }
        sub_end[i] = i + size;
    }
    if (anc) {
        for (int i = 0; i < n; ++i) {
            for (int j = 0; j < n_stride; ++j) anc[(size_t)i * n_stride + j] = 0;
            for (int u = perm[i];; u = parent[u]) {
                anc[(size_t)i * n_stride + dfs_of[u]] = 1;
                if (parent[u] == -1) break;
            }
        }
    }
    return OR_OK;
}

/* Batched wrapper; rows beyond n_nodes[b] are left untouched. status[b] gets
 * the per-request code. Returns the OR of all codes. */
int or_tree_build_batch(int B, int n_max, const int32_t *n_nodes, const int32_t *parent,
                        const int32_t *tokens, int32_t *perm, int32_t *dfs_of, int32_t *dparent,
                        int32_t *dtoken, int32_t *depth, int32_t *sub_end, uint8_t *anc,
                        int32_t *status) {
    int all = 0;
    for (int b = 0; b < B; ++b) {
        size_t o = (size_t)b * n_max;
        int n = n_nodes[b];
        int rc = (n < 1 || n > n_max)
                     ? OR_BAD_TREE
                     : or_tree_build(n, parent + o, tokens ? tokens + o : NULL, n_max, perm + o,
                                     dfs_of + o, dparent + o, dtoken + o, depth + o, sub_end + o,
                                     anc ? anc + (size_t)b * n_max * n_max : NULL);
        if (status) status[b] = rc;
        all |= rc;
    }
    return all;
}

/* Expansion configuration <k1..km> ([SI] sec. 3, Fig. 3): every node at depth
 * i-1 receives k_i children. Nodes are numbered in level order (root 0, then
 * the whole of depth 1, ...), children of a node consecutive, in the order the
 * drafter ranked them. Returns the node count, or -1 if it exceeds n_cap. */
int or_widths_parent(int m, const int32_t *widths, int n_cap, int32_t *parent) {
    int level_start = 0, level_n = 1, n = 1;
    if (n_cap < 1) return -1;
    parent[0] = -1;
    for (int l = 0; l < m; ++l) {
        int k = widths[l];
        if (k < 1) return -1;
        int next_start = n;
        for (int j = 0; j < level_n; ++j)
            for (int c = 0; c < k + (OR_MUTANT == 13 && l == 1); ++c) {
                if (n >= n_cap) return -1;
                parent[n++] = level_start + j;
            }
        level_start = next_start;
        level_n *= k;
    }
    return n;
}

/* Top-k expansion from the drafter ([SI] sec. 3, Fig. 3: the SSM expands each
 * node of depth i-1 into its k_i most likely next tokens). For the expansion
 * tree <k1..km> in level order (or_widths_parent), node u's children take, in
 * order, the k most probable tokens of drafter row u (ssm [B][NQ][V]), ties to
 * the lower token id: sort every token of the row by (probability desc, id
 * asc) and take the first k. tokens[b][0] = root_token[b]. A row with a
 * non-finite entry gives its children token -1 and sets OR_NONFINITE.
 * Returns the status bits. */
static const float *g_row;
static int by_prob_then_id(const void *a, const void *b) {
    int x = *(const int *)a, y = *(const int *)b;
    double px = g_row[x], py = g_row[y];
    if (px > py) return -1;
    if (px < py) return 1;
    return (x > y) - (x < y);
}

int or_topk_expand(int B, int n_max, int NQ, int V, int m, const int32_t *widths, const int32_t *root_token,
                   const float *ssm, int32_t *tokens) {
    int32_t *par = (int32_t *)malloc(sizeof(int32_t) * (size_t)n_max);
    int *ids = (int *)malloc(sizeof(int) * (size_t)V);
    int all = 0;
    int n = or_widths_parent(m, widths, n_max, par);
    if (n < 0) { free(par); free(ids); return OR_BAD_ARG; }
    for (int b = 0; b < B; ++b) {
        int32_t *tok = tokens + (size_t)b * n_max;
        for (int v = 0; v < n_max; ++v) tok[v] = -1;
        tok[0] = root_token[b];
        for (int u = 0; u < n; ++u) {
            int first = -1, k = 0;
            for (int v = 1; v < n; ++v)
                if (par[v] == u) { if (first < 0) first = v; ++k; }
            if (k == 0) continue;
            if (u >= NQ) { all |= OR_BAD_ARG; continue; }
            const float *row = ssm + ((size_t)b * NQ + u) * V;
            int bad = 0;
            for (int x = 0; x < V; ++x) { ids[x] = x; if (!isfinite(row[x])) bad = 1; }
            if (bad) { all |= OR_NONFINITE; continue; }
            g_row = row;
            qsort(ids, (size_t)V, sizeof(int), by_prob_then_id);
            for (int c = 0; c < k && c < V; ++c) tok[first + c] = ids[c];
        }
    }
    free(par);
    free(ids);
    return all;
}

/* Merge of chains ([SI] Def. 3.2): every node stands for one distinct token
 * sequence; insert the chains one after another into a trie rooted at the
 * committed token. New nodes are numbered in creation order. src[v] gives the
 * first (chain * len + position) that created node v (-1 for the root); that
 * chain's drafter supplies the proposal distribution of v. Returns the node
 * count or -1 when n_cap is too small. */
int or_merge_chains(int C, int len, const int32_t *chains, int32_t root_token, int n_cap,
                    int32_t *parent, int32_t *tokens, int32_t *src) {
    int n = 1;
    if (n_cap < 1) return -1;
    parent[0] = -1;
    tokens[0] = root_token;
    src[0] = -1;
    for (int c = 0; c < C; ++c) {
        int u = 0;
        for (int p = 0; p < len; ++p) {
            int32_t t = chains[(size_t)c * len + p];
            int found = -1;
            for (int v = 1; v < n; ++v)
                if ((OR_MUTANT == 11 || parent[v] == u) && tokens[v] == t) { found = v; break; }
            if (found < 0) {
                if (n >= n_cap) return -1;
                parent[n] = u;
                tokens[n] = t;
                src[n] = c * len + p;
                found = n++;
            }
            u = found;
        }
    }
    return n;
}

/* ------------------------------------------------------------------------- */
/* Tree attention ([SI] Eq. 1-4, Def. 4.1; topology-aware mask, sec. 4.2).   */
/* ------------------------------------------------------------------------- */

static double load_elem(const void *base, size_t idx, int dtype) {
    if (dtype == 0) return (double)((const float *)base)[idx];
    /* bfloat16: the upper 16 bits of an IEEE binary32 */
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* TreeAttention(u) = Attention(S_u): the query of node u attends the verified
 * prefix (cache rows 0..P_b-1 of its head) and the keys/values of the nodes on
 * the root..u path, which come from k_new / v_new (the pass's fresh K/V). It
 * never reads the cache's tree region, so it checks the layout independently.
 *
 * q, k_new, v_new : [B][n_max][H][d] (input node order), dtype 0=f32 1=bf16
 * k_cache, v_cache: [B][H][L_max][d], rows 0..prefix_len[b]-1 used
 * rows          : n_rows triples (b, h, v) to evaluate
 * out           : [n_rows][d] fp64
 */
int or_tree_attention_rows(int B, int H, int d, int n_max, int L_max, int dtype, const void *q,
                           const void *k_new, const void *v_new, const void *k_cache,
                           const void *v_cache, const int32_t *prefix_len, const int32_t *n_nodes,
                           const int32_t *parent, double scale, int n_rows, const int32_t *rows,
                           double *out, int nthreads) {
    int bad = 0;
    for (int r = 0; r < n_rows; ++r) {
        int b = rows[3 * r], h = rows[3 * r + 1], v = rows[3 * r + 2];
        if (b < 0 || b >= B || h < 0 || h >= H || v < 0 || v >= n_nodes[b] || n_nodes[b] > 4096) bad = 1;
        else if (prefix_len[b] < 0 || prefix_len[b] > L_max) bad = 1;
        else if (check_tree(n_nodes[b], parent + (size_t)b * n_max)) bad = 1;
    }
    if (bad) return OR_BAD_ARG;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int r = 0; r < n_rows; ++r) {
        int b = rows[3 * r], h = rows[3 * r + 1], v = rows[3 * r + 2];
        int P = prefix_len[b];
        const int32_t *par = parent + (size_t)b * n_max;
        /* the root..v path, root first */
        int path[4096];
        int plen = 0;
        for (int u = v;; u = par[u]) {
            if (!(OR_MUTANT == 4 && u == v)) path[plen++] = u;
            if (par[u] == -1) break;
        }
        int L = P + plen;
        double *s = (double *)malloc(sizeof(double) * (size_t)L);
        size_t qo = (((size_t)b * n_max + v) * H + h) * (size_t)d;
        double mx = -INFINITY;
        for (int j = 0; j < L; ++j) {
            double acc = 0.0;
            if (j < P) {
                size_t ko = (((size_t)b * H + h) * L_max + j) * (size_t)d;
                for (int e = 0; e < d; ++e) acc += load_elem(q, qo + e, dtype) * load_elem(k_cache, ko + e, dtype);
            } else {
                int a = path[plen - 1 - (j - P)];
                size_t ko = (((size_t)b * n_max + a) * H + h) * (size_t)d;
                for (int e = 0; e < d; ++e) acc += load_elem(q, qo + e, dtype) * load_elem(k_new, ko + e, dtype);
            }
            s[j] = acc * (OR_MUTANT == 5 ? scale * scale : scale);
            if (s[j] > mx) mx = s[j];
        }
        double z = 0.0;
        for (int j = 0; j < L; ++j) {
            s[j] = exp(s[j] - mx);
            z += s[j];
        }
        double *o = out + (size_t)r * d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        for (int j = 0; j < L; ++j) {
            double w = s[j] / z;
            if (j < P) {
                size_t vo = (((size_t)b * H + h) * L_max + j) * (size_t)d;
                for (int e = 0; e < d; ++e) o[e] += w * load_elem(v_cache, vo + e, dtype);
            } else {
                int a = path[plen - 1 - (j - P)];
                size_t vo = (((size_t)b * n_max + a) * H + h) * (size_t)d;
                for (int e = 0; e < d; ++e) o[e] += w * load_elem(v_new, vo + e, dtype);
            }
        }
        free(s);
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Verification ([SI] Algorithm 2).                                           */
/* ------------------------------------------------------------------------- */

/* children of u in input order */
static int children_of(int n, const int32_t *parent, int u, int32_t *ch) {
    int k = 0;
    for (int v = 0; v < n; ++v)
        if (parent[v] == u) ch[k++] = v;
    return k;
}

static int row_finite(const float *row, int V) {
    for (int x = 0; x < V; ++x)
        if (!isfinite(row[x])) return 0;
    return 1;
}

/* argmax with ties broken to the lowest token id */
static int argmax_row(const float *row, int V) {
    int best = 0;
    for (int x = 1; x < V; ++x)
        if (OR_MUTANT == 6 ? row[x] >= row[best] : row[x] > row[best]) best = x;
    return best;
}

/* VerifyGreedy: O(u) = argmax of the target logits at u. From the root, move to
 * the first child whose token equals O(u), appending that token; at the first
 * node with no such child (a leaf included) append O(u) and stop.
 * logits: [B][n_max][V] in input node order. out_tokens/out_path: [B][n_max+1];
 * out_path holds the input ids of the root and of every accepted node.
 * argmax_out (optional): [B][n_max]. */
int or_verify_greedy(int B, int n_max, int V, const int32_t *n_nodes, const int32_t *parent,
                     const int32_t *tokens, const float *logits, int32_t *out_tokens,
                     int32_t *out_path, int32_t *out_count, int32_t *argmax_out, int32_t *status) {
    int all = 0;
    int32_t *ch = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_max + 1));
    for (int b = 0; b < B; ++b) {
        int n = n_nodes[b];
        const int32_t *par = parent + (size_t)b * n_max;
        const int32_t *tok = tokens + (size_t)b * n_max;
        int32_t *ot = out_tokens + (size_t)b * (n_max + 1);
        int32_t *op = out_path + (size_t)b * (n_max + 1);
        int rc = (n < 1 || n > n_max) ? OR_BAD_TREE : check_tree(n, par);
        if (!rc)
            for (int v = 0; v < n; ++v)
                if (!row_finite(logits + ((size_t)b * n_max + v) * V, V)) rc |= OR_NONFINITE;
        out_count[b] = 0;
        if (rc) { if (status) status[b] = rc; all |= rc; continue; }
        if (argmax_out)
            for (int v = 0; v < n; ++v)
                argmax_out[(size_t)b * n_max + v] = argmax_row(logits + ((size_t)b * n_max + v) * V, V);
        int u = find_root(n, par), cnt = 0;
        op[0] = u;
        for (;;) {
            int o = argmax_row(logits + ((size_t)b * n_max + u) * V, V);
            int k = children_of(n, par, u, ch), next = -1;
            for (int i = 0; i < k; ++i)
                if (tok[ch[i]] == o) { next = ch[i]; break; }
            ot[cnt++] = o;
            if (next < 0 || (OR_MUTANT == 7 && cnt > 1)) break;
            op[cnt] = next;
            u = next;
        }
        out_count[b] = cnt;
        if (status) status[b] = 0;
    }
    free(ch);
    return all;
}

/* Target distribution at a node: p = softmax(logits / T), max-subtracted. */
static void softmax_t(const float *row, int V, double T, double *p) {
    double m = -INFINITY, z = 0.0;
    for (int x = 0; x < V; ++x)
        if ((double)row[x] > m) m = (double)row[x];
    for (int x = 0; x < V; ++x) {
        p[x] = exp(OR_MUTANT == 12 ? ((double)row[x] - m) * T : ((double)row[x] - m) / T);
        z += p[x];
    }
    for (int x = 0; x < V; ++x) p[x] /= z;
}

/* Rejection of a child whose drafter distribution is q: the residual becomes
 * norm(max(0, r - q)) ([SI] Algorithm 2 residual step; [UI] residual
 * distribution). Returns 1 if the normaliser was not positive, in which case r
 * is left unchanged (the zero-normaliser guard of [WK]). */
static double resid_term(double r, double q, int is_x) {
    double t = r - ((OR_MUTANT == 1 && !is_x) ? 0.0 : q);
    if (OR_MUTANT == 9) return t;
    return t > 0.0 ? t : 0.0;
}

static int residual_step(int V, double *r, const float *q, int x_rej) {
    double z = 0.0;
    for (int x = 0; x < V; ++x) z += resid_term(r[x], (double)q[x], x == x_rej);
    if (!(z > 0.0)) return 1;
    for (int x = 0; x < V; ++x) r[x] = resid_term(r[x], (double)q[x], x == x_rej) / z;
    return 0;
}

/* Acceptance probability of child token x proposed by q against residual r:
 * min(1, r(x) / q(x)); q(x) = 0 counts as always accepted. */
static double accept_prob(const double *r, const float *q, int x) {
    double qx = (double)q[x];
    if (qx <= 0.0) return 1.0;
    double a = r[x] / qx;
    return a < 1.0 ? a : 1.0;
}

/* Inverse CDF of the (unnormalised) distribution r with the uniform u: the
 * first x with C(x) > u * S, S = sum r. *margin receives the distance of u*S to
 * the two cumulative sums bracketing the choice, divided by S. */
static int inverse_cdf(int V, const double *r, double u, double *margin) {
    double S = 0.0;
    for (int x = 0; x < V; ++x) S += r[x];
    double target = u * S, c = 0.0;
    for (int x = 0; x < V; ++x) {
        double prev = c;
        c += r[x];
        if (c > target && r[x] > 0.0) {
            double m1 = target - prev, m2 = c - target;
            if (margin) *margin = (m1 < m2 ? m1 : m2) / S;
            return OR_MUTANT == 8 ? (x + 1) % V : x;
        }
    }
    for (int x = V - 1; x >= 0; --x)
        if (r[x] > 0.0) {
            if (margin) *margin = 0.0;
            return x;
        }
    if (margin) *margin = 0.0;
    return 0;
}

/* The law of one MSS node, for the exactness checks: given the target p at a
 * node and k children (tokens x_i, drafter rows q_i), returns a_i, the
 * probability of accepting child i given children 1..i-1 were rejected, and the
 * final residual r_k from which the node samples when all k are rejected.
 * Uses the same residual / acceptance helpers as or_verify_mss.
 * Returns the number of zero-normaliser guards taken. */
int or_mss_node_trace(int V, const double *p, int k, const int32_t *child_tok, const float *q,
                      double *a_out, double *resid_out) {
    int guards = 0;
    for (int x = 0; x < V; ++x) resid_out[x] = p[x];
    for (int i = 0; i < k; ++i) {
        const float *qi = q + (size_t)i * V;
        a_out[i] = accept_prob(OR_MUTANT == 2 ? p : resid_out, qi, child_tok[i]);
        guards += residual_step(V, resid_out, qi, child_tok[i]);
    }
    return guards;
}

/* VerifyStochastic / multi-step speculative sampling ([SI] Algorithm 2):
 *   u <- root; r <- p_u
 *   for each child c of u in order: a = min(1, r(x_c)/q_c(x_c));
 *       if uniforms[0][c] <= a: append x_c, u <- c, restart with r <- p_c
 *       else r <- norm(max(0, r - q_c))
 *   no child accepted (a leaf included): append the inverse-CDF sample of r
 *   with uniforms[1][u] and stop.
 * logits: [B][NP][V]; node v uses row p_row[v] (identity when p_row is NULL).
 * ssm:    [B][NQ][V]; child c is tested against row q_row[c].
 * lm_pos[b]: index in out_tokens of the first decision whose margin is below
 *            margin_eps (out_count[b] if none); min_margin[b]: smallest margin.
 */
int or_verify_mss(int B, int n_max, int V, const int32_t *n_nodes, const int32_t *parent,
                  const int32_t *tokens, const float *logits, const int32_t *p_row, int NP,
                  const float *ssm, const int32_t *q_row, int NQ, const float *uniforms,
                  double temperature, int32_t *out_tokens, int32_t *out_path, int32_t *out_count,
                  int32_t *lm_pos, double *min_margin, int32_t *status, double margin_eps) {
    int all = 0;
    if (!(temperature > 0.0) || V < 1) return OR_BAD_ARG;
    double *r = (double *)malloc(sizeof(double) * (size_t)V);
    double *p0 = (double *)malloc(sizeof(double) * (size_t)V);
    int32_t *ch = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_max + 1));
    for (int b = 0; b < B; ++b) {
        int n = n_nodes[b];
        const int32_t *par = parent + (size_t)b * n_max;
        const int32_t *tok = tokens + (size_t)b * n_max;
        const float *ua = uniforms + (size_t)b * 2 * n_max;
        const float *us = ua + n_max;
        int32_t *ot = out_tokens + (size_t)b * (n_max + 1);
        int32_t *op = out_path + (size_t)b * (n_max + 1);
        int rc = (n < 1 || n > n_max) ? OR_BAD_TREE : check_tree(n, par);
        out_count[b] = 0;
        if (lm_pos) lm_pos[b] = 0;
        if (min_margin) min_margin[b] = INFINITY;
        /* row indices and tokens are checked for every node up front; finiteness
         * only for the values the walk reads: the target row of each visited
         * node, q(x) of each tested child, the whole drafter row of each
         * rejected child */
        if (!rc)
            for (int v = 0; v < n; ++v) {
                int pr = p_row ? p_row[(size_t)b * n_max + v] : v;
                if (pr < 0 || pr >= NP) rc |= OR_INDEX;
                if (par[v] >= 0) {
                    int qr = q_row[(size_t)b * n_max + v];
                    if (qr < 0 || qr >= NQ) rc |= OR_INDEX;
                    if (tok[v] < 0 || tok[v] >= V) rc |= OR_INDEX;
                }
            }
        if (rc) { if (status) status[b] = rc; all |= rc; continue; }
        int u = find_root(n, par), cnt = 0, first_low = -1, flags = 0;
        double mm = INFINITY;
        op[0] = u;
        for (;;) {
            int pr = p_row ? p_row[(size_t)b * n_max + u] : u;
            if (!row_finite(logits + ((size_t)b * NP + pr) * V, V)) { flags |= OR_NONFINITE; break; }
            softmax_t(logits + ((size_t)b * NP + pr) * V, V, temperature, r);
            memcpy(p0, r, sizeof(double) * (size_t)V);
            int k = children_of(n, par, u, ch), next = -1;
            for (int i = 0; i < k; ++i) {
                int c = ch[i];
                const float *qc = ssm + ((size_t)b * NQ + q_row[(size_t)b * n_max + c]) * V;
                if (!isfinite(qc[tok[c]])) { flags |= OR_NONFINITE; break; }
                double a = accept_prob(OR_MUTANT == 2 ? p0 : r, qc, tok[c]);
                double mg = fabs((double)ua[c] - a);
                if (mg < mm) mm = mg;
                if (mg < margin_eps && first_low < 0) first_low = cnt;
                if ((double)ua[c] <= a) { next = c; break; }
                if (!row_finite(qc, V)) { flags |= OR_NONFINITE; break; }
                if (residual_step(V, r, qc, tok[c])) flags |= OR_ZERO_RESID;
            }
            if (flags & OR_NONFINITE) break;
            if (next >= 0) {
                ot[cnt++] = tok[next];
                op[cnt] = next;
                u = next;
                continue;
            }
            double mg;
            int t = inverse_cdf(V, r, (double)us[u], &mg);
            if (mg < mm) mm = mg;
            if (mg < margin_eps && first_low < 0) first_low = cnt;
            ot[cnt++] = t;
            break;
        }
        if (flags & OR_NONFINITE) cnt = 0;
        out_count[b] = cnt;
        if (lm_pos) lm_pos[b] = first_low < 0 ? cnt : first_low;
        if (min_margin) min_margin[b] = mm;
        if (status) status[b] = flags;
        all |= flags;
    }
    free(r);
    free(p0);
    free(ch);
    return all;
}

/* Naive sampling ([SI] sec. 4.3, the comparison of Theorem 4.3): at u draw t
 * from p_u by inverse CDF with uniforms[1][u]; if t is the token of a child
 * (the first such child), append it and move there; otherwise append t and
 * stop. Used only by the Theorem 4.3 checks. */
int or_verify_naive(int B, int n_max, int V, const int32_t *n_nodes, const int32_t *parent,
                    const int32_t *tokens, const float *logits, double temperature,
                    const float *uniforms, int32_t *out_tokens, int32_t *out_count) {
    if (!(temperature > 0.0)) return OR_BAD_ARG;
    double *p = (double *)malloc(sizeof(double) * (size_t)V);
    int32_t *ch = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_max + 1));
    int all = 0;
    for (int b = 0; b < B; ++b) {
        int n = n_nodes[b];
        const int32_t *par = parent + (size_t)b * n_max;
        const int32_t *tok = tokens + (size_t)b * n_max;
        const float *us = uniforms + (size_t)b * 2 * n_max + n_max;
        int32_t *ot = out_tokens + (size_t)b * (n_max + 1);
        out_count[b] = 0;
        if (n < 1 || n > n_max || check_tree(n, par)) { all |= OR_BAD_TREE; continue; }
        int u = find_root(n, par), cnt = 0;
        for (;;) {
            softmax_t(logits + ((size_t)b * n_max + u) * V, V, temperature, p);
            int t = inverse_cdf(V, p, (double)us[u], NULL);
            int k = children_of(n, par, u, ch), next = -1;
            for (int i = 0; i < k; ++i)
                if (tok[ch[i]] == t) { next = ch[i]; break; }
            ot[cnt++] = t;
            if (next < 0) break;
            u = next;
        }
        out_count[b] = cnt;
    }
    free(p);
    free(ch);
    return all;
}

/* Accepted-path compaction ([SI] sec. 4.2: only accepted tokens keep their
 * KV-cache entries). Path node i (root first, count nodes) moves from cache row
 * P + dfs(path[i]) to row P + i; the new verified length is P + count.
 * Works on a copy the caller supplies: cache [B][H][L_max][d] of elem_bytes. */
int or_kv_commit(int B, int H, int d, int L_max, int n_max, int elem_bytes, void *k_cache,
                 void *v_cache, const int32_t *prefix_len, const int32_t *dfs_of,
                 const int32_t *out_path, const int32_t *out_count, int32_t *new_prefix_len) {
    size_t row = (size_t)d * elem_bytes;
    unsigned char *tmp = (unsigned char *)malloc(row * (size_t)(n_max + 1) * 2);
    for (int b = 0; b < B; ++b) {
        int P = prefix_len[b], cnt = out_count[b];
        new_prefix_len[b] = P + cnt;
        for (int h = 0; h < H; ++h) {
            unsigned char *kb = (unsigned char *)k_cache + ((size_t)b * H + h) * L_max * row;
            unsigned char *vb = (unsigned char *)v_cache + ((size_t)b * H + h) * L_max * row;
            for (int i = 0; i < cnt; ++i) {
                int src = P + dfs_of[(size_t)b * n_max + out_path[(size_t)b * (n_max + 1) + i]];
                memcpy(tmp + (size_t)(2 * i) * row, kb + (size_t)src * row, row);
                memcpy(tmp + (size_t)(2 * i + 1) * row, vb + (size_t)src * row, row);
            }
            for (int i = 0; i < cnt; ++i) {
                memcpy(kb + (size_t)(P + i) * row, tmp + (size_t)(2 * i) * row, row);
                memcpy(vb + (size_t)(P + i) * row, tmp + (size_t)(2 * i + 1) * row, row);
            }
        }
    }
    free(tmp);
    return OR_OK;
}

int or_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
