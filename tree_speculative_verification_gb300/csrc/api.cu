// api.cu -- the C ABI of libtreespec: argument checks, workspace sizing and
// dispatch to the kernels. Every entry point is declared, with its meaning,
// layouts and error behaviour, in include/treespec.h.
#include <stdarg.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "ts_internal.cuh"

namespace {

thread_local char g_err[512] = "";

ts_status fail(ts_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}

ts_status ok() {
    g_err[0] = 0;
    return TS_OK;
}

ts_status cuda_result(cudaError_t e, const char *what) {
    if (e != cudaSuccess) return fail(TS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
    return ok();
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

ts_status check_tree(const ts_tree *t, const char *who) {
    if (!t) return fail(TS_ERR_INVALID_ARG, "%s: tree is NULL", who);
    if (t->B < 1) return fail(TS_ERR_INVALID_ARG, "%s: tree B=%d must be >= 1", who, t->B);
    if (t->n_max < 1 || t->n_max > TS_MAX_NODES)
        return fail(TS_ERR_INVALID_ARG, "%s: tree n_max=%d outside [1, %d]", who, t->n_max, TS_MAX_NODES);
    if (!t->n_nodes || !t->perm || !t->dfs_of || !t->parent || !t->token || !t->depth || !t->sub_end || !t->anc)
        return fail(TS_ERR_INVALID_ARG, "%s: a tree array is NULL", who);
    return TS_OK;
}

ts_status check_attn_shape(const char *who, const ts_tree *t, int H, int d, int L_max, ts_dtype dt) {
    if (H < 1) return fail(TS_ERR_INVALID_ARG, "%s: H=%d must be >= 1", who, H);
    if (d != 64 && d != 128) return fail(TS_ERR_UNSUPPORTED, "%s: head_dim %d (supported: 64, 128)", who, d);
    if (dt != TS_F32 && dt != TS_BF16) return fail(TS_ERR_INVALID_ARG, "%s: unknown dtype %d", who, (int)dt);
    if (L_max < t->n_max) return fail(TS_ERR_INVALID_ARG, "%s: L_max=%d below n_max=%d", who, L_max, t->n_max);
    if ((long long)t->B * H * L_max >= (1LL << 31))
        return fail(TS_ERR_INVALID_ARG, "%s: B*H*L_max = %lld rows exceeds 2^31", who, (long long)t->B * H * L_max);
    return TS_OK;
}

}  // namespace

namespace ts {
// Records the message returned by treespec_last_error() for entry points
// defined in other translation units.
ts_status set_error(ts_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return st;
}
}  // namespace ts

namespace ts {
// The host checks of tree_attention (tree, shape, NULL pointers, alignment),
// shared with tree_attention_noalloc so that both reject before enqueuing anything.
ts_status check_attention_args(const void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *prefix_len, const ts_tree *t, int H, int d, int L_max, ts_dtype dtype,
                               const char *who) {
    ts_status st = check_tree(t, who);
    if (st) return st;
    if ((st = check_attn_shape(who, t, H, d, L_max, dtype))) return st;
    if (!out || !q || !k_cache || !v_cache || !prefix_len) return fail(TS_ERR_INVALID_ARG, "%s: NULL pointer", who);
    if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(TS_ERR_INVALID_ARG, "%s: q, out and caches must be 16-byte aligned", who);
    return TS_OK;
}

bool pdl_enabled() {
    static const bool on = [] {
        const char *e = getenv("TREESPEC_PDL");
        return !(e && *e && atoi(e) == 0);
    }();
    return on;
}
}  // namespace ts

extern "C" {

const char *treespec_last_error(void) { return g_err; }

const char *treespec_version(void) { return "treespec 0.1 (sm_103a)"; }

// Expansion configuration <k1..km> -> level layout (shared by tree_build and
// tree_expand_topk); false with a message on bad widths.
static bool widths_param(const int32_t *widths, int m, int n_max, ts::WidthsParam &w, const char *who) {
    if (m < 0 || m > 16) {
        ts::set_error(TS_ERR_INVALID_ARG, "%s: %d expansion levels (at most 16)", who, m);
        return false;
    }
    w = ts::WidthsParam{};
    w.m = m;
    w.level_start[0] = 0;
    w.level_start[1] = 1;
    long long level_n = 1, n = 1;
    for (int l = 0; l < m; ++l) {
        if (widths[l] < 1) {
            ts::set_error(TS_ERR_INVALID_ARG, "%s: widths[%d]=%d must be >= 1", who, l, widths[l]);
            return false;
        }
        w.width[l] = widths[l];
        level_n *= widths[l];
        n += level_n;
        if (n > n_max) {
            ts::set_error(TS_ERR_INVALID_ARG, "%s: expansion tree has more than n_max=%d nodes", who, n_max);
            return false;
        }
        w.level_start[l + 2] = (int)n;
    }
    w.n = (int)n;
    w.sub[m] = 1;
    for (int l = m - 1; l >= 0; --l) w.sub[l] = 1 + w.width[l] * w.sub[l + 1];
    return true;
}

ts_status tree_build(const ts_tree *t, const int32_t *tokens, const int32_t *parent, const int32_t *n_nodes,
                     const int32_t *widths, int m, const int32_t *prefix_len, uint32_t *status,
                     cudaStream_t stream) {
    ts_status st = check_tree(t, "tree_build");
    if (st) return st;
    if (!tokens) return fail(TS_ERR_INVALID_ARG, "tree_build: tokens is NULL");
    if (widths) {
        ts::WidthsParam w;
        if (!widths_param(widths, m, t->n_max, w, "tree_build")) return TS_ERR_INVALID_ARG;
        return cuda_result(ts::launch_tree_build_widths(*t, tokens, w, prefix_len, status, stream), "tree_build");
    }
    if (!parent || !n_nodes) return fail(TS_ERR_INVALID_ARG, "tree_build: parent mode needs parent and n_nodes");
    return cuda_result(ts::launch_tree_build_parent(*t, tokens, parent, n_nodes, prefix_len, status, stream),
                       "tree_build");
}

ts_status tree_expand_topk(int32_t *tokens, const int32_t *root_token, const float *ssm_probs, int NQ, int B,
                           int n_max, const int32_t *widths, int m, int V, uint32_t *status, cudaStream_t stream) {
    if (!tokens || !root_token || !ssm_probs || !widths) return fail(TS_ERR_INVALID_ARG, "tree_expand_topk: NULL pointer");
    if (B < 1 || n_max < 1 || n_max > TS_MAX_NODES)
        return fail(TS_ERR_INVALID_ARG, "tree_expand_topk: B=%d, n_max=%d (1..%d)", B, n_max, TS_MAX_NODES);
    if (V < 1) return fail(TS_ERR_INVALID_ARG, "tree_expand_topk: V=%d must be >= 1", V);
    ts::WidthsParam w;
    if (!widths_param(widths, m, n_max, w, "tree_expand_topk")) return TS_ERR_INVALID_ARG;
    const int n_internal = w.level_start[m];   // every node above the last level has children
    if (NQ < n_internal)
        return fail(TS_ERR_INVALID_ARG, "tree_expand_topk: NQ=%d drafter rows, %d internal nodes", NQ, n_internal);
    // one CTA per internal node (one for the root alone when m = 0: it writes the root token)
    return cuda_result(ts::launch_expand_topk(tokens, root_token, ssm_probs, NQ, B, n_max, w,
                                              n_internal > 0 ? n_internal : 1, V, status, stream),
                       "tree_expand_topk");
}

ts_status tree_build_chains(const ts_tree *t, const int32_t *root_token, const int32_t *chains, int C, int len,
                            int32_t *tokens_out, int32_t *p_row, int32_t *q_row, const int32_t *prefix_len,
                            uint32_t *status, cudaStream_t stream) {
    ts_status st = check_tree(t, "tree_build_chains");
    if (st) return st;
    if (!root_token || !chains) return fail(TS_ERR_INVALID_ARG, "tree_build_chains: root_token/chains is NULL");
    if (C < 1 || len < 1) return fail(TS_ERR_INVALID_ARG, "tree_build_chains: C=%d len=%d must be >= 1", C, len);
    if (1LL + (long long)C * len > t->n_max)
        return fail(TS_ERR_INVALID_ARG, "tree_build_chains: 1 + C*len = %lld exceeds n_max=%d", 1LL + (long long)C * len,
                    t->n_max);
    return cuda_result(ts::launch_tree_build_chains(*t, root_token, chains, C, len, tokens_out, p_row, q_row,
                                                    prefix_len, status, stream),
                       "tree_build_chains");
}

ts_status tree_build_append(const ts_tree *t, const int32_t *tokens, const int32_t *widths, int m,
                            const int32_t *prefix_len, void *k_cache, void *v_cache, const void *k_new,
                            const void *v_new, int H, int d, int L_max, ts_dtype dtype, uint32_t *status,
                            cudaStream_t stream) {
    ts_status st = check_tree(t, "tree_build_append");
    if (st) return st;
    if ((st = check_attn_shape("tree_build_append", t, H, d, L_max, dtype))) return st;
    if (!tokens || !widths || !prefix_len || !k_cache || !v_cache || !k_new || !v_new)
        return fail(TS_ERR_INVALID_ARG, "tree_build_append: NULL pointer");
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
        return fail(TS_ERR_INVALID_ARG, "tree_build_append: caches and new K/V must be 16-byte aligned");
    ts::WidthsParam w;
    if (!widths_param(widths, m, t->n_max, w, "tree_build_append")) return TS_ERR_INVALID_ARG;
    const int esize = dtype == TS_BF16 ? 2 : 4;
    return cuda_result(ts::launch_build_append_widths(*t, tokens, w, prefix_len, k_cache, v_cache, k_new, v_new, H,
                                                      d, L_max, esize, status, stream),
                       "tree_build_append");
}

ts_status kv_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new, const int32_t *prefix_len,
                    const ts_tree *t, int H, int d, int L_max, ts_dtype dtype, uint32_t *status,
                    cudaStream_t stream) {
    ts_status st = check_tree(t, "kv_append");
    if (st) return st;
    if ((st = check_attn_shape("kv_append", t, H, d, L_max, dtype))) return st;
    if (!k_cache || !v_cache || !k_new || !v_new || !prefix_len)
        return fail(TS_ERR_INVALID_ARG, "kv_append: NULL pointer");
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
        return fail(TS_ERR_INVALID_ARG, "kv_append: caches and new K/V must be 16-byte aligned");
    const int esize = dtype == TS_BF16 ? 2 : 4;
    return cuda_result(ts::launch_kv_append(k_cache, v_cache, k_new, v_new, prefix_len, *t, H, d, L_max, esize,
                                            status, stream),
                       "kv_append");
}

ts_status tree_attention(void *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *prefix_len, const ts_tree *t, int H, int d, int L_max, ts_dtype dtype,
                         float scale, void *ws, size_t ws_bytes, uint32_t *status, cudaStream_t stream) {
    ts_status st = ts::check_attention_args(out, q, k_cache, v_cache, prefix_len, t, H, d, L_max, dtype,
                                            "tree_attention");
    if (st) return st;
    if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d);
    if (dtype == TS_F32)
        return cuda_result(ts::launch_attn_f32((float *)out, (const float *)q, (const float *)k_cache,
                                               (const float *)v_cache, prefix_len, *t, H, d, L_max, scale, status,
                                               stream),
                           "tree_attention");
    const ts::AttnPlan plan = ts::attn_plan(t->B, H, t->n_max, d, L_max, dtype);
    if (!ws || ws_bytes < plan.ws_bytes)
        return fail(TS_ERR_INVALID_ARG, "tree_attention: workspace of %zu bytes needed, %zu given", plan.ws_bytes,
                    ws ? ws_bytes : (size_t)0);
    if (!aligned16(ws)) return fail(TS_ERR_INVALID_ARG, "tree_attention: workspace must be 16-byte aligned");
    const char *why = nullptr;
    cudaError_t e = ts::launch_attn_bf16(out, q, k_cache, v_cache, prefix_len, *t, H, d, L_max, scale, plan, ws,
                                         status, stream, &why);
    if (why) return fail(TS_ERR_CUDA, "tree_attention: %s", why);
    return cuda_result(e, "tree_attention");
}

ts_status tree_attention_append(void *out, const void *q, void *k_cache, void *v_cache, const void *k_new,
                                const void *v_new, const int32_t *prefix_len, const ts_tree *t, int H, int d,
                                int L_max, ts_dtype dtype, float scale, void *ws, size_t ws_bytes, uint32_t *status,
                                cudaStream_t stream) {
    ts_status st = ts::check_attention_args(out, q, k_cache, v_cache, prefix_len, t, H, d, L_max, dtype,
                                            "tree_attention_append");
    if (st) return st;
    if (!k_new || !v_new) return fail(TS_ERR_INVALID_ARG, "tree_attention_append: NULL pointer");
    if (!aligned16(k_new) || !aligned16(v_new))
        return fail(TS_ERR_INVALID_ARG, "tree_attention_append: new K/V must be 16-byte aligned");
    const ts::AttnPlan plan = dtype == TS_BF16 ? ts::attn_plan(t->B, H, t->n_max, d, L_max, dtype) : ts::AttnPlan{};
    if (dtype == TS_BF16 && (!ws || ws_bytes < plan.ws_bytes))
        return fail(TS_ERR_INVALID_ARG, "tree_attention_append: workspace of %zu bytes needed, %zu given",
                    plan.ws_bytes, ws ? ws_bytes : (size_t)0);
    if (dtype == TS_BF16 && !aligned16(ws))
        return fail(TS_ERR_INVALID_ARG, "tree_attention_append: workspace must be 16-byte aligned");
    if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d);
    if (dtype == TS_BF16 && plan.tq) {   // one launch: the persistent kernel appends as it goes
        const char *why = nullptr;
        cudaError_t e = ts::launch_attn_tq(out, q, k_cache, v_cache, prefix_len, *t, H, L_max, scale, (unsigned *)ws,
                                           status, stream, &why, ts::PagedArgs(), k_new, v_new);
        if (why) return fail(TS_ERR_CUDA, "tree_attention_append: %s", why);
        return cuda_result(e, "tree_attention_append");
    }
    const int esize = dtype == TS_BF16 ? 2 : 4;
    cudaError_t e = ts::launch_kv_append(k_cache, v_cache, k_new, v_new, prefix_len, *t, H, d, L_max, esize, status,
                                         stream);
    if (e != cudaSuccess) return cuda_result(e, "tree_attention_append");
    if (dtype == TS_F32)
        return cuda_result(ts::launch_attn_f32((float *)out, (const float *)q, (const float *)k_cache,
                                               (const float *)v_cache, prefix_len, *t, H, d, L_max, scale, status,
                                               stream),
                           "tree_attention_append");
    const char *why = nullptr;
    e = ts::launch_attn_bf16(out, q, k_cache, v_cache, prefix_len, *t, H, d, L_max, scale, plan, ws, status, stream,
                             &why);
    if (why) return fail(TS_ERR_CUDA, "tree_attention_append: %s", why);
    return cuda_result(e, "tree_attention_append");
}

ts_status verify_greedy(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *argmax_out,
                        const float *logits, const ts_tree *t, int V, void *ws, size_t ws_bytes, uint32_t *status,
                        cudaStream_t stream) {
    ts_status st = check_tree(t, "verify_greedy");
    if (st) return st;
    if (!out_tokens || !out_path || !out_count || !logits)
        return fail(TS_ERR_INVALID_ARG, "verify_greedy: NULL pointer");
    if (V < 1) return fail(TS_ERR_INVALID_ARG, "verify_greedy: V=%d must be >= 1", V);
    const size_t need = ts::greedy_ws_bytes(t->B, t->n_max, V);
    if (!ws || ws_bytes < need)
        return fail(TS_ERR_INVALID_ARG, "verify_greedy: workspace of %zu bytes needed, %zu given", need,
                    ws ? ws_bytes : (size_t)0);
    return cuda_result(ts::launch_verify_greedy(out_tokens, out_path, out_count, argmax_out, logits, *t, V, ws,
                                                status, stream),
                       "verify_greedy");
}

ts_status verify_mss(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *out_lowmargin,
                     const float *target_logits, const int32_t *p_row, int NP, const float *ssm_probs,
                     const int32_t *q_row, int NQ, const float *uniforms, float temperature, const ts_tree *t, int V,
                     uint32_t *status, cudaStream_t stream) {
    ts_status st = check_tree(t, "verify_mss");
    if (st) return st;
    if (!out_tokens || !out_path || !out_count || !target_logits || !ssm_probs || !q_row || !uniforms)
        return fail(TS_ERR_INVALID_ARG, "verify_mss: NULL pointer");
    if (V < 1) return fail(TS_ERR_INVALID_ARG, "verify_mss: V=%d must be >= 1", V);
    if (!(temperature > 0.f)) return fail(TS_ERR_INVALID_ARG, "verify_mss: temperature must be > 0");
    if (NQ < 1) return fail(TS_ERR_INVALID_ARG, "verify_mss: NQ=%d must be >= 1", NQ);
    if (!p_row && NP < t->n_max)
        return fail(TS_ERR_INVALID_ARG, "verify_mss: without p_row, NP=%d must be >= n_max=%d", NP, t->n_max);
    if (NP < 1) return fail(TS_ERR_INVALID_ARG, "verify_mss: NP=%d must be >= 1", NP);
    if (V % 4 == 0 && !aligned16(target_logits))
        return fail(TS_ERR_INVALID_ARG, "verify_mss: target_logits must be 16-byte aligned");
    return cuda_result(ts::launch_verify_mss(out_tokens, out_path, out_count, out_lowmargin, target_logits, p_row, NP,
                                             ssm_probs, q_row, NQ, uniforms, temperature, *t, V, status, stream),
                       "verify_mss");
}

ts_status verify_naive(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *out_lowmargin,
                       const float *target_logits, const int32_t *p_row, int NP, const float *uniforms,
                       float temperature, const ts_tree *t, int V, uint32_t *status, cudaStream_t stream) {
    ts_status st = check_tree(t, "verify_naive");
    if (st) return st;
    if (!out_tokens || !out_path || !out_count || !target_logits || !uniforms)
        return fail(TS_ERR_INVALID_ARG, "verify_naive: NULL pointer");
    if (V < 1) return fail(TS_ERR_INVALID_ARG, "verify_naive: V=%d must be >= 1", V);
    if (!(temperature > 0.f)) return fail(TS_ERR_INVALID_ARG, "verify_naive: temperature must be > 0");
    if (!p_row && NP < t->n_max)
        return fail(TS_ERR_INVALID_ARG, "verify_naive: without p_row, NP=%d must be >= n_max=%d", NP, t->n_max);
    if (NP < 1) return fail(TS_ERR_INVALID_ARG, "verify_naive: NP=%d must be >= 1", NP);
    if (V % 4 == 0 && !aligned16(target_logits))
        return fail(TS_ERR_INVALID_ARG, "verify_naive: target_logits must be 16-byte aligned");
    return cuda_result(ts::launch_verify_naive(out_tokens, out_path, out_count, out_lowmargin, target_logits, p_row,
                                               NP, uniforms, temperature, *t, V, status, stream),
                       "verify_naive");
}

ts_status kv_commit(void *k_cache, void *v_cache, const int32_t *prefix_len, int32_t *new_prefix_len,
                    const int32_t *out_path, const int32_t *out_count, const ts_tree *t, int H, int d, int L_max,
                    ts_dtype dtype, uint32_t *status, cudaStream_t stream) {
    ts_status st = check_tree(t, "kv_commit");
    if (st) return st;
    if ((st = check_attn_shape("kv_commit", t, H, d, L_max, dtype))) return st;
    if (!k_cache || !v_cache || !prefix_len || !new_prefix_len || !out_path || !out_count)
        return fail(TS_ERR_INVALID_ARG, "kv_commit: NULL pointer");
    if (new_prefix_len == prefix_len) return fail(TS_ERR_INVALID_ARG, "kv_commit: new_prefix_len aliases prefix_len");
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(TS_ERR_INVALID_ARG, "kv_commit: caches must be 16-byte aligned");
    const int esize = dtype == TS_BF16 ? 2 : 4;
    return cuda_result(ts::launch_kv_commit(k_cache, v_cache, prefix_len, new_prefix_len, out_path, out_count, *t, H,
                                            d, L_max, esize, status, stream),
                       "kv_commit");
}

// ---- paged cache -------------------------------------------------------------
static ts_status check_paged(const ts_paged_kv *kv, const ts_tree *t, int H, int d, const char *who) {
    if (!kv || !kv->k_pages || !kv->v_pages || !kv->block_table) return fail(TS_ERR_INVALID_ARG, "%s: NULL cache", who);
    if (kv->num_pages < 1 || kv->max_pages < 1)
        return fail(TS_ERR_INVALID_ARG, "%s: num_pages=%d, max_pages=%d", who, kv->num_pages, kv->max_pages);
    if ((long long)kv->num_pages * H * TS_PAGE_KEYS >= (1LL << 31))
        return fail(TS_ERR_INVALID_ARG, "%s: 2^31 cache rows or more", who);
    if (!aligned16(kv->k_pages) || !aligned16(kv->v_pages))
        return fail(TS_ERR_INVALID_ARG, "%s: pages must be 16-byte aligned", who);
    return check_attn_shape(who, t, H, d, kv->max_pages * TS_PAGE_KEYS, TS_BF16);
}

static ts::PagedArgs paged_args(const ts_paged_kv *kv) {
    ts::PagedArgs pg;
    pg.bt = kv->block_table;
    pg.max_pages = kv->max_pages;
    pg.num_pages = kv->num_pages;
    return pg;
}

ts_status kv_append_paged(const ts_paged_kv *kv, const void *k_new, const void *v_new, const int32_t *prefix_len,
                          const ts_tree *t, int H, int d, uint32_t *status, cudaStream_t stream) {
    ts_status st = check_tree(t, "kv_append_paged");
    if (st || (st = check_paged(kv, t, H, d, "kv_append_paged"))) return st;
    if (!k_new || !v_new || !prefix_len) return fail(TS_ERR_INVALID_ARG, "kv_append_paged: NULL pointer");
    if (!aligned16(k_new) || !aligned16(v_new))
        return fail(TS_ERR_INVALID_ARG, "kv_append_paged: k_new and v_new must be 16-byte aligned");
    return cuda_result(ts::launch_kv_append(kv->k_pages, kv->v_pages, k_new, v_new, prefix_len, *t, H, d,
                                            kv->max_pages * TS_PAGE_KEYS, 2, status, stream, paged_args(kv)),
                       "kv_append_paged");
}

ts_status tree_attention_paged(void *out, const void *q, const ts_paged_kv *kv, const int32_t *prefix_len,
                               const ts_tree *t, int H, int d, float scale, void *ws, size_t ws_bytes,
                               uint32_t *status, cudaStream_t stream) {
    ts_status st = check_tree(t, "tree_attention_paged");
    if (st || (st = check_paged(kv, t, H, d, "tree_attention_paged"))) return st;
    if (!out || !q || !prefix_len) return fail(TS_ERR_INVALID_ARG, "tree_attention_paged: NULL pointer");
    if (!aligned16(out) || !aligned16(q))
        return fail(TS_ERR_INVALID_ARG, "tree_attention_paged: q and out must be 16-byte aligned");
    if (!(scale > 0.f)) scale = 1.0f / sqrtf((float)d);
    const int L_max = kv->max_pages * TS_PAGE_KEYS;
    const ts::AttnPlan plan = ts::attn_plan(t->B, H, t->n_max, d, L_max, TS_BF16);
    if (!ws || ws_bytes < plan.ws_bytes)
        return fail(TS_ERR_INVALID_ARG, "tree_attention_paged: workspace of %zu bytes needed, %zu given",
                    plan.ws_bytes, ws ? ws_bytes : (size_t)0);
    if (!aligned16(ws)) return fail(TS_ERR_INVALID_ARG, "tree_attention_paged: workspace must be 16-byte aligned");
    const char *why = nullptr;
    cudaError_t e = ts::launch_attn_bf16(out, q, kv->k_pages, kv->v_pages, prefix_len, *t, H, d, L_max, scale, plan,
                                         ws, status, stream, &why, paged_args(kv));
    if (why) return fail(TS_ERR_CUDA, "tree_attention_paged: %s", why);
    return cuda_result(e, "tree_attention_paged");
}

ts_status kv_commit_paged(const ts_paged_kv *kv, const int32_t *prefix_len, int32_t *new_prefix_len,
                          const int32_t *out_path, const int32_t *out_count, const ts_tree *t, int H, int d,
                          uint32_t *status, cudaStream_t stream) {
    ts_status st = check_tree(t, "kv_commit_paged");
    if (st || (st = check_paged(kv, t, H, d, "kv_commit_paged"))) return st;
    if (!prefix_len || !new_prefix_len || !out_path || !out_count)
        return fail(TS_ERR_INVALID_ARG, "kv_commit_paged: NULL pointer");
    if (new_prefix_len == prefix_len)
        return fail(TS_ERR_INVALID_ARG, "kv_commit_paged: new_prefix_len aliases prefix_len");
    return cuda_result(ts::launch_kv_commit(kv->k_pages, kv->v_pages, prefix_len, new_prefix_len, out_path, out_count,
                                            *t, H, d, kv->max_pages * TS_PAGE_KEYS, 2, status, stream,
                                            paged_args(kv)),
                       "kv_commit_paged");
}

size_t treespec_workspace_size(ts_op op, int B, int H, int n_max, int d, int L_max, int V) {
    if (B < 1 || n_max < 1 || n_max > TS_MAX_NODES) return 0;
    switch (op) {
        case TS_OP_ATTENTION:
            if (H < 1 || (d != 64 && d != 128) || L_max < n_max) return 0;
            return ts::attn_plan(B, H, n_max, d, L_max, TS_BF16).ws_bytes;
        case TS_OP_VERIFY_GREEDY:
            return ts::greedy_ws_bytes(B, n_max, V);
        default:
            return 0;
    }
}

const char *treespec_attention_kernel(int B, int H, int n_max, int d, int L_max, ts_dtype dtype) {
    if (B < 1 || H < 1 || n_max < 1 || n_max > TS_MAX_NODES || (d != 64 && d != 128) || L_max < n_max ||
        (dtype != TS_F32 && dtype != TS_BF16))
        return "";
    return ts::attn_plan(B, H, n_max, d, L_max, dtype).kernel;
}

ts_status treespec_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream) {
    if (!ws || ws_bytes == 0) return ok();
    return cuda_result(cudaMemsetAsync(ws, 0, ws_bytes, stream), "treespec_workspace_init");
}

}  // extern "C"
