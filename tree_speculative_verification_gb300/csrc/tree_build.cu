// tree_build.cu -- depth-first linearisation of speculated token trees.
//
// SpecInfer (arXiv 2305.09781) sec. 4.2 / Fig. 4: the tree's nodes sit in one
// KV cache after the verified prefix in depth-first order; sec. 3 / Fig. 3:
// expansion configuration <k1..km>; Def. 3.2: merge of drafter sequences.
// "Speculative decoding" concept page, Implementation sketch: position id =
// prefix length + depth.
//
// One CTA of TS_MAX_NODES threads per request; thread v owns input node v.
// The DFS index of v is the sum, over the nodes on its root path, of
// 1 + (sizes of the earlier siblings), which needs only subtree sizes and
// sibling order -- no sequential traversal.
#include <climits>
#include <math.h>

#include "ts_internal.cuh"

namespace ts {
namespace {

struct Smem {
    int par[kMaxNodes];
    int tok[kMaxNodes];
    int size[kMaxNodes];
    int depth[kMaxNodes];
    int off[kMaxNodes];
    int dfs[kMaxNodes];
    int slot_node[kMaxNodes];
    int roots;
    int bad;
};

__device__ void write_empty(const ts_tree &t, int b) {
    const int n_max = t.n_max, W = TS_MASK_WORDS(n_max);
    for (int i = threadIdx.x; i < n_max; i += blockDim.x) {
        size_t o = (size_t)b * n_max + i;
        t.perm[o] = -1;
        t.dfs_of[o] = -1;
        t.parent[o] = -1;
        t.token[o] = -1;
        t.depth[o] = -1;
        if (t.pos) t.pos[o] = -1;
        t.sub_end[o] = -1;
        for (int w = 0; w < W; ++w) t.anc[o * W + w] = 0u;
    }
}

// Linearise the tree held in sm.par / sm.tok (n nodes). Writes every row of
// request b, including padding, and t.n_nodes[b].
__device__ void linearize(const ts_tree &t, int b, int n, Smem &sm, int P, uint32_t *status) {
    const int v = threadIdx.x;
    if (v == 0) { sm.roots = 0; sm.bad = 0; }
    __syncthreads();
    if (v < n) {
        int p = sm.par[v];
        if (p == -1) atomicAdd(&sm.roots, 1);
        else if (p < 0 || p >= n || p == v) sm.bad = 1;
    }
    __syncthreads();
    if (v == 0 && sm.roots != 1) sm.bad = 1;
    __syncthreads();
    if (!sm.bad && v < n) {          // every node must reach the root within n steps
        int u = v, steps = 0;
        while (sm.par[u] != -1 && steps <= n) { u = sm.par[u]; ++steps; }
        if (sm.par[u] != -1) sm.bad = 1;
        sm.depth[v] = steps;
        sm.size[v] = 1;
    }
    __syncthreads();
    if (sm.bad) {
        write_empty(t, b);
        if (v == 0) { t.n_nodes[b] = 0; flag(status, TS_STATUS_BAD_TREE); }
        return;
    }
    if (v < n)   // count v in the subtree of each proper ancestor
        for (int u = sm.par[v]; u != -1; u = sm.par[u]) atomicAdd(&sm.size[u], 1);
    __syncthreads();
    if (v < n) {
        int p = sm.par[v], o = 0;
        if (p != -1) {
            o = 1;
            for (int w = 0; w < v; ++w)
                if (sm.par[w] == p) o += sm.size[w];
        }
        sm.off[v] = o;
    }
    __syncthreads();
    if (v < n) {
        int i = 0;
        for (int u = v; u != -1; u = sm.par[u]) i += sm.off[u];
        sm.dfs[v] = i;
    }
    __syncthreads();
    const int n_max = t.n_max, W = TS_MASK_WORDS(n_max);
    if (v < n) {
        const int i = sm.dfs[v];
        const size_t o = (size_t)b * n_max + i;
        t.perm[o] = v;
        t.dfs_of[(size_t)b * n_max + v] = i;
        t.parent[o] = sm.par[v] < 0 ? -1 : sm.dfs[sm.par[v]];
        t.token[o] = sm.tok[v];
        t.depth[o] = sm.depth[v];
        if (t.pos) t.pos[o] = P + sm.depth[v];
        t.sub_end[o] = i + sm.size[v];
        uint32_t words[kMaxWords];
#pragma unroll
        for (int w = 0; w < kMaxWords; ++w) words[w] = 0u;
        for (int u = v; u != -1; u = sm.par[u]) {
            int j = sm.dfs[u];
            words[j >> 5] |= 1u << (j & 31);
        }
        for (int w = 0; w < W; ++w) t.anc[o * W + w] = words[w];
    } else if (v < n_max) {
        const size_t o = (size_t)b * n_max + v;
        t.perm[o] = -1;
        t.dfs_of[o] = -1;
        t.parent[o] = -1;
        t.token[o] = -1;
        t.depth[o] = -1;
        if (t.pos) t.pos[o] = -1;
        t.sub_end[o] = -1;
        for (int w = 0; w < W; ++w) t.anc[o * W + w] = 0u;
    }
    if (v == 0) t.n_nodes[b] = n;
}

__global__ void __launch_bounds__(kMaxNodes) k_build_parent(ts_tree t, const int32_t *tokens,
                                                            const int32_t *parent, const int32_t *n_nodes,
                                                            const int32_t *prefix_len, uint32_t *status) {
    __shared__ Smem sm;
    const int b = blockIdx.x, v = threadIdx.x;
    const int n = n_nodes[b];
    pdl_wait();
    pdl_trigger();
    const int P = prefix_len ? prefix_len[b] : 0;
    if (n < 1 || n > t.n_max) {
        __syncthreads();
        write_empty(t, b);
        if (v == 0) { t.n_nodes[b] = 0; flag(status, TS_STATUS_BAD_TREE); }
        return;
    }
    if (v < n) {
        sm.par[v] = parent[(size_t)b * t.n_max + v];
        sm.tok[v] = tokens[(size_t)b * t.n_max + v];
    }
    __syncthreads();
    linearize(t, b, n, sm, P, status);
}

// Expansion trees (sec. 3, Fig. 3): every node at depth d has width[d]
// children, numbered level by level, so a node's place in depth-first order is
// mixed-radix arithmetic on the subtree sizes sub[]: thread i takes
// depth-first position i, walks down from the root choosing child
// (rest - 1) / sub[d + 1] at each depth, and gets its input id, depth, parent,
// subtree end and ancestors without shared memory or barriers.
// Tree arrays of request b, DFS position i (one thread per position).
__device__ __forceinline__ void build_widths_node(const ts_tree &t, const int32_t *tokens, const WidthsParam &w,
                                                  int P, int b, int i) {
    const int n = w.n, n_max = t.n_max, W = TS_MASK_WORDS(n_max);
    const size_t o = (size_t)b * n_max + i;
    if (i < n) {
        int d = 0, pos = 0, par = -1, idx = 0;   // current node: depth, DFS position, parent position, index in level
        int rest = i;                            // DFS offset of the target inside the current subtree
        int path[17];                            // DFS positions on the root path
        path[0] = 0;
#pragma unroll
        for (int l = 0; l < 16; ++l)
            if (l < w.m && rest > 0) {
                const int c = (rest - 1) / w.sub[l + 1];
                par = pos;
                pos = pos + 1 + c * w.sub[l + 1];
                rest = rest - 1 - c * w.sub[l + 1];
                idx = idx * w.width[l] + c;
                d = l + 1;
                path[d] = pos;
            }
        const int v = w.level_start[d] + idx;
        t.perm[o] = v;
        t.dfs_of[(size_t)b * n_max + v] = i;
        t.parent[o] = par;
        t.token[o] = tokens[(size_t)b * n_max + v];
        t.depth[o] = d;
        if (t.pos) t.pos[o] = P + d;
        t.sub_end[o] = i + w.sub[d];
        for (int wd = 0; wd < W; ++wd) {
            uint32_t bits = 0u;
#pragma unroll
            for (int l = 0; l <= 16; ++l)
                if (l <= d && (path[l] >> 5) == wd) bits |= 1u << (path[l] & 31);
            t.anc[o * W + wd] = bits;
        }
    } else if (i < n_max) {
        t.perm[o] = -1;
        t.dfs_of[o] = -1;
        t.parent[o] = -1;
        t.token[o] = -1;
        t.depth[o] = -1;
        if (t.pos) t.pos[o] = -1;
        t.sub_end[o] = -1;
        for (int wd = 0; wd < W; ++wd) t.anc[o * W + wd] = 0u;
    }
    if (i == 0) t.n_nodes[b] = n;
}

__global__ void __launch_bounds__(kMaxNodes) k_build_widths(ts_tree t, const int32_t *tokens, WidthsParam w,
                                                            const int32_t *prefix_len, uint32_t *status) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    build_widths_node(t, tokens, w, prefix_len ? prefix_len[b] : 0, b, threadIdx.x);
    (void)status;
}

// Depth-first position of the node with level-order id v of an expansion tree:
// v sits at level d with index idx in it, whose mixed-radix digits c_0 .. c_{d-1}
// (radices widths[0..d-1]) are the child ranks on its root path; every step
// down passes the node itself and c_l whole subtrees of the level below.
__device__ __forceinline__ int widths_dfs_of(const WidthsParam &w, int v) {
    int d = 0;
#pragma unroll
    for (int l = 1; l <= 16; ++l)
        if (l <= w.m && v >= w.level_start[l]) d = l;
    int idx = v - w.level_start[d], pos = 0;
    for (int l = d - 1; l >= 0; --l) {   // digits from the last level up
        const int c = idx % w.width[l];
        idx /= w.width[l];
        pos += 1 + c * w.sub[l + 1];
    }
    return pos;
}

// tree_build for an expansion tree and kv_append in one launch: CTA (h, b)
// copies head h of request b's new K/V rows to cache rows P + dfs(v) (the
// positions are arithmetic, so the copy does not wait for the tree arrays),
// and the CTAs of head 0 also write the tree arrays. The results equal the two
// separate calls'.
__global__ void __launch_bounds__(kMaxNodes) k_build_append_widths(ts_tree t, const int32_t *tokens, WidthsParam w,
                                                                   const int32_t *prefix_len, uint4 *k_cache,
                                                                   uint4 *v_cache, const uint4 *k_new,
                                                                   const uint4 *v_new, int H, int row_vec, int L_max,
                                                                   uint32_t *status) {
    const int b = blockIdx.y, h = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    const int P = prefix_len[b], n = w.n;
    if (h == 0) build_widths_node(t, tokens, w, P, b, threadIdx.x);
    if (P < 0 || P + n > L_max) {
        if (h == 0 && threadIdx.x == 0) flag(status, TS_STATUS_INDEX);
        return;
    }
    __shared__ int dfs_s[kMaxNodes];
    for (int v = threadIdx.x; v < n; v += kMaxNodes) dfs_s[v] = widths_dfs_of(w, v);
    __syncthreads();
    const size_t base_row = ((size_t)b * H + h) * L_max + P;
    const int total = n * row_vec;
    for (int base = threadIdx.x; base < total; base += 4 * kMaxNodes) {
        uint4 kv[4], vv[4];
        size_t dst[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int idx = base + k * kMaxNodes;
            if (idx < total) {
                const int v = idx / row_vec, c = idx - v * row_vec;
                const size_t src = (((size_t)b * t.n_max + v) * H + h) * row_vec + c;
                dst[k] = (base_row + dfs_s[v]) * row_vec + c;
                kv[k] = __ldcs(k_new + src);
                vv[k] = __ldcs(v_new + src);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (base + k * kMaxNodes < total) {
                k_cache[dst[k]] = kv[k];
                v_cache[dst[k]] = vv[k];
            }
    }
}

// Def. 3.2 merge, data-parallel: slot s = (chain c, position p). The slot
// opens a new node iff no earlier chain holds the same tokens 0..p; the new
// nodes are numbered by slot order (creation order), the root being node 0.
__global__ void __launch_bounds__(kMaxNodes) k_build_chains(ts_tree t, const int32_t *root_token,
                                                            const int32_t *chains, int C, int len,
                                                            int32_t *tokens_out, int32_t *p_row,
                                                            int32_t *q_row, const int32_t *prefix_len,
                                                            uint32_t *status) {
    __shared__ Smem sm;
    __shared__ int is_new[kMaxNodes];
    __shared__ int canon[kMaxNodes];
    __shared__ int n_sh;
    const int b = blockIdx.x, s = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const int S = C * len;
    const int32_t *ch = chains + (size_t)b * S;
    const int P = prefix_len ? prefix_len[b] : 0;
    if (s < S) {
        const int c = s / len, p = s % len;
        int cs = c;
        for (int c2 = 0; c2 < c; ++c2) {
            bool same = true;
            for (int q = 0; q <= p && same; ++q) same = ch[c2 * len + q] == ch[c * len + q];
            if (same) { cs = c2; break; }
        }
        canon[s] = cs * len + p;
        is_new[s] = cs == c;
    }
    __syncthreads();
    if (s < S && is_new[s]) {
        int id = 1;
        for (int s2 = 0; s2 < s; ++s2) id += is_new[s2];
        sm.slot_node[s] = id;
    }
    __syncthreads();
    if (s < S && !is_new[s]) sm.slot_node[s] = sm.slot_node[canon[s]];
    if (s == 0) {
        int cnt = 1;
        for (int s2 = 0; s2 < S; ++s2) cnt += is_new[s2];
        n_sh = cnt;
    }
    __syncthreads();
    const int n = n_sh;
    const size_t base = (size_t)b * t.n_max;
    if (s < S && is_new[s]) {
        const int v = sm.slot_node[s], p = s % len;
        sm.par[v] = p == 0 ? 0 : sm.slot_node[s - 1];
        sm.tok[v] = ch[s];
        if (p_row) p_row[base + v] = 1 + s;
        if (q_row) q_row[base + v] = s;
    }
    if (s == 0) {
        sm.par[0] = -1;
        sm.tok[0] = root_token[b];
        if (p_row) p_row[base] = 0;
        if (q_row) q_row[base] = -1;
    }
    for (int v = n + s; v < t.n_max; v += blockDim.x) {
        if (p_row) p_row[base + v] = -1;
        if (q_row) q_row[base + v] = -1;
        if (tokens_out) tokens_out[base + v] = -1;
    }
    __syncthreads();
    if (tokens_out && s < n) tokens_out[base + s] = sm.tok[s];
    linearize(t, b, n, sm, P, status);
}

// Top-k expansion (sec. 3, Fig. 3: the SSM expands each node of depth i-1
// into its k_i most likely next tokens). One CTA per (internal node u,
// request): u's children, consecutive in level order, take the k best tokens
// of drafter row u in the order (probability desc, id asc). Pass r keeps the
// best entry that ranks strictly below the pass r-1 pick in that order, so k
// passes over the row need no list of picked tokens.
constexpr int kExpandThreads = 256;

__device__ __forceinline__ bool ranks_above(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kExpandThreads) k_expand_topk(int32_t *tokens, const int32_t *root_token,
                                                                const float *ssm, int NQ, WidthsParam w, int V,
                                                                int n_max, bool vec4, uint32_t *status) {
    const int u = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    if (u == 0 && tid == 0) tokens[(size_t)b * n_max] = root_token[b];
    int l = 0;
    while (l < w.m && u >= w.level_start[l + 1]) ++l;
    if (l >= w.m) return;   // a leaf (only for m = 0: the root alone)
    const int k = w.width[l];
    const int first = w.level_start[l + 1] + (u - w.level_start[l]) * k;
    const float *row = ssm + ((size_t)b * NQ + u) * V;
    __shared__ float s_v[kExpandThreads / 32];
    __shared__ int s_i[kExpandThreads / 32];
    __shared__ int s_nf;
    __shared__ float pick_v;
    __shared__ int pick_i;
    if (tid == 0) s_nf = 0;
    float lv = INFINITY;
    int li = -1;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = INT_MAX;
        bool nf = false;
        auto take = [&](float x, int i) {
            if (r == 0 && !isfinite(x)) nf = true;
            if ((x < lv || (x == lv && i > li)) && ranks_above(x, i, bv, bi)) { bv = x; bi = i; }
        };
        if (vec4) {
            const float4 *r4 = reinterpret_cast<const float4 *>(row);
            for (int g = tid; g < (V >> 2); g += kExpandThreads) {
                const float4 a = __ldg(r4 + g);
                take(a.x, 4 * g); take(a.y, 4 * g + 1); take(a.z, 4 * g + 2); take(a.w, 4 * g + 3);
            }
        } else {
            for (int i = tid; i < V; i += kExpandThreads) take(__ldg(row + i), i);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ranks_above(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        nf = __any_sync(0xffffffffu, nf);
        if ((tid & 31) == 0) {
            s_v[tid >> 5] = bv;
            s_i[tid >> 5] = bi;
            if (nf) s_nf = 1;
        }
        __syncthreads();
        if (tid == 0) {
            for (int q = 1; q < kExpandThreads / 32; ++q)
                if (ranks_above(s_v[q], s_i[q], bv, bi)) { bv = s_v[q]; bi = s_i[q]; }
            pick_v = bv;
            pick_i = bi < V ? bi : -1;   // fewer than k tokens in the row
        }
        __syncthreads();
        if (s_nf) {   // a non-finite drafter value: the children get no token
            if (tid < k) tokens[(size_t)b * n_max + first + tid] = -1;
            if (tid == 0) flag(status, TS_STATUS_NONFINITE);
            return;
        }
        lv = pick_v;
        li = pick_i;
        if (tid == 0) tokens[(size_t)b * n_max + first + r] = li;
        __syncthreads();   // pick_v / pick_i are rewritten by the next pass
        if (li < 0) return;
    }
}

}  // namespace

cudaError_t launch_tree_build_parent(const ts_tree &t, const int32_t *tokens, const int32_t *parent,
                                     const int32_t *n_nodes, const int32_t *prefix_len, uint32_t *status,
                                     cudaStream_t s) {
    return launch(k_build_parent, dim3(t.B), dim3(kMaxNodes), 0, s, t, tokens, parent, n_nodes, prefix_len, status);
}

cudaError_t launch_tree_build_widths(const ts_tree &t, const int32_t *tokens, const WidthsParam &w,
                                     const int32_t *prefix_len, uint32_t *status, cudaStream_t s) {
    return launch(k_build_widths, dim3(t.B), dim3(kMaxNodes), 0, s, t, tokens, w, prefix_len, status);
}

cudaError_t launch_build_append_widths(const ts_tree &t, const int32_t *tokens, const WidthsParam &w,
                                       const int32_t *prefix_len, void *k_cache, void *v_cache, const void *k_new,
                                       const void *v_new, int H, int d, int L_max, int esize, uint32_t *status,
                                       cudaStream_t s) {
    const int row_vec = d * esize / 16;
    return launch(k_build_append_widths, dim3(H, t.B), dim3(kMaxNodes), 0, s, t, tokens, w, prefix_len,
                  (uint4 *)k_cache, (uint4 *)v_cache, (const uint4 *)k_new, (const uint4 *)v_new, H, row_vec, L_max,
                  status);
}

cudaError_t launch_tree_build_chains(const ts_tree &t, const int32_t *root_token, const int32_t *chains, int C,
                                     int len, int32_t *tokens_out, int32_t *p_row, int32_t *q_row,
                                     const int32_t *prefix_len, uint32_t *status, cudaStream_t s) {
    return launch(k_build_chains, dim3(t.B), dim3(kMaxNodes), 0, s, t, root_token, chains, C, len, tokens_out, p_row,
                  q_row, prefix_len, status);
}

cudaError_t launch_expand_topk(int32_t *tokens, const int32_t *root_token, const float *ssm, int NQ, int B,
                              int n_max, const WidthsParam &w, int n_internal, int V, uint32_t *status,
                              cudaStream_t s) {
    const bool vec4 = (V % 4 == 0) && ((uintptr_t)ssm % 16 == 0);
    return launch(k_expand_topk, dim3(n_internal, B), dim3(kExpandThreads), 0, s, tokens, root_token, ssm, NQ, w, V,
                  n_max, vec4, status);
}

}  // namespace ts
