// kv.cu -- shared tree KV cache: append the pass's K/V in depth-first order,
// and commit the accepted path.
//
// SpecInfer (arXiv 2305.09781) sec. 4.2: one KV cache holds the verified
// prefix followed by every tree node in depth-first order; after
// verification only the accepted tokens keep their cache entries.
#include "ts_internal.cuh"

namespace ts {
namespace {

// cache[b][h][P + dfs_of[v]] = new[b][v][h], 16-byte vectors.
__global__ void __launch_bounds__(128) k_kv_append(uint4 *k_cache, uint4 *v_cache, const uint4 *k_new,
                                                   const uint4 *v_new, const int32_t *prefix_len, ts_tree t,
                                                   int H, int row_vec, int L_max, uint32_t *status) {
    const int b = blockIdx.y, h = blockIdx.x;
    const int n = t.n_nodes[b], P = prefix_len[b];
    if (n <= 0) return;
    if (P < 0 || P + n > L_max) {
        if (h == 0 && threadIdx.x == 0) flag(status, TS_STATUS_INDEX);
        return;
    }
    const int32_t *dfs_of = t.dfs_of + (size_t)b * t.n_max;
    const size_t cache_base = ((size_t)b * H + h) * L_max + P;
    const int total = n * row_vec;
    for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
        const int v = idx / row_vec, c = idx - v * row_vec;
        const size_t src = (((size_t)b * t.n_max + v) * H + h) * row_vec + c;
        const size_t dst = (cache_base + dfs_of[v]) * row_vec + c;
        k_cache[dst] = k_new[src];
        v_cache[dst] = v_new[src];
    }
}

// One warp per (b, h). Path node i moves from row P + dfs(path[i]) to row
// P + i. Since dfs(path[i]) >= i (a node's DFS index is at least its depth),
// handling the rows in increasing i never overwrites a row still to be read,
// and every lane touches the same 16-byte column in every row.
__global__ void __launch_bounds__(32) k_kv_commit(uint4 *k_cache, uint4 *v_cache, const int32_t *prefix_len,
                                                  int32_t *new_prefix_len, const int32_t *out_path,
                                                  const int32_t *out_count, ts_tree t, int H, int row_vec,
                                                  int L_max, uint32_t *status) {
    const int b = blockIdx.y, h = blockIdx.x, lane = threadIdx.x;
    const int n = t.n_nodes[b], P = prefix_len[b];
    int cnt = out_count[b];
    bool ok = n > 0 && cnt >= 0 && cnt <= n && P >= 0 && P + n <= L_max;
    const int32_t *path = out_path + (size_t)b * (t.n_max + 1);
    const int32_t *dfs_of = t.dfs_of + (size_t)b * t.n_max;
    for (int i = 0; ok && i < cnt; ++i) ok = path[i] >= 0 && path[i] < n;
    if (!ok) {
        if (h == 0 && lane == 0) {
            if (cnt != 0 || (n > 0 && (P < 0 || P + n > L_max))) flag(status, TS_STATUS_INDEX);
            new_prefix_len[b] = P;
        }
        return;
    }
    const size_t base = ((size_t)b * H + h) * L_max + P;
    for (int i = 0; i < cnt; ++i) {
        const int src_row = dfs_of[path[i]];
        if (src_row == i) continue;
        for (int c = lane; c < row_vec; c += 32) {
            k_cache[(base + i) * row_vec + c] = k_cache[(base + src_row) * row_vec + c];
            v_cache[(base + i) * row_vec + c] = v_cache[(base + src_row) * row_vec + c];
        }
    }
    if (h == 0 && lane == 0) new_prefix_len[b] = P + cnt;
}

}  // namespace

cudaError_t launch_kv_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                             const int32_t *prefix_len, const ts_tree &t, int H, int d, int L_max, int esize,
                             uint32_t *status, cudaStream_t s) {
    const int row_vec = d * esize / 16;
    dim3 grid(H, t.B);
    k_kv_append<<<grid, 128, 0, s>>>((uint4 *)k_cache, (uint4 *)v_cache, (const uint4 *)k_new,
                                     (const uint4 *)v_new, prefix_len, t, H, row_vec, L_max, status);
    return cudaGetLastError();
}

cudaError_t launch_kv_commit(void *k_cache, void *v_cache, const int32_t *prefix_len, int32_t *new_prefix_len,
                             const int32_t *out_path, const int32_t *out_count, const ts_tree &t, int H, int d,
                             int L_max, int esize, uint32_t *status, cudaStream_t s) {
    const int row_vec = d * esize / 16;
    dim3 grid(H, t.B);
    k_kv_commit<<<grid, 32, 0, s>>>((uint4 *)k_cache, (uint4 *)v_cache, prefix_len, new_prefix_len, out_path,
                                    out_count, t, H, row_vec, L_max, status);
    return cudaGetLastError();
}

}  // namespace ts
