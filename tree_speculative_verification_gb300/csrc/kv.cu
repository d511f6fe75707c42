// kv.cu -- shared tree KV cache: append the pass's K/V in depth-first order,
// and commit the accepted path.
//
// SpecInfer (arXiv 2305.09781) sec. 4.2: one KV cache holds the verified
// prefix followed by every tree node in depth-first order; after
// verification only the accepted tokens keep their cache entries.
#include "ts_internal.cuh"

namespace ts {
namespace {

constexpr int kKvThreads = 256;

// cache[b][h][P + dfs_of[v]] = new[b][v][h], 16-byte vectors; one CTA per
// (head, request), the request's depth-first map staged in shared memory and
// four independent copies in flight per thread.
__global__ void __launch_bounds__(kKvThreads) k_kv_append(uint4 *k_cache, uint4 *v_cache, const uint4 *k_new,
                                                          const uint4 *v_new, const int32_t *prefix_len, ts_tree t,
                                                          int H, int row_vec, int L_max, uint32_t *status,
                                                          PagedArgs pg) {
    const int b = blockIdx.y, h = blockIdx.x;
    pdl_wait();
    pdl_trigger();
    const int n = t.n_nodes[b], P = prefix_len[b];
    if (n <= 0) return;
    if (P < 0 || P + n > L_max) {
        if (h == 0 && threadIdx.x == 0) flag(status, TS_STATUS_INDEX);
        return;
    }
    // cache row of every node (row P + its depth-first index)
    __shared__ long long dst_s[kMaxNodes];
    __shared__ int bad_s;
    if (threadIdx.x == 0) bad_s = 0;
    __syncthreads();
    for (int v = threadIdx.x; v < n; v += kKvThreads) {
        dst_s[v] = cache_row(pg, b, h, H, L_max, P + t.dfs_of[(size_t)b * t.n_max + v]);
        if (dst_s[v] < 0) bad_s = 1;
    }
    __syncthreads();
    if (bad_s) {
        if (h == 0 && threadIdx.x == 0) flag(status, TS_STATUS_INDEX);
        return;
    }
    const int total = n * row_vec;
    for (int base = threadIdx.x; base < total; base += 4 * kKvThreads) {
        uint4 kv[4], vv[4];
        size_t dst[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int idx = base + k * kKvThreads;
            if (idx < total) {
                const int v = idx / row_vec, c = idx - v * row_vec;
                const size_t src = (((size_t)b * t.n_max + v) * H + h) * row_vec + c;
                dst[k] = (size_t)dst_s[v] * row_vec + c;
                kv[k] = __ldcs(k_new + src);
                vv[k] = __ldcs(v_new + src);
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
            if (base + k * kKvThreads < total) {
                k_cache[dst[k]] = kv[k];
                v_cache[dst[k]] = vv[k];
            }
    }
}

// One CTA per (request, group of kCommitHeads heads): one wave of CTAs for
// the workloads' batches, and one short chain of dependent loads per CTA.
// Path node i moves from row P + dfs(path[i]) to row P + i. The counts, the
// path and the request's whole depth-first map are fetched in one round trip;
// then the moves go in rounds of increasing path index, each round reading all
// its 16-byte pieces and, after a barrier, writing them. A round's destinations
// (rows P + i) are never a later round's sources, because a node's DFS index
// is at least its depth, dfs(path[i']) >= i' > i; rows already in place
// (dfs(path[i]) == i) are not copied. Measured in a graph (LLaMA-7B-shaped
// layer, 8 requests x 32 heads): one 256-thread CTA per (head, request) 1.7
// us, one 512-thread CTA per request 2.8 us.
constexpr int kCommitThreads = 256, kCommitPer = 4, kCommitHeads = 8;

__global__ void __launch_bounds__(kCommitThreads) k_kv_commit(uint4 *k_cache, uint4 *v_cache, const int32_t *prefix_len,
                                                              int32_t *new_prefix_len, const int32_t *out_path,
                                                              const int32_t *out_count, ts_tree t, int H, int row_vec,
                                                              int L_max, uint32_t *status, PagedArgs pg) {
    const int b = blockIdx.x, tid = threadIdx.x;
    const int h0 = blockIdx.y * kCommitHeads, hn = min(H - h0, kCommitHeads);   // this CTA's heads
    const bool lead = blockIdx.y == 0;   // writes the new prefix length and the status
    pdl_wait();
    pdl_trigger();
    __shared__ int dfs_s[kMaxNodes], src_s[kMaxNodes + 1];
    __shared__ long long from_s[kMaxNodes + 1], to_s[kMaxNodes + 1];   // cache rows of head 0
    __shared__ int bad_s;
    const int n = t.n_nodes[b], P = prefix_len[b], cnt = out_count[b];
    const int32_t *path = out_path + (size_t)b * (t.n_max + 1);
    // cnt <= n_max <= kMaxNodes = kCommitThreads: one path entry and one
    // depth-first index per thread, fetched with the counts
    static_assert(kCommitThreads >= kMaxNodes, "a thread per path entry and per node");
    const int v_mine = tid < t.n_max ? path[tid] : -1;
    const int dfs_mine = tid < t.n_max ? t.dfs_of[(size_t)b * t.n_max + tid] : -1;
    if (tid == 0) bad_s = !(n > 0 && cnt >= 0 && cnt <= n && P >= 0 && P + n <= L_max);
    if (tid < t.n_max) dfs_s[tid] = dfs_mine;
    __syncthreads();
    if (!bad_s && tid < cnt) {
        if (v_mine < 0 || v_mine >= n) bad_s = 1;
        else src_s[tid] = dfs_s[v_mine];
    }
    __syncthreads();
    if (bad_s) {
        if (tid == 0 && lead) {
            if (cnt != 0 || (n > 0 && (P < 0 || P + n > L_max))) flag(status, TS_STATUS_INDEX);
            new_prefix_len[b] = P;
        }
        return;
    }
    // rows of head h are those of head 0 plus h * hs (dense strips of L_max
    // rows, or pages holding TS_PAGE_KEYS rows of every head)
    const long long hs = pg.bt ? TS_PAGE_KEYS : L_max;
    if (tid < cnt) {
        from_s[tid] = cache_row(pg, b, 0, H, L_max, P + src_s[tid]);
        to_s[tid] = cache_row(pg, b, 0, H, L_max, P + tid);
        if (from_s[tid] < 0 || to_s[tid] < 0) bad_s = 1;
    }
    __syncthreads();
    if (bad_s) {
        if (tid == 0 && lead) {
            flag(status, TS_STATUS_INDEX);
            new_prefix_len[b] = P;
        }
        return;
    }
    const int per_i = hn * row_vec;   // pieces of one path node, this CTA's heads
    const int total = cnt * per_i;
    for (int r0 = 0; r0 < total; r0 += kCommitThreads * kCommitPer) {
        uint4 kx[kCommitPer], vx[kCommitPer];
        size_t dst[kCommitPer];
        bool mv[kCommitPer];
#pragma unroll
        for (int k = 0; k < kCommitPer; ++k) {
            const int idx = r0 + k * kCommitThreads + tid;
            mv[k] = false;
            if (idx < total) {
                const int i = idx / per_i, rem = idx - i * per_i, h = h0 + rem / row_vec, c = rem % row_vec;
                if (src_s[i] != i) {
                    mv[k] = true;
                    const size_t src = (size_t)(from_s[i] + h * hs) * row_vec + c;
                    dst[k] = (size_t)(to_s[i] + h * hs) * row_vec + c;
                    kx[k] = k_cache[src];
                    vx[k] = v_cache[src];
                }
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kCommitPer; ++k)
            if (mv[k]) {
                k_cache[dst[k]] = kx[k];
                v_cache[dst[k]] = vx[k];
            }
        __syncthreads();
    }
    if (tid == 0 && lead) new_prefix_len[b] = P + cnt;
}

}  // namespace

cudaError_t launch_kv_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                             const int32_t *prefix_len, const ts_tree &t, int H, int d, int L_max, int esize,
                             uint32_t *status, cudaStream_t s, const PagedArgs &pg) {
    const int row_vec = d * esize / 16;
    dim3 grid(H, t.B);
    return launch(k_kv_append, grid, dim3(kKvThreads), 0, s, (uint4 *)k_cache, (uint4 *)v_cache, (const uint4 *)k_new,
                  (const uint4 *)v_new, prefix_len, t, H, row_vec, L_max, status, pg);
}

cudaError_t launch_kv_commit(void *k_cache, void *v_cache, const int32_t *prefix_len, int32_t *new_prefix_len,
                             const int32_t *out_path, const int32_t *out_count, const ts_tree &t, int H, int d,
                             int L_max, int esize, uint32_t *status, cudaStream_t s, const PagedArgs &pg) {
    const int row_vec = d * esize / 16;
    return launch(k_kv_commit, dim3(t.B, (H + kCommitHeads - 1) / kCommitHeads), dim3(kCommitThreads), 0, s,
                  (uint4 *)k_cache, (uint4 *)v_cache, prefix_len,
                  new_prefix_len, out_path, out_count, t, H, row_vec, L_max, status, pg);
}

}  // namespace ts
