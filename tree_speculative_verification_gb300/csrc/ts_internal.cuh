// ts_internal.cuh -- shared internals of libtreespec (kernel launchers, device helpers).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/treespec.h"

namespace ts {

constexpr int kMaxNodes = TS_MAX_NODES;
constexpr int kMaxWords = TS_MASK_WORDS(TS_MAX_NODES);

// Bounded waits: a spin gives up after this many clock64 cycles (about 2 s at
// 2 GHz), records TS_STATUS_TIMEOUT and lets the kernel return.
constexpr long long kWaitCycles = 4000000000LL;

__device__ __forceinline__ void flag(uint32_t *status, uint32_t bits) {
    if (status) atomicOr(status, bits);
}

// ---- programmatic dependent launch ------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialization: it may be scheduled while the kernel before it on the stream
// is still running, and pdl_wait() -- the first thing each kernel does before
// it reads or writes global memory -- blocks until that kernel has completed
// and its writes are visible. pdl_trigger() lets the next kernel be scheduled
// early. Both are no-ops without a programmatic neighbour.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

bool pdl_enabled();   // false when TREESPEC_PDL=0

template <typename... K, typename... A>
cudaError_t launch(void (*kern)(K...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

// ---- launchers (one per .cu file) -------------------------------------------
struct WidthsParam {
    int m;
    int n;                 // total node count
    int level_start[17];   // start id of each level, level_start[m+1] = n
    int width[16];
    int sub[17];           // size of a subtree rooted at depth d (sub[m] = 1)
};

cudaError_t launch_tree_build_parent(const ts_tree &t, const int32_t *tokens, const int32_t *parent,
                                     const int32_t *n_nodes, const int32_t *prefix_len,
                                     uint32_t *status, cudaStream_t s);
cudaError_t launch_build_append_widths(const ts_tree &t, const int32_t *tokens, const WidthsParam &w,
                                       const int32_t *prefix_len, void *k_cache, void *v_cache, const void *k_new,
                                       const void *v_new, int H, int d, int L_max, int esize, uint32_t *status,
                                       cudaStream_t s);
cudaError_t launch_tree_build_widths(const ts_tree &t, const int32_t *tokens, const WidthsParam &w,
                                     const int32_t *prefix_len, uint32_t *status, cudaStream_t s);
cudaError_t launch_tree_build_chains(const ts_tree &t, const int32_t *root_token, const int32_t *chains,
                                     int C, int len, int32_t *tokens_out, int32_t *p_row, int32_t *q_row,
                                     const int32_t *prefix_len, uint32_t *status, cudaStream_t s);

cudaError_t launch_expand_topk(int32_t *tokens, const int32_t *root_token, const float *ssm, int NQ, int B,
                              int n_max, const WidthsParam &w, int n_internal, int V, uint32_t *status,
                              cudaStream_t s);

// Row addressing of the KV cache: dense [B][H][L_max][d] when bt is null, else
// pages of TS_PAGE_KEYS rows ([page][H][TS_PAGE_KEYS][d]) listed per request in
// bt [B][max_pages]. Returns the cache row of (b, h, logical row r), or -1 for
// a page id outside [0, num_pages).
struct PagedArgs {
    const int32_t *bt = nullptr;
    int max_pages = 0, num_pages = 0;
};
__device__ __forceinline__ long long cache_row(const PagedArgs &pg, int b, int h, int H, int L_max, int r) {
    if (!pg.bt) return ((long long)b * H + h) * L_max + r;
    const int page = pg.bt[(size_t)b * pg.max_pages + r / TS_PAGE_KEYS];
    if (page < 0 || page >= pg.num_pages) return -1;
    return ((long long)page * H + h) * TS_PAGE_KEYS + r % TS_PAGE_KEYS;
}

cudaError_t launch_kv_append(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                             const int32_t *prefix_len, const ts_tree &t, int H, int d, int L_max,
                             int esize, uint32_t *status, cudaStream_t s, const PagedArgs &pg = PagedArgs());
cudaError_t launch_kv_commit(void *k_cache, void *v_cache, const int32_t *prefix_len, int32_t *new_prefix_len,
                             const int32_t *out_path, const int32_t *out_count, const ts_tree &t, int H,
                             int d, int L_max, int esize, uint32_t *status, cudaStream_t s,
                             const PagedArgs &pg = PagedArgs());

// Split-KV plan shared by the size query and the launch.
struct AttnPlan {
    int splits;          // CTAs per (b, h) at most
    int chunk_tiles;     // 64-key tiles per CTA
    int n_pad;           // node rows kept per partial
    size_t ws_bytes;     // workspace bytes the launch uses
    const char *kernel;  // name of the kernel the launch uses
    bool tq = false;     // the persistent 128-key-tile tcgen05 kernel
    size_t zero_bytes = 0;   // leading workspace bytes that must be zero before a launch (counters)
};
// Workspace of the persistent tcgen05 kernel: its item queue, two unsigned
// counters (next item, CTAs finished) that the last CTA returns to zero.
constexpr size_t kTqQueueBytes = 256;
AttnPlan attn_plan(int B, int H, int n_max, int d, int L_max, ts_dtype dt);

cudaError_t launch_attn_f32(float *out, const float *q, const float *k_cache, const float *v_cache,
                            const int32_t *prefix_len, const ts_tree &t, int H, int d, int L_max,
                            float scale, uint32_t *status, cudaStream_t s);
// Persistent tcgen05 kernel with 128-key tiles (head_dim 128, at most 128
// nodes); queue = the plan's workspace (kTqQueueBytes, zero before the launch).
// With k_new / v_new (dense cache only) the same launch also appends the new
// K/V rows to the cache (kv_append), in a tenth warp of each CTA.
cudaError_t launch_attn_tq(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *prefix_len, const ts_tree &t, int H, int L_max, float scale,
                           unsigned *queue, uint32_t *status, cudaStream_t s, const char **why, const PagedArgs &pg,
                           const void *k_new = nullptr, const void *v_new = nullptr);
cudaError_t launch_attn_bf16(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *prefix_len, const ts_tree &t, int H, int d, int L_max,
                             float scale, const AttnPlan &plan, void *ws, uint32_t *status, cudaStream_t s,
                             const char **why, const PagedArgs &pg = PagedArgs());

size_t greedy_ws_bytes(int B, int n_max, int V);
cudaError_t launch_verify_greedy(int32_t *out_tokens, int32_t *out_path, int32_t *out_count,
                                 int32_t *argmax_out, const float *logits, const ts_tree &t, int V, void *ws,
                                 uint32_t *status, cudaStream_t s);
cudaError_t launch_verify_mss(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *out_lowmargin,
                              const float *logits, const int32_t *p_row, int NP, const float *ssm,
                              const int32_t *q_row, int NQ, const float *uniforms, float temperature,
                              const ts_tree &t, int V, uint32_t *status, cudaStream_t s);

cudaError_t launch_verify_naive(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *out_lowmargin,
                                const float *logits, const int32_t *p_row, int NP, const float *uniforms,
                                float temperature, const ts_tree &t, int V, uint32_t *status, cudaStream_t s);

int num_sms();

ts_status set_error(ts_status st, const char *fmt, ...);
ts_status check_attention_args(const void *out, const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *prefix_len, const ts_tree *t, int H, int d, int L_max, ts_dtype dtype,
                               const char *who);

}  // namespace ts
