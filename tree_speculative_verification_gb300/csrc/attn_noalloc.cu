// attn_noalloc.cu -- tree_attention for callers that cannot allocate device memory.
//
// Some callers are not allowed to allocate device memory themselves: plugin or
// callback code that runs inside a host framework which owns every device
// allocation and forbids cudaMalloc on its execution path, or serving loops
// that must not allocate once they are warmed up. They still own their inputs
// and outputs, but cannot provide the split-KV workspace tree_attention needs.
// This entry point takes that workspace from a fixed scratch array compiled
// into the library instead.
//
// The array lives in device memory of every GPU on which the library's device
// code is loaded, for the life of the process, and holds
// TS_NOALLOC_SCRATCH_BYTES. Every call on a device shares it: its contents are
// whatever the previous call left, so the counters the chosen kernel needs at
// zero (split counters, or the persistent kernel's item queue) are cleared on
// the call's stream before each launch, and calls whose kernels overlap on the
// GPU (different streams, no ordering between them) race on it.
#include <mutex>

#include "ts_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_scratch[TS_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device. The host-side name
// g_scratch is only a stand-in for the symbol, not a device address: the
// address has to come from cudaGetSymbolAddress, once per device, with that
// device current.
cudaError_t scratch_ptr(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ts_status tree_attention_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                                            const int32_t *prefix_len, const ts_tree *t, int H, int d, int L_max,
                                            ts_dtype dtype, float scale, uint32_t *status, cudaStream_t stream) {
    // every check tree_attention makes, before anything is enqueued
    ts_status st = ts::check_attention_args(out, q, k_cache, v_cache, prefix_len, t, H, d, L_max, dtype,
                                            "tree_attention_noalloc");
    if (st) return st;
    if (dtype != TS_BF16)   // the fp32 kernel uses no workspace: nothing to replace
        return tree_attention(out, q, k_cache, v_cache, prefix_len, t, H, d, L_max, dtype, scale, nullptr, 0, status,
                              stream);
    const ts::AttnPlan plan = ts::attn_plan(t->B, H, t->n_max, d, L_max, dtype);
    if (plan.ws_bytes > TS_NOALLOC_SCRATCH_BYTES || plan.zero_bytes > plan.ws_bytes)
        return ts::set_error(TS_ERR_INVALID_ARG,
                             "tree_attention_noalloc: these sizes need %zu bytes of scratch, the built-in scratch "
                             "holds %zu (use tree_attention with a caller-provided workspace)",
                             plan.ws_bytes, (size_t)TS_NOALLOC_SCRATCH_BYTES);
    void *ws = nullptr;
    cudaError_t e = scratch_ptr(&ws);
    if (e != cudaSuccess)
        return ts::set_error(TS_ERR_CUDA, "tree_attention_noalloc: cudaGetSymbolAddress failed: %s",
                             cudaGetErrorString(e));
    // the plan's counters (split counters, or the persistent kernel's item
    // queue) must start at zero; the previous call may have left anything
    if (plan.zero_bytes > 0) {
        e = cudaMemsetAsync(ws, 0, plan.zero_bytes, stream);
        if (e != cudaSuccess)
            return ts::set_error(TS_ERR_CUDA, "tree_attention_noalloc: clearing the scratch failed: %s",
                                 cudaGetErrorString(e));
    }
    return tree_attention(out, q, k_cache, v_cache, prefix_len, t, H, d, L_max, dtype, scale, ws,
                          (size_t)TS_NOALLOC_SCRATCH_BYTES, status, stream);
}
