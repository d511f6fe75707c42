// attn_f32.cu -- fp32 tree attention (reference-precision variant).
//
// TreeAttention(u) = Attention(S_u) (SpecInfer, arXiv 2305.09781, Def. 4.1):
// node u attends the verified prefix and the nodes on its root path, the
// topology-aware mask of sec. 4.2 taken from the ancestor-or-self bitmask.
// One CTA per (head, request), one warp per node, lanes split the head
// dimension; online softmax over the visible keys. Meant for small fp32
// problems (the bf16 path is the bandwidth-optimised one).
#include <math.h>

#include "ts_internal.cuh"

namespace ts {
namespace {

template <int D>
__global__ void __launch_bounds__(256) k_attn_f32(float *out, const float *q, const float *k_cache,
                                                  const float *v_cache, const int32_t *prefix_len, ts_tree t,
                                                  int H, int L_max, float scale, uint32_t *status) {
    constexpr int PER = D / 32;
    const int h = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const int n = t.n_nodes[b], P = prefix_len[b];
    if (n <= 0) return;
    if (P < 0 || P + n > L_max) {
        if (h == 0 && threadIdx.x == 0) flag(status, TS_STATUS_INDEX);
        return;
    }
    const int n_max = t.n_max, W = TS_MASK_WORDS(n_max);
    const float *kb = k_cache + ((size_t)b * H + h) * L_max * D;
    const float *vb = v_cache + ((size_t)b * H + h) * L_max * D;
    for (int i = warp; i < n; i += 8) {
        const int v = t.perm[(size_t)b * n_max + i];
        const uint32_t *anc = t.anc + ((size_t)b * n_max + i) * W;
        const float *qr = q + (((size_t)b * n_max + v) * H + h) * D;
        float qv[PER], acc[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) { qv[e] = qr[lane + 32 * e]; acc[e] = 0.f; }
        float m = -INFINITY, l = 0.f;
        const int L = P + n;
        for (int j = 0; j < L; ++j) {
            if (j >= P) {
                const int a = j - P;
                if (!((anc[a >> 5] >> (a & 31)) & 1u)) continue;
            }
            const float *kr = kb + (size_t)j * D;
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) s = fmaf(qv[e], kr[lane + 32 * e], s);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            s *= scale;
            const float mn = fmaxf(m, s);
            const float alpha = expf(m - mn), p = expf(s - mn);
            l = l * alpha + p;
            const float *vr = vb + (size_t)j * D;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = fmaf(acc[e], alpha, p * vr[lane + 32 * e]);
            m = mn;
        }
        float *orow = out + (((size_t)b * n_max + v) * H + h) * D;
        const float inv = 1.f / l;
#pragma unroll
        for (int e = 0; e < PER; ++e) orow[lane + 32 * e] = acc[e] * inv;
    }
}

}  // namespace

cudaError_t launch_attn_f32(float *out, const float *q, const float *k_cache, const float *v_cache,
                            const int32_t *prefix_len, const ts_tree &t, int H, int d, int L_max, float scale,
                            uint32_t *status, cudaStream_t s) {
    dim3 grid(H, t.B);
    if (d == 64)
        return launch(k_attn_f32<64>, grid, dim3(256), 0, s, out, q, k_cache, v_cache, prefix_len, t, H, L_max, scale,
                      status);
    return launch(k_attn_f32<128>, grid, dim3(256), 0, s, out, q, k_cache, v_cache, prefix_len, t, H, L_max, scale,
                  status);
}

}  // namespace ts
