// attn_f32.cu -- fp32 tree attention (reference-precision variant).
//
// TreeAttention(u) = Attention(S_u) (SpecInfer, arXiv 2305.09781, Def. 4.1):
// node u attends the verified prefix and the nodes on its root path, the
// topology-aware mask of sec. 4.2 taken from the ancestor-or-self bitmask.
// One CTA per (head, request), one warp per node; keys in chunks of 32: each
// lane scores one key of the chunk, one maximum and one sum per chunk (online
// softmax), then P V with the lanes over the head dimension. Meant for small
// fp32 problems (the bf16 path is the bandwidth-optimised one).
#include <math.h>

#include "ts_internal.cuh"

namespace ts {
namespace {

template <int D>
__global__ void __launch_bounds__(256, 1) k_attn_f32(float *out, const float *q, const float *k_cache,
                                                  const float *v_cache, const int32_t *prefix_len, ts_tree t,
                                                  int H, int L_max, float scale, uint32_t *status) {
    constexpr int PER = D / 32;
    const int h = blockIdx.x, b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __shared__ __align__(16) float q_s[8][D];   // each warp's current node row
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
    const int L = P + n;
    for (int i = warp; i < n; i += 8) {
        const int v = t.perm[(size_t)b * n_max + i];
        const uint32_t *anc = t.anc + ((size_t)b * n_max + i) * W;
        const float *qr = q + (((size_t)b * n_max + v) * H + h) * D;
#pragma unroll
        for (int e = 0; e < PER; ++e) q_s[warp][lane + 32 * e] = qr[lane + 32 * e];
        __syncwarp();
        float acc[PER];
#pragma unroll
        for (int e = 0; e < PER; ++e) acc[e] = 0.f;
        float m = -INFINITY, l = 0.f;
        // 32 keys at a time: lane j scores key c + j, one maximum and one sum per
        // chunk, then P V with the lanes over the head dimension
        for (int c = 0; c < L; c += 32) {
            const int j = c + lane;
            bool vis = j < L;
            if (vis && j >= P) vis = (anc[(j - P) >> 5] >> ((j - P) & 31)) & 1u;
            float s = -INFINITY;
            if (vis) {
                const float4 *kr = reinterpret_cast<const float4 *>(kb + (size_t)j * D);
                const float4 *q4 = reinterpret_cast<const float4 *>(q_s[warp]);
                float d = 0.f;
#pragma unroll
                for (int e = 0; e < D / 4; ++e) {
                    const float4 kv = kr[e], qv = q4[e];
                    d = fmaf(qv.x, kv.x, d); d = fmaf(qv.y, kv.y, d); d = fmaf(qv.z, kv.z, d); d = fmaf(qv.w, kv.w, d);
                }
                s = d * scale;
            }
            float mc = s;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
            if (mc == -INFINITY) continue;   // no visible key in this chunk
            const float mn = fmaxf(m, mc);
            const float alpha = expf(m - mn);   // 0 while nothing was accumulated
            const float p = vis ? expf(s - mn) : 0.f;
            float ps = p;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            l = l * alpha + ps;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] *= alpha;
            const int kn = min(32, L - c);
            for (int k = 0; k < kn; ++k) {
                const float pk = __shfl_sync(0xffffffffu, p, k);
                if (pk != 0.f) {
                    const float *vr = vb + (size_t)(c + k) * D;
#pragma unroll
                    for (int e = 0; e < PER; ++e) acc[e] = fmaf(pk, vr[lane + 32 * e], acc[e]);
                }
            }
            m = mn;
        }
        float *orow = out + (((size_t)b * n_max + v) * H + h) * D;
        const float inv = 1.f / l;
#pragma unroll
        for (int e = 0; e < PER; ++e) orow[lane + 32 * e] = acc[e] * inv;
        __syncwarp();   // q_s is rewritten for the warp's next node
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
