// verify.cu -- tree verification kernels (SpecInfer, arXiv 2305.09781, sec. 4.3,
// Algorithm 2: VerifyGreedy and VerifyStochastic / multi-step speculative
// sampling; residual norm(max(0, p - q)) as in "How Speculative Decoding in
// LLM Serving Actually Works").
//
// verify_greedy: node-parallel. Every (request, node, vocab segment) CTA
//   streams its slice of the target logits once (argmax, lowest id on ties);
//   the last CTA of a request merges the segments and walks the tree.
// verify_mss / verify_naive: walk-first. One 1024-thread CTA per request follows Algorithm 2
//   and touches only the rows on the accepted path (the target row of each
//   visited node, the drafter rows of its tested children); each step is a
//   block-wide reduction over the vocabulary. Elementwise work is fp32; sums
//   are per-thread compensated (Kahan) fp32, merged as float-float across
//   threads (k_walk, rows in shared memory) or in fp64 across warps (k_mss,
//   the form for rows that do not fit shared memory).
#include <float.h>
#include <math.h>

#include "attn_common.cuh"
#include "ts_internal.cuh"

namespace ts {
namespace {

// ---------------------------------------------------------------- greedy ----
constexpr int kMaxSeg = 8;
constexpr int kGreedyBulkMin = 16384;   // segments from this size on arrive by bulk copy

struct ArgPart {
    float val;
    int idx;   // -1: the segment held a non-finite value
};

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__device__ __forceinline__ void consider(float x, int i, float &bv, int &bi, bool &nf) {
    if (!isfinite(x)) nf = true;
    if (x > bv) { bv = x; bi = i; }   // indices arrive in increasing order per thread
}

// mode 0: scalar loads; 1: float4 loads, eight in flight per thread; 2: the
// segment by one bulk copy into shared memory (dynamic shared memory of the
// segment's size)
template <int kGreedyThreads>
__global__ void __launch_bounds__(kGreedyThreads) k_greedy(int32_t *out_tokens, int32_t *out_path,
                                                           int32_t *out_count, int32_t *argmax_out,
                                                           const float *logits, ts_tree t, int V, int seg,
                                                           int mode, unsigned *counters, ArgPart *parts,
                                                           uint32_t *status) {
    extern __shared__ __align__(16) float4 gseg[];
    __shared__ __align__(8) unsigned long long gbar;
    const int b = blockIdx.y;
    const int v = blockIdx.x / seg, sg = blockIdx.x % seg;
    pdl_wait();
    pdl_trigger();
    const int n = t.n_nodes[b];
    const int n_max = t.n_max;
    if (n <= 0) {
        if (blockIdx.x == 0 && threadIdx.x == 0) out_count[b] = 0;
        return;
    }
    if (v >= n) return;
    const float *row = logits + ((size_t)b * n_max + v) * V;
    float bv = -FLT_MAX;
    int bi = INT_MAX;
    bool nf = false, tmo = false;
    if (mode == 2) {
        const int V4 = V >> 2, per = (V4 + seg - 1) / seg;
        const int g0 = sg * per, g1 = min(V4, g0 + per);
        const uint32_t bar = smem_u32(&gbar);
        if (threadIdx.x == 0) {
            mbar_init(bar, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            mbar_expect_tx(bar, (uint32_t)(g1 - g0) * 16u);
            if (g1 > g0) bulk_g2s(smem_u32(gseg), reinterpret_cast<const float4 *>(row) + g0, (uint32_t)(g1 - g0) * 16u, bar);
        }
        __syncthreads();
        if (!mbar_wait_bounded(bar, 0)) {
            tmo = true;
        } else {
            for (int g = threadIdx.x; g < g1 - g0; g += kGreedyThreads) {
                const float4 a = gseg[g];
                consider(a.x, 4 * (g0 + g), bv, bi, nf);
                consider(a.y, 4 * (g0 + g) + 1, bv, bi, nf);
                consider(a.z, 4 * (g0 + g) + 2, bv, bi, nf);
                consider(a.w, 4 * (g0 + g) + 3, bv, bi, nf);
            }
        }
    } else if (mode == 1) {
        // all of a thread's loads (up to 8 x 16 bytes) in flight at once
        const int V4 = V >> 2, per = (V4 + seg - 1) / seg;
        const int g0 = sg * per, g1 = min(V4, g0 + per);
        const float4 *r4 = reinterpret_cast<const float4 *>(row);
        for (int base = g0 + threadIdx.x; base < g1; base += 8 * kGreedyThreads) {
            float4 a[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int g = base + k * kGreedyThreads;
                if (g < g1) a[k] = __ldcs(r4 + g);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int g = base + k * kGreedyThreads;
                if (g < g1) {
                    const float xs[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (!isfinite(xs[e])) nf = true;
                        if (better(xs[e], 4 * g + e, bv, bi)) { bv = xs[e]; bi = 4 * g + e; }
                    }
                }
            }
        }
    } else {
        const int per = (V + seg - 1) / seg;
        const int i0 = sg * per, i1 = min(V, i0 + per);
        for (int i = i0 + threadIdx.x; i < i1; i += kGreedyThreads) consider(row[i], i, bv, bi, nf);
    }
    // block reduction of (value, index), lowest index on ties
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    nf = __any_sync(0xffffffffu, nf);
    tmo = __any_sync(0xffffffffu, tmo);
    __shared__ float s_v[kGreedyThreads / 32];
    __shared__ int s_i[kGreedyThreads / 32];
    __shared__ int s_nf;
    __shared__ bool s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) s_nf = 0;
    __syncthreads();
    if (lane == 0) {
        s_v[warp] = bv;
        s_i[warp] = bi;
        if (nf || tmo) atomicOr(&s_nf, tmo ? 2 : 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int k = 1; k < kGreedyThreads / 32; ++k)
            if (better(s_v[k], s_i[k], bv, bi)) { bv = s_v[k]; bi = s_i[k]; }
        if (s_nf & 2) flag(status, TS_STATUS_TIMEOUT);
        ArgPart p;
        p.val = bv;
        p.idx = s_nf ? -1 : bi;
        parts[((size_t)b * n_max + v) * seg + sg] = p;
        // release of this CTA's partial, acquire of the others' for the last one
        unsigned prev;
        asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(prev) : "l"(&counters[b]) : "memory");
        s_last = prev == (unsigned)(n * seg - 1);
    }
    __syncthreads();
    if (!s_last) return;
    // ---- last CTA of request b: merge segments, then walk (Algorithm 2, VerifyGreedy)
    __shared__ int am[kMaxNodes];
    __shared__ int s_perm[kMaxNodes], s_tok[kMaxNodes], s_se[kMaxNodes];
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    for (int w = threadIdx.x; w < n; w += kGreedyThreads) {
        const size_t o = (size_t)b * n_max + w;
        s_perm[w] = t.perm[o];
        s_tok[w] = t.token[o];
        s_se[w] = t.sub_end[o];
        float cv = -FLT_MAX;
        int ci = INT_MAX;
        bool bad = false;
        ArgPart pp[kMaxSeg];   // all segment results of the node fetched at once
#pragma unroll
        for (int k = 0; k < kMaxSeg; ++k)
            if (k < seg) {
                pp[k].val = __ldcg(&parts[o * seg + k].val);
                pp[k].idx = __ldcg(&parts[o * seg + k].idx);
            }
#pragma unroll
        for (int k = 0; k < kMaxSeg; ++k)
            if (k < seg) {
                if (pp[k].idx < 0) bad = true;
                else if (better(pp[k].val, pp[k].idx, cv, ci)) { cv = pp[k].val; ci = pp[k].idx; }
            }
        am[w] = bad ? -1 : ci;
        if (bad) s_bad = 1;
        if (argmax_out) argmax_out[o] = am[w];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        counters[b] = 0u;   // leave the workspace zeroed for the next call
        int32_t *ot = out_tokens + (size_t)b * (n_max + 1);
        int32_t *op = out_path + (size_t)b * (n_max + 1);
        if (s_bad) {
            out_count[b] = 0;
            flag(status, TS_STATUS_NONFINITE);
        } else {
            int u = 0, cnt = 0;
            op[0] = s_perm[0];
            for (int step = 0; step < n; ++step) {
                const int o = am[s_perm[u]];
                int next = -1;
                for (int c = u + 1; c < s_se[u]; c = s_se[c])
                    if (s_tok[c] == o) { next = c; break; }
                ot[cnt++] = o;
                if (next < 0) break;
                op[cnt] = s_perm[next];
                u = next;
            }
            out_count[b] = cnt;
        }
    }
}

// ------------------------------------------------------------------- MSS ----
constexpr int kMssThreads = 1024;
constexpr int kMssWarps = kMssThreads / 32;
constexpr float kL2E = 1.4426950408889634f;

// float-float accumulation (Knuth two-sum)
__device__ __forceinline__ void ff_add(float &hi, float &lo, float bh, float bl) {
    float s = hi + bh;
    float v = s - hi;
    float e = (hi - (s - v)) + (bh - v);
    e += lo + bl;
    hi = s + e;
    lo = e - (hi - s);
}

__device__ __forceinline__ void kahan(float &sum, float &comp, float x) {
    float y = x - comp;
    float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
}

struct MssShared {
    double red_d[kMssWarps];
    float red_f[kMssWarps];
    int red_i[kMssWarps];
    float wh[kMssWarps], wl[kMssWarps];     // float-float warp totals of the CDF scan
    float cq[kMaxNodes];                    // q_c(x_c) of each child of the current node
    float cu[kMaxNodes];                    // its accept uniform
    int depth[kMaxNodes];
    int perm[kMaxNodes];
    int tok[kMaxNodes];
    int sub_end[kMaxNodes];
    int prow[kMaxNodes];
    int qrow[kMaxNodes];
    const float *rej_q[kMaxNodes];
    float rej_S[kMaxNodes];
    double bcast_d;
    double base;
    float bcast_f;
    float us;                               // the final-sample uniform of the current node
    int bcast_i;
    int pick;
    int token;
    int lowm;                               // decisions of the walk with a margin below kLowMargin
};
// A decision is reported as low-margin when the device's own margin is below
// this: |u - a| for an accept test, the distance of u * S to the cumulative
// sums on either side of the drawn token, over S, for a sample.
constexpr double kLowMargin = 1e-6;
constexpr size_t kMssHeader = (sizeof(MssShared) + 15) & ~(size_t)15;

// The residual of the current node. With the shared-memory row (R != nullptr)
// R[y] holds it directly; otherwise it is recomputed from the logits and the
// drafter rows of the rejections applied so far:
//   R_0(y) = e(y) = 2^((l_y / T - m) log2 e),  R_{j+1}(y) = max(0, R_j(y) - S_j q_j(y))
// with S_j = sum_y R_j(y); r_j = R_j / S_j is the normalised residual.
struct Resid {
    const float *row;
    float invT, m;
    const float *const *rq;
    const float *rS;
    int nrej;
    const float *R;
};

__device__ __forceinline__ float e_of(float l, float invT, float m) { return exp2f((l * invT - m) * kL2E); }

__device__ __forceinline__ float resid_recompute(const Resid &r, int y) {
    float v = e_of(__ldg(r.row + y), r.invT, r.m);
    for (int j = 0; j < r.nrej; ++j) v = fmaxf(0.f, __fmaf_rn(-r.rS[j], __ldg(r.rq[j] + y), v));
    return v;
}

__device__ __forceinline__ float resid_at(const Resid &r, int y) { return r.R ? r.R[y] : resid_recompute(r, y); }

__device__ double block_sum(MssShared &sm, float hi, float lo) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float bh = __shfl_xor_sync(0xffffffffu, hi, o);
        float bl = __shfl_xor_sync(0xffffffffu, lo, o);
        ff_add(hi, lo, bh, bl);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sm.red_d[warp] = (double)hi + (double)lo;
    __syncthreads();
    if (warp == 0) {
        double x = sm.red_d[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) sm.bcast_d = x;
    }
    __syncthreads();
    double r = sm.bcast_d;
    __syncthreads();
    return r;
}

__device__ float block_max(MssShared &sm, float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sm.red_f[warp] = x;
    __syncthreads();
    if (warp == 0) {
        float y = sm.red_f[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, o));
        if (lane == 0) sm.bcast_f = y;
    }
    __syncthreads();
    float r = sm.bcast_f;
    __syncthreads();
    return r;
}

__device__ int block_or(MssShared &sm, int x) {
    x = __any_sync(0xffffffffu, x);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sm.red_i[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int y = __any_sync(0xffffffffu, sm.red_i[lane]);
        if (lane == 0) sm.bcast_i = y;
    }
    __syncthreads();
    int r = sm.bcast_i;
    __syncthreads();
    return r;
}

// One CTA per request, walking the tree as Algorithm 2 does. SMEM_R keeps the
// residual row of the current node in shared memory (vocabularies up to ~53K
// entries): the exps are taken once per visited node and a rejection is one
// in-place pass over R and one drafter row. NAIVE: naive sampling instead
// (SpecInfer sec. 4.3): at each visited node draw x from p by the same inverse
// CDF, move to the first child whose token is x, else append x and stop; no
// drafter rows are read.
template <bool SMEM_R, bool NAIVE>
__global__ void __launch_bounds__(kMssThreads, 1) k_mss(int32_t *out_tokens, int32_t *out_path, int32_t *out_count,
                                                        int32_t *out_lowmargin, const float *logits,
                                                        const int32_t *p_row, int NP,
                                                        const float *ssm, const int32_t *q_row, int NQ,
                                                        const float *uniforms, float invT, ts_tree t, int V,
                                                        uint32_t *status) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    MssShared &sm = *reinterpret_cast<MssShared *>(smem_raw);
    float *Rs = SMEM_R ? reinterpret_cast<float *>(smem_raw + kMssHeader) : nullptr;
    const int b = blockIdx.x, tid = threadIdx.x;
    pdl_wait();
    pdl_trigger();
    const int n = t.n_nodes[b];
    const int n_max = t.n_max;
    int32_t *ot = out_tokens + (size_t)b * (n_max + 1);
    int32_t *op = out_path + (size_t)b * (n_max + 1);
    if (n <= 0) {
        if (tid == 0) {
            out_count[b] = 0;
            if (out_lowmargin) out_lowmargin[b] = 0;
        }
        return;
    }
    if (tid == 0) sm.lowm = 0;
    // tree and row indices into shared memory; index checks for every node
    int bad_index = 0;
    for (int i = tid; i < n; i += kMssThreads) {
        const size_t o = (size_t)b * n_max + i;
        const int v = t.perm[o];
        sm.perm[i] = v;
        sm.tok[i] = t.token[o];
        sm.sub_end[i] = t.sub_end[o];
        sm.depth[i] = t.depth[o];
        const int pr = p_row ? p_row[(size_t)b * n_max + v] : v;
        sm.prow[i] = pr;
        if (pr < 0 || pr >= NP) bad_index = 1;
        if (i > 0 && NAIVE) {
            if (sm.tok[i] < 0 || sm.tok[i] >= V) bad_index = 1;
        } else if (i > 0) {
            const int qr = q_row[(size_t)b * n_max + v];
            sm.qrow[i] = qr;
            if (qr < 0 || qr >= NQ || sm.tok[i] < 0 || sm.tok[i] >= V) bad_index = 1;
        }
    }
    __syncthreads();
    if (block_or(sm, bad_index)) {
        if (tid == 0) {
            out_count[b] = 0;
            if (out_lowmargin) out_lowmargin[b] = 0;
            flag(status, TS_STATUS_INDEX);
        }
        return;
    }
    const float *u_acc = uniforms + (size_t)b * 2 * n_max;
    const float *u_smp = u_acc + n_max;
    const bool vec = (V & 3) == 0;
    const int V4 = V >> 2;
    int u = 0, cnt = 0, nonfinite = 0;
    if (tid == 0) op[0] = sm.perm[0];

    for (int step = 0; step < n; ++step) {
        const float *row = logits + ((size_t)b * NP + sm.prow[u]) * V;
        // the values the walk tests at this node, fetched in parallel now rather
        // than one at a time later: q_c(x_c) and the accept uniform of every
        // child, the final-sample uniform of u
        {
            const int du = sm.depth[u], se_u = sm.sub_end[u];
            for (int i = u + 1 + tid; !NAIVE && i < se_u; i += kMssThreads)
                if (sm.depth[i] == du + 1) {
                    sm.cq[i] = __ldg(ssm + ((size_t)b * NQ + sm.qrow[i]) * V + sm.tok[i]);
                    sm.cu[i] = __ldg(u_acc + sm.perm[i]);
                }
            if (tid == kMssThreads - 1) sm.us = __ldg(u_smp + sm.perm[u]);
        }
        // pass 1: max of the tempered logits, finiteness (and the tempered row kept)
        float mx = -FLT_MAX;
        int nf = 0;
        if (vec) {
            // four independent 16-byte loads in flight per thread
            const float4 *r4 = reinterpret_cast<const float4 *>(row);
            for (int g0 = tid; g0 < V4; g0 += 4 * kMssThreads) {
                float4 a[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (g0 + k * kMssThreads < V4) a[k] = __ldg(r4 + g0 + k * kMssThreads);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int g = g0 + k * kMssThreads;
                    if (g < V4) {
                        nf |= !isfinite(a[k].x) | !isfinite(a[k].y) | !isfinite(a[k].z) | !isfinite(a[k].w);
                        a[k].x *= invT; a[k].y *= invT; a[k].z *= invT; a[k].w *= invT;
                        mx = fmaxf(mx, fmaxf(fmaxf(a[k].x, a[k].y), fmaxf(a[k].z, a[k].w)));
                        if (SMEM_R) reinterpret_cast<float4 *>(Rs)[g] = a[k];
                    }
                }
            }
        } else {
            for (int y0 = tid; y0 < V; y0 += 4 * kMssThreads) {
                float a[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (y0 + k * kMssThreads < V) a[k] = __ldg(row + y0 + k * kMssThreads);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int y = y0 + k * kMssThreads;
                    if (y < V) {
                        nf |= !isfinite(a[k]);
                        mx = fmaxf(mx, a[k] * invT);
                        if (SMEM_R) Rs[y] = a[k] * invT;
                    }
                }
            }
        }
        // one reduction for both: a non-finite logit makes the maximum +inf
        const float m = block_max(sm, nf ? INFINITY : mx);
        if (m == INFINITY) { nonfinite = 1; break; }
        // pass 2: e = 2^((l/T - m) log2 e) and Z = sum e
        float s = 0.f, cc = 0.f;
        if (SMEM_R) {
            if (vec) {
                for (int g = tid; g < V4; g += kMssThreads) {
                    float4 a = reinterpret_cast<float4 *>(Rs)[g];
                    a.x = exp2f((a.x - m) * kL2E); a.y = exp2f((a.y - m) * kL2E);
                    a.z = exp2f((a.z - m) * kL2E); a.w = exp2f((a.w - m) * kL2E);
                    kahan(s, cc, a.x); kahan(s, cc, a.y); kahan(s, cc, a.z); kahan(s, cc, a.w);
                    reinterpret_cast<float4 *>(Rs)[g] = a;
                }
            } else {
                for (int y = tid; y < V; y += kMssThreads) {
                    const float e = exp2f((Rs[y] - m) * kL2E);
                    Rs[y] = e;
                    kahan(s, cc, e);
                }
            }
        } else {
            for (int y = tid; y < V; y += kMssThreads) kahan(s, cc, e_of(__ldg(row + y), invT, m));
        }
        double S = block_sum(sm, s, -cc);

        // children in input order: u+1, sub_end[u+1], ... below sub_end[u]
        int nrej = 0;
        int accepted = -1;
        for (int c = u + 1; !NAIVE && c < sm.sub_end[u]; c = sm.sub_end[c]) {
            const float *qc = ssm + ((size_t)b * NQ + sm.qrow[c]) * V;
            const int x = sm.tok[c];
            const Resid rr{row, invT, m, sm.rej_q, sm.rej_S, nrej, Rs};
            if (tid == 0) {
                const float qx = sm.cq[c];
                int acc = 0, bad = !isfinite(qx);
                if (!bad) {
                    double a = 1.0;
                    if (qx > 0.f) a = fmin(1.0, (double)resid_at(rr, x) / (S * (double)qx));
                    acc = (double)sm.cu[c] <= a;
                    if (fabs((double)sm.cu[c] - a) < kLowMargin) ++sm.lowm;
                }
                sm.pick = bad ? -2 : acc;
            }
            __syncthreads();
            const int verdict = sm.pick;
            __syncthreads();
            if (verdict == -2) { nonfinite = 1; break; }
            if (verdict == 1) { accepted = c; break; }
            // rejection: R' = max(0, R - S q_c), S' = sum R'
            const float Sf = (float)S;
            float s2 = 0.f, c2 = 0.f;
            int bad = 0;
            if (SMEM_R && vec && ((uintptr_t)qc & 15u) == 0) {
                const float4 *q4 = reinterpret_cast<const float4 *>(qc);
                float4 *R4 = reinterpret_cast<float4 *>(Rs);
                for (int g0 = tid; g0 < V4; g0 += 4 * kMssThreads) {
                    float4 qv[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (g0 + k * kMssThreads < V4) qv[k] = __ldg(q4 + g0 + k * kMssThreads);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int g = g0 + k * kMssThreads;
                        if (g < V4) {
                            bad |= !isfinite(qv[k].x) | !isfinite(qv[k].y) | !isfinite(qv[k].z) | !isfinite(qv[k].w);
                            float4 r = R4[g];
                            r.x = fmaxf(0.f, __fmaf_rn(-Sf, qv[k].x, r.x));
                            r.y = fmaxf(0.f, __fmaf_rn(-Sf, qv[k].y, r.y));
                            r.z = fmaxf(0.f, __fmaf_rn(-Sf, qv[k].z, r.z));
                            r.w = fmaxf(0.f, __fmaf_rn(-Sf, qv[k].w, r.w));
                            R4[g] = r;
                            kahan(s2, c2, r.x); kahan(s2, c2, r.y); kahan(s2, c2, r.z); kahan(s2, c2, r.w);
                        }
                    }
                }
            } else if (SMEM_R) {
                for (int y0 = tid; y0 < V; y0 += 4 * kMssThreads) {
                    float qv[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (y0 + k * kMssThreads < V) qv[k] = __ldg(qc + y0 + k * kMssThreads);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int y = y0 + k * kMssThreads;
                        if (y < V) {
                            bad |= !isfinite(qv[k]);
                            const float v = fmaxf(0.f, __fmaf_rn(-Sf, qv[k], Rs[y]));
                            Rs[y] = v;
                            kahan(s2, c2, v);
                        }
                    }
                }
            } else {
                for (int y = tid; y < V; y += kMssThreads) {
                    const float qy = __ldg(qc + y);
                    bad |= !isfinite(qy);
                    kahan(s2, c2, fmaxf(0.f, __fmaf_rn(-Sf, qy, resid_recompute(rr, y))));
                }
            }
            // one reduction for both: a non-finite drafter value makes the sum NaN
            const double Snew = block_sum(sm, bad ? NAN : s2, bad ? 0.f : -c2);
            if (isnan(Snew)) { nonfinite = 1; break; }
            if (Snew > 0.0) {
                if (tid == 0) {
                    sm.rej_q[nrej] = qc;
                    sm.rej_S[nrej] = Sf;
                }
                __syncthreads();
                ++nrej;
                S = Snew;
            } else {
                if (tid == 0) flag(status, TS_STATUS_ZERO_RESID);   // keep the residual unchanged
                if (SMEM_R) {     // the in-place pass overwrote it: rebuild R from the applied rejections
                    const Resid keep{row, invT, m, sm.rej_q, sm.rej_S, nrej, nullptr};
                    for (int y = tid; y < V; y += kMssThreads) Rs[y] = resid_recompute(keep, y);
                    __syncthreads();
                }
            }
        }
        if (nonfinite) break;
        if (accepted >= 0) {
            if (tid == 0) {
                ot[cnt] = sm.tok[accepted];
                op[cnt + 1] = sm.perm[accepted];
            }
            ++cnt;
            u = accepted;
            __syncthreads();   // the next node's pass 1 overwrites R
            continue;
        }
        // inverse CDF of the residual: the first y with C(y) > u * S. Each thread
        // sums a contiguous segment (compensated fp32), a float-float block scan
        // gives every segment's starting point, the segment holding u * S is
        // found by a bracket test, and warp 0 scans inside it.
        const Resid rr{row, invT, m, sm.rej_q, sm.rej_S, nrej, Rs};
        const int per = vec ? (V4 + kMssThreads - 1) / kMssThreads : (V + kMssThreads - 1) / kMssThreads;
        const int unit = vec ? 4 : 1;
        const int warp = tid >> 5, lane = tid & 31;
        float sh, sl;
        {
            const int y0 = tid * per * unit, y1 = min(V, y0 + per * unit);
            float s3 = 0.f, c3 = 0.f;
            for (int y = y0; y < y1; ++y) kahan(s3, c3, resid_at(rr, y));
            sh = s3;
            sl = -c3;
        }
        float ih = sh, il = sl;     // inclusive warp scan (float-float)
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float bh = __shfl_up_sync(0xffffffffu, ih, o), bl = __shfl_up_sync(0xffffffffu, il, o);
            if (lane >= o) ff_add(ih, il, bh, bl);
        }
        if (lane == 31) {
            sm.wh[warp] = ih;
            sm.wl[warp] = il;
        }
        if (tid == 0) sm.pick = INT_MAX;
        __syncthreads();
        if (warp == 0) {            // exclusive scan of the 32 warp totals
            const float oh = sm.wh[lane], ol = sm.wl[lane];
            float xh = oh, xl = ol;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float bh = __shfl_up_sync(0xffffffffu, xh, o), bl = __shfl_up_sync(0xffffffffu, xl, o);
                if (lane >= o) ff_add(xh, xl, bh, bl);
            }
            if (lane == 31) sm.bcast_d = (double)xh + (double)xl;   // total mass
            ff_add(xh, xl, -oh, -ol);
            __syncwarp();
            sm.wh[lane] = xh;
            sm.wl[lane] = xl;
        }
        __syncthreads();
        float ph = ih, pl = il;
        ff_add(ph, pl, -sh, -sl);
        ff_add(ph, pl, sm.wh[warp], sm.wl[warp]);
        const double total = sm.bcast_d;
        const double target = (double)sm.us * total;
        const double lo_c = (double)ph + (double)pl, hi_c = lo_c + ((double)sh + (double)sl);
        if (hi_c > lo_c && lo_c <= target && target < hi_c) atomicMin(&sm.pick, tid);
        __syncthreads();
        if (sm.pick == INT_MAX) {   // rounding left no bracket: the last segment with mass
            __syncthreads();
            if (tid == 0) sm.pick = -1;
            __syncthreads();
            if (hi_c > lo_c) atomicMax(&sm.pick, tid);
            __syncthreads();
        }
        const int pick = sm.pick;
        if (tid == pick) sm.base = lo_c;
        __syncthreads();
        if (warp == 0) {
            int chosen = -1, last_pos = -1;
            double margin = 0.0;   // stays 0 when rounding left no bracket (the fallback pick)
            if (pick >= 0) {
                const int ys = pick * per * unit, ye = min(V, ys + per * unit);
                double carry = sm.base;
                for (int y0 = ys; y0 < ye && chosen < 0; y0 += 32) {
                    const int y = y0 + lane;
                    const float r = y < ye ? resid_at(rr, y) : 0.f;
                    float ch = r, cl = 0.f;   // inclusive scan of this 32-wide slice
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float bh = __shfl_up_sync(0xffffffffu, ch, o), bl = __shfl_up_sync(0xffffffffu, cl, o);
                        if (lane >= o) ff_add(ch, cl, bh, bl);
                    }
                    const double cum = carry + ((double)ch + (double)cl);
                    const unsigned hit = __ballot_sync(0xffffffffu, r > 0.f && cum > target);
                    const unsigned pos = __ballot_sync(0xffffffffu, r > 0.f);
                    if (hit) {
                        const int hl = __ffs(hit) - 1;
                        chosen = y0 + hl;
                        // C(t) and C(t - 1) of the drawn token t, from the lane that holds it
                        const double c_t = __shfl_sync(0xffffffffu, cum, hl);
                        const double c_prev = c_t - (double)__shfl_sync(0xffffffffu, r, hl);
                        margin = total > 0.0 ? fmin(target - c_prev, c_t - target) / total : 0.0;
                    } else if (pos) {
                        last_pos = y0 + 31 - __clz(pos);
                    }
                    carry += (double)__shfl_sync(0xffffffffu, ch, 31) + (double)__shfl_sync(0xffffffffu, cl, 31);
                }
            }
            if (chosen < 0) chosen = last_pos >= 0 ? last_pos : 0;
            if (lane == 0) {
                ot[cnt] = chosen;
                sm.token = chosen;
                if (margin < kLowMargin) ++sm.lowm;
            }
        }
        ++cnt;
        if (!NAIVE) break;
        // naive sampling: continue at the first child holding the drawn token
        __syncthreads();
        if (tid == 0) {
            int next = -1;
            for (int c = u + 1; c < sm.sub_end[u]; c = sm.sub_end[c])
                if (sm.tok[c] == sm.token) { next = c; break; }
            sm.pick = next;
            if (next >= 0) op[cnt] = sm.perm[next];
        }
        __syncthreads();
        const int next = sm.pick;
        __syncthreads();   // the next node's pass 1 overwrites R and pick
        if (next < 0) break;
        u = next;
    }
    __syncthreads();
    if (tid == 0) {
        if (nonfinite) {
            out_count[b] = 0;
            flag(status, TS_STATUS_NONFINITE);
        } else {
            out_count[b] = cnt;
        }
        if (out_lowmargin) out_lowmargin[b] = sm.lowm;
    }
}

// -------------------------------------------------- MSS / naive walk, fast form ----
// The same walk (Algorithm 2, VerifyStochastic; or naive sampling) for rows
// that fit shared memory with V a multiple of 4 and 16-byte aligned rows:
//  * warp w owns the contiguous float4 range [w C4, (w + 1) C4) of the
//    vocabulary in every pass (lane-consecutive 16-byte shared-memory accesses,
//    no bank conflicts), so the per-warp partial sums of a pass are also the
//    coarse level of the inverse CDF, and no warp ever touches another's range;
//  * each warp's range of the visited node's target row arrives by its own
//    bulk copy (TMA engine) into the residual buffer R, on the warp's own
//    mbarrier, and the warp takes its maximum, its exponentials relative to
//    that maximum and their sum as soon as its range has landed. R stays
//    relative to its warp's maximum (factor f_w to the row maximum) until the
//    first rejection pass rescales it; the tests and the final sample apply
//    f_w where it still does;
//  * a reduction is two barriers: every warp publishes its float-float
//    partial, then warp 0 alone combines the 32 partials (row maximum, S),
//    takes the child's test or the coarse level of the final sample, and
//    publishes the verdict, which every warp reads after the second barrier.
// Elementwise arithmetic is fp32 (the hardware exp2); sums are fp32 over a
// float4, compensated across float4s, float-float across threads; ratio and
// CDF tests in fp32 / float-float (no fp64 in per-thread code: GB300's fp64
// rate is low).
constexpr int kWalkThreads = 1024;
constexpr int kWalkWarps = kWalkThreads / 32;

// Verdicts of the deciding warp (a child index >= 0: that child is accepted)
constexpr int kVReject = -1;      // the tested child is rejected: its rejection pass follows
constexpr int kVSample = -2;      // no child left to test: the final sample follows
constexpr int kVZero = -3;        // the rejection left a zero normaliser: the residual is rebuilt
constexpr int kVNonfinite = -4;   // a non-finite target or drafter value
constexpr int kVTimeout = -5;     // a row copy did not complete

struct WalkShared {
    float red_mx[kWalkWarps];               // the warps' published partials
    float red_hi[kWalkWarps], red_lo[kWalkWarps];
    int red_bad[kWalkWarps];
    int bad[kWalkWarps];                    // the warps' index checks
    float f[kWalkWarps];                    // each warp's factor to the row maximum
    float cq[kMaxNodes];                    // q_c(x_c) of each child of the current node
    float cu[kMaxNodes];                    // its accept uniform
    int depth[kMaxNodes];
    int perm[kMaxNodes];
    int tok[kMaxNodes];
    int sub_end[kMaxNodes];
    int prow[kMaxNodes];
    int qrow[kMaxNodes];
    const float *rej_q[kMaxNodes];
    float rej_S[kMaxNodes];
    float Sh, Sl;                           // the current normaliser S (float-float)
    float m;                                // the row's tempered maximum (natural units)
    float rx;                               // R at the token of the child tested next
    float us;                               // the final-sample uniform of the current node
    int nrej;                               // rejections applied to the current residual
    int verdict;
    int chosen;
    int lowm;
    // the final sample's coarse level: the warp whose range holds the target,
    // whether rounding left no bracket, the warp's exclusive prefix, the target
    // u * total (float-float) and the total
    int ws, fb;
    float bh, bl, tgh, tgl, toth;
    unsigned long long wbar[kWalkWarps];    // completion of each warp's bulk copy of its range
};
constexpr size_t kWalkHeader = (sizeof(WalkShared) + 127) & ~(size_t)127;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ void warp_ff_sum(float &h, float &l) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float bh = __shfl_xor_sync(0xffffffffu, h, o), bl = __shfl_xor_sync(0xffffffffu, l, o);
        ff_add(h, l, bh, bl);
    }
}

// a > b for normalised float-float values
__device__ __forceinline__ bool ff_gt(float ah, float al, float bh, float bl) {
    return ah > bh || (ah == bh && al > bl);
}

// (h, l) * x as float-float (exact product of the high part, plus the low part's)
__device__ __forceinline__ void ff_mul_f(float h, float l, float x, float &oh, float &ol) {
    const float p = h * x;
    const float e = __fmaf_rn(h, x, -p) + l * x;
    oh = p + e;
    ol = e - (oh - p);
}

// A warp's partial of a reduction into its slots: its float-float sum (h, l),
// its maximum mx and the OR of its flags. The block barrier follows.
__device__ __forceinline__ void walk_publish(WalkShared &sm, float h, float l, float mx, int flag) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    warp_ff_sum(h, l);
    flag = __reduce_or_sync(0xffffffffu, flag);
    if (lane == 0) {
        sm.red_hi[warp] = h;
        sm.red_lo[warp] = l;
        sm.red_mx[warp] = mx;
        sm.red_bad[warp] = flag;
    }
}

// The test of child c (Algorithm 2: accept with probability
// min(1, p(x_c) / q_c(x_c)), p = R / S), by lane 0 of the deciding warp;
// kVSample when c is not a child of the current node.
__device__ void walk_test(WalkShared &sm, int c, int se_u, bool local, int C4) {
    if (c < 0 || c >= se_u) {
        sm.verdict = kVSample;
        return;
    }
    const float qx = sm.cq[c];
    if (!isfinite(qx)) {
        sm.verdict = kVNonfinite;
        return;
    }
    const float Sf = sm.Sh + sm.Sl;
    float rxv = sm.rx;
    if (local) rxv *= sm.f[(sm.tok[c] >> 2) / C4];   // R relative to the maximum of the warp holding x_c
    float a = 1.f;
    if (qx > 0.f) a = fminf(1.f, rxv / (Sf * qx));
    const float uc = sm.cu[c];
    if (fabsf(uc - a) < (float)kLowMargin) ++sm.lowm;
    sm.verdict = uc <= a ? c : kVReject;
}

// The deciding warp: the coarse level of the inverse CDF, from the warps'
// partials (times f while R is relative to the warps' maxima): the first warp
// whose inclusive prefix exceeds u * total.
__device__ void walk_coarse(WalkShared &sm, bool local) {
    const int lane = threadIdx.x & 31;
    float oh = sm.red_hi[lane], ol = sm.red_lo[lane];
    if (local) ff_mul_f(oh, ol, sm.f[lane], oh, ol);
    float ih = oh, il = ol;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float bh = __shfl_up_sync(0xffffffffu, ih, o), bl = __shfl_up_sync(0xffffffffu, il, o);
        if (lane >= o) ff_add(ih, il, bh, bl);
    }
    const float toth = __shfl_sync(0xffffffffu, ih, 31), totl = __shfl_sync(0xffffffffu, il, 31);
    float tgh, tgl;
    ff_mul_f(toth, totl, sm.us, tgh, tgl);
    const unsigned hitw = __ballot_sync(0xffffffffu, oh > 0.f && ff_gt(ih, il, tgh, tgl));
    const unsigned posw = __ballot_sync(0xffffffffu, oh > 0.f);
    const int ws = hitw ? __ffs(hitw) - 1 : (posw ? 31 - __clz(posw) : 0);
    float bh = __shfl_sync(0xffffffffu, ih, ws), bl = __shfl_sync(0xffffffffu, il, ws);
    ff_add(bh, bl, -__shfl_sync(0xffffffffu, oh, ws), -__shfl_sync(0xffffffffu, ol, ws));
    if (lane == 0) {
        sm.ws = ws;
        sm.fb = hitw == 0;
        sm.bh = bh;
        sm.bl = bl;
        sm.tgh = tgh;
        sm.tgl = tgl;
        sm.toth = toth;
    }
}

// The deciding warp after a node's statistics: the row maximum M (log2
// units), f_w = 2^(M_w - M), S = sum_w S_w f_w, then the first child's test
// (or the final sample's coarse level).
__device__ void walk_decide_stats(WalkShared &sm, int c_first, int se_u, int C4, bool naive) {
    const int lane = threadIdx.x & 31;
    const int flags = __reduce_or_sync(0xffffffffu, sm.red_bad[lane]);
    const float ml = sm.red_mx[lane];
    const float M = warp_max(ml);
    const float fl = exp2f(ml - M);   // 0 for a warp with an empty range (ml = -inf)
    float h, l;
    ff_mul_f(sm.red_hi[lane], sm.red_lo[lane], fl, h, l);
    warp_ff_sum(h, l);
    sm.f[lane] = fl;
    __syncwarp();
    if (lane == 0) {
        sm.Sh = h;
        sm.Sl = l;
        sm.m = M * 0.6931471805599453f;
        sm.nrej = 0;
        if (flags & 2) sm.verdict = kVTimeout;
        else if (flags & 1) sm.verdict = kVNonfinite;
        else if (naive) sm.verdict = kVSample;
        else walk_test(sm, c_first, se_u, true, C4);
    }
    __syncwarp();
    if (sm.verdict == kVSample) walk_coarse(sm, true);
}

// The deciding warp after child c's rejection pass: S' = sum of the residual;
// a NaN sum means a non-finite drafter value; S' > 0 records the rejection
// and tests child c_next; S' = 0 asks for the residual to be rebuilt.
__device__ void walk_decide_resid(WalkShared &sm, const float *q_c, int c_next, int se_u, int C4, uint32_t *status) {
    const int lane = threadIdx.x & 31;
    float h = sm.red_hi[lane], l = sm.red_lo[lane];
    warp_ff_sum(h, l);
    if (lane == 0) {
        if (isnan(h)) {
            sm.verdict = kVNonfinite;
        } else if (h > 0.f) {
            sm.rej_q[sm.nrej] = q_c;
            sm.rej_S[sm.nrej] = sm.Sh + sm.Sl;
            ++sm.nrej;
            sm.Sh = h;
            sm.Sl = l;
            walk_test(sm, c_next, se_u, false, C4);
        } else {
            flag(status, TS_STATUS_ZERO_RESID);
            sm.verdict = kVZero;
        }
    }
    __syncwarp();
    if (sm.verdict == kVSample) walk_coarse(sm, false);
}

// The deciding warp after the residual was rebuilt (S unchanged): the test of
// child c_next.
__device__ void walk_decide_rebuilt(WalkShared &sm, int c_next, int se_u, int C4) {
    const int lane = threadIdx.x & 31;
    if (lane == 0) walk_test(sm, c_next, se_u, false, C4);
    __syncwarp();
    if (sm.verdict == kVSample) walk_coarse(sm, false);
}

template <bool NAIVE>
__global__ void __launch_bounds__(kWalkThreads, 1) k_walk(int32_t *out_tokens, int32_t *out_path, int32_t *out_count,
                                                          int32_t *out_lowmargin, const float *logits,
                                                          const int32_t *p_row, int NP, const float *ssm,
                                                          const int32_t *q_row, int NQ, const float *uniforms,
                                                          float invT, ts_tree t, int V, uint32_t *status) {
    extern __shared__ __align__(128) unsigned char walk_smem[];
    WalkShared &sm = *reinterpret_cast<WalkShared *>(walk_smem);
    float *R = reinterpret_cast<float *>(walk_smem + kWalkHeader);
    float4 *R4 = reinterpret_cast<float4 *>(R);
    const int b = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t wbar = smem_u32(&sm.wbar[warp]);
    pdl_wait();
    pdl_trigger();
    const int n = t.n_nodes[b];
    const int n_max = t.n_max;
    int32_t *ot = out_tokens + (size_t)b * (n_max + 1);
    int32_t *op = out_path + (size_t)b * (n_max + 1);
    if (n <= 0) {
        if (tid == 0) {
            out_count[b] = 0;
            if (out_lowmargin) out_lowmargin[b] = 0;
        }
        return;
    }
    if (tid == 0) {
        sm.lowm = 0;
        for (int w = 0; w < kWalkWarps; ++w) mbar_init(smem_u32(&sm.wbar[w]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // tree and row indices into shared memory; index checks for every node
    int bad_index = 0;
    for (int i = tid; i < n; i += kWalkThreads) {
        const size_t o = (size_t)b * n_max + i;
        const int v = t.perm[o];
        sm.perm[i] = v;
        sm.tok[i] = t.token[o];
        sm.sub_end[i] = t.sub_end[o];
        sm.depth[i] = t.depth[o];
        const int pr = p_row ? p_row[(size_t)b * n_max + v] : v;
        sm.prow[i] = pr;
        if (pr < 0 || pr >= NP) bad_index = 1;
        if (i > 0 && NAIVE) {
            if (sm.tok[i] < 0 || sm.tok[i] >= V) bad_index = 1;
        } else if (i > 0) {
            const int qr = q_row[(size_t)b * n_max + v];
            sm.qrow[i] = qr;
            if (qr < 0 || qr >= NQ || sm.tok[i] < 0 || sm.tok[i] >= V) bad_index = 1;
        }
    }
    bad_index = __any_sync(0xffffffffu, bad_index);
    if (lane == 0) sm.bad[warp] = bad_index;
    __syncthreads();
    if (__any_sync(0xffffffffu, sm.bad[lane])) {
        if (tid == 0) {
            out_count[b] = 0;
            if (out_lowmargin) out_lowmargin[b] = 0;
            flag(status, TS_STATUS_INDEX);
        }
        return;
    }
    const float *u_acc = uniforms + (size_t)b * 2 * n_max;
    const float *u_smp = u_acc + n_max;
    const int V4 = V >> 2;
    const int C4 = (V4 + kWalkWarps - 1) / kWalkWarps;          // float4s of a warp's chunk
    const int g0 = min(V4, warp * C4), g1 = min(V4, g0 + C4);     // this warp's chunk
    const float a2 = invT * kL2E;
    int u = 0, cnt = 0, nonfinite = 0, timeout = 0;
    uint32_t visit = 0;   // bulk copies so far (mbarrier phase)
    if (tid == 0) op[0] = sm.perm[0];

    for (int step = 0; step < n; ++step) {
        const float *row = logits + ((size_t)b * NP + sm.prow[u]) * V;
        const int du = sm.depth[u], se_u = sm.sub_end[u];
        const int c_first = u + 1 < se_u ? u + 1 : -1;
        // this warp's range of the node's row into R by bulk copy (the warp's
        // earlier accesses of its range are behind the last barrier; the proxy
        // fence orders them before the copy). An empty range completes at once.
        if (lane == 0) {
            fence_async_smem();
            mbar_expect_tx(wbar, (uint32_t)(g1 - g0) * 16u);
            if (g1 > g0)
                bulk_g2s(smem_u32(R4 + g0), reinterpret_cast<const float4 *>(row) + g0, (uint32_t)(g1 - g0) * 16u,
                         wbar);
        }
        // meanwhile: the values the tests read (q_c(x_c), accept uniforms; at
        // most one node per thread: n <= kMaxNodes <= threads) and the
        // final-sample uniform, into registers now and into shared memory after
        // the passes, so that their latency hides under the passes. (Pulling the
        // first child's drafter and target rows into L2 here measured slower:
        // each warp's range then lands 1 us later, merge workload 54.2 vs 48.0
        // us per call.)
        const int ti = u + 1 + tid;
        const bool tchild = !NAIVE && ti < se_u && sm.depth[ti] == du + 1;
        float t_q = 0.f, t_u = 0.f;
        if (tchild) {
            t_q = __ldg(ssm + ((size_t)b * NQ + sm.qrow[ti]) * V + sm.tok[ti]);
            t_u = __ldg(u_acc + sm.perm[ti]);
        }
        const float t_us = tid == kWalkThreads - 1 ? __ldg(u_smp + sm.perm[u]) : 0.f;
        const bool landed = mbar_wait_warp(wbar, visit & 1u);
        ++visit;
        // the warp's maximum (invT > 0) and finiteness: x * 0 + z stays 0 unless
        // x is NaN or infinite
        float mx = -FLT_MAX, z = 0.f;
        if (landed)
            for (int g = g0 + lane; g < g1; g += 32) {
                const float4 a = R4[g];
                mx = fmaxf(mx, fmaxf(fmaxf(a.x, a.y), fmaxf(a.z, a.w)));
                z = __fmaf_rn(a.x, 0.f, z); z = __fmaf_rn(a.y, 0.f, z);
                z = __fmaf_rn(a.z, 0.f, z); z = __fmaf_rn(a.w, 0.f, z);
            }
        mx = warp_max(mx);
        const int nf = __any_sync(0xffffffffu, z != 0.f);
        // e = 2^(l a2 - Mw), a2 = log2(e) / T, Mw = max(l) a2, into R (one FMA and
        // the hardware exp2 an entry), their sum; R at the first child's token
        const float Mw = mx * a2;
        const int x_first = (!NAIVE && c_first >= 0) ? sm.tok[c_first] : -1;
        float s = 0.f, cc = 0.f;
        if (landed && !nf)
            for (int g = g0 + lane; g < g1; g += 32) {
                float4 a = R4[g];
                a.x = ex2(__fmaf_rn(a.x, a2, -Mw)); a.y = ex2(__fmaf_rn(a.y, a2, -Mw));
                a.z = ex2(__fmaf_rn(a.z, a2, -Mw)); a.w = ex2(__fmaf_rn(a.w, a2, -Mw));
                kahan(s, cc, (a.x + a.y) + (a.z + a.w));
                R4[g] = a;
            }
        __syncwarp();
        if (lane == 0 && x_first >= 0 && (x_first >> 2) >= g0 && (x_first >> 2) < g1) sm.rx = R[x_first];
        if (tchild) {
            sm.cq[ti] = t_q;
            sm.cu[ti] = t_u;
        }
        if (tid == kWalkThreads - 1) sm.us = t_us;
        walk_publish(sm, s, -cc, Mw, (nf ? 1 : 0) | (landed ? 0 : 2));
        __syncthreads();
        if (warp == 0) walk_decide_stats(sm, c_first, se_u, C4, NAIVE);
        __syncthreads();
        int v = sm.verdict;
        if (v == kVTimeout) { timeout = 1; break; }
        // R relative to each warp's maximum (factor fw) until a rejection pass
        // rescales it to the row maximum
        bool local = true;
        float fw = sm.f[warp];
        // children in input order: u+1, sub_end[u+1], ... below sub_end[u]
        int c = c_first;
        while (v == kVReject) {
            // child c rejected: R' = max(0, R - S q_c), S' = sum R'; R' at the next child's token
            const float Sf = sm.Sh + sm.Sl;
            const float *qc = ssm + ((size_t)b * NQ + sm.qrow[c]) * V;
            const float4 *q4 = reinterpret_cast<const float4 *>(qc);
            const int c_next = sm.sub_end[c] < se_u ? sm.sub_end[c] : -1;
            const int x_next = c_next >= 0 ? sm.tok[c_next] : -1;
            float s2 = 0.f, c2 = 0.f, zq = 0.f;   // zq: NaN once a drafter value is not finite
            for (int g00 = g0 + lane; g00 < g1; g00 += 4 * 32) {
                float4 qv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (g00 + 32 * j < g1) qv[j] = __ldg(q4 + g00 + 32 * j);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int g = g00 + 32 * j;
                    if (g < g1) {
                        zq = __fmaf_rn(qv[j].x, 0.f, zq); zq = __fmaf_rn(qv[j].y, 0.f, zq);
                        zq = __fmaf_rn(qv[j].z, 0.f, zq); zq = __fmaf_rn(qv[j].w, 0.f, zq);
                        float4 r = R4[g];
                        r.x = fmaxf(0.f, __fmaf_rn(-Sf, qv[j].x, r.x * fw));
                        r.y = fmaxf(0.f, __fmaf_rn(-Sf, qv[j].y, r.y * fw));
                        r.z = fmaxf(0.f, __fmaf_rn(-Sf, qv[j].z, r.z * fw));
                        r.w = fmaxf(0.f, __fmaf_rn(-Sf, qv[j].w, r.w * fw));
                        R4[g] = r;
                        kahan(s2, c2, (r.x + r.y) + (r.z + r.w));
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && x_next >= 0 && (x_next >> 2) >= g0 && (x_next >> 2) < g1) sm.rx = R[x_next];
            // a non-finite drafter value makes the partial NaN
            const bool bad = __any_sync(0xffffffffu, zq != 0.f);
            walk_publish(sm, bad ? NAN : s2, bad ? 0.f : -c2, 0.f, 0);
            __syncthreads();
            if (warp == 0) walk_decide_resid(sm, qc, c_next, se_u, C4, status);
            __syncthreads();
            local = false;   // R is now relative to the row maximum
            fw = 1.f;
            v = sm.verdict;
            if (v == kVZero) {
                // zero normaliser: keep the residual unchanged (rebuilt from the
                // rejections applied so far: the in-place pass overwrote it)
                const Resid keep{row, invT, sm.m, sm.rej_q, sm.rej_S, sm.nrej, nullptr};
                float s3 = 0.f, c3 = 0.f;
                for (int g = g0 + lane; g < g1; g += 32) {
                    float4 r;
                    r.x = resid_recompute(keep, 4 * g);
                    r.y = resid_recompute(keep, 4 * g + 1);
                    r.z = resid_recompute(keep, 4 * g + 2);
                    r.w = resid_recompute(keep, 4 * g + 3);
                    R4[g] = r;
                    kahan(s3, c3, (r.x + r.y) + (r.z + r.w));
                }
                __syncwarp();
                if (lane == 0 && x_next >= 0 && (x_next >> 2) >= g0 && (x_next >> 2) < g1) sm.rx = R[x_next];
                walk_publish(sm, s3, -c3, 0.f, 0);
                __syncthreads();
                if (warp == 0) walk_decide_rebuilt(sm, c_next, se_u, C4);
                __syncthreads();
                v = sm.verdict;
            }
            c = c_next;
        }
        if (v == kVNonfinite) { nonfinite = 1; break; }
        if (v >= 0) {   // child v accepted
            if (tid == 0) {
                ot[cnt] = sm.tok[v];
                op[cnt + 1] = sm.perm[v];
            }
            ++cnt;
            u = v;
            continue;
        }
        // ---- the final sample: the first y with C(y) > u * S, inside the range
        // of warp sm.ws (the coarse level is the deciding warp's)
        if (warp == sm.ws) {
            const bool fallback = sm.fb;
            const float bh = sm.bh, bl = sm.bl, tgh = sm.tgh, tgl = sm.tgl, toth = sm.toth;
            // lane j sums the float4s [g0 + j K, g0 + (j + 1) K) of the chunk
            const int K = (g1 - g0 + 31) / 32;
            const int a0 = min(g1, g0 + lane * K), a1 = min(g1, a0 + K);
            float lh = 0.f, ll = 0.f;
            for (int g = a0; g < a1; ++g) {
                const float4 r = R4[g];
                ff_add(lh, ll, r.x * fw, 0.f); ff_add(lh, ll, r.y * fw, 0.f);
                ff_add(lh, ll, r.z * fw, 0.f); ff_add(lh, ll, r.w * fw, 0.f);
            }
            float jh = lh, jl = ll;   // inclusive scan over the lanes
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float xh = __shfl_up_sync(0xffffffffu, jh, o), xl = __shfl_up_sync(0xffffffffu, jl, o);
                if (lane >= o) ff_add(jh, jl, xh, xl);
            }
            float ch = bh, cl = bl;   // C before this lane's range
            ff_add(ch, cl, jh, jl);
            ff_add(ch, cl, -lh, -ll);
            float eh = bh, el = bl;   // C after it
            ff_add(eh, el, jh, jl);
            const unsigned hitl = fallback ? 0u : __ballot_sync(0xffffffffu, lh > 0.f && ff_gt(eh, el, tgh, tgl));
            const unsigned posl = __ballot_sync(0xffffffffu, lh > 0.f);
            const int wl = hitl ? __ffs(hitl) - 1 : (posl ? 31 - __clz(posl) : -1);
            if (lane == wl) {
                int chosen = -1, last_pos = -1;
                float margin = 0.f;
                for (int y = 4 * a0; y < 4 * a1 && chosen < 0; ++y) {
                    const float r = R[y] * fw;
                    if (r > 0.f) {
                        float nh = ch, nl = cl;
                        ff_add(nh, nl, r, 0.f);
                        if (hitl && ff_gt(nh, nl, tgh, tgl)) {
                            chosen = y;
                            float d1h = tgh, d1l = tgl, d2h = nh, d2l = nl;
                            ff_add(d1h, d1l, -ch, -cl);
                            ff_add(d2h, d2l, -tgh, -tgl);
                            margin = fminf(d1h + d1l, d2h + d2l) / toth;
                        }
                        last_pos = y;
                        ch = nh;
                        cl = nl;
                    }
                }
                if (chosen < 0) chosen = last_pos;   // rounding left no bracket: the last token with mass
                sm.chosen = chosen;
                if (!(margin >= (float)kLowMargin)) ++sm.lowm;
            } else if (wl < 0 && lane == 0) {
                sm.chosen = 0;   // no mass anywhere (not reachable with S > 0)
                ++sm.lowm;
            }
        }
        __syncthreads();
        const int chosen = sm.chosen;
        if (tid == 0) ot[cnt] = chosen;
        ++cnt;
        if (!NAIVE) break;
        // naive sampling: continue at the first child holding the drawn token
        int next = -1;
        for (int c2 = u + 1; c2 < se_u; c2 = sm.sub_end[c2])
            if (sm.tok[c2] == chosen) { next = c2; break; }
        if (next < 0) break;
        if (tid == 0) op[cnt] = sm.perm[next];
        u = next;
        __syncthreads();   // sm.chosen is rewritten at the next node
    }
    // a row copy may still be in flight after a timeout: each warp waits for its
    // own (bounded) before the block exits
    if (timeout && lane == 0) mbar_wait_bounded(wbar, (visit - 1) & 1u);
    __syncthreads();
    if (tid == 0) {
        if (timeout) {
            out_count[b] = 0;
            flag(status, TS_STATUS_TIMEOUT);
        } else if (nonfinite) {
            out_count[b] = 0;
            flag(status, TS_STATUS_NONFINITE);
        } else {
            out_count[b] = cnt;
        }
        if (out_lowmargin) out_lowmargin[b] = sm.lowm;
    }
}

}  // namespace

size_t greedy_ws_bytes(int B, int n_max, int V) {
    (void)V;
    size_t counters = ((size_t)B * sizeof(unsigned) + 255) / 256 * 256;
    return counters + (size_t)B * n_max * kMaxSeg * sizeof(ArgPart);
}

cudaError_t launch_verify_greedy(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *argmax_out,
                                 const float *logits, const ts_tree &t, int V, void *ws, uint32_t *status,
                                 cudaStream_t s) {
    const int rows = t.B * t.n_max;
    const bool vec4 = (V % 4 == 0) && ((uintptr_t)logits % 16 == 0);
    unsigned *counters = (unsigned *)ws;
    ArgPart *parts = (ArgPart *)((char *)ws + ((size_t)t.B * sizeof(unsigned) + 255) / 256 * 256);
    // bulk copies: 256-thread CTAs, segments for two resident CTAs per SM over
    // all rows (at most 96 KB a segment), when a segment is 16 KB or more and the
    // grid is about one wave (LLaMA-7B-shaped rows: 8.0 -> 6.8 us a call). Larger
    // grids keep small 128-thread CTAs without shared memory: beside the
    // attention of a long-context step they give back SMs sooner (step 369 us
    // against 378 us with 64 KB segments, though the call alone is 15.0 against
    // 12.1 us)
    int seg = (2 * num_sms() + rows - 1) / rows;
    seg = max(1, min(kMaxSeg, max(seg, (int)(((size_t)V * 4 + 98303) / 98304))));
    const size_t seg_bytes = (size_t)(((V >> 2) + seg - 1) / seg) * 16;
    if (vec4 && seg_bytes >= (size_t)kGreedyBulkMin && seg_bytes <= 98304 && (long long)rows * seg <= 3LL * num_sms()) {
        cudaError_t e = cudaFuncSetAttribute(k_greedy<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)seg_bytes);
        if (e != cudaSuccess) return e;
        return launch(k_greedy<256>, dim3(t.n_max * seg, t.B), dim3(256), seg_bytes, s, out_tokens, out_path, out_count,
                      argmax_out, logits, t, V, seg, 2, counters, parts, status);
    }
    // vocab segments per node row: as many as fit one wave of resident CTAs (a
    // second, partial wave doubles the time of this latency-bound pass), and no
    // segment shorter than 2048 entries
    static int occ = 0;
    if (occ == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k_greedy<128>, 128, 0) != cudaSuccess) {
        cudaGetLastError();
        occ = 4;
    }
    const int slots = num_sms() * (occ > 0 ? occ : 1);
    seg = max(1, min(kMaxSeg, min(slots / rows, max(1, V / 2048))));
    return launch(k_greedy<128>, dim3(t.n_max * seg, t.B), dim3(128), 0, s, out_tokens, out_path, out_count,
                  argmax_out, logits, t, V, seg, vec4 ? 1 : 0, counters, parts, status);
}

template <bool NAIVE>
cudaError_t launch_walk(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *out_lowmargin,
                        const float *logits,
                        const int32_t *p_row, int NP, const float *ssm, const int32_t *q_row, int NQ,
                        const float *uniforms, float temperature, const ts_tree &t, int V, uint32_t *status,
                        cudaStream_t s) {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    // the fast form: rows by bulk copy (V a multiple of 4, 16-byte aligned rows)
    const size_t walk_smem = kWalkHeader + (size_t)V * sizeof(float);
    const bool aligned = ((uintptr_t)logits & 15u) == 0 && (NAIVE || ((uintptr_t)ssm & 15u) == 0);
    if (V % 4 == 0 && aligned && walk_smem <= (size_t)optin) {
        cudaError_t e = cudaFuncSetAttribute(k_walk<NAIVE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)walk_smem);
        if (e != cudaSuccess) return e;
        return launch(k_walk<NAIVE>, dim3(t.B), dim3(kWalkThreads), walk_smem, s, out_tokens, out_path, out_count,
                      out_lowmargin, logits, p_row, NP, ssm, q_row, NQ, uniforms, 1.0f / temperature, t, V, status);
    }
    const size_t with_row = kMssHeader + (size_t)((V + 3) & ~3) * sizeof(float);
    if (with_row <= (size_t)optin) {
        cudaError_t e =
            cudaFuncSetAttribute(k_mss<true, NAIVE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)with_row);
        if (e != cudaSuccess) return e;
        return launch(k_mss<true, NAIVE>, dim3(t.B), dim3(kMssThreads), with_row, s, out_tokens, out_path, out_count,
                      out_lowmargin, logits, p_row, NP, ssm, q_row, NQ, uniforms, 1.0f / temperature, t, V, status);
    }
    return launch(k_mss<false, NAIVE>, dim3(t.B), dim3(kMssThreads), (size_t)kMssHeader, s, out_tokens, out_path,
                  out_count, out_lowmargin, logits, p_row, NP, ssm, q_row, NQ, uniforms, 1.0f / temperature, t, V,
                  status);
}

cudaError_t launch_verify_mss(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *out_lowmargin,
                              const float *logits, const int32_t *p_row, int NP, const float *ssm,
                              const int32_t *q_row, int NQ, const float *uniforms, float temperature,
                              const ts_tree &t, int V, uint32_t *status, cudaStream_t s) {
    return launch_walk<false>(out_tokens, out_path, out_count, out_lowmargin, logits, p_row, NP, ssm, q_row, NQ,
                              uniforms, temperature, t, V, status, s);
}

cudaError_t launch_verify_naive(int32_t *out_tokens, int32_t *out_path, int32_t *out_count, int32_t *out_lowmargin,
                                const float *logits, const int32_t *p_row, int NP, const float *uniforms,
                                float temperature, const ts_tree &t, int V, uint32_t *status, cudaStream_t s) {
    return launch_walk<true>(out_tokens, out_path, out_count, out_lowmargin, logits, p_row, NP, nullptr, nullptr, 1,
                             uniforms, temperature, t, V, status, s);
}

}  // namespace ts
