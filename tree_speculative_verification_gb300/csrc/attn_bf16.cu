// attn_bf16.cu -- split-KV tree attention, bf16 in / fp32 accumulate.
//
// What it computes: TreeAttention(u) = Attention(S_u) for every node u of the
// token tree (SpecInfer, arXiv 2305.09781, Def. 4.1, Eq. 1-4), all nodes of a
// (request, head) in one pass over that head's KV cache, whose rows are the
// verified prefix followed by the tree nodes in depth-first order (sec. 4.2).
// A key j is visible to node i iff j < P (prefix) or key j - P is an ancestor
// of i or i itself (the topology-aware causal mask of sec. 4.2); the mask is a
// bit test on the ancestor bitmask, evaluated in registers.
//
// GB300 design:
//  * The prefix K/V stream is the whole cost (HBM bound). Each CTA owns one
//    (request, head, key chunk) and streams 64-key K and V tiles with TMA
//    (cp.async.bulk.tensor, 128-byte swizzle) into a 3-stage mbarrier ring.
//  * Tensor cores in swap-AB orientation: S^T = K Q^T puts 16 keys on the M
//    side and the few tree nodes (8 per n-tile) on the N side, so a 21-node
//    tree pads to 24 columns, not 32 rows. P^T is moved from the accumulator
//    layout to the B-operand layout with movmatrix; O^T = V^T P^T.
//  * With ragged prefixes the grid rows take the requests longest first (the
//    rank of P_b + n_b, computed by every CTA from the B counts), so that the
//    longest (request, head) pairs start in the first wave of CTAs.
//  * Online softmax per node column in the exp2 domain; the CTA's partial
//    (max, sum, O) goes to the workspace and the last CTA of the (request,
//    head) -- found with an atomic counter, no waiting -- merges the splits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "attn_common.cuh"
#include "ts_internal.cuh"

namespace ts {
namespace {

constexpr int TK = 64;       // keys per pipeline tile
constexpr int kMaxSplits = 64;

// STG_: TMA ring stages; QR_: Q fragments held in registers for the whole pass
// (else re-read from shared memory per k-step pair, 48 registers fewer at 24
// nodes); MINB_: CTAs per SM the register allocation must allow. Measured on
// GB300 (21 nodes, 2048-key prefix, 256 pairs): <3, regs, 1> 50.7 us,
// <3, smem, 2> 51.0, <2, regs, 2> 52.5, <2, smem, 2> 53.0, <2, smem, 3> with
// three CTAs per SM 58.8 -- more warps per SM do not help this kernel.
template <int D_, int NT_, int NG_, int KS_, int STG_ = 3, bool QR_ = true, int MINB_ = 1>
struct Cfg {
    static constexpr int D = D_, NT = NT_, NG = NG_, KS = KS_, STG = STG_, MINB = MINB_;
    static constexpr bool QR = QR_;
    static constexpr int WARPS = NG * KS, THREADS = WARPS * 32;
    static constexpr int NODES = NG * NT * 8;            // node columns held (padded)
    static constexpr int BOXES = D / 64;                  // 64-column (128-byte) TMA boxes per row
    static constexpr int BOX_BYTES = TK * 128;
    static constexpr int TILE_BYTES = BOXES * BOX_BYTES;  // one K or V tile
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int KEYS_PER_WARP = TK / KS;
    static constexpr int CHUNKS = KEYS_PER_WARP / 16;
    static constexpr int Q_BYTES = NODES * D * 2;
    static constexpr int ANC_BYTES = NODES * kMaxWords * 4;
    static constexpr int NT8P = NT * 8 + 4;               // padded node stride of the merge slots
    static constexpr int SLOT_FLOATS = 2 * NT * 8 + D * NT8P;
    static constexpr int OFF_Q = STG * STAGE_BYTES;
    static constexpr int OFF_ANC = OFF_Q + Q_BYTES;
    static constexpr int OFF_PERM = OFF_ANC + ANC_BYTES;
    static constexpr int OFF_BAR = OFF_PERM + NODES * 4;
    static constexpr int OFF_MISC = OFF_BAR + 2 * STG * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;     // + slack for 1024-byte alignment
    static_assert(NG * (KS - 1) * SLOT_FLOATS * 4 <= STG * STAGE_BYTES, "merge slots exceed stage memory");
    static_assert(KEYS_PER_WARP % 16 == 0, "warp key slice must be a multiple of 16");
};

// ------------------------------------------------------------ PTX helpers ---
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ---------------------------------------------------------------- kernel ----

// After a CTA has published its partial (max, sum, unnormalised O) for key
// split sidx of (b, h), the CTA that arrives last on the (b, h) counter merges
// all S_b partials by log-sum-exp and writes the bf16 rows. No CTA waits: the
// others return. Called by every thread of the CTA.
template <int D>
__device__ void merge_splits(const AttnArgs &a, int b, int h, int n, int S_b, const int *perm_s, int *flag_s,
                             int nthreads) {
    const int tid = threadIdx.x;
    const size_t bh = (size_t)b * a.H + h;
    __threadfence();
    __syncthreads();
    if (tid == 0) flag_s[0] = atomicAdd(&a.counters[bh], 1u) == (unsigned)(S_b - 1);
    __syncthreads();
    if (!flag_s[0]) return;
    __threadfence();
    const int n_max = a.t.n_max;
    // Each thread merges up to four (node, dim pair) items at a time, four splits
    // at a time, with every load of a group issued before any is used.
    constexpr int IT = 4, SG = 4;
    const int items = n * (D / 2);
    for (int idx0 = tid; idx0 < items; idx0 += IT * nthreads) {
        float M[IT], Ls[IT], o0[IT], o1[IT];
        int ii[IT], dd[IT];
#pragma unroll
        for (int q = 0; q < IT; ++q) {
            const int idx = idx0 + q * nthreads;
            ii[q] = idx < items ? idx / (D / 2) : -1;
            dd[q] = idx < items ? (idx % (D / 2)) * 2 : 0;
            M[q] = -INFINITY;
            Ls[q] = o0[q] = o1[q] = 0.f;
        }
        for (int s0 = 0; s0 < S_b; s0 += SG) {
            float ms[IT][SG], ls[IT][SG];
            float2 ov[IT][SG];
#pragma unroll
            for (int q = 0; q < IT; ++q)
#pragma unroll
                for (int k = 0; k < SG; ++k) {
                    const int sp = s0 + k;
                    if (ii[q] >= 0 && sp < S_b) {
                        const float *pml = a.part_ml + (bh * a.splits + sp) * 2 * a.n_pad;
                        ms[q][k] = __ldcg(pml + ii[q]);
                        ls[q][k] = __ldcg(pml + a.n_pad + ii[q]);
                        ov[q][k] = __ldcg((const float2 *)(a.part_o + ((bh * a.splits + sp) * a.n_pad + ii[q]) * D + dd[q]));
                    } else {
                        ms[q][k] = -INFINITY;
                        ls[q][k] = 0.f;
                        ov[q][k] = make_float2(0.f, 0.f);
                    }
                }
#pragma unroll
            for (int q = 0; q < IT; ++q)
#pragma unroll
                for (int k = 0; k < SG; ++k) {
                    const float mn = fmaxf(M[q], ms[q][k]);
                    const float fo = M[q] == mn ? 1.f : exp2f(M[q] - mn);   // 0 from -inf
                    const float fs = ms[q][k] == mn ? 1.f : exp2f(ms[q][k] - mn);
                    Ls[q] = Ls[q] * fo + ls[q][k] * fs;
                    o0[q] = o0[q] * fo + ov[q][k].x * fs;
                    o1[q] = o1[q] * fo + ov[q][k].y * fs;
                    M[q] = mn;
                }
        }
#pragma unroll
        for (int q = 0; q < IT; ++q)
            if (ii[q] >= 0) {
                const float inv = Ls[q] > 0.f ? 1.f / Ls[q] : 0.f;
                *(__nv_bfloat162 *)(a.out + (((size_t)b * n_max + perm_s[ii[q]]) * a.H + h) * D + dd[q]) =
                    __floats2bfloat162_rn(o0[q] * inv, o1[q] * inv);
            }
    }
    if (tid == 0) a.counters[bh] = 0u;   // leave the workspace zeroed
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, C::MINB) k_attn_bf16(const __grid_constant__ CUtensorMap map_k,
                                                                   const __grid_constant__ CUtensorMap map_v,
                                                                   const __grid_constant__ CUtensorMap map_k8,
                                                                   const __grid_constant__ CUtensorMap map_v8,
                                                                   AttnArgs a) {
    constexpr int D = C::D, NT = C::NT, KS = C::KS, STAGES = C::STG;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sm_base = smem_u32(sm);
    uint32_t *anc_s = (uint32_t *)(sm + C::OFF_ANC);
    int *perm_s = (int *)(sm + C::OFF_PERM);
    int *misc = (int *)(sm + C::OFF_MISC);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int grp = warp / KS, ks = warp % KS;
    const int g = lane >> 2, tq = lane & 3;
    const int h = blockIdx.x, sidx = blockIdx.z;
    const ts_tree &t = a.t;
    pdl_wait();
    pdl_trigger();
    const int b = request_by_rank(a, blockIdx.y, (int *)(sm + C::OFF_Q));
    const int n = t.n_nodes[b], P = a.prefix_len[b];
    if (n <= 0) return;
    if (P < 0 || P + n > a.L_max) {
        if (sidx == 0 && h == 0 && tid == 0) flag(a.status, TS_STATUS_INDEX);
        return;
    }
    const int L = P + n;
    const int chunk_keys = a.chunk_tiles * TK;
    const int S_b = (L + chunk_keys - 1) / chunk_keys;
    if (sidx >= S_b) return;
    const int k_begin = sidx * chunk_keys, k_end = min(L, k_begin + chunk_keys);
    const int ntiles = (k_end - k_begin + TK - 1) / TK;
    const uint32_t bar0 = sm_base + C::OFF_BAR;

    if (tid == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar0 + 8 * s, 1);                              // full: TMA bytes landed
            mbar_init(bar0 + 8 * (STAGES + s), C::WARPS);            // empty: every warp done
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    static_assert(TK == TS_PAGE_KEYS, "one key tile is one page");
    // one tile into its stage; the chunk's last tile, when it holds fewer than
    // TK keys, comes in 8-row pieces (one swizzle atom each), so no more than 7
    // rows past the chunk's end are read
    auto issue = [&](int it, int row) {
        const int st = it % STAGES;
        const uint32_t kdst = sm_base + st * C::STAGE_BYTES, vdst = kdst + C::TILE_BYTES;
        const uint32_t bar = bar0 + 8 * st;
        const int nv = min(TK, k_end - (k_begin + it * TK));
        if (nv == TK) {
            mbar_expect_tx(bar, C::STAGE_BYTES);
#pragma unroll
            for (int bx = 0; bx < C::BOXES; ++bx) {
                tma_load_2d(kdst + bx * C::BOX_BYTES, &map_k, bx * 64, row, bar);
                tma_load_2d(vdst + bx * C::BOX_BYTES, &map_v, bx * 64, row, bar);
            }
        } else {
            mbar_expect_tx(bar, 2u * C::BOXES * (uint32_t)((nv + 7) & ~7) * 128u);
#pragma unroll
            for (int bx = 0; bx < C::BOXES; ++bx)
                for (int r8 = 0; r8 < nv; r8 += 8) {
                    tma_load_2d(kdst + bx * C::BOX_BYTES + r8 * 128, &map_k8, bx * 64, row + r8, bar);
                    tma_load_2d(vdst + bx * C::BOX_BYTES + r8 * 128, &map_v8, bx * 64, row + r8, bar);
                }
        }
    };
    if (tid == 0) {
        int rows[STAGES];
#pragma unroll
        for (int it = 0; it < STAGES; ++it)   // every page id in flight before the first use
            if (it < ntiles) rows[it] = tile_row(a, b, h, k_begin + it * TK);
#pragma unroll
        for (int it = 0; it < STAGES; ++it)
            if (it < ntiles) issue(it, rows[it]);
    }

    // Q rows of the CTA's nodes (DFS order) into swizzled shared memory; ancestor masks
    const int n_max = t.n_max, W = TS_MASK_WORDS(n_max);
    for (int r = tid; r < C::NODES; r += C::THREADS) perm_s[r] = r < n ? t.perm[(size_t)b * n_max + r] : -1;
    __syncthreads();
    {
        constexpr int CH = D / 8;   // 16-byte chunks per row
        uint4 *qs = (uint4 *)(sm + C::OFF_Q);
        for (int idx = tid; idx < C::NODES * CH; idx += C::THREADS) {
            const int r = idx / CH, c = idx % CH;
            uint4 val = make_uint4(0u, 0u, 0u, 0u);
            if (r < n) {
                const uint4 *src = (const uint4 *)(a.q + (((size_t)b * n_max + perm_s[r]) * a.H + h) * D);
                val = src[c];
            }
            qs[r * CH + (c ^ (r & 7))] = val;
        }
        for (int idx = tid; idx < C::NODES * kMaxWords; idx += C::THREADS) {
            const int r = idx / kMaxWords, w = idx % kMaxWords;
            anc_s[idx] = (r < n && w < W) ? t.anc[((size_t)b * n_max + r) * W + w] : 0u;
        }
    }
    __syncthreads();

    // Q as B operand fragments: for k-step pair (kk, kk + 1) and node tile j,
    // one ldmatrix.x4 from the swizzled Q rows; held in registers for the
    // whole pass (QR) or re-read at every use
    const int node0 = grp * NT * 8;
    const uint32_t qbase = sm_base + C::OFF_Q;
    auto load_q = [&](int j, int kk, uint32_t &q0, uint32_t &q1, uint32_t &q2, uint32_t &q3) {
        const int r = node0 + j * 8 + (lane & 7);
        const int c = kk * 2 + (lane >> 3);
        ldsm_x4(qbase + r * (D * 2) + ((c ^ (r & 7)) << 4), q0, q1, q2, q3);
    };
    uint32_t qf[C::QR ? NT : 1][C::QR ? D / 16 : 1][2];
    if constexpr (C::QR) {
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int kk = 0; kk < D / 16; kk += 2) load_q(j, kk, qf[j][kk][0], qf[j][kk][1], qf[j][kk + 1][0], qf[j][kk + 1][1]);
    }

    float oacc[D / 16][NT][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) oacc[mt][j][e] = 0.f;
    float m_run[NT][2], l_run[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        m_run[j][0] = m_run[j][1] = -INFINITY;
        l_run[j][0] = l_run[j][1] = 0.f;
    }

    // Main loop. Stage st of the ring is refilled by thread 0 once every warp
    // has released it (empty barrier, one arrival per warp), so warps are not
    // coupled by a CTA-wide barrier per tile.
    const uint32_t ebar0 = bar0 + 8 * STAGES;
    const float c = a.scale_log2;
    int timed_out = 0;
    for (int it = 0; it < ntiles; ++it) {
        const int st = it % STAGES;
        const uint32_t phase = (uint32_t)(it / STAGES) & 1u;
        // the row of the tile issued at the end of this iteration, fetched now
        const int next_row = (tid == 0 && it + STAGES < ntiles) ? tile_row(a, b, h, k_begin + (it + STAGES) * TK) : 0;
        if (!mbar_wait_bounded(bar0 + 8 * st, phase)) { timed_out = 1; break; }
        const int key_base = k_begin + it * TK;
        unsigned char *ktile = sm + st * C::STAGE_BYTES;
        unsigned char *vtile = ktile + C::TILE_BYTES;
        if (key_base + TK > k_end) {
            // last tile: rows past the chunk may hold anything (even NaN); zero
            // their V so that a zero probability multiplies a zero
            for (int idx = tid; idx < TK * C::BOXES * 8; idx += C::THREADS) {
                const int r = idx / (C::BOXES * 8), rem = idx % (C::BOXES * 8);
                if (key_base + r >= k_end)
                    *(uint4 *)(vtile + (rem / 8) * C::BOX_BYTES + r * 128 + (rem % 8) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncthreads();
        }
        const uint32_t kb_addr = smem_u32(ktile), vb_addr = smem_u32(vtile);
#pragma unroll
        for (int ch16 = 0; ch16 < C::CHUNKS; ++ch16) {
            const int kb = ks * C::KEYS_PER_WARP + ch16 * 16;
            const int key0 = key_base + kb;
            if (key0 >= k_end) break;
            // S^T = K Q^T : 16 keys x (NT*8) nodes, raw dot products
            float sacc[NT][4];
#pragma unroll
            for (int j = 0; j < NT; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
            uint32_t qp[C::QR ? 1 : NT][4];
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int r = kb + (lane & 7) + (((lane >> 3) & 1) << 3);
                const int chn = 2 * (kk & 3) + (lane >> 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(kb_addr + (kk >> 2) * C::BOX_BYTES + swz(r, chn), a0, a1, a2, a3);
                if constexpr (C::QR) {
#pragma unroll
                    for (int j = 0; j < NT; ++j) mma_bf16(sacc[j], a0, a1, a2, a3, qf[j][kk][0], qf[j][kk][1]);
                } else {
                    if ((kk & 1) == 0)
#pragma unroll
                        for (int j = 0; j < NT; ++j) load_q(j, kk, qp[j][0], qp[j][1], qp[j][2], qp[j][3]);
#pragma unroll
                    for (int j = 0; j < NT; ++j)
                        mma_bf16(sacc[j], a0, a1, a2, a3, qp[j][(kk & 1) * 2], qp[j][(kk & 1) * 2 + 1]);
                }
            }
            // the mask is needed only where the chunk reaches the tree rows or the chunk end
            if (key0 + 16 > P || key0 + 16 > k_end) {
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int key = key0 + g + ((e >> 1) << 3);
                        const int node = node0 + j * 8 + 2 * tq + (e & 1);
                        bool vis = key < k_end;
                        if (vis && key >= P) {
                            const int tk = key - P;
                            vis = (anc_s[node * kMaxWords + (tk >> 5)] >> (tk & 31)) & 1u;
                        }
                        if (!vis) sacc[j][e] = -INFINITY;
                    }
            }
            // column max over the 16 keys (raw scores; the scale is positive)
            float cmax[NT][2];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                cmax[j][0] = fmaxf(sacc[j][0], sacc[j][2]);
                cmax[j][1] = fmaxf(sacc[j][1], sacc[j][3]);
#pragma unroll
                for (int x = 0; x < 2; ++x) {
                    float v = cmax[j][x];
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
                    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
                    cmax[j][x] = v * c;
                }
            }
            // online rescale, only when some column's running max moved
            bool grow = false;
#pragma unroll
            for (int j = 0; j < NT; ++j) grow |= (cmax[j][0] > m_run[j][0]) | (cmax[j][1] > m_run[j][1]);
            if (__any_sync(0xffffffffu, grow)) {
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    float al[2];
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const float mn = fmaxf(m_run[j][x], cmax[j][x]);
                        al[x] = mn == m_run[j][x] ? 1.f : exp2f(m_run[j][x] - mn);
                        m_run[j][x] = mn;
                    }
                    l_run[j][0] *= al[0];
                    l_run[j][1] *= al[1];
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        oacc[mt][j][0] *= al[0];
                        oacc[mt][j][1] *= al[1];
                        oacc[mt][j][2] *= al[0];
                        oacc[mt][j][3] *= al[1];
                    }
                }
            }
            // P^T (bf16) in the B-operand layout; p = exp2(s * c - m); the row sums
            // take the fp32 probabilities, O their bf16 roundings
            uint32_t pb[NT][2];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const float mu0 = m_run[j][0] == -INFINITY ? 0.f : m_run[j][0];
                const float mu1 = m_run[j][1] == -INFINITY ? 0.f : m_run[j][1];
                const float p0 = ex2(__fmaf_rn(sacc[j][0], c, -mu0)), p1 = ex2(__fmaf_rn(sacc[j][1], c, -mu1));
                const float p2 = ex2(__fmaf_rn(sacc[j][2], c, -mu0)), p3 = ex2(__fmaf_rn(sacc[j][3], c, -mu1));
                const __nv_bfloat162 b01 = __floats2bfloat162_rn(p0, p1), b23 = __floats2bfloat162_rn(p2, p3);
                l_run[j][0] += p0 + p2;
                l_run[j][1] += p1 + p3;
                pb[j][0] = movm_t(*reinterpret_cast<const uint32_t *>(&b01));
                pb[j][1] = movm_t(*reinterpret_cast<const uint32_t *>(&b23));
            }
            // O^T += V^T P^T
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                const int r = kb + (lane & 7) + ((lane >> 4) << 3);
                const int chn = 2 * (mt & 3) + ((lane >> 3) & 1);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_t(vb_addr + (mt >> 2) * C::BOX_BYTES + swz(r, chn), a0, a1, a2, a3);
#pragma unroll
                for (int j = 0; j < NT; ++j) mma_bf16(oacc[mt][j], a0, a1, a2, a3, pb[j][0], pb[j][1]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ebar0 + 8 * st);
        if (tid == 0 && it + STAGES < ntiles) {
            if (!mbar_wait_bounded(ebar0 + 8 * st, phase)) { timed_out = 1; break; }
            issue(it + STAGES, next_row);
        }
    }
    if (__syncthreads_or(timed_out)) {
        if (tid == 0) flag(a.status, TS_STATUS_TIMEOUT);
        return;
    }

    // ---- merge the KS key-split warps of each node group (through smem)
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            float v = l_run[j][x];
            v += __shfl_xor_sync(0xffffffffu, v, 4);
            v += __shfl_xor_sync(0xffffffffu, v, 8);
            v += __shfl_xor_sync(0xffffffffu, v, 16);
            l_run[j][x] = v;
        }
    float *slots = (float *)sm;
    if (KS > 1) {
        if (ks > 0) {
            float *sl = slots + (grp * (KS - 1) + (ks - 1)) * C::SLOT_FLOATS;
            float *sm_m = sl, *sm_l = sl + NT * 8, *sm_o = sl + 2 * NT * 8;
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int nc = j * 8 + 2 * tq;
                if (g == 0) {
                    sm_m[nc] = m_run[j][0];
                    sm_m[nc + 1] = m_run[j][1];
                    sm_l[nc] = l_run[j][0];
                    sm_l[nc + 1] = l_run[j][1];
                }
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    *(float2 *)(sm_o + (mt * 16 + g) * C::NT8P + nc) = make_float2(oacc[mt][j][0], oacc[mt][j][1]);
                    *(float2 *)(sm_o + (mt * 16 + g + 8) * C::NT8P + nc) = make_float2(oacc[mt][j][2], oacc[mt][j][3]);
                }
            }
        }
        __syncthreads();
        if (ks == 0) {
            for (int k = 0; k < KS - 1; ++k) {
                const float *sl = slots + (grp * (KS - 1) + k) * C::SLOT_FLOATS;
                const float *sm_m = sl, *sm_l = sl + NT * 8, *sm_o = sl + 2 * NT * 8;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const int nc = j * 8 + 2 * tq;
                    float fs[2], fo[2];
#pragma unroll
                    for (int x = 0; x < 2; ++x) {
                        const float mo = sm_m[nc + x];
                        const float mn = fmaxf(m_run[j][x], mo);
                        fs[x] = m_run[j][x] == -INFINITY ? 0.f : exp2f(m_run[j][x] - mn);
                        fo[x] = mo == -INFINITY ? 0.f : exp2f(mo - mn);
                        l_run[j][x] = l_run[j][x] * fs[x] + sm_l[nc + x] * fo[x];
                        m_run[j][x] = mn;
                    }
#pragma unroll
                    for (int mt = 0; mt < D / 16; ++mt) {
                        const float2 u0 = *(const float2 *)(sm_o + (mt * 16 + g) * C::NT8P + nc);
                        const float2 u1 = *(const float2 *)(sm_o + (mt * 16 + g + 8) * C::NT8P + nc);
                        oacc[mt][j][0] = oacc[mt][j][0] * fs[0] + u0.x * fo[0];
                        oacc[mt][j][1] = oacc[mt][j][1] * fs[1] + u0.y * fo[1];
                        oacc[mt][j][2] = oacc[mt][j][2] * fs[0] + u1.x * fo[0];
                        oacc[mt][j][3] = oacc[mt][j][3] * fs[1] + u1.y * fo[1];
                    }
                }
            }
        }
        __syncthreads();
    }

    const size_t bh = (size_t)b * a.H + h;
    if (S_b == 1) {
        // normalise and write bf16 rows out[b][perm[i]][h][:], staged per warp in smem
        if (ks == 0) {
            __nv_bfloat16 *stage = (__nv_bfloat16 *)(sm + C::OFF_Q) + grp * NT * 8 * D;   // Q is no longer needed
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int nc = j * 8 + 2 * tq;
                const float inv0 = l_run[j][0] > 0.f ? 1.f / l_run[j][0] : 0.f;
                const float inv1 = l_run[j][1] > 0.f ? 1.f / l_run[j][1] : 0.f;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                    stage[nc * D + mt * 16 + g] = __float2bfloat16_rn(oacc[mt][j][0] * inv0);
                    stage[(nc + 1) * D + mt * 16 + g] = __float2bfloat16_rn(oacc[mt][j][1] * inv1);
                    stage[nc * D + mt * 16 + g + 8] = __float2bfloat16_rn(oacc[mt][j][2] * inv0);
                    stage[(nc + 1) * D + mt * 16 + g + 8] = __float2bfloat16_rn(oacc[mt][j][3] * inv1);
                }
            }
            __syncwarp();
            constexpr int CH = D / 8;
            for (int idx = lane; idx < NT * 8 * CH; idx += 32) {
                const int r = idx / CH, c = idx % CH;
                const int i = node0 + r;
                if (i < n)
                    ((uint4 *)(a.out + (((size_t)b * n_max + perm_s[i]) * a.H + h) * D))[c] = ((const uint4 *)stage)[r * CH + c];
            }
        }
        return;
    }

    // ---- split: publish the partial, the last CTA of (b, h) merges
    if (ks == 0) {
        const size_t ps = bh * a.splits + sidx;
        float *pml = a.part_ml + ps * 2 * a.n_pad;
        float *po = a.part_o + ps * a.n_pad * D;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int nc = node0 + j * 8 + 2 * tq;
            if (g == 0) {
                pml[nc] = m_run[j][0];
                pml[nc + 1] = m_run[j][1];
                pml[a.n_pad + nc] = l_run[j][0];
                pml[a.n_pad + nc + 1] = l_run[j][1];
            }
#pragma unroll
            for (int mt = 0; mt < D / 16; ++mt) {
                po[(size_t)nc * D + mt * 16 + g] = oacc[mt][j][0];
                po[(size_t)(nc + 1) * D + mt * 16 + g] = oacc[mt][j][1];
                po[(size_t)nc * D + mt * 16 + g + 8] = oacc[mt][j][2];
                po[(size_t)(nc + 1) * D + mt * 16 + g + 8] = oacc[mt][j][3];
            }
        }
    }
    merge_splits<D>(a, b, h, n, S_b, perm_s, misc, C::THREADS);
}


// ------------------------------------------------------------------ host ----

struct Variant {
    int nodes, threads, smem;
    const char *name;
    const void *fn;
    cudaError_t (*launch)(dim3, const CUtensorMap *, const AttnArgs &, cudaStream_t);
};

// maps: K and V with 64-row boxes, then K and V with 8-row boxes
template <class C>
cudaError_t launch_cfg(dim3 grid, const CUtensorMap *m, const AttnArgs &a, cudaStream_t s) {
    return launch(k_attn_bf16<C>, grid, dim3(C::THREADS), C::SMEM, s, m[0], m[1], m[2], m[3], a);
}

template <class C>
const char *cfg_name() {
    static char buf[48];
    static const bool once =
        (C::STG == 3 && C::QR && C::MINB == 1
             ? snprintf(buf, sizeof buf, "k_attn_bf16<%d,%d,%d,%d>", C::D, C::NT, C::NG, C::KS)
             : snprintf(buf, sizeof buf, "k_attn_bf16<%d,%d,%d,%d,%d,%d,%d>", C::D, C::NT, C::NG, C::KS, C::STG,
                        (int)C::QR, C::MINB),
         true);
    (void)once;
    return buf;
}

template <class C>
Variant variant() {
    return Variant{C::NODES, C::THREADS, C::SMEM, cfg_name<C>(), (const void *)k_attn_bf16<C>, launch_cfg<C>};
}

template <int D>
Variant pick(int n_max) {
    if (n_max <= 24) return variant<Cfg<D, 3, 1, 4>>();
    if (n_max <= 32) return variant<Cfg<D, 4, 1, 4>>();
    if (n_max <= 48) return variant<Cfg<D, 3, 2, 4>>();
    if (n_max <= 64) return variant<Cfg<D, 4, 2, 2>>();
    if (n_max <= 96) return variant<Cfg<D, 3, 4, 2>>();
    if (n_max <= 128) return variant<Cfg<D, 4, 4, 2>>();
    if (n_max <= 192) return variant<Cfg<D, 3, 8, 1>>();
    return variant<Cfg<D, 4, 8, 1>>();
}

// Kernel choice for head_dim 128: trees of 33..128 nodes go to the persistent
// 128-key-tile tcgen05 kernel (k_attn_tq, attn_tq.cu). Smaller trees go to it
// too, except when the (request, head) pairs fill exactly one wave of the
// mma.sync kernel's two CTAs per SM (SMs < pairs <= 2 SMs). Measured on GB300
// for 21-node trees over a 2048-key prefix (32 heads): batch 4 (128 pairs)
// tcgen05 29.6 us vs mma.sync 50.4 us (which must split keys to fill the
// SMs); batch 8 (256 pairs) 53.7 vs 51.4 us; batch 16 (512 pairs) 98.9 vs
// 96.9 us; merged-chain trees over ragged prefixes (512 pairs) 113.0 vs
// 117.4 us (the persistent kernel's queue balances the ragged items). Head
// dim 64 and trees of more than 128 nodes: the mma.sync kernel.
// TREESPEC_ATTN_KERNEL=mma or tq forces one of them where its limits allow.
bool use_tq(int d, int n_max, long long pairs) {
    if (d != 128 || n_max > 128) return false;
    const char *e = getenv("TREESPEC_ATTN_KERNEL");
    if (e && *e) return strcmp(e, "tq") == 0;
    if (n_max > 32) return true;
    const long long sms = num_sms();
    return !(pairs > sms && pairs <= 2 * sms);
}

Variant pick_variant(int d, int n_max) { return d == 64 ? pick<64>(n_max) : pick<128>(n_max); }

int occupancy(const Variant &v) {
    int occ = 0;
    cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, v.fn, v.threads, v.smem) != cudaSuccess || occ < 1) {
        cudaGetLastError();
        occ = 1;
    }
    return occ;
}

}  // namespace

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 152;
    }
    return n > 0 ? n : 152;
}

AttnPlan attn_plan(int B, int H, int n_max, int d, int L_max, ts_dtype dt) {
    AttnPlan p{1, 1, 0, 0, "k_attn_f32"};
    if (dt != TS_BF16) return p;
    if (use_tq(d, n_max, (long long)B * H)) {
        p.tq = true;
        p.n_pad = 128;
        p.kernel = "k_attn_tq";
        p.ws_bytes = kTqQueueBytes;   // the item queue's two counters
        p.zero_bytes = kTqQueueBytes;
        return p;
    }
    const Variant v = pick_variant(d, n_max);
    p.kernel = v.name;
    const int tiles = (L_max + TK - 1) / TK;
    const long long pairs = (long long)B * H;
    const long long slots = (long long)num_sms() * occupancy(v);
    // Split the key axis only when the (request, head) pairs fill at most half
    // a wave of CTA slots, into equal chunks. Measured on GB300 (llama7b layer,
    // 256 pairs of 33 tiles on 304 slots): no split 58 us; two equal chunks
    // 1.7x slower; chunks of 28 and 5 tiles dispatched longest-first 71 us.
    long long chunk = tiles;
    if (2 * pairs <= slots) chunk = (tiles + (slots + pairs - 1) / pairs - 1) / ((slots + pairs - 1) / pairs);
    if (const char *e = getenv("TREESPEC_ATTN_SPLITS"))   // equal chunks, this many
        if (*e) {
            int sp = atoi(e);
            sp = sp < 1 ? 1 : (sp > tiles ? tiles : sp);
            chunk = (tiles + sp - 1) / sp;
        }
    const long long min_chunk = (tiles + kMaxSplits - 1) / kMaxSplits;
    if (chunk < min_chunk) chunk = min_chunk;
    p.chunk_tiles = (int)chunk;
    p.splits = (tiles + p.chunk_tiles - 1) / p.chunk_tiles;
    p.n_pad = v.nodes;
    const size_t counters = ((size_t)pairs * 4 + 255) / 256 * 256;
    p.ws_bytes = p.splits > 1 ? counters + (size_t)pairs * p.splits * p.n_pad * (2 + d) * 4 : counters;
    p.zero_bytes = counters;
    return p;
}

cudaError_t launch_attn_bf16(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *prefix_len, const ts_tree &t, int H, int d, int L_max, float scale,
                             const AttnPlan &plan, void *ws, uint32_t *status, cudaStream_t s, const char **why,
                             const PagedArgs &pg) {
    if (plan.tq)
        return launch_attn_tq(out, q, k_cache, v_cache, prefix_len, t, H, L_max, scale, (unsigned *)ws, status, s, why,
                              pg);
    const Variant v = pick_variant(d, t.n_max);
    CUtensorMap maps[4];
    // the TMA view: every cache row, [B*H*L_max] dense or [num_pages*H*64] paged;
    // 64-row boxes, and 8-row boxes for a chunk's ragged last tile
    const long long rows = pg.bt ? (long long)pg.num_pages * H * TS_PAGE_KEYS : (long long)t.B * H * L_max;
    if (!make_map(&maps[0], k_cache, d, rows, TK) || !make_map(&maps[1], v_cache, d, rows, TK) ||
        !make_map(&maps[2], k_cache, d, rows, 8) || !make_map(&maps[3], v_cache, d, rows, 8)) {
        *why = "cuTensorMapEncodeTiled failed for the KV cache";
        return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem);
    if (e != cudaSuccess) return e;
    AttnArgs a;
    a.out = (__nv_bfloat16 *)out;
    a.q = (const __nv_bfloat16 *)q;
    a.prefix_len = prefix_len;
    a.t = t;
    a.H = H;
    a.L_max = L_max;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.chunk_tiles = plan.chunk_tiles;
    a.splits = plan.splits;
    a.n_pad = plan.n_pad;
    const size_t pairs = (size_t)t.B * H;
    const size_t counters = (pairs * 4 + 255) / 256 * 256;
    a.counters = (unsigned *)ws;
    a.part_ml = (float *)((char *)ws + counters);
    a.part_o = a.part_ml + pairs * plan.splits * 2 * plan.n_pad;
    a.status = status;
    a.bt = pg.bt;
    a.max_pages = pg.max_pages;
    a.num_pages = pg.num_pages;
    // longest-first dispatch of the requests (TREESPEC_ATTN_LPT=0: request order)
    const char *lp = getenv("TREESPEC_ATTN_LPT");
    a.lpt = !(lp && *lp && atoi(lp) == 0);
    // split index slowest: every first (longest) chunk is dispatched before any later one
    dim3 grid(H, t.B, plan.splits);
    return v.launch(grid, maps, a, s);
}

}  // namespace ts
