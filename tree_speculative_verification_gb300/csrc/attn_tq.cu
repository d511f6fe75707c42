// attn_tq.cu -- persistent tcgen05 tree attention with 128-key tiles, for trees
// of up to 128 nodes and head_dim 128.
//
// What it computes: TreeAttention(u) = Attention(S_u) for every node u of the
// token tree (SpecInfer, arXiv 2305.09781, Def. 4.1, Eq. 1-4): node i sees every
// prefix key and the tree keys of its ancestors and itself (the topology-aware
// causal mask of sec. 4.2, a bit test on the ancestor bitmask).
//
// GB300 design. Each CTA (one per SM) walks (request, head) items taken from a
// queue in the workspace (an atomic counter), its first item included, so that
// CTAs which start late -- their SM still held by a kernel of another stream --
// take fewer and shorter items instead of holding a long one to the end (a
// fixed first item per CTA made the merge-workload step, whose sampling walk
// holds 16 SMs, 131 us instead of 119 us). Items are handed out longest
// request first. The K/V ring, the two score buffers and the softmax run on
// across item boundaries.
//   warp 0    TMA producer and item queue (lane 0): claims the next item one
//             item ahead and publishes it in a 4-slot shared-memory ring
//             (mbarriers iready / ifree) that the other roles read; loads
//             128-key K and V tiles into a 3-stage ring (64 KB a stage), as
//             128-key boxes, or 64-key boxes (a paged cache: one page each;
//             and with the append in the launch), and pulls the tile after
//             each one into L2
//   warp 1    MMA issuer (lane 0): S = Q K^T (M = 128 node rows, N = 128 keys,
//             K = 128 dims) with Q read from TMEM; O += P V (M = 128, N = 128
//             dims, K = 128 keys) with P read from TMEM
//   warps 2-9 softmax. A warp reaches only its own TMEM lane quarter. Trees
//             of more than 64 nodes (DUP = false): the two warps of a quarter
//             share its 32 node rows, one taking key columns 0-63 of the tile,
//             the other 64-127. Trees of up to 64 nodes (DUP = true): lanes
//             64-127 hold a second copy of Q's rows 0-63, so all four quarters
//             (all four SM sub-partitions) work; the four warps of a node row
//             take 32 keys each, each copy of the row gets zero P for the 64
//             keys the other copy takes, and O's rows r and r + 64 are two
//             partial sums the epilogue adds through shared memory. The warps
//             of a row exchange their partial maxima (and at the end their
//             sums) through shared memory, so all apply the same running max;
//             each writes its bf16 P over the scores it came from, loads the
//             next item's Q rows into the other Q buffer, and at the end of an
//             item normalises and writes its part of each output row.
//   warp 10   (FUSED, tree_attention_append) the KV append: reads each
//             published item and copies its new K/V rows into the cache rows
//             P + dfs, an item ahead of the producer, which waits for them
//             (mbarrier tready) before it loads the item's tiles with tree keys.
// TMEM (512 columns): S0 [0,128) S1 [128,256) (fp32 scores; P in bf16 pairs:
// keys 0-63 at [x*128, +32) and 64-127 at [x*128+64, +32), or with DUP key block
// kb (32 keys) at [x*128 + kb*32, +16)), O [256,384), Q0 [384,448), Q1 [448,512)
// (bf16 pairs). Every wait is bounded; on a timeout the CTA keeps its barrier
// schedule, sets TS_STATUS_TIMEOUT and frees its TMEM.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "attn_common.cuh"
#include "ts_internal.cuh"

namespace ts {
namespace {

struct TqCfg {
    static constexpr int D = 128, TKT = 128, HALF = 64, STAGES = 3, NODES = 128, SM_WARPS = 8;
    static constexpr int THREADS = 64 + 32 * SM_WARPS;
    static constexpr int BOX_BYTES = HALF * 128;          // one TMA box: 64 key rows x 128 bytes
    static constexpr int OPB = TKT * 128;                 // a 64-dim half of a 128-key operand
    static constexpr int TILE_BYTES = 2 * OPB;            // K (or V) of 128 keys x 128 dims
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;    // K then V
    static constexpr int OFF_MX = STAGES * STAGE_BYTES;   // partial row maxima [2 parities][4 slots][128]
    static constexpr int OFF_LS = OFF_MX + 2 * 4 * NODES * 4;   // partial row sums [4 slots][128]
    static constexpr int XO_STRIDE = 33;                  // padded row of the O exchange
    static constexpr int OFF_XO = OFF_LS + 4 * NODES * 4; // upper-copy O chunks [2 quarters][2 halves][32][33]
    static constexpr int REQ_CACHE = 512;                 // (n, P) of the first requests, in shared memory
    static constexpr int OFF_REQ = OFF_XO + 4 * 32 * XO_STRIDE * 4;
    static constexpr int RING = 4;                        // published items (the queue's shared-memory ring)
    static constexpr int NBAR = 2 * STAGES + 2 + 2 + 2 + 2 + 1 + 1 + 3 * RING;
    static constexpr int OFF_ORDER = OFF_REQ + REQ_CACHE * 8;   // requests longest first
    static constexpr int OFF_BAR = OFF_ORDER + REQ_CACHE * 4;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    // misc ints: [0] TMEM base, [1] timeout, [4..8) item ring, [8..24) the softmax
    // warps' votes on a ring slot (two sets of eight)
    static constexpr int MISC_RING = 4, MISC_VOTE = 8;
    static constexpr int SMEM = OFF_MISC + 128 + 1024;
    static constexpr uint32_t TMEM_COLS = 512, S_COL = 0, O_COL = 256, Q_COL = 384;
};

struct TqItem {
    int b, h, n, P, L, ntiles;
};

// Item p = b * H + h; (n, P) from the shared-memory copy when b is in it.
__device__ __forceinline__ TqItem tq_item(const AttnArgs &a, const int2 *req, int p) {
    TqItem it;
    it.b = p / a.H;
    it.h = p - it.b * a.H;
    if (it.b < TqCfg::REQ_CACHE) {
        const int2 r = req[it.b];
        it.n = r.x;
        it.P = r.y;
    } else {
        it.n = a.t.n_nodes[it.b];
        it.P = a.prefix_len[it.b];
    }
    it.L = it.P + it.n;
    const bool ok = it.n > 0 && it.n <= TqCfg::NODES && it.P >= 0 && it.L <= a.L_max;
    it.ntiles = ok ? (it.L + TqCfg::TKT - 1) / TqCfg::TKT : 0;
    return it;
}

// A 32-bit global load issued here (the asm is not moved), its result waited
// for only where it is first used.
__device__ __forceinline__ int ld_early(const int32_t *p) {
    int v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// Ancestor words (up to four) of node row `row` of an item, loaded early; zero past n.
struct TqAnc {
    uint32_t w0, w1, w2, w3;
};
__device__ __forceinline__ TqAnc tq_anc(const AttnArgs &a, const TqItem &it, int row, bool any) {
    TqAnc r{0u, 0u, 0u, 0u};
    if (!any || row >= it.n) return r;
    const int W = TS_MASK_WORDS(a.t.n_max);
    const int32_t *ar = (const int32_t *)a.t.anc + ((size_t)it.b * a.t.n_max + row) * W;
    r.w0 = (uint32_t)ld_early(ar);
    if (W > 1) r.w1 = (uint32_t)ld_early(ar + 1);
    if (W > 2) r.w2 = (uint32_t)ld_early(ar + 2);
    if (W > 3) r.w3 = (uint32_t)ld_early(ar + 3);
    return r;
}

// Named barrier of the two softmax warps that share a TMEM lane quarter.
__device__ __forceinline__ void pair_sync(int quarter) {
    asm volatile("bar.sync %0, 64;" ::"r"(2 + quarter) : "memory");
}

// Named barrier of the four softmax warps of lane quarters lq and lq + 2 (the
// two copies of node rows lq*32 .. +32 when rows are duplicated).
__device__ __forceinline__ void group_sync(int lq) {
    asm volatile("bar.sync %0, 128;" ::"r"(6 + lq) : "memory");
}

// Named barrier of the eight softmax warps.
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 10, 256;" ::: "memory"); }

// Visibility of the keys k0 .. k0 + 63 of an item for one node row, bit e for
// key k0 + e: prefix keys visible, tree key t visible iff ancestor bit t (lo:
// bits 0-63, hi: 64-127), nothing from L on. Needs k0 + 64 > P.
__device__ __forceinline__ unsigned long long tq_window(unsigned long long lo, unsigned long long hi, int k0, int P,
                                                        int L) {
    const int t0 = k0 - P;   // tree index of the first key, > -64
    unsigned long long win;
    if (t0 >= 0) {
        win = t0 >= 64 ? (t0 >= 128 ? 0ull : hi >> (t0 - 64)) : (t0 == 0 ? lo : (lo >> t0) | (hi << (64 - t0)));
    } else {
        win = (lo << (-t0)) | ((1ull << (-t0)) - 1ull);
    }
    const int valid = L - k0;   // keys before L
    if (valid < 64) win &= valid <= 0 ? 0ull : (1ull << valid) - 1ull;
    return win;
}

// The 128-byte half (dims hf*64 .. +64) of the Q row of DFS row `row` of an
// item, given that row's node index r = perm[b][row] (null past n).
__device__ __forceinline__ const uint4 *tq_q_src(const AttnArgs &a, const TqItem &it, int row, int r, int hf) {
    if (row >= it.n || r < 0) return nullptr;
    return (const uint4 *)(a.q + (((size_t)it.b * a.t.n_max + r) * a.H + it.h) * TqCfg::D + hf * 64);
}

// One softmax warp's half of an item's Q rows (rows quarter*32 + lane; zero
// past n) into TMEM Q buffer qb.
__device__ __forceinline__ void tq_load_q(const uint4 *src, uint32_t tmem, int quarter, int hf, int qb) {
    uint32_t qw[32];
#pragma unroll
    for (int c4 = 0; c4 < 8; ++c4) {
        const uint4 v = src ? __ldg(src + c4) : make_uint4(0u, 0u, 0u, 0u);
        qw[4 * c4] = v.x;
        qw[4 * c4 + 1] = v.y;
        qw[4 * c4 + 2] = v.z;
        qw[4 * c4 + 3] = v.w;
    }
    tc_st32u(tmem + ((uint32_t)(quarter * 32) << 16) + TqCfg::Q_COL + qb * 64 + hf * 32, qw);
    tc_wait_st();
}

// DUP: every tree of the launch has at most 64 nodes, and TMEM lanes 64-127
// hold a second copy of rows 0-63 (see the file comment). FUSED: the call
// also appends the tree's new K/V rows to the cache (kv_append): a tenth warp
// copies each item's rows from the new K/V into the cache rows P + dfs (an
// item ahead of the TMA producer, which waits for them before it loads the
// item's tiles that hold tree keys; they are then read back from L2).
// PAGED: the cache is in pages of 64 keys, each tile loaded as 64-key boxes
// through the block table. A dense cache takes 128-key boxes (an SM moves
// more bytes a second in fewer, larger boxes: LLaMA-7B-shaped items at batch
// 2 26.0 -> 22.3 us, the long-context layer 347.6 -> 337.1 us; an item's last
// tile is then loaded whole, its rows past the item's keys masked as before),
// except with the append in the launch, which keeps 64-key boxes (the
// OPT-30B-shaped launch measured 345.1 us with them, 352.1 us with 128-key
// boxes, under ncu).
template <bool DUP, bool FUSED, bool PAGED>
__global__ void __launch_bounds__(TqCfg::THREADS + (FUSED ? 32 : 0), 1)
    k_attn_tq(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v, AttnArgs a) {
    using C = TqCfg;
    constexpr int D = C::D;
    constexpr int NTHR = C::THREADS + (FUSED ? 32 : 0);
    constexpr bool BOX64 = PAGED || FUSED;   // 64-key boxes (else 128-key)
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sm_base = smem_u32(sm);
    volatile int *misc = (volatile int *)(sm + C::OFF_MISC);   // [0] TMEM base, [1] timeout
    float *mx_s = (float *)(sm + C::OFF_MX);
    float *ls_s = (float *)(sm + C::OFF_LS);
    int2 *req_s = (int2 *)(sm + C::OFF_REQ);
    int *order_s = (int *)(sm + C::OFF_ORDER);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int pairs = a.t.B * a.H;
    pdl_wait();
    pdl_trigger();

    const uint32_t full = sm_base + C::OFF_BAR, empty = full + 8 * C::STAGES;
    const uint32_t sfull = empty + 8 * C::STAGES, pfull = sfull + 16, pvdone = pfull + 16;
    const uint32_t qready = pvdone + 16, ofree = qready + 16, fin = ofree + 8;
    const uint32_t iready = fin + 8, ifree = iready + 8 * C::RING, tready = ifree + 8 * C::RING;
    volatile int *ring = misc + C::MISC_RING;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32((void *)misc)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 32) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(full + 8 * s, 1);
            mbar_init(empty + 8 * s, 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(sfull + 8 * x, 1);
            mbar_init(pfull + 8 * x, C::SM_WARPS);
            mbar_init(pvdone + 8 * x, 1);
            mbar_init(qready + 8 * x, C::SM_WARPS);
        }
        mbar_init(ofree, C::SM_WARPS);
        mbar_init(fin, 1);
        for (int r = 0; r < C::RING; ++r) {
            mbar_init(iready + 8 * r, 1);
            // the MMA issuer, every softmax warp (and the tree-row warp)
            mbar_init(ifree + 8 * r, 1 + C::SM_WARPS + (FUSED ? 1 : 0));
            mbar_init(tready + 8 * r, 1);   // the item's tree rows are in the cache
        }
        misc[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // every role reads the requests' (n, P) at each item: one copy in shared memory
    for (int b = tid; b < a.t.B && b < C::REQ_CACHE; b += NTHR) req_s[b] = make_int2(a.t.n_nodes[b], a.prefix_len[b]);
    __syncthreads();
    // the producer hands out the requests' items longest first (keys P + n,
    // ties to the lower request), so that with ragged prefixes the last items
    // of the launch are short ones; request order when B exceeds the cache
    const bool lpt = a.t.B <= C::REQ_CACHE;
    for (int b = tid; lpt && b < a.t.B; b += NTHR) {
        const int kb = req_s[b].x > 0 ? req_s[b].x + req_s[b].y : -1;
        int rank = 0;
        for (int o = 0; o < a.t.B; ++o) {
            const int ko = req_s[o].x > 0 ? req_s[o].x + req_s[o].y : -1;
            rank += ko > kb || (ko == kb && o < b);
        }
        order_s[rank] = b;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = (uint32_t)misc[0];

    if (warp == 0) {
        if (lane == 0) {   // ---------------------------------------------- TMA producer, item queue
            // the next item with key tiles from the queue, -1 when none is left
            auto claim = [&]() -> int {
                for (int q = (int)atomicAdd(&a.counters[0], 1u); q < pairs; q = (int)atomicAdd(&a.counters[0], 1u)) {
                    const int p = lpt ? order_s[q / a.H] * a.H + q % a.H : q;   // the q-th item, longest first
                    const TqItem it = tq_item(a, req_s, p);
                    if (it.ntiles > 0) return p;
                    if (it.n > 0 && it.h == 0) flag(a.status, TS_STATUS_INDEX);
                }
                return -1;
            };
            // item k of this CTA into ring slot k % RING, once the item that used
            // the slot before has been released by every reader
            auto publish = [&](int k, int p) -> bool {
                const int r = k % C::RING;
                if (k >= C::RING && !mbar_wait_bounded(ifree + 8 * r, (uint32_t)(k / C::RING - 1) & 1u)) return false;
                ring[r] = p;
                mbar_arrive(iready + 8 * r);
                return true;
            };
            int g = 0, k = 0;
            int p = claim();
            bool ok = publish(0, p);
            while (ok && p >= 0) {
                const int pn = claim();   // published before this item's tiles: readers see it an item early
                if (!publish(k + 1, pn)) {
                    ok = false;
                    break;
                }
                const TqItem it = tq_item(a, req_s, p);
                bool rows_ready = !FUSED;
                for (int j = 0; j < it.ntiles; ++j, ++g) {
                    const int st = g % C::STAGES, key0 = j * C::TKT;
                    const bool h1 = key0 + C::HALF < it.L;   // the tile's second 64 keys hold any key
                    if (!rows_ready && key0 + C::TKT > it.P) {   // the first tile with tree keys
                        if (!mbar_wait_bounded(tready + 8 * (k % C::RING), (uint32_t)(k / C::RING) & 1u)) {
                            ok = false;
                            break;
                        }
                        rows_ready = true;
                    }
                    // rows (page ids) fetched before the wait
                    const int row0 = tile_row(a, it.b, it.h, key0);
                    const int row1 = BOX64 && h1 ? tile_row(a, it.b, it.h, key0 + C::HALF) : 0;
                    if (g >= C::STAGES && !mbar_wait_bounded(empty + 8 * st, (uint32_t)((g / C::STAGES) - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    const uint32_t kdst = sm_base + st * C::STAGE_BYTES, vdst = kdst + C::TILE_BYTES;
                    if constexpr (BOX64) {
                        mbar_expect_tx(full + 8 * st, (h1 ? 2 : 1) * 4 * C::BOX_BYTES);
                        for (int kh = 0; kh < (h1 ? 2 : 1); ++kh) {
                            const int row = kh ? row1 : row0;
#pragma unroll
                            for (int dh = 0; dh < 2; ++dh) {
                                tma_load_2d(kdst + dh * C::OPB + kh * C::BOX_BYTES, &map_k, dh * 64, row, full + 8 * st);
                                tma_load_2d(vdst + dh * C::OPB + kh * C::BOX_BYTES, &map_v, dh * 64, row, full + 8 * st);
                            }
                        }
                    } else {   // one 128-key box per 64-dim half of K and of V
                        mbar_expect_tx(full + 8 * st, 8 * C::BOX_BYTES);
#pragma unroll
                        for (int dh = 0; dh < 2; ++dh) {
                            tma_load_2d(kdst + dh * C::OPB, &map_k, dh * 64, row0, full + 8 * st);
                            tma_load_2d(vdst + dh * C::OPB, &map_v, dh * 64, row0, full + 8 * st);
                        }
                    }
                    {   // the tile after this one (this item's, else the next item's) into L2, so that
                        // its ring load finds it there: OPT-30B-shaped layer 334 -> 323 us (two
                        // tiles ahead 329 us, four 341 us)
                        int pj = j + 1;
                        TqItem pit = it;
                        if (pj >= it.ntiles) {
                            pj -= it.ntiles;
                            if (pn >= 0) pit = tq_item(a, req_s, pn);
                            else pj = -1;
                        }
                        if (pj >= 0 && pj < pit.ntiles) {
                            const int pk0 = pj * C::TKT;
                            for (int kh = 0; kh < (BOX64 && pk0 + C::HALF < pit.L ? 2 : 1); ++kh) {
                                const int prow = tile_row(a, pit.b, pit.h, pk0 + kh * C::HALF);
#pragma unroll
                                for (int dh = 0; dh < 2; ++dh) {
                                    tma_prefetch_2d(&map_k, dh * 64, prow);
                                    tma_prefetch_2d(&map_v, dh * 64, prow);
                                }
                            }
                        }
                    }
                }
                p = pn;
                ++k;
            }
            if (!ok) misc[1] = 1;
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {   // ---------------------------------------------- MMA issuer
            constexpr uint32_t idesc_s = idesc_bf16(128, C::TKT, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, D, true);
            bool ok = true;
            // S of tile g into score buffer g & 1, A = Q buffer qb; the buffer's
            // previous P (tile g - 2) must have been consumed by its PV
            auto issue_s = [&](int g, int qb) -> bool {
                const int st = g % C::STAGES, x = g & 1;
                if (!mbar_wait_bounded(full + 8 * st, (uint32_t)(g / C::STAGES) & 1u)) return false;
                if (g >= 2 && !mbar_wait_bounded(pvdone + 8 * x, (uint32_t)((g - 2) >> 1) & 1u)) return false;
                tc_fence_after();
                const uint32_t kbase = sm_base + st * C::STAGE_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t bd = smem_desc_sw128(kbase + (kk >> 2) * C::OPB + (kk & 3) * 32, 16, 1024);
                    tc_mma_ts(tmem + C::S_COL + x * C::TKT, tmem + C::Q_COL + qb * 64 + kk * 8, bd, idesc_s, kk > 0);
                }
                tc_commit(sfull + 8 * x);
                return true;
            };
            // O += P V for tile g; the first tile of item u (u >= 1) starts O afresh
            // once item u - 1's output has been read out of it
            auto issue_pv = [&](int g, bool first, int u) -> bool {
                const int st = g % C::STAGES, x = g & 1;
                if (first && u >= 1 && !mbar_wait_bounded(ofree, (uint32_t)(u - 1) & 1u)) return false;
                if (!mbar_wait_bounded(pfull + 8 * x, (uint32_t)(g >> 1) & 1u)) return false;
                tc_fence_after();
                const uint32_t vbase = sm_base + st * C::STAGE_BYTES + C::TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < C::TKT / 16; ++kk) {
                    const uint64_t bd = smem_desc_sw128(vbase + kk * 2048, C::OPB, 1024);
                    // P of keys 16kk .. +16: at 64-key halves (cols 0-31, 64-95), or with
                    // duplicated rows at 32-key blocks (cols 0-15, 32-47, 64-79, 96-111)
                    const uint32_t pc = DUP ? (kk >> 1) * 32 + (kk & 1) * 8 : (kk >> 2) * 64 + (kk & 3) * 8;
                    tc_mma_ts(tmem + C::O_COL, tmem + C::S_COL + x * C::TKT + pc, bd, idesc_pv,
                              (!first || kk > 0) ? 1u : 0u);
                }
                tc_commit(empty + 8 * st);
                tc_commit(pvdone + 8 * x);
                return true;
            };
            // S(g + 1) is issued before PV(g), also across item boundaries
            int g = 0, u = 0, pend_g = -1, pend_u = 0;
            bool pend_first = false;
            for (; ok; ++u) {
                const int r = u % C::RING;
                if (!mbar_wait_bounded(iready + 8 * r, (uint32_t)(u / C::RING) & 1u)) { ok = false; break; }
                const int p = ring[r];
                mbar_arrive(ifree + 8 * r);
                if (p < 0) break;
                const TqItem it = tq_item(a, req_s, p);
                const int qb = u & 1;
                if (!mbar_wait_bounded(qready + 8 * qb, (uint32_t)(u >> 1) & 1u)) { ok = false; break; }
                tc_fence_after();
                for (int j = 0; j < it.ntiles && ok; ++j, ++g) {
                    if (!issue_s(g, qb)) { ok = false; break; }
                    if (pend_g >= 0 && !issue_pv(pend_g, pend_first, pend_u)) { ok = false; break; }
                    pend_g = g;
                    pend_first = j == 0;
                    pend_u = u;
                }
            }
            if (ok && pend_g >= 0) ok = issue_pv(pend_g, pend_first, pend_u);
            if (!ok) misc[1] = 1;
            tc_commit(fin);   // completes once every MMA issued above has finished
            if (!mbar_wait_bounded(fin, 0)) misc[1] = 1;
        }
        __syncwarp();
    } else if (FUSED && warp == 2 + C::SM_WARPS) {   // -------------------- tree rows into the cache
        // item u of this CTA: its n new K/V rows (input order, 256 bytes each)
        // to cache rows P + dfs(v), eight rows per batch with every load of a
        // batch in flight; then a proxy fence (the TMA reads them back) and
        // tready of the item's ring slot
        bool ok = true;
        for (int u = 0; ok; ++u) {
            const int r = u % C::RING;
            if (!mbar_wait_warp(iready + 8 * r, (uint32_t)(u / C::RING) & 1u)) {
                ok = false;
                break;
            }
            const int p = ring[r];
            if (p >= 0) {
                const TqItem it = tq_item(a, req_s, p);
                const int n_max = a.t.n_max;
                const size_t crow = ((size_t)it.b * a.H + it.h) * a.L_max + it.P;   // the item's row P
                const int c = lane & 15;
                for (int r0 = 0; r0 < it.n; r0 += 8) {
                    uint4 kv[4], vv[4];
                    size_t dst[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int v = r0 + 2 * j + (lane >> 4);
                        dst[j] = ~(size_t)0;
                        if (v < it.n) {
                            const size_t src = (((size_t)it.b * n_max + v) * a.H + it.h) * (D / 8) + c;
                            dst[j] = (crow + __ldg(a.t.dfs_of + (size_t)it.b * n_max + v)) * (D / 8) + c;
                            kv[j] = __ldcs(a.k_new + src);
                            vv[j] = __ldcs(a.v_new + src);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (dst[j] != ~(size_t)0) {
                            a.k_cache_w[dst[j]] = kv[j];
                            a.v_cache_w[dst[j]] = vv[j];
                        }
                }
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(tready + 8 * r);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(ifree + 8 * r);
            if (p < 0) break;
        }
        if (!ok && lane == 0) misc[1] = 1;
    } else {   // ------------------------------------------------------ softmax
        const int quarter = warp & 3, hf = (warp - 2) >> 2;
        const int prow = quarter * 32 + lane;                  // this lane's TMEM row
        const int row = DUP ? (prow & 63) : prow;              // its node row
        const bool upper = DUP && quarter >= 2;                // the second copy of the row
        const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
        const int n_max = a.t.n_max;
        const float c = a.scale_log2;
        // 32-key blocks of a tile this warp scores (two, or one with duplicated
        // rows) and, with duplicated rows, the block whose P it zeroes
        constexpr int NKB = DUP ? 1 : 2;
        const int kb0 = DUP ? 2 * (quarter >> 1) + hf : 2 * hf;
        const int kbz = quarter >= 2 ? hf : 2 + hf;
        float *xo = (float *)(sm + C::OFF_XO) + ((quarter & 1) * 2 + hf) * 32 * C::XO_STRIDE + lane * C::XO_STRIDE;
        bool ok = true;
        // ring slot k (item k of this CTA). Every softmax warp votes with what it
        // read (INT_MIN: its wait gave up) and all take the common verdict, so
        // that the warps sharing named barriers always walk the same items.
        volatile int *vote = misc + C::MISC_VOTE;
        auto read_slot = [&](int k) -> int {
            const int r = k % C::RING;
            int v = INT_MIN;
            if (ok && mbar_wait_warp(iready + 8 * r, (uint32_t)(k / C::RING) & 1u)) v = ring[r];
            if (lane == 0) vote[(k & 1) * C::SM_WARPS + (warp - 2)] = v;
            softmax_sync();   // two vote sets: set k & 1 is rewritten only after every warp passed read k + 1
            int agreed = vote[(k & 1) * C::SM_WARPS];
            for (int w = 1; w < C::SM_WARPS; ++w)
                if (vote[(k & 1) * C::SM_WARPS + w] != agreed) agreed = INT_MIN;
            if (agreed == INT_MIN) {
                ok = false;
                return -1;
            }
            return agreed;
        };
        int p = read_slot(0);
        int perm_cur = -1;   // perm[b][row] of the current item
        TqAnc anc_cur{0u, 0u, 0u, 0u};   // its ancestor words of this row
        if (p >= 0) {        // Q of the first item
            const TqItem it = tq_item(a, req_s, p);
            perm_cur = row < it.n ? a.t.perm[(size_t)it.b * n_max + row] : -1;
            anc_cur = tq_anc(a, it, row, true);
            tq_load_q(tq_q_src(a, it, row, perm_cur, hf), tmem, quarter, hf, 0);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(qready);
        }
        int g = 0;
        for (int u = 0; p >= 0; ++u) {
            const TqItem it = tq_item(a, req_s, p);
            const int nxt = read_slot(u + 1);
            const TqItem itn = nxt >= 0 ? tq_item(a, req_s, nxt) : it;
            // the next item's perm entry and ancestor words issued now (used an
            // item later), an L2 prefetch of its Q row a tile later, the Q load
            // itself two tiles after that: global latency off the softmax's path
            const int perm_nxt = nxt >= 0 && row < itn.n ? ld_early(a.t.perm + (size_t)itn.b * n_max + row) : -1;
            const TqAnc anc_nxt = tq_anc(a, itn, row, nxt >= 0);
            const bool active = (row & ~31) < it.n;
            const unsigned long long anc_lo = (unsigned long long)anc_cur.w0 | ((unsigned long long)anc_cur.w1 << 32);
            const unsigned long long anc_hi = (unsigned long long)anc_cur.w2 | ((unsigned long long)anc_cur.w3 << 32);
            float m_run = -INFINITY, l_run = 0.f;
            const int jq = it.ntiles - 1 < 3 ? it.ntiles - 1 : 3;   // after this tile, the next item's Q
            const int jp = jq < 1 ? jq : 1;                           // after this tile, its L2 prefetch
            for (int j = 0; j < it.ntiles; ++j, ++g) {
                const int x = g & 1;
                if (ok && !mbar_wait_warp(sfull + 8 * x, (uint32_t)(g >> 1) & 1u)) ok = false;
                tc_fence_after();
                const int key_base = j * C::TKT, k0 = key_base + kb0 * 32;   // this warp's first key
                const uint32_t sb = tl + C::S_COL + x * C::TKT;
                float sv[32 * NKB];
                float mh = -INFINITY;
                if (ok && active) {
                    tc_ld32(sb + kb0 * 32, *reinterpret_cast<float(*)[32]>(&sv[0]));
                    if constexpr (NKB == 2) tc_ld32(sb + (kb0 + 1) * 32, *reinterpret_cast<float(*)[32]>(&sv[32]));
                    tc_wait_ld();
                    if (k0 + 32 * NKB > it.P) {   // tree keys or keys past the end in these blocks
                        const unsigned long long win = tq_window(anc_lo, anc_hi, k0, it.P, it.L);
                        const uint32_t wl = (uint32_t)win, wh = (uint32_t)(win >> 32);
#pragma unroll
                        for (int e = 0; e < 32 * NKB; ++e)
                            if (!(((e < 32 ? wl : wh) >> (e & 31)) & 1u)) sv[e] = -INFINITY;
                    }
                    float mx4[4] = {sv[0], sv[1], sv[2], sv[3]};
#pragma unroll
                    for (int e = 4; e < 32 * NKB; ++e) mx4[e & 3] = fmaxf(mx4[e & 3], sv[e]);
                    mh = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c;
                }
                // the partial maxima of the row's warps: all take the same row max
                float mo;
                if constexpr (DUP) {
                    mx_s[((g & 1) * 4 + kb0) * C::NODES + row] = mh;
                    group_sync(quarter & 1);
                    mo = fmaxf(fmaxf(mx_s[((g & 1) * 4) * C::NODES + row], mx_s[((g & 1) * 4 + 1) * C::NODES + row]),
                               fmaxf(mx_s[((g & 1) * 4 + 2) * C::NODES + row], mx_s[((g & 1) * 4 + 3) * C::NODES + row]));
                } else {
                    mx_s[((g & 1) * 4 + hf) * C::NODES + row] = mh;
                    pair_sync(quarter);
                    mo = mx_s[((g & 1) * 4 + (hf ^ 1)) * C::NODES + row];
                }
                if (ok && active) {
                    const float mt = fmaxf(mh, mo);
                    float alpha = 1.f;
                    bool resc = false;
                    if (m_run == -INFINITY) {
                        m_run = mt;                          // nothing accumulated yet for this row
                    } else if (mt > m_run + 8.f) {
                        alpha = exp2f(m_run - mt);
                        m_run = mt;
                        resc = true;
                    }
                    if (__any_sync(0xffffffffu, resc)) {
                        // the previous PV must have landed in O before O is rescaled
                        const int gp = g - 1;
                        if (j >= 1 && !mbar_wait_warp(pvdone + 8 * (gp & 1), (uint32_t)(gp >> 1) & 1u)) ok = false;
                        tc_fence_after();
                        if (ok) {
#pragma unroll
                            for (int q2 = 0; q2 < 2; ++q2) {
                                float o[32];
                                tc_ld32(tl + C::O_COL + hf * 64 + q2 * 32, o);
                                tc_wait_ld();
#pragma unroll
                                for (int e = 0; e < 32; ++e) o[e] *= alpha;
                                tc_st32(tl + C::O_COL + hf * 64 + q2 * 32, o);
                            }
                            tc_wait_st();
                        }
                        l_run *= alpha;
                    }
                    if (ok) {
                        const float mu = m_run == -INFINITY ? 0.f : m_run;
                        float ls[4] = {0.f, 0.f, 0.f, 0.f};
                        uint32_t pk[16 * NKB];
#pragma unroll
                        for (int e = 0; e < 32 * NKB; e += 2) {
                            // the row sum takes the fp32 probabilities, P V their bf16 roundings
                            const float p0 = ex2(__fmaf_rn(sv[e], c, -mu)), p1 = ex2(__fmaf_rn(sv[e + 1], c, -mu));
                            const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
                            pk[e >> 1] = *reinterpret_cast<const uint32_t *>(&pb);
                            ls[(e >> 1) & 3] += p0 + p1;
                        }
                        l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                        if constexpr (DUP) {
                            // P over the first 16 columns of the scored block; this copy of
                            // the row takes no part in the other copy's keys
                            tc_st16u(sb + kb0 * 32, pk);
                            uint32_t zr[16];
#pragma unroll
                            for (int e = 0; e < 16; ++e) zr[e] = 0u;
                            tc_st16u(sb + kbz * 32, zr);
                        } else {
                            tc_st32u(sb + hf * 64, pk);   // P over the first 32 columns of this half
                        }
                        tc_wait_st();
                    }
                }
                if (key_base + C::TKT > it.L) {
                    // last tile of the item: zero the V rows past its keys (they may
                    // hold anything, even NaN, or stale rows of an earlier tile)
                    const int st = g % C::STAGES;
                    if (ok && !mbar_wait_warp(full + 8 * st, (uint32_t)(g / C::STAGES) & 1u)) ok = false;
                    unsigned char *vt = sm + st * C::STAGE_BYTES + C::TILE_BYTES;
                    const int r0 = it.L - key_base;
                    for (int idx = tid - 64; ok && idx < (C::TKT - r0) * 16; idx += 32 * C::SM_WARPS) {
                        const int r = r0 + (idx >> 4), c16 = idx & 15;
                        *(uint4 *)(vt + (c16 >> 3) * C::OPB + r * 128 + ((c16 & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_async_smem();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pfull + 8 * x);
                if (j == jp && nxt >= 0) {
                    const uint4 *qs = tq_q_src(a, itn, row, perm_nxt, hf);
                    if (qs) asm volatile("prefetch.global.L2 [%0];" ::"l"(qs));
                }
                if (j == jq && nxt >= 0) {
                    // the next item's Q rows into the other Q buffer: every S of the
                    // item that used it finished before this item's first S
                    if (ok) tq_load_q(tq_q_src(a, itn, row, perm_nxt, hf), tmem, quarter, hf, (u + 1) & 1);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(qready + 8 * ((u + 1) & 1));
                }
            }
            // ---- epilogue: O holds the item once its last PV has finished
            const int gl = g - 1;
            if (ok && !mbar_wait_warp(pvdone + 8 * (gl & 1), (uint32_t)(gl >> 1) & 1u)) ok = false;
            tc_fence_after();
            float lsum;
            if constexpr (DUP) {
                ls_s[kb0 * C::NODES + row] = l_run;
                group_sync(quarter & 1);
                lsum = (ls_s[row] + ls_s[C::NODES + row]) + (ls_s[2 * C::NODES + row] + ls_s[3 * C::NODES + row]);
            } else {
                ls_s[hf * C::NODES + row] = l_run;
                pair_sync(quarter);
                lsum = ls_s[row] + ls_s[C::NODES + row];
            }
            const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
            uint4 *dst = nullptr;
            if (ok && active && !upper && row < it.n && perm_cur >= 0)
                dst = (uint4 *)(a.out + (((size_t)it.b * n_max + perm_cur) * a.H + it.h) * D + hf * 64);
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {   // 32 dims at a time
                float o[32];
                if (ok && active) {
                    tc_ld32(tl + C::O_COL + hf * 64 + q2 * 32, o);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0.f;
                }
                if (q2 == 1) {   // O is read out: the next item's first PV may overwrite it
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(ofree);
                }
                if constexpr (DUP) {   // the upper copy's partial row goes to its lower twin
                    if (upper) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) xo[e] = o[e];
                    }
                    group_sync(quarter & 1);
                    if (!upper) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] += xo[e];
                    }
                    group_sync(quarter & 1);
                }
                if (dst) {
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        float d0, d1;
                        uint4 v;
                        v.x = pack_bf16(o[8 * c8] * inv, o[8 * c8 + 1] * inv, d0, d1);
                        v.y = pack_bf16(o[8 * c8 + 2] * inv, o[8 * c8 + 3] * inv, d0, d1);
                        v.z = pack_bf16(o[8 * c8 + 4] * inv, o[8 * c8 + 5] * inv, d0, d1);
                        v.w = pack_bf16(o[8 * c8 + 6] * inv, o[8 * c8 + 7] * inv, d0, d1);
                        dst[q2 * 4 + c8] = v;
                    }
                }
            }
            if (lane == 0) mbar_arrive(ifree + 8 * (u % C::RING));   // the item's ring slot may be reused
            p = nxt;
            perm_cur = perm_nxt;
            anc_cur = anc_nxt;
        }
        if (!ok) misc[1] = 1;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
    if (tid == 0) {
        if (misc[1]) flag(a.status, TS_STATUS_TIMEOUT);
        // the last CTA to finish returns the queue to zero for the next launch:
        // every CTA counted here has stopped claiming items
        __threadfence();
        if (atomicAdd(&a.counters[1], 1u) == gridDim.x - 1) {
            a.counters[0] = 0u;
            a.counters[1] = 0u;
        }
    }
}

}  // namespace

cudaError_t launch_attn_tq(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *prefix_len, const ts_tree &t, int H, int L_max, float scale,
                           unsigned *queue, uint32_t *status, cudaStream_t s, const char **why, const PagedArgs &pg,
                           const void *k_new, const void *v_new) {
    CUtensorMap mk, mv;
    // the TMA view: every cache row, [B*H*L_max] dense or [num_pages*H*64] paged
    const long long rows = pg.bt ? (long long)pg.num_pages * H * TS_PAGE_KEYS : (long long)t.B * H * L_max;
    const int box_rows = pg.bt || k_new ? TqCfg::HALF : TqCfg::TKT;   // the kernel's BOX64
    if (!make_map(&mk, k_cache, TqCfg::D, rows, box_rows) || !make_map(&mv, v_cache, TqCfg::D, rows, box_rows)) {
        *why = "cuTensorMapEncodeTiled failed for the KV cache";
        return cudaErrorInvalidValue;
    }
    const bool dup = t.n_max <= 64, fused = k_new != nullptr;
    if (fused && pg.bt) {
        *why = "the fused append takes a dense cache";
        return cudaErrorInvalidValue;
    }
    const bool paged = pg.bt != nullptr;
    const void *fn = fused   ? (dup ? (const void *)k_attn_tq<true, true, false> : (const void *)k_attn_tq<false, true, false>)
                     : paged ? (dup ? (const void *)k_attn_tq<true, false, true> : (const void *)k_attn_tq<false, false, true>)
                             : (dup ? (const void *)k_attn_tq<true, false, false> : (const void *)k_attn_tq<false, false, false>);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, TqCfg::SMEM);
    if (e != cudaSuccess) return e;
    AttnArgs a;
    a.out = (__nv_bfloat16 *)out;
    a.q = (const __nv_bfloat16 *)q;
    a.prefix_len = prefix_len;
    a.t = t;
    a.H = H;
    a.L_max = L_max;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.chunk_tiles = 0;
    a.splits = 1;
    a.n_pad = TqCfg::NODES;
    a.counters = queue;   // [0] next item, [1] CTAs finished
    a.part_ml = nullptr;
    a.part_o = nullptr;
    a.status = status;
    a.bt = pg.bt;
    a.max_pages = pg.max_pages;
    a.num_pages = pg.num_pages;
    a.k_new = (const uint4 *)k_new;
    a.v_new = (const uint4 *)v_new;
    a.k_cache_w = (uint4 *)const_cast<void *>(k_cache);
    a.v_cache_w = (uint4 *)const_cast<void *>(v_cache);
    const int pairs = t.B * H;
    const int grid = pairs < num_sms() ? pairs : num_sms();
    if (grid < 1) return cudaSuccess;
    const dim3 block(TqCfg::THREADS + (fused ? 32 : 0));
    if (fused) {
        if (dup) return launch(k_attn_tq<true, true, false>, dim3(grid), block, TqCfg::SMEM, s, mk, mv, a);
        return launch(k_attn_tq<false, true, false>, dim3(grid), block, TqCfg::SMEM, s, mk, mv, a);
    }
    if (paged) {
        if (dup) return launch(k_attn_tq<true, false, true>, dim3(grid), block, TqCfg::SMEM, s, mk, mv, a);
        return launch(k_attn_tq<false, false, true>, dim3(grid), block, TqCfg::SMEM, s, mk, mv, a);
    }
    if (dup) return launch(k_attn_tq<true, false, false>, dim3(grid), block, TqCfg::SMEM, s, mk, mv, a);
    return launch(k_attn_tq<false, false, false>, dim3(grid), block, TqCfg::SMEM, s, mk, mv, a);
}

}  // namespace ts
