// attn_kt.cu -- tree attention for small trees (at most 32 nodes, head_dim 128)
// on the tcgen05 tensor cores with the key axis on the MMA's M side.
//
// What it computes: TreeAttention(u) = Attention(S_u) for every node u of the
// token tree (SpecInfer, arXiv 2305.09781, Def. 4.1, Eq. 1-4) over the shared
// KV cache of sec. 4.2 (verified prefix, then the tree in depth-first order).
// Key j is visible to node u iff j < P or key j - P is an ancestor of u or u
// itself (the topology-aware causal mask of sec. 4.2).
//
// GB300 design:
//  * Work split: the 128-key tiles of all (request, head) pairs, laid end to
//    end in (request, head, tile) order, are cut into gridDim.x equal ranges,
//    one per persistent CTA (one CTA per SM), so every SM streams the same
//    number of K/V bytes whatever the pair count and the prefix lengths. A
//    pair cut by a range boundary leaves partials (reference max, row sum,
//    unnormalised O) in the workspace; the CTA that arrives last on the
//    pair's counter merges them. No CTA waits for another.
//  * Per tile, two MMAs with fp32 accumulators in TMEM:
//      S^T = K Q^T      M = 128 keys, N = 32 nodes, K = 128 dims
//      O^T += V^T P^T   M = 128 dims, N = 32 nodes, K = 128 keys
//    Each is split into two accumulator chains (over dims, over keys) whose
//    MMAs are issued alternately and summed when read: with N = 32 an MMA is
//    short, and eight MMAs into one accumulator would run at the latency of
//    one dependent MMA after another.
//    K, Q and P^T are K-major, V is MN-major -- all in the 128-byte swizzled
//    layout TMA writes -- so a tree of 21 nodes pads to 32 columns, not to
//    128 rows. Node columns are in input order (Q rows are read without the
//    depth-first permutation; the mask is translated instead).
//  * Memory: K and V tiles (32 KB each) in separate rings: K, read only by
//    the first MMA, is freed as soon as that MMA completes (2 slots); V waits
//    for the softmax and the second MMA (4 slots). L2 prefetches further ahead
//    measured slower on GB300 and are not used.
//  * Softmax: eight warps; the two warps on a TMEM lane quarter own the 32
//    keys of that quarter and split the 32 node columns, 16 each. Scores are
//    exponentiated (ex2.approx) against a reference max per node that moves
//    only when a score exceeds it by more than 2^8 -- one vote of the eight
//    warps per tile, the threshold compared on the raw score -- so a tile
//    needs no cross-thread max; each thread keeps partial row sums of its
//    own key, summed across the warps once per pair segment. Lane pairs
//    exchange values so that each thread writes whole 4-byte words of P^T,
//    32 banks per warp store.
//  * Warps: 0 TMA producer (lane 0) and TMEM owner; 1 MMA issuer (lane 0),
//    which polls the ring and the softmax and issues whichever MMA is ready;
//    2-9 softmax and epilogue; 10 loads each segment's Q rows and
//    descendant masks into a double buffer. Every wait is bounded; TMEM is
//    freed on every exit path.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <stdlib.h>

#include "attn_common.cuh"
#include "ts_internal.cuh"

namespace ts {
namespace {

struct KtCfg {
    static constexpr int D = 128, TKT = 128, NODES = 32;
    static constexpr int KS = 2, VS = 4;                  // K and V ring slots (K is freed right after S^T)
        static constexpr int SM_WARPS = 8;                    // softmax warps 2..9
    static constexpr int LOADER_WARP = 10;
    static constexpr int THREADS = 11 * 32;
    static constexpr int REGION = TKT * 128;              // 128 key rows x 64 dims
    static constexpr int TILE_BYTES = 2 * REGION;         // K (or V) of one tile
    static constexpr int OFF_V = KS * TILE_BYTES;
    static constexpr int QREG = NODES * 128;              // 32 node rows x 64 dims
    static constexpr int Q_BYTES = 2 * QREG;
    static constexpr int PREG = NODES * 128;              // 32 node rows x 64 keys
    static constexpr int P_BYTES = 2 * PREG;
    static constexpr int OFF_Q = OFF_V + VS * TILE_BYTES;  // two Q buffers
    static constexpr int OFF_P = OFF_Q + 2 * Q_BYTES;     // two P^T buffers
    static constexpr int OFF_META = OFF_P + 2 * P_BYTES;  // per Q buffer: descendant masks [32]
    static constexpr int OFF_RED = OFF_META + 2 * NODES * 4;       // [2 halves][4 quarters][16]
    static constexpr int OFF_VOTE = OFF_RED + 2 * 4 * 16 * 4;      // [2][8] vote slots
    static constexpr int NBAR = 2 * KS + 2 * VS + 8 * 2 + 1;
    static constexpr int OFF_BAR = OFF_VOTE + 2 * SM_WARPS * 4;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM = OFF_MISC + 64 + 1024;     // + alignment slack (misc: 4 ints, then 5 long longs)
    // TMEM columns: S [0,128) two tiles x two chains, O [128,256) two segments x two chains
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr int S_COL = 0, O_COL = 128, CHAIN = 32, BUF = 64;
    static constexpr float THR = 8.0f;                    // log2 headroom above the reference max
    static constexpr int PART_FLOATS = NODES * D + 2 * NODES;   // one partial: O [32][128], max[32], sum[32]
};
static_assert(KtCfg::SMEM <= 232448, "shared memory of the small-tree kernel");

// Tiles of request b (0 for an empty or out-of-range request).
__device__ __forceinline__ int kt_tiles(const AttnArgs &a, int b, int &P, int &n) {
    n = a.t.n_nodes[b];
    P = a.prefix_len[b];
    if (n <= 0 || P < 0 || P + n > a.L_max) return 0;
    return (P + n + KtCfg::TKT - 1) / KtCfg::TKT;
}

struct Seg {
    int b, h, j0, j1, tiles, P, n, slot;
    long long gp;   // global index of the pair's first tile
    bool whole;
};

// Walks the CTA's tile range [s_begin, s_end) as segments, one per (request,
// head) pair it touches. The range's last segment comes first (it is the
// start of a pair whose rest another CTA finished at its own start), so that
// the pairs cut by range boundaries are merged early, where the K/V stream
// of this and the other CTAs hides the merge, not at the end of the kernel.
// Every role of the CTA runs its own copy.
struct SegIter {
    long long g, g_end, gb, s_begin;
    int b, tiles, P, n;
    // the range's last segment: pair (last_b, last_h) from tile last_j0 on
    int last_b, last_h, last_j0, last_j1, last_tiles, last_P, last_n;
    long long last_gp;
    bool last_pending;
    __device__ void init(const AttnArgs &a, long long sb, long long se, int b0, long long gb0, int b1, long long gb1) {
        s_begin = g = sb;
        g_end = se;
        b = b0;
        gb = gb0;
        tiles = b0 < a.t.B ? kt_tiles(a, b0, P, n) : 0;
        last_pending = false;
        if (se > sb && b1 < a.t.B) {
            last_b = b1;
            last_tiles = kt_tiles(a, b1, last_P, last_n);
            last_h = (int)((se - 1 - gb1) / last_tiles);
            last_gp = gb1 + (long long)last_h * last_tiles;
            const long long start = last_gp > sb ? last_gp : sb;
            if (start > sb) {   // more than one segment: the last goes first
                last_pending = true;
                last_j0 = (int)(start - last_gp);
                last_j1 = (int)(se - last_gp);
                g_end = start;
            }
        }
    }
    __device__ bool next(const AttnArgs &a, Seg &s) {
        if (last_pending) {
            last_pending = false;
            s.b = last_b;
            s.h = last_h;
            s.j0 = last_j0;
            s.j1 = last_j1;
            s.gp = last_gp;
            s.tiles = last_tiles;
            s.P = last_P;
            s.n = last_n;
            s.whole = s.j0 == 0 && s.j1 == last_tiles;
            s.slot = 1;
            return true;
        }
        while (g < g_end) {
            const long long span = (long long)a.H * tiles;
            if (g >= gb + span) {
                gb += span;
                if (++b >= a.t.B) return false;
                tiles = kt_tiles(a, b, P, n);
                continue;
            }
            const long long off = g - gb;
            s.b = b;
            s.h = (int)(off / tiles);
            s.j0 = (int)(off % tiles);
            s.gp = gb + (long long)s.h * tiles;
            const long long stop = s.gp + tiles < g_end ? s.gp + tiles : g_end;
            s.j1 = (int)(stop - s.gp);
            s.tiles = tiles;
            s.P = P;
            s.n = n;
            s.whole = s.j0 == 0 && s.j1 == tiles;
            s.slot = g == s_begin ? 0 : 1;
            g = stop;
            return true;
        }
        return false;
    }
};

// Walks the CTA's tiles one at a time: global tile count t, segment index
// si and the tile's place in its segment.
struct TileCursor {
    SegIter it;
    Seg sg;
    int j, t, si;
    bool has;
    __device__ void init(const SegIter &i0, const AttnArgs &a) {
        it = i0;
        t = 0;
        si = -1;
        next_seg(a);
    }
    __device__ void next_seg(const AttnArgs &a) {
        has = it.next(a, sg);
        if (has) {
            j = sg.j0;
            ++si;
        }
    }
    __device__ void advance(const AttnArgs &a) {
        ++t;
        if (++j >= sg.j1) next_seg(a);
    }
    __device__ bool first() const { return j == sg.j0; }
    __device__ bool last() const { return j == sg.j1 - 1; }
    __device__ int row(const AttnArgs &a) const { return (sg.b * a.H + sg.h) * a.L_max + j * KtCfg::TKT; }
};

// First tile of CTA c when T tiles are cut into G ranges, and the CTA that
// holds tile g.
__device__ __forceinline__ long long range_start(long long T, int c, int G) { return T * c / G; }
__device__ __forceinline__ int range_of(long long T, long long g, int G) {
    return (int)(((g + 1) * G + T - 1) / T) - 1;
}

__device__ __forceinline__ void named_sync_softmax() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// One vote per softmax warp (bit-OR of the eight warps' values), the same
// result in every softmax thread.
__device__ __forceinline__ int group_vote(volatile int *slots, int &parity, int sw, int v) {
    if ((threadIdx.x & 31) == 0) slots[parity * 8 + sw] = v;
    named_sync_softmax();
    const volatile int *q = slots + parity * 8;
    const int r = (q[0] | q[1] | q[2] | q[3]) | (q[4] | q[5] | q[6] | q[7]);
    parity ^= 1;
    return r;
}

// Lanes c and c + 16 end up with the maximum (or sum) over the warp's 32
// lanes of element c of v: 16 shuffles across the half-warps, then 15 to
// transpose.
template <bool MAX>
__device__ __forceinline__ float reduce16(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, v[i], 16);
        v[i] = MAX ? fmaxf(v[i], o) : v[i] + o;
    }
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1) {
        const bool up = lane & w;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float send = up ? v[i] : v[i + w];
            const float keep = up ? v[i + w] : v[i];
            const float got = __shfl_xor_sync(0xffffffffu, send, w);
            v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

__device__ __forceinline__ void sts_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts_zero16(uint32_t addr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
}

__global__ void __launch_bounds__(KtCfg::THREADS, 1) k_attn_kt(const __grid_constant__ CUtensorMap map_k,
                                                               const __grid_constant__ CUtensorMap map_v, AttnArgs a) {
    using C = KtCfg;
    constexpr int D = C::D;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const uint32_t sm_base = smem_u32(sm);
    volatile int *misc = (volatile int *)(sm + C::OFF_MISC);   // [0] TMEM base, [1] timeout, [2] merge flag
    long long *sched = (long long *)(sm + C::OFF_MISC + 16);  // T, first tile of b0, b0, first tile of b1, b1
    uint32_t *meta = (uint32_t *)(sm + C::OFF_META);          // [qb][32] descendant masks
    float *red = (float *)(sm + C::OFF_RED);                  // [half][quarter][16]
    volatile int *vote = (volatile int *)(sm + C::OFF_VOTE);  // [2][8]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = gridDim.x, cta = blockIdx.x;
    const int H = a.H, n_max = a.t.n_max, W = TS_MASK_WORDS(n_max);

    const uint32_t kfull = sm_base + C::OFF_BAR, kempty = kfull + 8 * C::KS;
    const uint32_t vfull = kempty + 8 * C::KS, vempty = vfull + 8 * C::VS;
    const uint32_t sfull = vempty + 8 * C::VS, sfree = sfull + 16, pfull = sfree + 16, pfree = pfull + 16;
    const uint32_t qfull = pfree + 16, qfree = qfull + 16, odone = qfree + 16, ofree = odone + 16;
    const uint32_t fin = ofree + 16;

    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32((void *)misc)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (tid == 32) {
        for (int s = 0; s < C::KS; ++s) {
            mbar_init(kfull + 8 * s, 1);
            mbar_init(kempty + 8 * s, 1);
        }
        for (int s = 0; s < C::VS; ++s) {
            mbar_init(vfull + 8 * s, 1);
            mbar_init(vempty + 8 * s, 1);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(sfull + 8 * x, 1);
            mbar_init(sfree + 8 * x, C::SM_WARPS);
            mbar_init(pfull + 8 * x, C::SM_WARPS);
            mbar_init(pfree + 8 * x, 1);
            mbar_init(qfull + 8 * x, 1);
            mbar_init(qfree + 8 * x, 1 + C::SM_WARPS);   // the MMA issuer's commit + every softmax warp
            mbar_init(odone + 8 * x, 1);
            mbar_init(ofree + 8 * x, C::SM_WARPS);
        }
        mbar_init(fin, 1);
        misc[1] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    pdl_wait();
    pdl_trigger();
    if (warp == C::LOADER_WARP) {
        // ---- schedule: total tiles T and the request holding this CTA's first tile
        const int B = a.t.B;
        long long tot = 0;
        for (int base = 0; base < B; base += 32) {
            const int b = base + lane;
            int P = 0, n = 0, tl = 0;
            if (b < B) {
                tl = kt_tiles(a, b, P, n);
                if (n > 0 && tl == 0 && cta == 0) flag(a.status, TS_STATUS_INDEX);
            }
            int s = tl;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            tot += s;
        }
        const long long T = tot * H, s0 = range_start(T, cta, G), s1 = range_start(T, cta + 1, G);
        long long acc = 0, gb0 = T, gb1 = T;
        int b0 = B, b1 = B;
        for (int base = 0; base < B && (b0 == B || b1 == B); base += 32) {
            const int b = base + lane;
            int P = 0, n = 0;
            const int tl = b < B ? kt_tiles(a, b, P, n) : 0;
            int incl = tl;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const long long start = acc + (long long)H * (incl - tl);
            const bool hit0 = tl > 0 && s0 >= start && s0 < start + (long long)H * tl;
            const bool hit1 = tl > 0 && s1 - 1 >= start && s1 - 1 < start + (long long)H * tl;
            const unsigned m0 = __ballot_sync(0xffffffffu, hit0), m1 = __ballot_sync(0xffffffffu, hit1);
            if (m0) {
                const int src = __ffs(m0) - 1;
                b0 = base + src;
                gb0 = __shfl_sync(0xffffffffu, start, src);
            }
            if (m1) {
                const int src = __ffs(m1) - 1;
                b1 = base + src;
                gb1 = __shfl_sync(0xffffffffu, start, src);
            }
            acc += (long long)H * __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            sched[0] = T;
            sched[1] = gb0;
            sched[2] = b0;
            sched[3] = gb1;
            sched[4] = b1;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = (uint32_t)misc[0];
    const long long T = sched[0];
    SegIter it0;
    it0.init(a, range_start(T, cta, G), range_start(T, cta + 1, G), (int)sched[2], sched[1], (int)sched[4], sched[3]);

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------------ TMA producer
            TileCursor cur;
            cur.init(it0, a);
            bool ok = true;
            while (ok && cur.has) {
                const int t = cur.t, ks = t % C::KS, vs = t % C::VS;
                const int y = cur.row(a);
                if (t >= C::KS && !mbar_wait_bounded(kempty + 8 * ks, (uint32_t)((t / C::KS) - 1) & 1u)) {
                    ok = false;
                    break;
                }
                const uint32_t kdst = sm_base + ks * C::TILE_BYTES;
                mbar_expect_tx(kfull + 8 * ks, C::TILE_BYTES);
                tma_load_2d(kdst, &map_k, 0, y, kfull + 8 * ks);
                tma_load_2d(kdst + C::REGION, &map_k, 64, y, kfull + 8 * ks);
                if (t >= C::VS && !mbar_wait_bounded(vempty + 8 * vs, (uint32_t)((t / C::VS) - 1) & 1u)) {
                    ok = false;
                    cur.advance(a);   // K of this tile is in flight: drained below
                    break;
                }
                const uint32_t vdst = sm_base + C::OFF_V + vs * C::TILE_BYTES;
                mbar_expect_tx(vfull + 8 * vs, C::TILE_BYTES);
                tma_load_2d(vdst, &map_v, 0, y, vfull + 8 * vs);
                tma_load_2d(vdst + C::REGION, &map_v, 64, y, vfull + 8 * vs);
                cur.advance(a);
            }
            if (!ok) misc[1] = 1;
            // no copy may still be landing in shared memory when the CTA exits (a V copy
            // not issued for the last tile is waited for in vain only after a timeout)
            const int t = cur.t;
            for (int k = t - C::KS < 0 ? 0 : t - C::KS; k < t; ++k)
                if (!mbar_wait_bounded(kfull + 8 * (k % C::KS), (uint32_t)(k / C::KS) & 1u)) misc[1] = 1;
            for (int k = t - C::VS < 0 ? 0 : t - C::VS; k < t; ++k)
                if (!mbar_wait_bounded(vfull + 8 * (k % C::VS), (uint32_t)(k / C::VS) & 1u)) misc[1] = 1;
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ------------------------------------------------ MMA issuer
            constexpr uint32_t idesc_s = idesc_bf16(128, C::NODES, false, false);
            constexpr uint32_t idesc_pv = idesc_bf16(128, C::NODES, false, true);
            // cursor s: the next S^T = K Q^T; cursor p: the next O^T += V^T P^T (always behind s).
            // Each is issued as soon as its inputs are ready, so a stage is released
            // without waiting for the next tile's data.
            TileCursor cs, cp;
            cs.init(it0, a);
            cp.init(it0, a);
            bool ok = true;
            long long t_prog = clock64();
            while (cs.has || cp.t < cs.t) {
                bool prog = false;
                if (cs.has) {
                    const int t = cs.t, x = t & 1, ks = t % C::KS, qb = cs.si & 1;
                    if ((!cs.first() || mbar_test(qfull + 8 * qb, (uint32_t)(cs.si >> 1) & 1u)) &&
                        (t < 2 || mbar_test(sfree + 8 * x, (uint32_t)((t >> 1) - 1) & 1u)) &&
                        mbar_test(kfull + 8 * ks, (uint32_t)(t / C::KS) & 1u)) {
                        tc_fence_after();
                        const uint32_t kbase = sm_base + ks * C::TILE_BYTES;
                        const uint32_t qbase = sm_base + C::OFF_Q + qb * C::Q_BYTES;
                        // two independent accumulator chains (dims 0-63 and 64-127), issued
                        // alternately so that consecutive MMAs never wait on each other
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
                            for (int ch = 0; ch < 2; ++ch) {
                                const uint64_t ad = smem_desc_sw128(kbase + ch * C::REGION + k4 * 32, 16, 1024);
                                const uint64_t bd = smem_desc_sw128(qbase + ch * C::QREG + k4 * 32, 16, 1024);
                                tc_mma(tmem + C::S_COL + x * C::BUF + ch * C::CHAIN, ad, bd, idesc_s, k4 > 0 ? 1u : 0u);
                            }
                        tc_commit(sfull + 8 * x);
                        tc_commit(kempty + 8 * ks);
                        if (cs.last()) tc_commit(qfree + 8 * qb);
                        cs.advance(a);
                        prog = true;
                    }
                }
                if (cp.t < cs.t) {
                    const int t = cp.t, x = t & 1, vs = t % C::VS, ob = cp.si & 1;
                    if (mbar_test(pfull + 8 * x, (uint32_t)(t >> 1) & 1u) &&
                        mbar_test(vfull + 8 * vs, (uint32_t)(t / C::VS) & 1u) &&
                        (!cp.first() || cp.si < 2 || mbar_test(ofree + 8 * ob, (uint32_t)((cp.si >> 1) - 1) & 1u))) {
                        tc_fence_after();
                        const uint32_t vbase = sm_base + C::OFF_V + vs * C::TILE_BYTES;
                        const uint32_t pbase = sm_base + C::OFF_P + x * C::P_BYTES;
                        const bool first = cp.first();
                        // two independent chains (keys 0-63 and 64-127), issued alternately
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
                            for (int ch = 0; ch < 2; ++ch) {
                                const int kk = ch * 4 + k4;
                                const uint64_t ad = smem_desc_sw128(vbase + kk * 2048, C::REGION, 1024);
                                const uint64_t bd = smem_desc_sw128(pbase + ch * C::PREG + k4 * 32, 16, 1024);
                                tc_mma(tmem + C::O_COL + ob * C::BUF + ch * C::CHAIN, ad, bd, idesc_pv,
                                       (first && k4 == 0) ? 0u : 1u);
                            }
                        tc_commit(pfree + 8 * x);
                        tc_commit(vempty + 8 * vs);
                        if (cp.last()) tc_commit(odone + 8 * ob);
                        cp.advance(a);
                        prog = true;
                    }
                }
                if (prog) {
                    t_prog = clock64();
                } else if (clock64() - t_prog > kWaitCycles) {
                    ok = false;
                    break;
                }
            }
            if (!ok) misc[1] = 1;
            // every MMA of this CTA has completed before TMEM is freed
            tc_commit(fin);
            if (!mbar_wait_bounded(fin, 0)) misc[1] = 1;
        }
    } else if (warp == C::LOADER_WARP) {   // ------------------------------------ segment loader
        SegIter it = it0;
        Seg sg;
        int si = 0;
        while (it.next(a, sg)) {
            const int qb = si & 1;
            if (si >= 2 && !mbar_wait_warp(qfree + 8 * qb, (uint32_t)((si >> 1) - 1) & 1u)) {
                if (lane == 0) misc[1] = 1;
                break;
            }
            const size_t rb = (size_t)sg.b * n_max;
            const bool real = lane < sg.n;
            // Q row of input node `lane` into the 128-byte swizzled K-major layout
            const uint4 *qrow = reinterpret_cast<const uint4 *>(a.q + ((rb + lane) * H + sg.h) * D);
            uint4 qv[16];
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) qv[ch] = real ? __ldg(qrow + ch) : make_uint4(0u, 0u, 0u, 0u);
            // ancestors of input node `lane` as depth-first positions; tree key i (position
            // i) is visible to node c iff bit i of anc_c
            const int dfs = real ? a.t.dfs_of[rb + lane] : 0;
            const uint32_t anc = real ? a.t.anc[(rb + dfs) * W] : 0u;
            uint32_t desc = 0u;
#pragma unroll
            for (int c = 0; c < 32; ++c) desc |= ((__shfl_sync(0xffffffffu, anc, c) >> lane) & 1u) << c;
            meta[qb * 32 + lane] = desc;
            unsigned char *qs = sm + C::OFF_Q + qb * C::Q_BYTES;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch)
                *reinterpret_cast<uint4 *>(qs + (ch >> 3) * C::QREG + swz(lane, ch & 7)) = qv[ch];
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(qfull + 8 * qb);
            ++si;
        }
    } else {   // ---------------------------------------------------------------- softmax warps 2-9
        const int sw = warp - 2;          // vote slot
        const int wq = warp & 3;          // TMEM lane quarter
        const int hf = sw >> 2;           // node half: columns 16 hf .. 16 hf + 15
        const int r = wq * 32 + lane;     // key of the tile / head dim of O^T
        const uint32_t tl = tmem + ((uint32_t)(wq * 32) << 16) + 16 * hf;
        const float sc = a.scale_log2;
        int vpar = 0;
        SegIter it = it0;
        Seg sg;
        int t = 0, si = 0;
        float mref[16], lp[16];
        bool ok = true;
        // P^T word address pieces: the lane pair (r, r + 1) shares one 4-byte word per node
        const int kb = r & ~1, kk = kb & 63;
        const uint32_t p_off = (uint32_t)((kb >> 6) * C::PREG + (kk & 7) * 2);
        const int chunk = kk >> 3;
        const bool odd = lane & 1;
        while (ok && it.next(a, sg)) {
            const int qb = si & 1, ob = si & 1;
            const uint32_t *desc_s = meta + qb * 32;
            bool wok = mbar_wait_warp(qfull + 8 * qb, (uint32_t)(si >> 1) & 1u);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                mref[i] = -INFINITY;
                lp[i] = 0.f;
            }
            const int L = sg.P + sg.n;
            for (int j = sg.j0; j < sg.j1; ++j, ++t) {
                const int x = t & 1, vs = t % C::VS;
                wok = wok && mbar_wait_warp(sfull + 8 * x, (uint32_t)(t >> 1) & 1u);
                wok = wok && (t < 2 || mbar_wait_warp(pfree + 8 * x, (uint32_t)((t >> 1) - 1) & 1u));
                float s[16];
                {
                    float s1[16];
                    tc_fence_after();
                    tc_ld16(tl + C::S_COL + x * C::BUF, s);
                    tc_ld16(tl + C::S_COL + x * C::BUF + C::CHAIN, s1);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) s[i] += s1[i];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sfree + 8 * x);
                const int key = j * C::TKT + r;
                // keys visible to the half's 16 nodes (bit i: node 16 hf + i)
                uint32_t vis = 0xFFFFu;
                if ((j + 1) * C::TKT > sg.P)   // a tile with tree keys or keys past the end
                    vis = key >= L ? 0u : (key < sg.P ? 0xFFFFu : (desc_s[key - sg.P] >> (16 * hf)) & 0xFFFFu);
                // z = score * c - reference max (0 while a node has none): the exponent of p
                // and the test for a move; a node without a reference always moves
                bool over = false;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const bool none = mref[i] == -INFINITY;
                    s[i] = __fmaf_rn(s[i], sc, none ? 0.f : -mref[i]);
                    over |= ((vis >> i) & 1u) && (s[i] > C::THR || none);
                }
                const int v = group_vote(vote, vpar, sw, (wok ? 0 : 1) | (__any_sync(0xffffffffu, over) ? 2 : 0));
                if (v & 1) {
                    ok = false;
                    break;
                }
                if ((v & 2) || j == sg.j0) {
                    // ---- new reference max of the half's nodes (over the four lane quarters)
                    float mx[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        mx[i] = ((vis >> i) & 1u) ? s[i] + (mref[i] == -INFINITY ? 0.f : mref[i]) : -INFINITY;
                    red[(hf * 4 + wq) * 16 + (lane & 15)] = reduce16<true>(mx);
                    bool rok = true;
                    if (j > sg.j0) rok = mbar_wait_warp(pfree + 8 * ((t - 1) & 1), (uint32_t)((t - 1) >> 1) & 1u);
                    if (group_vote(vote, vpar, sw, rok ? 0 : 1) & 1) {
                        ok = false;
                        break;
                    }
                    float f[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float *rr = red + hf * 64 + i;
                        const float m = fmaxf(fmaxf(rr[0], rr[16]), fmaxf(rr[32], rr[48]));
                        const float mn = fmaxf(mref[i], m);
                        f[i] = mn == mref[i] ? 1.f : ex2(mref[i] - mn);
                        if (mn != mref[i]) s[i] += (mref[i] == -INFINITY ? 0.f : mref[i]) - mn;   // re-base z
                        mref[i] = mn;
                        lp[i] *= f[i];
                    }
                    if (j > sg.j0) {   // the previous tile's O^T MMA is complete: O^T *= f per node column
                        tc_fence_after();
#pragma unroll 1
                        for (int ch = 0; ch < 2; ++ch) {
                            float o[16];
                            tc_ld16(tl + C::O_COL + ob * C::BUF + ch * C::CHAIN, o);
                            tc_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) o[i] *= f[i];
                            tc_st16(tl + C::O_COL + ob * C::BUF + ch * C::CHAIN, o);
                        }
                        tc_wait_st();
                    }
                    named_sync_softmax();   // red[] is read by all before it is written again
                }
                // ---- P^T (bf16): word (key kb, key kb + 1) of each node row, K-major 128-byte swizzle
                float (&p)[16] = s;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    p[i] = ((vis >> i) & 1u) ? ex2(s[i]) : 0.f;
                    lp[i] += p[i];
                }
                const uint32_t pb = sm_base + C::OFF_P + x * C::P_BYTES + p_off;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    // the even lane writes node i, the odd lane node 8 + ((i + 4) & 7): different
                    // swizzle phases, so the warp's 32 words land in 32 banks
                    const int io = 8 + ((i + 4) & 7);
                    const float got = __shfl_xor_sync(0xffffffffu, odd ? p[i] : p[io], 1);
                    const int c = 16 * hf + (odd ? io : i);
                    __nv_bfloat162 w = odd ? __floats2bfloat162_rn(got, p[io]) : __floats2bfloat162_rn(p[i], got);
                    sts_u32(pb + c * 128 + (((chunk ^ (c & 7)) & 7) << 4), *reinterpret_cast<uint32_t *>(&w));
                }
                if ((j + 1) * C::TKT > L) {
                    // V rows past the pair's last key may hold anything: once the tile's V has
                    // landed, zero them (P is 0 there, and 0 * NaN would not be)
                    const bool vok = mbar_wait_warp(vfull + 8 * vs, (uint32_t)(t / C::VS) & 1u);
                    if (!vok && lane == 0) misc[1] = 1;
                    if (vok && key >= L) {
                        const uint32_t vrow = sm_base + C::OFF_V + vs * C::TILE_BYTES + hf * C::REGION + r * 128;
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) sts_zero16(vrow + ch * 16);
                    }
                }
                tc_fence_before();
                fence_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(pfull + 8 * x);
            }
            if (!ok) break;
            // ---- epilogue of the segment: row sums over the 128 keys, O^T, output or partial
            const bool eok = mbar_wait_warp(odone + 8 * ob, (uint32_t)(si >> 1) & 1u);
            red[(hf * 4 + wq) * 16 + (lane & 15)] = reduce16<false>(lp);
            if (group_vote(vote, vpar, sw, eok ? 0 : 1) & 1) {
                ok = false;
                break;
            }
            float o[16], l[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float *rr = red + hf * 64 + i;
                l[i] = (rr[0] + rr[16]) + (rr[32] + rr[48]);
            }
            {
                float o1[16];
                tc_fence_after();
                tc_ld16(tl + C::O_COL + ob * C::BUF, o);
                tc_ld16(tl + C::O_COL + ob * C::BUF + C::CHAIN, o1);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] += o1[i];
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(ofree + 8 * ob);
            const int n = sg.n, b = sg.b, h = sg.h;
            if (sg.whole) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int c = 16 * hf + i;
                    if (c < n) {
                        const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
                        a.out[(((size_t)b * n_max + c) * H + h) * D + r] = __float2bfloat16_rn(o[i] * inv);
                    }
                }
            } else {
                float *part = a.part_o + ((size_t)cta * 2 + sg.slot) * C::PART_FLOATS;
#pragma unroll
                for (int i = 0; i < 16; ++i) part[(16 * hf + i) * D + r] = o[i];
                if (wq == 0 && lane < 16) {
                    // thread `lane` publishes node 16 hf + lane's reference max and row sum
                    float mm = mref[0], ll = l[0];
#pragma unroll
                    for (int i = 1; i < 16; ++i)
                        if (lane == i) {
                            mm = mref[i];
                            ll = l[i];
                        }
                    part[C::NODES * D + 16 * hf + lane] = mm;
                    part[C::NODES * D + C::NODES + 16 * hf + lane] = ll;
                }
                named_sync_softmax();   // every thread's partial stores precede the release below
                // the pair's contributors: the CTAs c_first..c_last whose ranges are not
                // empty (with fewer tiles than CTAs, empty ranges sit between them)
                const int c_first = range_of(T, sg.gp, G), c_last = range_of(T, sg.gp + sg.tiles - 1, G);
                if (sw == 0 && lane == 0) {
                    int need = 0;
                    for (int cc = c_first; cc <= c_last; ++cc) need += range_start(T, cc + 1, G) > range_start(T, cc, G);
                    __threadfence();   // release: the CTA's partial (ordered by the barrier) before the count
                    const unsigned prev = atomicAdd(&a.counters[(size_t)b * H + h], 1u);
                    __threadfence();   // acquire: the other contributors' partials after the count
                    misc[2] = prev == (unsigned)(need - 1);
                }
                named_sync_softmax();
                if (misc[2]) {
                    // ---- last contributor: merge the partials of the contributing CTAs, eight
                    // nodes at a time; all loads of a contributor are issued before any is used
#pragma unroll 1
                    for (int i0 = 0; i0 < 16; i0 += 8) {
                        float M[8], Ls[8], acc[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            M[i] = -INFINITY;
                            Ls[i] = 0.f;
                            acc[i] = 0.f;
                        }
                        for (int cc = c_first; cc <= c_last; ++cc) {
                            if (range_start(T, cc + 1, G) == range_start(T, cc, G)) continue;   // empty range
                            const int slot = range_start(T, cc, G) >= sg.gp ? 0 : 1;
                            const float *pp = a.part_o + ((size_t)cc * 2 + slot) * C::PART_FLOATS;
                            float pm[8], pl[8], po[8];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const int c = 16 * hf + i0 + i;
                                pm[i] = __ldcg(pp + C::NODES * D + c);
                                pl[i] = __ldcg(pp + C::NODES * D + C::NODES + c);
                                po[i] = __ldcg(pp + c * D + r);
                            }
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float mn = fmaxf(M[i], pm[i]);
                                const float fo = M[i] == mn ? 1.f : ex2(M[i] - mn);    // 0 from -inf
                                const float fp = pm[i] == mn ? 1.f : ex2(pm[i] - mn);
                                Ls[i] = Ls[i] * fo + pl[i] * fp;
                                acc[i] = acc[i] * fo + po[i] * fp;
                                M[i] = mn;
                            }
                        }
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const int c = 16 * hf + i0 + i;
                            if (c < n) {
                                const float inv = Ls[i] > 0.f ? 1.f / Ls[i] : 0.f;
                                a.out[(((size_t)b * n_max + c) * H + h) * D + r] = __float2bfloat16_rn(acc[i] * inv);
                            }
                        }
                    }
                    if (sw == 0 && lane == 0) a.counters[(size_t)b * H + h] = 0u;   // leave the workspace zeroed
                }
                named_sync_softmax();   // misc[2] is read by all before the next segment writes it
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(qfree + 8 * qb);
            ++si;
        }
        if (!ok && lane == 0) misc[1] = 1;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS) : "memory");
    if (misc[1] && tid == 0) flag(a.status, TS_STATUS_TIMEOUT);
}

}  // namespace

size_t attn_kt_ws_bytes(int B, int H) {
    const size_t counters = ((size_t)B * H * 4 + 255) / 256 * 256;
    return counters + (size_t)num_sms() * 2 * KtCfg::PART_FLOATS * sizeof(float);
}

cudaError_t launch_attn_kt(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *prefix_len, const ts_tree &t, int H, int L_max, float scale, void *ws,
                           uint32_t *status, cudaStream_t s, const char **why) {
    CUtensorMap mk, mv;
    const long long rows = (long long)t.B * H * L_max;
    if (rows + KtCfg::TKT >= (1LL << 31)) {
        *why = "KV cache of 2^31 rows or more";
        return cudaErrorInvalidValue;
    }
    if (!make_map(&mk, k_cache, KtCfg::D, rows, KtCfg::TKT) || !make_map(&mv, v_cache, KtCfg::D, rows, KtCfg::TKT)) {
        *why = "cuTensorMapEncodeTiled failed for the KV cache";
        return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(k_attn_kt, cudaFuncAttributeMaxDynamicSharedMemorySize, KtCfg::SMEM);
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
    a.n_pad = KtCfg::NODES;
    const size_t counters = ((size_t)t.B * H * 4 + 255) / 256 * 256;
    a.counters = (unsigned *)ws;
    a.part_o = (float *)((char *)ws + counters);
    a.part_ml = nullptr;
    a.status = status;
    // one CTA per SM; TREESPEC_ATTN_CTAS=k uses k CTAs (at most one per SM),
    // which moves the range boundaries that cut pairs into partials
    int G = num_sms();
    if (const char *e = getenv("TREESPEC_ATTN_CTAS"))
        if (*e && atoi(e) >= 1 && atoi(e) < G) G = atoi(e);
    return launch(k_attn_kt, dim3(G), dim3(KtCfg::THREADS), KtCfg::SMEM, s, mk, mv, a);
}

}  // namespace ts
