// Backward kernels for tree/DAG-packed paged attention (sm_103a, tcgen05 + TMA).
//
// With P = softmax over vis(r) recomputed from the saved logsumexp and delta = <dO, O>:
//   dS = P * (dO V^T - delta),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO
// (the adjoint of the forward in Octopus arXiv 2611.06956 Section 3.3 Eq. 4; gradients of a
// shared prefix row or a mounted row are summed over all of its readers -- Octopus Section 3.4
// "differentiable mount edges", HARTS arXiv 2608.28158 Section 3.4 gather backward).
//
// Four launches:
//   delta_kernel   per (query block, KV head, 128-lane query tile): each lane's -lse * log2(e)
//                  and -delta = -<dO, O>, one 1 KB table per tile              (HBM-bound)
//   dq_kernel      query-major: one CTA per (query block, KV head, 128-lane query tile);
//                  walks the block's packed key tiles like the forward
//   dkdv_kernel    key-major: one CTA per (key-tile chunk, KV head); walks the query blocks
//                  that read the tile (the plan's transpose), both 128-lane query tiles each;
//                  dK and dV accumulate in TMEM and are written once -- to the pool, or to a
//                  partial slot when the tile's readers were split into several chunks
//   reduce_kernel  sums each split tile's partial slots in a fixed order (deterministic)
#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------------------------ delta
// One CTA per (query block, KV head, 128-lane query tile); thread m handles query lane m,
// i.e. row (head hl, row rl) with 128 t + m = hl R + rl.  It writes the tile's 1 KB unit
// table: [m] = -lse * log2(e) (-inf for padding lanes, so that P = 0 there) and
// [128 + m] = -delta = -<dO, O> of that row, negated so that both backward kernels add
// them (P = exp2(S scale log2e + [m]), dS = P (dP + [128 + m])).  The dK/dV loader copies
// the halves with one bulk copy each.
template <int D>
__global__ void __launch_bounds__(128) delta_kernel(const BwdParams p) {
    const int t = blockIdx.x & 1, g = (blockIdx.x >> 1) % p.Hkv, qb = (blockIdx.x >> 1) / p.Hkv;
    const int m = threadIdx.x, m_flat = 128 * t + m;
    const int hl = m_flat / p.R, rl = m_flat % p.R, h = g * p.G + hl;
    const int q_row0 = __ldg(p.blocks + 4 * qb), n_rows = __ldg(p.blocks + 4 * qb + 1);
    const bool valid = rl < n_rows && debug_in_range(q_row0 + rl, 0, p.N, p.status);
    float nlse2 = -INFINITY, acc = 0.f;
    if (valid) {
        const int r = q_row0 + rl;
        const size_t base = (static_cast<size_t>(r) * p.Hq + h) * D;
        const uint4 *a = reinterpret_cast<const uint4 *>(p.d_o + base);
        const uint4 *b = reinterpret_cast<const uint4 *>(p.o + base);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) {
            const uint4 x = __ldg(a + i), y = __ldg(b + i);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 fx = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xs[k]));
                const float2 fy = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&ys[k]));
                acc = fmaf(fx.x, fy.x, acc);
                acc = fmaf(fx.y, fy.y, acc);
            }
        }
        nlse2 = -__ldg(p.lse + static_cast<size_t>(h) * p.N + r) * kLog2e;
    }
    float *tab = p.utab + (static_cast<size_t>(g * p.n_blocks + qb) * 2 + t) * 256;
    tab[m] = nlse2;
    tab[128 + m] = -acc;
}

// One 128-lane query tile t of a block: rows (head, row) flattened as m = hl * R + rl, i.e.
// 128 / QB consecutive heads x QB rows (QB = min(R, 128)), loaded as one box of the rank-4
// view {64 elements, rows, heads, 64-element chunks} of a [N, Hq, D] tensor.  The box lands
// chunk-major ([chunk][head][row][128 B], chunk stride 16 KB): the K-major 128-byte-swizzled
// layout the MMA descriptors read.  One 32 KB box instead of 4 boxes of 8 KB: the TMA unit
// moves large boxes from L2 about three times faster than 8 KB ones.
__device__ __forceinline__ void load_q_tile(uint32_t dst, const CUtensorMap *tm, int t, int g, int G, int R,
                                            int q_row0, uint32_t bar) {
    const int m0 = 128 * t, hl = m0 / R, r0 = m0 % R;
    tma_load_4d(dst, tm, 0, q_row0 + r0, g * G + hl, 0, bar);
}

template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t sA, uint32_t sB, uint32_t idesc) {
    // D[128 x 128] = A[128 x D] * B[128 x D]^T, both K-major 128-byte-swizzled tiles
    // descriptors are built once; advancing along K only moves the 14-bit start-address field
    const uint64_t a0 = sdesc_sw128(sA, 16, 1024), b0 = sdesc_sw128(sB, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t koff = static_cast<uint64_t>(((kk >> 2) * (kTileRows * 128) + (kk & 3) * 32) >> 4);
        mma_ss(d_tmem, a0 + koff, b0 + koff, idesc, kk > 0 ? 1u : 0u);
    }
}

constexpr int kDqThreads = 384;    // dQ: warps 0-3 / 4-7 elementwise groups, 8 loads, 9 / 10 / 11 MMA (S, dP, dQ)
constexpr int kDkvThreads = 352;   // dK/dV: warps 9 and 10 each issue one of the two MMA chains
constexpr int kQStages = 3;        // dK/dV: Q stages (a Q tile is last read by dK)
constexpr int kDoStages = 2;       // dK/dV: dO stages (a dO tile is last read by dV)
constexpr int kKStages = 3;        // dQ: K stages (K is held until the dQ MMAs)
constexpr int kVStages = 3;        // dQ: V stages (V is released after the dP MMAs)

template <int D>
__device__ __forceinline__ void issue_tk(uint32_t d_tmem, uint32_t a_tmem, uint32_t sB, uint32_t idesc) {
    // D[128 x N] = A[128 x D] (bf16 rows resident in TMEM) * B[N x D]^T (K-major smem tile):
    // only B is read from shared memory
    const uint64_t b0 = sdesc_sw128(sB, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
        mma_ts(d_tmem, a_tmem + kk * 8,
               b0 + static_cast<uint64_t>(((kk >> 2) * (kTileRows * 128) + (kk & 3) * 32) >> 4), idesc,
               kk > 0 ? 1u : 0u);
}

// D[128 x N] (+)= A[128 x 128] * B[128 x N], A in bf16 TMEM columns written by the two
// elementwise groups (group w's 64 K-columns packed into columns [64w, 64w + 32) of a_base),
// B the rows of an MN-major smem tile (N = D contiguous, LBO = one 64-column half).
__device__ __forceinline__ void issue_acc_split(uint32_t d_tmem, uint32_t a_base, uint32_t sB, uint32_t idesc,
                                                bool acc) {
    const uint64_t b0 = sdesc_sw128(sB, kTileRows * 128, 1024);
#pragma unroll
    for (int kk = 0; kk < kTileRows / 16; ++kk)
        mma_ts(d_tmem, a_base + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
               b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc, (acc || kk > 0) ? 1u : 0u);
}

// Half h of issue_acc_split: the K-columns [64w + 32h, 64w + 32h + 32) of both groups w.
__device__ __forceinline__ void issue_acc_half(uint32_t d_tmem, uint32_t a_base, uint32_t sB, uint32_t idesc, int h,
                                               bool acc) {
    const uint64_t b0 = sdesc_sw128(sB, kTileRows * 128, 1024);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int kk = 4 * (i >> 1) + 2 * h + (i & 1);
        mma_ts(d_tmem, a_base + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8),
               b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc, (acc || i > 0) ? 1u : 0u);
    }
}

// D[128 x N] (+)= A[128 x 128] * B[128 x N], A in bf16 TMEM columns [a_base, a_base + 64)
// (K-column k in column a_base + k / 2), B the rows of an MN-major smem tile.
__device__ __forceinline__ void issue_acc(uint32_t d_tmem, uint32_t a_base, uint32_t sB, uint32_t idesc, bool acc) {
    const uint64_t b0 = sdesc_sw128(sB, kTileRows * 128, 1024);
#pragma unroll
    for (int kk = 0; kk < kTileRows / 16; ++kk)
        mma_ts(d_tmem, a_base + kk * 8, b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc,
               (acc || kk > 0) ? 1u : 0u);
}

// Copy the 64-element chunks c = w, w + 2, ... of one bf16 row of D elements from global
// memory into this thread's TMEM lane (chunk c at column `taddr + 32 c`, two elements per
// 32-bit column: the layout tcgen05.mma reads A from).  The two elementwise groups (w = 0, 1)
// each copy half of the row.
template <int D>
__device__ __forceinline__ void row_to_tmem(uint32_t taddr, const __nv_bfloat16 *row, bool valid, int w) {
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
        if ((c & 1) != w) continue;
        uint32_t v[32];
        if (valid) {
            const uint4 *src = reinterpret_cast<const uint4 *>(row + 64 * c);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 x = __ldg(src + i);
                v[4 * i] = x.x; v[4 * i + 1] = x.y; v[4 * i + 2] = x.z; v[4 * i + 3] = x.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0u;
        }
        tmem_st32(taddr + 32 * c, v);
    }
}

// ------------------------------------------------------------------------------ dQ
template <int D>
struct DqLayout {
    static constexpr int kTile = 128 * D * 2;
    static constexpr int k_off = 0;
    static constexpr int v_off = k_off + kKStages * kTile;
    static constexpr int do_off = v_off + kVStages * kTile;   // the CTA's dO tile (read by every dP)
    static constexpr int bar_off = do_off + kTile;
    static constexpr int n_bars = 2 + 2 * kKStages + 2 * kVStages + 7;
    static constexpr int misc_off = bar_off + n_bars * 8;
    static constexpr int bytes = misc_off + 16 + 1024;
};

// One CTA = one 128-lane query tile (t) of one query block x one KV head.  The tile's Q rows
// stay in TMEM and its dO tile in shared memory for the CTA's lifetime.  Per key-tile entry
// j, with full-width (N = 128) MMAs:
//   MMA:  S_j = Q K_j^T (TS), dP_j = dO V_j^T (SS)                        (into TMEM)
//   EW :  read S_j (frees it: S_{j+1} starts), P_j = exp2(S_j scale log2e - lse) masked
//   EW :  read dP_j (frees it: dP_{j+1} starts), dS_j = P_j (dP_j - delta) as bf16 into
//         the dS columns, once dQ_{j-1} has read them                       -> ds_full
//   MMA:  dQ += dS_j K_j
// dS has TMEM columns of its own, so no MMA of entry j + 1 waits for dQ_j: while the
// elementwise groups work on entry j the tensor core runs S_{j+1}, dP_{j+1} and dQ_{j-1}.
// Three threads issue the MMAs -- warp 9: S, warp 10: dP, warp 11: dQ -- because issuing a
// batch blocks the thread while the tensor core's queue is full, and an issuer that also
// waits for dS_j would start S_{j+2} only after dQ_j (on the mount-heavy workload: one issuer
// 27.3 ms; S and dQ on one thread, dP on another, 23.0 ms; three issuers 21.65 ms, dQ
// bit-identical).  K_j is freed by the dQ issuer's commit: S_j, its other reader, finished
// before the groups could form dS_j.
// The two groups split each entry's 128 key columns (64 each); P stays in their registers
// between the phases.
template <int D>
__global__ void __launch_bounds__(kDqThreads, 1)
dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_k64,
          const __grid_constant__ CUtensorMap tm_v64, const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
    using L = DqLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int unit = blockIdx.x >> 1, t = blockIdx.x & 1;
    const int qb = __ldg(p.order + unit / p.Hkv), g = unit % p.Hkv;
    const int q_row0 = __ldg(p.blocks + 4 * qb), n_rows = __ldg(p.blocks + 4 * qb + 1);
    const int e0 = __ldg(p.fblk + 2 * qb), E = __ldg(p.fblk + 2 * qb + 1) - e0;
    const int4 *tiles = reinterpret_cast<const int4 *>(p.ftiles) + 2 * e0;   // two int4 per tile

    const uint32_t sK = sbase + L::k_off, sV = sbase + L::v_off, sDO = sbase + L::do_off;
    auto bar = [&](int i) { return sbase + L::bar_off + 8u * i; };
    const uint32_t q_ready = bar(0), do_full = bar(1);
    auto k_full = [&](int s) { return bar(2 + s); };
    auto k_empty = [&](int s) { return bar(2 + kKStages + s); };
    auto v_full = [&](int s) { return bar(2 + 2 * kKStages + s); };
    auto v_empty = [&](int s) { return bar(2 + 2 * kKStages + kVStages + s); };
    constexpr int kb = 2 + 2 * kKStages + 2 * kVStages;
    const uint32_t s_full = bar(kb), s_free = bar(kb + 1), dp_full = bar(kb + 2), dp_free = bar(kb + 3);
    const uint32_t ds_full = bar(kb + 4), ds_free = bar(kb + 5), o_full = bar(kb + 6);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc_off);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L::misc_off + 4);

    if (threadIdx.x == 0) {
        mbar_init(q_ready, 8);                // one arrival per elementwise warp
        mbar_init(do_full, 1);
        for (int s = 0; s < kKStages; ++s) { mbar_init(k_full(s), 1); mbar_init(k_empty(s), 1); }
        for (int s = 0; s < kVStages; ++s) { mbar_init(v_full(s), 1); mbar_init(v_empty(s), 1); }
        mbar_init(s_full, 1);
        mbar_init(s_free, 8);
        mbar_init(dp_full, 1);
        mbar_init(dp_free, 8);
        mbar_init(ds_full, 8);
        mbar_init(ds_free, 1);
        mbar_init(o_full, 3);                 // one commit from each MMA issuer
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns: Q [0, D/2) as bf16 pairs, dS [64, 128) as bf16 pairs (key k in column
    // 64 + k/2, so group w writes [64 + 32w, 96 + 32w)), dQ [128, 128 + D), S [256, 384),
    // dP [384, 512).
    constexpr uint32_t cQ = 0, cDS = 64, cDQ = 128, cS = 256, cDP = 384;

    if (warp == 8) {
        bool do_issued = false;
        if (lane == 0) {
            tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v); tma_prefetch_desc(&tm_do);
            tma_prefetch_desc(&tm_k64); tma_prefetch_desc(&tm_v64);
            if (E > 0) {
                mbar_arrive_expect_tx(do_full, L::kTile);
                load_q_tile(sDO, &tm_do, t, g, p.G, p.R, q_row0, do_full);
                do_issued = true;
            }
        }
        PackFeed f;
        const int oob = p.num_pages * p.page_size;
        int k_issued = 0, v_issued = 0;
        for (int j = 0; j < E; ++j) {
            if ((j & 31) == 0)
                pack_feed_fill(f, j, E, tiles, p.page_table, p.n_logical_pages, p.page_size, oob, lane, p.status);
            int y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = __shfl_sync(0xffffffffu, f.y[i], j & 31);
            const int fl = __shfl_sync(0xffffffffu, f.b.z, j & 31);
            const int ks = j % kKStages, vs = j % kVStages;
            bool ok = true;
            if (lane == 0 && j >= kKStages) ok = mbar_wait(k_empty(ks), ((j / kKStages) - 1) & 1, abort, p.status);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(k_full(ks), L::kTile);
                tma_packed_tile(sK + ks * L::kTile, &tm_k, &tm_k64, y, fl, p.page_size, g, D, k_full(ks));
            }
            k_issued = j + 1;
            if (lane == 0 && j >= kVStages) ok = mbar_wait(v_empty(vs), ((j / kVStages) - 1) & 1, abort, p.status);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(v_full(vs), L::kTile);
                tma_packed_tile(sV + vs * L::kTile, &tm_v, &tm_v64, y, fl, p.page_size, g, D, v_full(vs));
            }
            v_issued = j + 1;
        }
        if (lane == 0) {
            // wait for this warp's copies still in flight before the CTA can exit
            if (do_issued) mbar_wait(do_full, 0, nullptr, p.status);
            for (int d = (k_issued > kKStages ? k_issued - kKStages : 0); d < k_issued; ++d)
                mbar_wait(k_full(d % kKStages), (d / kKStages) & 1, nullptr, p.status);
            for (int d = (v_issued > kVStages ? v_issued - kVStages : 0); d < v_issued; ++d)
                mbar_wait(v_full(d % kVStages), (d / kVStages) & 1, nullptr, p.status);
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------------- MMA: S
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
            bool ok = E > 0 && mbar_wait(q_ready, 0, abort, p.status) && mbar_wait(k_full(0), 0, abort, p.status);
            if (ok) {
                tc_fence_after();
                issue_tk<D>(tmem + cS, tmem + cQ, sK, idesc_s);        // S_0 = Q K_0^T
                mma_commit(s_full);
            }
            for (int j = 0; ok && j + 1 < E; ++j) {
                const int ks1 = (j + 1) % kKStages;
                // S_{j+1} as soon as both groups have read S_j
                if (!(ok = mbar_wait(s_free, j & 1, abort, p.status) &&
                           mbar_wait(k_full(ks1), ((j + 1) / kKStages) & 1, abort, p.status)))
                    break;
                tc_fence_after();
                issue_tk<D>(tmem + cS, tmem + cQ, sK + ks1 * L::kTile, idesc_s);
                mma_commit(s_full);
            }
            mma_commit(o_full);
            mbar_wait(o_full, 0, nullptr, p.status);
        }
    } else if (warp == 11) {
        // ---------------------------------------------------------------- MMA: dQ
        if (lane == 0) {
            constexpr uint32_t idesc_o = idesc_bf16(128, D, 0, 1);
            bool ok = true;
            for (int j = 0; ok && j < E; ++j) {
                const int ks = j % kKStages;
                if (!(ok = mbar_wait(ds_full, j & 1, abort, p.status))) break;
                tc_fence_after();
                // S_j, the other reader of K_j, finished before the groups could form dS_j
                issue_acc(tmem + cDQ, tmem + cDS, sK + ks * L::kTile, idesc_o, j > 0);   // dQ += dS_j K_j
                mma_commit(k_empty(ks));
                mma_commit(ds_free);
            }
            mma_commit(o_full);
            mbar_wait(o_full, 0, nullptr, p.status);
        }
    } else if (warp == 10) {
        // ---------------------------------------------------------------- MMA: dP
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
            bool ok = E > 0 && mbar_wait(do_full, 0, abort, p.status) && mbar_wait(v_full(0), 0, abort, p.status);
            if (ok) {
                tc_fence_after();
                issue_qk<D>(tmem + cDP, sDO, sV, idesc_s);             // dP_0 = dO V_0^T
                mma_commit(dp_full);
                mma_commit(v_empty(0));
            }
            for (int j = 0; ok && j + 1 < E; ++j) {
                // dP_{j+1} as soon as both groups have read dP_j
                const int vs1 = (j + 1) % kVStages;
                if (!(ok = mbar_wait(dp_free, j & 1, abort, p.status) &&
                           mbar_wait(v_full(vs1), ((j + 1) / kVStages) & 1, abort, p.status)))
                    break;
                tc_fence_after();
                issue_qk<D>(tmem + cDP, sDO, sV + vs1 * L::kTile, idesc_s);
                mma_commit(dp_full);
                mma_commit(v_empty(vs1));
            }
            mma_commit(o_full);
            mbar_wait(o_full, 0, nullptr, p.status);
        }
    } else {
        // ---------------------------------------------------------------- elementwise (warps 0-7)
        const int w = warp >> 2, q4 = warp & 3;
        const int m_flat = 128 * t + 32 * q4 + lane;
        const int hl = m_flat / p.R, rl = m_flat % p.R;
        const int r_abs = q_row0 + rl, h = g * p.G + hl;
        const bool valid = rl < n_rows && debug_in_range(r_abs, 0, p.N, p.status);
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        // the two groups put this lane's Q row into TMEM, half each
        row_to_tmem<D>(tmem + lane_off + cQ, p.q + (static_cast<size_t>(r_abs) * p.Hq + h) * D, valid, w);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_ready);
        const float sl2 = p.scale_log2;
        const float *tab = p.utab + (static_cast<size_t>(g * p.n_blocks + qb) * 2 + t) * 256;
        const float nlse2 = tab[32 * q4 + lane];      // -lse * log2(e)
        const float ndelta = tab[128 + 32 * q4 + lane];  // -delta
        bool ok = true;
        WarpPackRecords recs;
        for (int j = 0; j < E; ++j) {
            int4 ra, rb;
            recs.get(tiles, j, E, lane, ra, rb);
            // ---------------- phase 1: P_j from S_j
            ok = __all_sync(0xffffffffu, mbar_wait(s_full, j & 1, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            float pf[64];
            {
                uint32_t sv[2][32];
                tmem_ld32(tmem + lane_off + cS + 64 * w, sv[0]);
                tmem_ld32(tmem + lane_off + cS + 64 * w + 32, sv[1]);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free);
                const uint64_t sc2 = f2_pack(sl2, sl2), nl2 = f2_pack(nlse2, nlse2);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x0, x1;
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[i >> 4][(2 * i) & 31]), __uint_as_float(sv[i >> 4][(2 * i + 1) & 31])),
                                     sc2, nl2), x0, x1);
                    pf[2 * i] = ex2(x0);
                    pf[2 * i + 1] = ex2(x1);
                }
                if (rb.z & kPackMask) {              // this group's slots 2w, 2w + 1: mask key columns
#pragma unroll
                    for (int sl = 0; sl < 2; ++sl) {
                        int lo, hi;
                        pack_slot_range(ra, rb, 2 * w + sl, r_abs, lo, hi);
                        if (lo > 0 || hi < kPieceRows) {
#pragma unroll
                            for (int c = 0; c < kPieceRows; ++c)
                                pf[kPieceRows * sl + c] = (c >= lo && c < hi) ? pf[kPieceRows * sl + c] : 0.f;
                        }
                    }
                }
            }
            // ---------------- phase 2: dS_j
            ok = __all_sync(0xffffffffu, mbar_wait(dp_full, j & 1, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            {
                uint32_t dpv[2][32];
                tmem_ld32(tmem + lane_off + cDP + 64 * w, dpv[0]);
                tmem_ld32(tmem + lane_off + cDP + 64 * w + 32, dpv[1]);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dp_free);
                uint32_t ds[2][16];
                const uint64_t nd2 = f2_pack(ndelta, ndelta);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float r0, r1;
                    f2_unpack(f2_mul(f2_pack(pf[2 * i], pf[2 * i + 1]),
                                     f2_add(f2_pack(__uint_as_float(dpv[i >> 4][(2 * i) & 31]), __uint_as_float(dpv[i >> 4][(2 * i + 1) & 31])),
                                            nd2)), r0, r1);
                    ds[i >> 4][i & 15] = pack_bf16(r0, r1);
                }
                // dQ_{j-1} must have read the dS columns before they are overwritten
                if (j > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait(ds_free, (j - 1) & 1, abort, p.status));
                    if (!ok) break;
                    tc_fence_after();
                }
                tmem_st16(tmem + lane_off + cDS + 32 * w, ds[0]);
                tmem_st16(tmem + lane_off + cDS + 32 * w + 16, ds[1]);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ds_full);
            }
        }
        ok = __all_sync(0xffffffffu, ok && mbar_wait(o_full, 0, abort, p.status));
        if (ok) {
            tc_fence_after();
            // each group writes half of the row's columns
            float *dst = p.dq + (static_cast<size_t>(r_abs) * p.Hq + h) * D + w * (D / 2);
#pragma unroll
            for (int c = 0; c < D / 64; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_off + cDQ + w * (D / 2) + 32 * c, v);
                tmem_wait_ld();
                if (valid) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d4[i] = make_float4(__uint_as_float(v[4 * i]) * p.scale, __uint_as_float(v[4 * i + 1]) * p.scale,
                                            __uint_as_float(v[4 * i + 2]) * p.scale, __uint_as_float(v[4 * i + 3]) * p.scale);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------------ dK, dV
template <int D>
struct DkvLayout {
    static constexpr int kTile = 128 * D * 2;
    static constexpr int k_off = 0;
    static constexpr int v_off = k_off + kTile;
    static constexpr int q_off = v_off + kTile;                    // kQStages Q tiles
    static constexpr int do_off = q_off + kQStages * kTile;        // kDoStages dO tiles
    // the unit's lse*log2(e) travels with its dO tile (read by the first elementwise phase, which
    // ends before dV can release the dO slot), its delta with its Q tile (read by the second
    // phase, which ends before dK releases the Q slot)
    static constexpr int lse_off = do_off + kDoStages * kTile;     // per dO stage: 128 floats
    static constexpr int dl_off = lse_off + kDoStages * 512;       // per Q stage: 128 floats
    static constexpr int bar_off = dl_off + kQStages * 512;
    static constexpr int n_bars = 1 + 2 * kQStages + 2 * kDoStages + 8;
    static constexpr int misc_off = bar_off + n_bars * 8;
    static constexpr int bytes = misc_off + 16;                     // the base is 1024-aligned
};

// One CTA = one key tile x one KV head x one chunk of the tile's readers.  K and V stay in
// shared memory.  Every (reader block, 128-lane query tile) is one unit, processed in two
// phases so that the tensor core always has work while the elementwise warps run:
//   MMA:  S^T = K Q^T, dP^T = V dO^T                       (128 x 128 each, into TMEM)
//   EW :  P^T = exp2(S^T log2e scale - lse) (masked), bf16 copy into TMEM, in two halves of
//         each group's columns                                     -> p_full, p_half1
//   MMA:  dV += P^T dO (the first halves' K-steps while EW exponentiates the second halves),
//         then the next unit's S^T                                 (while EW computes dS)
//   EW :  dS^T = P^T (dP^T - delta), bf16 copy into TMEM                        -> ds_full
//   MMA:  dK += dS^T Q,  then the next unit's dP^T            (while EW computes the next P)
// The two elementwise warpgroups split each unit's 128 query columns (64 each); P stays in
// their registers between the phases.  dV and dK accumulate in TMEM for the whole chunk and
// each key row of the tile is written once at the end.
// Q and dO have separate rings: a unit's dO is last read by dV (early in its period), its Q
// by dK (late), so three Q slots and two dO slots give both about two periods between the
// release of a slot and the first read of the tile loaded into it -- the load latency of a
// 32 KB tile on these access patterns is about 3,000 cycles.
// The two MMA chains have their own issuing threads -- warp 9: S^T(u+1) after dV(u) (both on
// the S^T columns), warp 10: dP^T(u+1) after dK(u) (the dP^T columns) -- because issuing a
// batch of MMAs blocks the thread until the tensor core has room, and one thread would only
// see the other chain's barrier after its own batch.  The tensor core runs MMAs in the order
// they reach it, so warp 10 issues dK(u) only once warp 9 has issued S^T(u + 1): the next
// phase-1 elementwise work waits for S^T(u + 1), not for dK(u) and dP^T(u + 1), which are
// needed only a phase later (a clock-stamped trace of one CTA on the mount-heavy workload:
// 3,510 cycles per unit without the ordering, 3,110 with it).  A Q or dO slot is read by MMAs
// of both chains, so its "empty" barrier takes one commit from each.
template <int D>
__global__ void __launch_bounds__(kDkvThreads, 1)
dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
    using L = DkvLayout<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    const uint32_t sbase = smem_u32(smem);
    if (sbase & 1023u) {                      // the layout has no alignment slack left
        if (threadIdx.x == 0) atomicOr(p.status, kStatusMisaligned);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int ci = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;
    const int tile = __ldg(p.chunks + 4 * ci), a0 = __ldg(p.chunks + 4 * ci + 1);
    const int n_ent = __ldg(p.chunks + 4 * ci + 2) - a0, slot = __ldg(p.chunks + 4 * ci + 3);
    const int4 *tinfo = reinterpret_cast<const int4 *>(p.t_info) + a0;   // block<<2|flags, first row, lo, hi
    const int U = 2 * n_ent;   // (entry, query tile) units

    const uint32_t sK = sbase + L::k_off, sV = sbase + L::v_off;
    auto sQ = [&](int s) { return sbase + L::q_off + s * L::kTile; };
    auto sDO = [&](int s) { return sbase + L::do_off + s * L::kTile; };
    float *lse_s = reinterpret_cast<float *>(smem + L::lse_off);      // [dO stage][128]
    float *dl_s = reinterpret_cast<float *>(smem + L::dl_off);        // [Q stage][128]
    auto bar = [&](int i) { return sbase + L::bar_off + 8u * i; };
    const uint32_t kv_full = bar(0);
    auto q_full = [&](int s) { return bar(1 + s); };
    auto q_empty = [&](int s) { return bar(1 + kQStages + s); };
    auto do_full = [&](int s) { return bar(1 + 2 * kQStages + s); };
    auto do_empty = [&](int s) { return bar(1 + 2 * kQStages + kDoStages + s); };
    constexpr int kb = 1 + 2 * kQStages + 2 * kDoStages;
    const uint32_t s_full = bar(kb), dp_full = bar(kb + 1), p_full = bar(kb + 2), ds_full = bar(kb + 3);
    const uint32_t o_full = bar(kb + 4);
    // S^T(u + 1) has been issued (two barriers, alternating by unit): the dK issuer waits for it
    auto s_issued = [&](int u) { return bar(kb + 5 + (u & 1)); };
    const uint32_t p_half1 = bar(kb + 7);   // second half of each group's P^T columns
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc_off);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L::misc_off + 4);

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        mbar_init(s_issued(0), 1);
        mbar_init(s_issued(1), 1);
        for (int s = 0; s < kQStages; ++s) { mbar_init(q_full(s), 1); mbar_init(q_empty(s), 2); }
        for (int s = 0; s < kDoStages; ++s) { mbar_init(do_full(s), 1); mbar_init(do_empty(s), 2); }
        mbar_init(s_full, 1);
        mbar_init(dp_full, 1);
        mbar_init(p_full, 8);                 // one arrival per elementwise warp
        mbar_init(p_half1, 8);
        mbar_init(ds_full, 8);
        mbar_init(o_full, 2);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM columns: S^T [0,128) | dP^T [128,256) | dV [256, 256+D) | dK [384, 384+D).
    // Group w's bf16 P^T (query columns [64w, 64w+64)) goes to S^T columns [64w, 64w+32),
    // its dS^T to dP^T columns [64w, 64w+32): inside its own half, so no group overwrites
    // scores the other group has not read yet.
    constexpr uint32_t cS = 0, cDP = 128, cDV = 256, cDK = 384;

    if (warp == 8) {
        // ---------------------------------------------------------------- loads (whole warp)
        const int ppt = kTileRows / p.page_size;
        int ky[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            ky[i] = i < ppt ? __ldg(p.tile_rows + tile * ppt + i) : 0;
            // (TA_DEBUG) a page of the tile past the strip's end has the row one past the pool,
            // which TMA zero-fills; any other row outside the pool is flagged and replaced by it
            const long long past = static_cast<long long>(p.num_pages) * p.page_size;
            if (!debug_in_range(ky[i], 0, past + 1, p.status)) ky[i] = static_cast<int>(past);
        }
        if (lane == 0) {
            tma_prefetch_desc(&tm_q); tma_prefetch_desc(&tm_do);
            tma_prefetch_desc(&tm_k); tma_prefetch_desc(&tm_v);
            mbar_arrive_expect_tx(kv_full, 2 * L::kTile);
            tma_kv_tile(sK, &tm_k, ky, ppt, p.page_size, g, D, kv_full);
            tma_kv_tile(sV, &tm_v, ky, ppt, p.page_size, g, D, kv_full);
        }
        int4 mine = make_int4(0, 0, 0, 0);   // lane i holds the reader info of entry (base + i)
        int q_issued = 0, do_issued = 0;
        for (int u = 0; u < U; ++u) {
            const int qs = u % kQStages, ds = u % kDoStages, t = u & 1, e = u >> 1;
            if ((u & 63) == 0 && e + lane < n_ent) mine = __ldg(tinfo + e + lane);
            const int qb = __shfl_sync(0xffffffffu, mine.x, e & 31) >> 2;
            const int q_row0 = __shfl_sync(0xffffffffu, mine.y, e & 31);
            bool ok = true;
            // Q first: S^T(u) is the first MMA to read the unit, dP^T(u) comes after it; the slots
            // free in the same order (dK(u-3) completes before dV(u-2))
            if (lane == 0 && u >= kQStages) ok = mbar_wait(q_empty(qs), ((u / kQStages) - 1) & 1, abort, p.status);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            const float *utab = p.utab + (static_cast<size_t>(g * p.n_blocks + qb) * 2 + t) * 256;
            if (lane == 0) {
                mbar_arrive_expect_tx(q_full(qs), L::kTile + 512);
                bulk_load(smem_u32(dl_s + qs * 128), utab + 128, 512, q_full(qs));
                load_q_tile(sQ(qs), &tm_q, t, g, p.G, p.R, q_row0, q_full(qs));
            }
            q_issued = u + 1;
            if (lane == 0 && u >= kDoStages) ok = mbar_wait(do_empty(ds), ((u / kDoStages) - 1) & 1, abort, p.status);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(do_full(ds), L::kTile + 512);
                bulk_load(smem_u32(lse_s + ds * 128), utab, 512, do_full(ds));
                load_q_tile(sDO(ds), &tm_do, t, g, p.G, p.R, q_row0, do_full(ds));
            }
            do_issued = u + 1;
        }
        if (lane == 0) {
            for (int d = (do_issued > kDoStages ? do_issued - kDoStages : 0); d < do_issued; ++d)
                mbar_wait(do_full(d % kDoStages), (d / kDoStages) & 1, nullptr, p.status);
            for (int d = (q_issued > kQStages ? q_issued - kQStages : 0); d < q_issued; ++d)
                mbar_wait(q_full(d % kQStages), (d / kQStages) & 1, nullptr, p.status);
            mbar_wait(kv_full, 0, nullptr, p.status);
        }
    } else if (warp == 9) {
        // ---------------------------------------------------------------- MMA: S^T, dV chain
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16(128, D, 0, 1);
            bool ok = U > 0 && mbar_wait(kv_full, 0, abort, p.status) && mbar_wait(q_full(0), 0, abort, p.status);
            if (ok) {
                tc_fence_after();
                issue_qk<D>(tmem + cS, sK, sQ(0), idesc_s);        // S^T = K Q^T
                mma_commit(s_full);
                mma_commit(q_empty(0));                            // this chain's read of Q(0)
            }
            for (int u = 0; ok && u < U; ++u) {
                const int ds = u % kDoStages, qs1 = (u + 1) % kQStages;
                // Q(u + 1) is checked before P^T(u): dV(u) and S^T(u + 1) then issue back to back
                if (u + 1 < U && !(ok = mbar_wait(q_full(qs1), ((u + 1) / kQStages) & 1, abort, p.status))) break;
                if (!(ok = mbar_wait(p_full, u & 1, abort, p.status))) break;
                tc_fence_after();
                issue_acc_half(tmem + cDV, tmem + cS, sDO(ds), idesc_o, 0, u > 0);  // dV += P^T dO, first halves
                if (!(ok = mbar_wait(p_half1, u & 1, abort, p.status))) break;
                tc_fence_after();
                issue_acc_half(tmem + cDV, tmem + cS, sDO(ds), idesc_o, 1, true);   // second halves
                mma_commit(do_empty(ds));
                if (u + 1 < U) {
                    issue_qk<D>(tmem + cS, sK, sQ(qs1), idesc_s);
                    mma_commit(s_full);
                    mma_commit(q_empty(qs1));
                }
                mbar_arrive(s_issued(u));   // the dK(u) MMAs queue behind S^T(u + 1)
            }
            mma_commit(o_full);
            mbar_wait(o_full, 0, nullptr, p.status);
        }
    } else if (warp == 10) {
        // ---------------------------------------------------------------- MMA: dP^T, dK chain
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16(128, D, 0, 1);
            bool ok = U > 0 && mbar_wait(kv_full, 0, abort, p.status) && mbar_wait(do_full(0), 0, abort, p.status);
            if (ok) {
                tc_fence_after();
                issue_qk<D>(tmem + cDP, sV, sDO(0), idesc_s);      // dP^T = V dO^T
                mma_commit(dp_full);
                mma_commit(do_empty(0));                           // this chain's read of dO(0)
            }
            for (int u = 0; ok && u < U; ++u) {
                const int qs = u % kQStages, ds1 = (u + 1) % kDoStages;
                // dO(u + 1) is checked first: dK(u) and dP^T(u + 1) then issue back to back
                if (u + 1 < U && !(ok = mbar_wait(do_full(ds1), ((u + 1) / kDoStages) & 1, abort, p.status))) break;
                if (!(ok = mbar_wait(ds_full, u & 1, abort, p.status) &&
                           mbar_wait(s_issued(u), (u >> 1) & 1, abort, p.status)))
                    break;
                tc_fence_after();
                issue_acc_split(tmem + cDK, tmem + cDP, sQ(qs), idesc_o, u > 0);    // dK += dS^T Q
                mma_commit(q_empty(qs));
                if (u + 1 < U) {
                    issue_qk<D>(tmem + cDP, sV, sDO(ds1), idesc_s);
                    mma_commit(dp_full);
                    mma_commit(do_empty(ds1));
                }
            }
            mma_commit(o_full);
            mbar_wait(o_full, 0, nullptr, p.status);
        }
    } else {
        // ---------------------------------------------------------------- elementwise (warps 0-7)
        const int w = warp >> 2, q4 = warp & 3;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const int row = 32 * q4 + lane;                 // key row within the tile
        const int jj = tile * kTileRows + row;          // its compact row
        const float sl2 = p.scale_log2;
        bool ok = true;
        WarpRecords recs;
        for (int u = 0; u < U; ++u) {
            const int ds = u % kDoStages, qs = u % kQStages;
            const int4 te = recs.get(tinfo, u >> 1, n_ent, lane);
            // s_full implies the unit's stages were loaded; waiting on their barriers as well makes
            // the bulk-copied lse / delta visible to this thread directly
            ok = __all_sync(0xffffffffu, mbar_wait(s_full, u & 1, abort, p.status) &&
                                             mbar_wait(do_full(ds), (u / kDoStages) & 1, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            const float4 *ls4 = reinterpret_cast<const float4 *>(lse_s + ds * 128 + 64 * w);
            const float4 *dl4 = reinterpret_cast<const float4 *>(dl_s + qs * 128 + 64 * w);
            const bool row_in = jj >= te.z && jj < te.w;
            const bool causal = (te.x & kEntryCausal) != 0;
            // query row of lane m of this group's columns: first row + ((128 t + 64 w + m) mod R)
            const int rbase = te.y, rmask = p.R - 1, mbase = 128 * (u & 1) + 64 * w;
            // ---------------- phase 1: P^T, in two halves of 32 query columns: the dV MMAs of
            // the first half run while the second is exponentiated
            float pf[64];
            {
                uint32_t sv[2][32];
                tmem_ld32(tmem + lane_off + cS + 64 * w, sv[0]);
                tmem_wait_ld_regs(sv[0]);
                tmem_ld32(tmem + lane_off + cS + 64 * w + 32, sv[1]);
                const uint64_t sc2 = f2_pack(sl2, sl2);
                const bool need_mask = causal || __any_sync(0xffffffffu, !row_in);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    if (h == 1) tmem_wait_ld_regs(sv[1]);
#pragma unroll
                    for (int i4 = 8 * h; i4 < 8 * h + 8; ++i4) {
                        const float4 l4 = ls4[i4];       // -lse * log2(e) of four query columns
                        float x0, x1, x2, x3;
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[h][4 * (i4 & 7)]), __uint_as_float(sv[h][4 * (i4 & 7) + 1])),
                                         sc2, f2_pack(l4.x, l4.y)), x0, x1);
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[h][4 * (i4 & 7) + 2]), __uint_as_float(sv[h][4 * (i4 & 7) + 3])),
                                         sc2, f2_pack(l4.z, l4.w)), x2, x3);
                        pf[4 * i4] = ex2(x0);
                        pf[4 * i4 + 1] = ex2(x1);
                        pf[4 * i4 + 2] = ex2(x2);
                        pf[4 * i4 + 3] = ex2(x3);
                    }
                    if (need_mask) {
#pragma unroll
                        for (int c = 32 * h; c < 32 * h + 32; ++c) {
                            const int r = rbase + ((mbase + c) & rmask);
                            pf[c] = (row_in && !(causal && jj > r)) ? pf[c] : 0.f;
                        }
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(pf[32 * h + 2 * i], pf[32 * h + 2 * i + 1]);
                    tmem_st16(tmem + lane_off + cS + 64 * w + 16 * h, pk);
                    tmem_wait_st();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(h == 0 ? p_full : p_half1);
                }
            }
            // ---------------- phase 2: dS^T
            ok = __all_sync(0xffffffffu, mbar_wait(dp_full, u & 1, abort, p.status) &&
                                             mbar_wait(q_full(qs), (u / kQStages) & 1, abort, p.status));
            if (!ok) break;
            tc_fence_after();
            {
                uint32_t dv[2][32];
                tmem_ld32(tmem + lane_off + cDP + 64 * w, dv[0]);
                tmem_ld32(tmem + lane_off + cDP + 64 * w + 32, dv[1]);
                tmem_wait_ld();
                uint32_t dk[2][16];
#pragma unroll
                for (int i4 = 0; i4 < 16; ++i4) {
                    const float4 d4 = dl4[i4];       // -delta of four query columns
                    float r0, r1, r2, r3;
                    f2_unpack(f2_mul(f2_pack(pf[4 * i4], pf[4 * i4 + 1]),
                                     f2_add(f2_pack(__uint_as_float(dv[i4 >> 3][4 * (i4 & 7)]), __uint_as_float(dv[i4 >> 3][4 * (i4 & 7) + 1])),
                                            f2_pack(d4.x, d4.y))), r0, r1);
                    f2_unpack(f2_mul(f2_pack(pf[4 * i4 + 2], pf[4 * i4 + 3]),
                                     f2_add(f2_pack(__uint_as_float(dv[i4 >> 3][4 * (i4 & 7) + 2]), __uint_as_float(dv[i4 >> 3][4 * (i4 & 7) + 3])),
                                            f2_pack(d4.z, d4.w))), r2, r3);
                    dk[i4 >> 3][2 * (i4 & 7)] = pack_bf16(r0, r1);
                    dk[i4 >> 3][2 * (i4 & 7) + 1] = pack_bf16(r2, r3);
                }
                tmem_st16(tmem + lane_off + cDP + 64 * w, dk[0]);
                tmem_st16(tmem + lane_off + cDP + 64 * w + 16, dk[1]);
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(ds_full);
            }
        }
        ok = __all_sync(0xffffffffu, ok && mbar_wait(o_full, 0, abort, p.status));
        if (ok) {
            tc_fence_after();
            // group 0 writes dK (scaled), group 1 writes dV
            float *dst;
            bool write = true;
            if (slot >= 0) {
                dst = p.partials + (static_cast<size_t>(slot) * p.Hkv + g) * 2 * kTileRows * D +
                      static_cast<size_t>(w * kTileRows + row) * D;
            } else {
                write = jj < p.N;
                const int l = jj / p.page_size;
                write = write && debug_in_range(l, 0, p.n_logical_pages, p.status);
                const int pg = write ? __ldg(p.page_table + l) : 0;
                write = write && debug_in_range(pg, 0, p.num_pages, p.status);
                const size_t prow = write ? static_cast<size_t>(pg) * p.page_size + jj % p.page_size : 0;
                dst = (w == 0 ? p.dk_pool : p.dv_pool) + (prow * p.Hkv + g) * D;
            }
            const float mul = w == 0 ? p.scale : 1.f;
            const uint32_t src = tmem + lane_off + (w == 0 ? cDK : cDV);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(src + 32 * c, v);
                tmem_wait_ld();
                if (write) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst + 32 * c);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        d4[i] = make_float4(__uint_as_float(v[4 * i]) * mul, __uint_as_float(v[4 * i + 1]) * mul,
                                            __uint_as_float(v[4 * i + 2]) * mul, __uint_as_float(v[4 * i + 3]) * mul);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------------------ reduce
// One CTA per (split tile, KV head): dK and dV of every row = sum of the tile's partial
// slots in slot order, written through the page table.
template <int D>
__global__ void __launch_bounds__(256) reduce_kernel(const BwdParams p) {
    const int ri = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;
    const int tile = __ldg(p.reduce + 4 * ri), s0 = __ldg(p.reduce + 4 * ri + 1), ns = __ldg(p.reduce + 4 * ri + 2);
    constexpr int V4 = D / 4;
    for (int idx = threadIdx.x; idx < 2 * kTileRows * V4; idx += blockDim.x) {
        const int which = idx / (kTileRows * V4), rem = idx % (kTileRows * V4);
        const int row = rem / V4, c4 = rem % V4;
        const int jj = tile * kTileRows + row;
        if (jj >= p.N) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < ns; ++s) {
            const float4 v = reinterpret_cast<const float4 *>(
                p.partials + ((static_cast<size_t>(s0 + s) * p.Hkv + g) * 2 + which) * kTileRows * D)[row * V4 + c4];
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        if (!debug_in_range(jj / p.page_size, 0, p.n_logical_pages, p.status)) continue;
        const int pg = __ldg(p.page_table + jj / p.page_size);
        if (!debug_in_range(pg, 0, p.num_pages, p.status)) continue;
        const size_t prow = static_cast<size_t>(pg) * p.page_size + jj % p.page_size;
        float *dst = (which == 0 ? p.dk_pool : p.dv_pool) + (prow * p.Hkv + g) * D;
        reinterpret_cast<float4 *>(dst)[c4] = acc;
    }
}

template <int D>
cudaError_t launch_bwd_d(const CUtensorMap &tm_q, const KvMaps &kv, const CUtensorMap &tm_do, const BwdParams &p,
                         int n_blocks, int n_chunks, int n_reduce, cudaStream_t stream, void *const *trace) {
    trace_record(trace, 2, stream);
    delta_kernel<D><<<static_cast<unsigned>(n_blocks) * p.Hkv * 2, 128, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dq_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DqLayout<D>::bytes);
    if (e != cudaSuccess) return e;
    trace_record(trace, 3, stream);
    dq_kernel<D><<<n_blocks * p.Hkv * 2, kDqThreads, DqLayout<D>::bytes, stream>>>(
        tm_q, kv.k_piece, kv.v_piece, kv.k_half, kv.v_half, tm_do, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dkdv_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, DkvLayout<D>::bytes);
    if (e != cudaSuccess) return e;
    trace_record(trace, 4, stream);
    dkdv_kernel<D><<<n_chunks * p.Hkv, kDkvThreads, DkvLayout<D>::bytes, stream>>>(tm_q, kv.k_page, kv.v_page,
                                                                                    tm_do, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    trace_record(trace, 5, stream);
    if (n_reduce > 0) {
        reduce_kernel<D><<<n_reduce * p.Hkv, 256, 0, stream>>>(p);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    trace_record(trace, 6, stream);
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_bwd(int D, const CUtensorMap &tm_q, const KvMaps &kv, const CUtensorMap &tm_do,
                       const BwdParams &p, int n_blocks, int n_chunks, int n_reduce, cudaStream_t stream,
                       void *const *trace) {
    if (D == 64) return launch_bwd_d<64>(tm_q, kv, tm_do, p, n_blocks, n_chunks, n_reduce, stream, trace);
    return launch_bwd_d<128>(tm_q, kv, tm_do, p, n_blocks, n_chunks, n_reduce, stream, trace);
}

}  // namespace treeattn
