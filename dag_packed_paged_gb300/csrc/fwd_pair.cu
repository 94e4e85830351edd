// Forward kernel on CTA pairs (sm_103a: tcgen05 cta_group::2, TMA, TMEM), head dim 128.
//
// Computes the same O and lse as fwd.cu -- for every row r of a query block and the G query
// heads of KV head g, O[r,h] = sum_{j in vis(r)} softmax_j(scale q[r,h].k[j,g]) v[j,g] over the
// key rows the plan's packed tiles list (Octopus arXiv 2611.06956 Section 3.3 Eq. 4 with the
// rectangular causal alignment after it; HARTS arXiv 2608.28158 Section 4.2 Eq. 21-22) -- with
// one work item (a query block, or one part of a split block: fwd.cu) x one KV head per pair
// of CTAs on neighbouring SMs (a cluster of two).
//
// The block's 256 MMA rows (R rows x G heads) are split between the two CTAs: CTA r holds query
// tile r (128 rows) in shared memory and owns the 128 TMEM lanes of those rows.  Every MMA is
// issued once for the pair (M = 256) by a thread of CTA 0:
//   S = Q K^T   A: each CTA's query tile;  B: the packed key tile, keys [64r, 64r + 64) in CTA r
//   O += P V    A: each CTA's P (bf16, in its TMEM);  B: V, head-dim columns [64r, 64r + 64) in CTA r
// so every SM loads half of each K and V tile and the pair uses it for 256 query rows, as the
// single-SM kernel does with two query tiles.  With one query tile per SM, TMEM holds three score
// buffers and O (3 x 128 + 128 = 512 columns): P(j) overwrites S(j) in place and is read by PV(j)
// before S(j + 3) reuses the buffer, so the scores of the next tiles are computed while the
// softmax of tile j runs.  The single-SM kernel's per-tile chain (softmax -> PV -> next S ->
// softmax) becomes softmax -> softmax.  With a finite running max the exponentials start as soon
// as the scores are loaded (the lazy rescale keeps the max unless a tile exceeds it by 2^8), the
// row maximum only deciding whether they are recomputed.
//
// Warps per CTA: 0-3 softmax of the CTA's query tile (one TMEM lane = one (row, head) per
// thread); 4 TMA producer (the CTA's query tile, its half of every K and V tile); 5 TMEM
// allocation (both CTAs) and, in CTA 0, the PV issuer; 6, in CTA 0, the S issuer.  One thread
// issuing every MMA with its commits and waits needs more cycles per tile than the tensor core
// (measured); the S issuer puts S(j + 3) behind PV(j) through a barrier that the PV issuer
// arrives on once PV(j) is issued.
// Barriers that gather both CTAs' work live in CTA 0: the full barriers of Q, K and V (each CTA's
// TMA signals CTA 0's barrier, whose expected bytes cover both halves) and P-ready (every softmax
// warp of both CTAs arrives).  The MMA commits of CTA 0 arrive on the barriers of both CTAs:
// scores ready, K/V stage free (after PV, which also tells the softmax that O is up to date),
// O final.
#include <cfloat>

#include "fwd_store.cuh"
#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

constexpr int kD = 128;
constexpr int kPS = 4;            // K/V half-tile stages
constexpr int kSB = 3;            // score buffers in TMEM (128 columns each; O takes the last 128)
constexpr uint32_t kOCol = kSB * 128;
constexpr int kPairThreads = 224;

struct PairLayout {
    static constexpr int kQ = 128 * kD * 2;        // the CTA's query tile: [2 chunks][128 rows][128 B]
    static constexpr int kKh = 64 * kD * 2;        // half a key tile: 64 keys, [2 chunks][64 rows][128 B]
    static constexpr int kVh = kTileRows * 64 * 2; // half a value tile: 64 head-dim columns, [128 keys][128 B]
    static constexpr int q_off = 0;
    static constexpr int k_off = q_off + kQ;
    static constexpr int v_off = k_off + kPS * kKh;
    static constexpr int bar_off = v_off + kPS * kVh;
    // q_full, k_full, v_full, kv_empty (per stage), s_full, p_full, pv_issued (per score buffer),
    // s_drain, o_full
    static constexpr int n_bars = 1 + 3 * kPS + 3 * kSB + 1 + 1;
    static constexpr int misc_off = bar_off + n_bars * 8;
    static constexpr int bytes = misc_off + 16 + 1024;     // + alignment slack
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_k64,
                const __grid_constant__ CUtensorMap tm_v64, const FwdParams p) {
    using L = PairLayout;
    constexpr int D = kD;
    extern __shared__ uint8_t smem_raw[];
    // both CTAs run the same kernel, so the aligned base (and every offset) is the same in both:
    // the pair MMAs read the peer's operands at the addresses given for this CTA's
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    const int pair = blockIdx.x >> 1;
    const int4 item = __ldg(reinterpret_cast<const int4 *>(p.items) + pair / p.Hkv);   // work item (fwd.cu)
    const int qb = item.x, e0 = item.y, E = item.z - item.y, slot = item.w;
    const int g = pair % p.Hkv;
    const int q_row0 = __ldg(p.blocks + 4 * qb), n_rows = __ldg(p.blocks + 4 * qb + 1);
    const int4 *tiles = reinterpret_cast<const int4 *>(p.ftiles) + 2 * e0;   // two int4 per tile

    const uint32_t sQ = sbase + L::q_off, sK = sbase + L::k_off, sV = sbase + L::v_off;
    auto bar = [&](int i) { return sbase + L::bar_off + 8u * i; };
    const uint32_t q_full = bar(0);
    auto k_full = [&](int s) { return bar(1 + s); };
    auto v_full = [&](int s) { return bar(1 + kPS + s); };
    auto kv_empty = [&](int s) { return bar(1 + 2 * kPS + s); };
    auto s_full = [&](int b) { return bar(1 + 3 * kPS + b); };
    auto p_full = [&](int b) { return bar(1 + 3 * kPS + kSB + b); };
    auto pv_issued = [&](int b) { return bar(1 + 3 * kPS + 2 * kSB + b); };
    const uint32_t s_drain = bar(1 + 3 * kPS + 3 * kSB);
    const uint32_t o_full = bar(2 + 3 * kPS + 3 * kSB);
    auto lead = [&](uint32_t a) { return mapa_shared(a, 0); };   // CTA 0's copy of a barrier
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc_off);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L::misc_off + 4);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kPS; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(v_full(s), 1);
            mbar_init(kv_empty(s), 1);
        }
        for (int b = 0; b < kSB; ++b) {
            mbar_init(s_full(b), 1);
            mbar_init(p_full(b), 8);         // 4 softmax warps x 2 CTAs
            mbar_init(pv_issued(b), 1);
        }
        mbar_init(s_drain, 1);
        mbar_init(o_full, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncwarp();
    cluster_sync();          // both CTAs' barriers exist before either CTA signals the other
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_k64);
            tma_prefetch_desc(&tm_v64);
            const int R = p.R, QB = R < 128 ? R : 128;
            if (leader) mbar_arrive_expect_tx(q_full, 2 * L::kQ);
            const uint32_t qbar = lead(q_full);
            for (int b = 0; b < 128 / QB; ++b) {
                const int m0 = 128 * static_cast<int>(rank) + b * QB, hl = m0 / R, r0 = m0 % R;
                for (int c = 0; c < D / 64; ++c)
                    tma_load_2d_pair(sQ + c * 16384 + b * QB * 128, &tm_q, (g * p.G + hl) * D + c * 64, q_row0 + r0,
                                     qbar);
            }
        }
        // the whole warp prefetches tile records and TMA rows 32 tiles at a time; lane 0 issues
        PackFeed f;
        const int oob = p.num_pages * p.page_size;
        const int h = static_cast<int>(rank);      // this CTA's half of each key tile (slots 2h, 2h + 1)
        int issued = 0;
        for (int j = 0; j < E; ++j) {
            if ((j & 31) == 0)
                pack_feed_fill(f, j, E, tiles, p.page_table, p.n_logical_pages, p.page_size, oob, lane, p.status);
            int y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = __shfl_sync(0xffffffffu, f.y[i], j & 31);
            const int fl = __shfl_sync(0xffffffffu, f.b.z, j & 31);
            const int st = j % kPS;
            bool ok = true;
            // the stage is free once PV(j - kPS) is done (S(j - kPS) finished before it)
            if (lane == 0 && j >= kPS) ok = mbar_wait(kv_empty(st), ((j / kPS) - 1) & 1, abort, p.status);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (lane == 0) {
                if (leader) {
                    mbar_arrive_expect_tx(k_full(st), 2 * L::kKh);
                    mbar_arrive_expect_tx(v_full(st), 2 * L::kVh);
                }
                const uint32_t kb = lead(k_full(st)), kdst = sK + st * L::kKh;
                if (fl & (kPackHalf64 << h)) {
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_2d_pair(kdst + c * (64 * 128), &tm_k64, g * D + c * 64, y[4 * h], kb);
                } else {
                    for (int s = 0; s < 2; ++s) {
                        const int k = 2 * h + s;
                        for (int c = 0; c < D / 64; ++c) {
                            tma_load_2d_pair(kdst + c * (64 * 128) + s * 32 * 128, &tm_k, g * D + c * 64, y[2 * k], kb);
                            if (p.page_size < 32)
                                tma_load_2d_pair(kdst + c * (64 * 128) + s * 32 * 128 + 16 * 128, &tm_k, g * D + c * 64,
                                                 y[2 * k + 1], kb);
                        }
                    }
                }
                const uint32_t vb = lead(v_full(st)), vdst = sV + st * L::kVh;
                const int x = g * D + h * 64;      // this CTA's 64 head-dim columns, all 128 keys
                for (int hh = 0; hh < 2; ++hh) {
                    if (fl & (kPackHalf64 << hh)) {
                        tma_load_2d_pair(vdst + hh * 64 * 128, &tm_v64, x, y[4 * hh], vb);
                    } else {
                        for (int s = 0; s < 2; ++s) {
                            const int k = 2 * hh + s;
                            tma_load_2d_pair(vdst + k * 32 * 128, &tm_v, x, y[2 * k], vb);
                            if (p.page_size < 32)
                                tma_load_2d_pair(vdst + k * 32 * 128 + 16 * 128, &tm_v, x, y[2 * k + 1], vb);
                        }
                    }
                }
            }
            issued = j + 1;
        }
        if (lane == 0 && leader) {
            // CTA 0's full barriers count both CTAs' bytes: once their last phases are complete no
            // copy of either CTA is in flight (the final cluster barrier keeps CTA 1 resident)
            for (int d = (issued > kPS ? issued - kPS : 0); d < issued; ++d) {
                mbar_wait(k_full(d % kPS), (d / kPS) & 1, nullptr, p.status);
                mbar_wait(v_full(d % kPS), (d / kPS) & 1, nullptr, p.status);
            }
            mbar_wait(q_full, 0, nullptr, p.status);
        }
    } else if (warp == 5 || warp == 6) {
        // ------------------------------------------------------------------ MMA issuers (CTA 0)
        auto commit_both = [&](uint32_t b) {
            mma_commit_pair(b);
            mma_commit_pair(mapa_shared(b, 1));
        };
        if (lane == 0 && leader && warp == 6) {
            // S(j) = Q K(j)^T into buffer j mod 3, behind PV(j - 3) (which reads P(j - 3) there)
            constexpr uint32_t idesc_s = idesc_bf16(256, kTileRows, 0, 0);
            const uint64_t a0 = sdesc_sw128(sQ, 16, 1024);
            bool ok = E > 0 && mbar_wait(q_full, 0, abort, p.status);
            for (int j = 0; ok && j < E; ++j) {
                const int b = j % kSB, st = j % kPS;
                if (j >= kSB && !(ok = mbar_wait(pv_issued(b), ((j - kSB) / kSB) & 1, abort, p.status))) break;
                if (!(ok = mbar_wait(k_full(st), (j / kPS) & 1, abort, p.status))) break;
                tc_fence_after();
                const uint64_t b0 = sdesc_sw128(sK + st * L::kKh, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t aoff = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    const uint64_t boff = static_cast<uint64_t>(((kk >> 2) * 8192 + (kk & 3) * 32) >> 4);
                    mma_ss_pair(tmem + b * 128, a0 + aoff, b0 + boff, idesc_s, kk > 0 ? 1u : 0u);
                }
                commit_both(s_full(b));
            }
            mma_commit_pair(s_drain);                        // this thread's MMAs, before TMEM is freed
            mbar_wait(s_drain, 0, nullptr, p.status);
        } else if (lane == 0 && leader) {
            // O += P(j) V(j), P(j) in the first 64 columns of buffer j mod 3 (key k in column k / 2)
            constexpr uint32_t idesc_o = idesc_bf16(256, D, 0, 1);
            bool ok = true;
            for (int j = 0; ok && j < E; ++j) {
                const int b = j % kSB, st = j % kPS;
                if (!(ok = mbar_wait(v_full(st), (j / kPS) & 1, abort, p.status))) break;
                if (!(ok = mbar_wait(p_full(b), (j / kSB) & 1, abort, p.status))) break;
                tc_fence_after();
                const uint64_t b0 = sdesc_sw128(sV + st * L::kVh, kTileRows * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk)
                    mma_ts_pair(tmem + kOCol, tmem + b * 128 + kk * 8,
                                b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
                commit_both(kv_empty(st));
                mbar_arrive(pv_issued(b));
            }
            commit_both(o_full);                                 // every MMA of the pair is done
            mbar_wait(o_full, 0, nullptr, p.status);             // drain before TMEM is released
        }
    } else {
        // ------------------------------------------------------------------ softmax (warps 0-3)
        const int q4 = warp;
        const int row = 32 * q4 + lane;            // TMEM lane = the CTA's query-tile row
        const int m_flat = 128 * static_cast<int>(rank) + row;
        const int hl = m_flat / p.R, rl = m_flat % p.R;
        const int r_abs = q_row0 + rl;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const uint32_t tO = tmem + lane_off + kOCol;
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        WarpPackRecords recs;
        // p = 2^(s scale log2e - m) for the row's 128 scores: the arguments two at a time, four
        // independent partial sums; returns the row sum and packs the values as bf16 pairs
        auto exps = [&](const float (&s)[kTileRows], float m, uint32_t (&pk)[kTileRows / 2]) {
            const float mref = m == -INFINITY ? 0.f : m;
            const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mref, -mref);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
            for (int c = 0; c < kTileRows / 2; ++c) {
                float xa, xb;
                f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), sc2, nm2), xa, xb);
                const float a = ex2(xa), bb = ex2(xb);
                acc[c & 3] = f2_add(acc[c & 3], f2_pack(a, bb));
                pk[c] = pack_bf16(a, bb);
            }
            float r0, r1, r2, r3, r4, r5, r6, r7;
            f2_unpack(acc[0], r0, r1);
            f2_unpack(acc[1], r2, r3);
            f2_unpack(acc[2], r4, r5);
            f2_unpack(acc[3], r6, r7);
            return ((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7));
        };
        for (int j = 0; ok && j < E; ++j) {
            const int b = j % kSB;
            const uint32_t tS = tmem + lane_off + b * 128;
            int4 ra, rb;
            recs.get(tiles, j, E, lane, ra, rb);
            ok = __all_sync(0xffffffffu, mbar_wait(s_full(b), (j / kSB) & 1, abort, p.status));
            if (!ok) break;                          // warp-uniform: tcgen05.ld/st are collective
            tc_fence_after();
            uint32_t sb[kTileRows];
#pragma unroll
            for (int c = 0; c < kTileRows / 32; ++c)
                tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sb[c * 32]));
            tmem_wait_ld();
            float s[kTileRows];
#pragma unroll
            for (int c = 0; c < kTileRows; ++c) s[c] = __uint_as_float(sb[c]);
            if (rb.z & kPackMask) {                   // some slot is partial, causal or empty
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    int lo, hi;
                    pack_slot_range(ra, rb, k, r_abs, lo, hi);
                    if (lo > 0 || hi < kPieceRows) {
#pragma unroll
                        for (int c = 0; c < kPieceRows; ++c)
                            if (c < lo || c >= hi) s[kPieceRows * k + c] = -INFINITY;
                    }
                }
            }
            // With a finite running max the probabilities are computed against it right away,
            // while the tile's maximum is still being formed: the lazy rescale keeps m unless
            // the tile exceeds it by more than 2^8, so in the common case these are the final
            // values; otherwise they are recomputed below.
            const bool spec = !__any_sync(0xffffffffu, m_used == -INFINITY);
            uint32_t pk[kTileRows / 2];
            float rs = 0.f;
            if (spec) rs = exps(s, m_used, pk);
            // row max: a tree of three-input maxima (16 independent chains, then a final fold)
            float a16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float m = max3(s[i], s[16 + i], s[32 + i]);
                m = max3(m, s[48 + i], s[64 + i]);
                m = max3(m, s[80 + i], s[96 + i]);
                a16[i] = fmaxf(m, s[112 + i]);
            }
            float mx = max3(max3(a16[0], a16[1], a16[2]), max3(a16[3], a16[4], a16[5]), max3(a16[6], a16[7], a16[8]));
            mx = max3(mx, max3(a16[9], a16[10], a16[11]), max3(a16[12], a16[13], a16[14]));
            mx = fmaxf(mx, a16[15]);
            const float m_new = fmaxf(m_used, mx * sl2);
            const bool need = m_new > m_used + 8.f;
            const bool any_need = __any_sync(0xffffffffu, need);
            if (!spec || any_need) {
                if (j == 0) {
                    if (need) m_used = m_new;
                } else if (any_need) {
                    // O holds PV(0 .. j-1); S(j) was issued behind PV(j-3) only, so wait for
                    // PV(j-1), whose completion frees its K/V stage (that barrier has completed
                    // either the phase of PV(j-1) or the one before it here)
                    const int st1 = (j - 1) % kPS;
                    ok = __all_sync(0xffffffffu, mbar_wait(kv_empty(st1), ((j - 1) / kPS) & 1, abort, p.status));
                    if (!ok) break;
                    tc_fence_after();
                    const float f = need ? ex2(m_used - m_new) : 1.f;
                    if (need) {
                        l *= f;
                        m_used = m_new;
                    }
#pragma unroll
                    for (int c = 0; c < D / 16; ++c) {
                        uint32_t v[16];
                        tmem_ld16(tO + c * 16, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                        tmem_st16(tO + c * 16, v);
                    }
                    tmem_wait_st();
                }
                rs = exps(s, m_used, pk);
            }
            l += rs;
            tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));   // P over the first 64 score columns
            tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();                            // the whole warp's P is in TMEM
            if (lane == 0) mbar_arrive_cluster(lead(p_full(b)));
        }
        ok = __all_sync(0xffffffffu, ok && mbar_wait(o_full, 0, abort, p.status));
        if (ok) {
            tc_fence_after();
            const bool valid = rl < n_rows && debug_in_range(r_abs, 0, p.N, p.status) &&
                               (slot < 0 || debug_in_range(slot, 0, p.n_slots, p.status));
            const int hh = g * p.G + hl;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float lse = (m_used + log2f(l)) * 0.69314718055994531f;
            if (slot < 0)
                store_o_row<D>(tO, valid, inv, p.o + (static_cast<size_t>(r_abs) * p.Hq + hh) * D,
                               p.lse + static_cast<size_t>(hh) * p.N + r_abs, lse);
            else
                store_partial_row<D>(tO, valid, inv, p, slot, g, m_flat, lse);
        }
    }

    tc_fence_before();
    __syncwarp();            // the barrier below is warp-aligned: reconverge the role branches
    cluster_sync();          // neither CTA frees TMEM or leaves while the pair's MMAs may touch it
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

}  // namespace

cudaError_t launch_fwd_pair(const CUtensorMap &tm_q, const KvMaps &kv, const FwdParams &p, int n_items,
                            cudaStream_t stream) {
    const int smem = PairLayout::bytes;
    cudaError_t err = cudaFuncSetAttribute(fwd_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    fwd_pair_kernel<<<2 * n_items * p.Hkv, kPairThreads, smem, stream>>>(tm_q, kv.k_piece, kv.v_piece, kv.k_half,
                                                                         kv.v_half, p);
    return cudaGetLastError();
}

}  // namespace treeattn
