// Forward kernel: tree/DAG-packed attention over a paged KV pool (sm_103a, tcgen05 + TMA).
//
// Computes, for every row r of one query block and the G query heads of one KV head g,
//   O[r,h] = sum_{j in vis(r)} softmax_j(scale q[r,h].k[j,g]) v[j,g],   lse[h,r] = ln sum exp
// (Octopus arXiv 2611.06956 Section 3.3 Eq. 4 with the rectangular causal alignment after it;
// HARTS arXiv 2608.28158 Section 4.2 Eq. 21-22), visiting only the packed key tiles the plan
// lists for the block -- 4 slots of 32 key rows each, gathered from the visible intervals --
// and masking each slot's rows outside its [lo, hi) and, on slots of the block's own rows,
// above the query row.
//
// One CTA = one work item (a query block, or a run of its packed tiles when the plan splits a
// long block: split-KV) of R rows x G heads = 256 query rows of the MMA, two 128-lane tiles,
// x one KV head.  A split item writes its normalised O and lse in fp32 to a partial slot, and
// fwd_combine_kernel merges the parts.  Warp roles:
//   warps 0-3  softmax for query tile 0 (one TMEM lane = one (row, head) per thread)
//   warps 4-7  softmax for query tile 1
//   warp 8     TMA producer: Q once, then K and V tiles slot by slot (a box per 32-row slot,
//              or per 64-row half when its two slots are one aligned run)
//   warp 9     tcgen05 MMA issuer: S_t = Q_t K^T into TMEM, O_t += P_t V with P read from TMEM
// TMEM (512 columns): S0 | S1 | O0 | O1; P_t (bf16 pairs) overwrites the first half of S_t.
// The two query tiles ping-pong so that one tile's softmax overlaps the other tile's MMAs.
// The running max is rescaled lazily (only when it grows by more than 2^8).
#include <cfloat>

#include "fwd_store.cuh"
#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

constexpr int kKS = 2;           // K stages
constexpr int kVS = 2;           // V stages
constexpr int kThreads = 320;

template <int D>
struct FwdLayout {
    static constexpr int kQTile = 128 * D * 2;            // bytes of one 128-row Q tile
    static constexpr int kKV = kTileRows * D * 2;          // bytes of one K or V tile
    static constexpr int q_off = 0;
    static constexpr int k_off = q_off + 2 * kQTile;
    static constexpr int v_off = k_off + kKS * kKV;
    static constexpr int bar_off = v_off + kVS * kKV;
    static constexpr int n_bars = 1 + 2 * kKS + 2 * kVS + 2 + 2 + 1;
    static constexpr int misc_off = bar_off + n_bars * 8;
    static constexpr int bytes = misc_off + 16 + 1024;     // + alignment slack
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
           const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_k64,
           const __grid_constant__ CUtensorMap tm_v64, const FwdParams p) {
    using L = FwdLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int4 item = __ldg(reinterpret_cast<const int4 *>(p.items) + blockIdx.x / p.Hkv);
    const int qb = item.x, e0 = item.y, E = item.z - item.y, slot = item.w;
    const int g = blockIdx.x % p.Hkv;
    const int q_row0 = __ldg(p.blocks + 4 * qb), n_rows = __ldg(p.blocks + 4 * qb + 1);
    const int4 *tiles = reinterpret_cast<const int4 *>(p.ftiles) + 2 * e0;   // two int4 per tile

    const uint32_t sQ = sbase + L::q_off, sK = sbase + L::k_off, sV = sbase + L::v_off;
    auto bar = [&](int i) { return sbase + L::bar_off + 8u * i; };
    const uint32_t q_full = bar(0);
    auto k_full = [&](int s) { return bar(1 + s); };
    auto k_empty = [&](int s) { return bar(1 + kKS + s); };
    auto v_full = [&](int s) { return bar(1 + 2 * kKS + s); };
    auto v_empty = [&](int s) { return bar(1 + 2 * kKS + kVS + s); };
    auto s_full = [&](int t) { return bar(1 + 2 * kKS + 2 * kVS + t); };
    auto p_full = [&](int t) { return bar(3 + 2 * kKS + 2 * kVS + t); };
    const uint32_t o_full = bar(5 + 2 * kKS + 2 * kVS);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc_off);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + L::misc_off + 4);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kKS; ++s) { mbar_init(k_full(s), 1); mbar_init(k_empty(s), 1); }
        for (int s = 0; s < kVS; ++s) { mbar_init(v_full(s), 1); mbar_init(v_empty(s), 1); }
        for (int t = 0; t < 2; ++t) { mbar_init(s_full(t), 1); mbar_init(p_full(t), 4); }   // one arrival per warp
        mbar_init(o_full, 1);
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

    if (warp == 8) {
        // ------------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_k64);
            tma_prefetch_desc(&tm_v64);
            const int R = p.R, QB = R < 128 ? R : 128;
            mbar_arrive_expect_tx(q_full, 2 * L::kQTile);
            for (int t = 0; t < 2; ++t)
                for (int b = 0; b < 128 / QB; ++b) {
                    const int m0 = 128 * t + b * QB, hl = m0 / R, r0 = m0 % R;
                    for (int c = 0; c < D / 64; ++c)
                        tma_load_2d(sQ + t * L::kQTile + c * 16384 + b * QB * 128, &tm_q,
                                    (g * p.G + hl) * D + c * 64, q_row0 + r0, q_full);
                }
        }
        // the whole warp prefetches tile records and TMA rows 32 tiles at a time; lane 0 issues
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
            const int ks = j % kKS, vs = j % kVS;
            bool ok = true;
            if (lane == 0 && j >= kKS) ok = mbar_wait(k_empty(ks), ((j / kKS) - 1) & 1, abort, p.status);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(k_full(ks), L::kKV);
                tma_packed_tile(sK + ks * L::kKV, &tm_k, &tm_k64, y, fl, p.page_size, g, D, k_full(ks));
            }
            k_issued = j + 1;
            if (lane == 0 && j >= kVS) ok = mbar_wait(v_empty(vs), ((j / kVS) - 1) & 1, abort, p.status);
            if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
            if (lane == 0) {
                mbar_arrive_expect_tx(v_full(vs), L::kKV);
                tma_packed_tile(sV + vs * L::kKV, &tm_v, &tm_v64, y, fl, p.page_size, g, D, v_full(vs));
            }
            v_issued = j + 1;
        }
        if (lane == 0) {
            // never leave the CTA with copies in flight: wait for the last phase of each stage
            for (int d = (k_issued > kKS ? k_issued - kKS : 0); d < k_issued; ++d)
                mbar_wait(k_full(d % kKS), (d / kKS) & 1, nullptr, p.status);
            for (int d = (v_issued > kVS ? v_issued - kVS : 0); d < v_issued; ++d)
                mbar_wait(v_full(d % kVS), (d / kVS) & 1, nullptr, p.status);
            mbar_wait(q_full, 0, nullptr, p.status);
        }
    } else if (warp == 9) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, kTileRows, 0, 0);
            constexpr uint32_t idesc_o = idesc_bf16(128, D, 0, 1);
            // descriptors are built once per tile; stepping along K only moves the 14-bit
            // start-address field, so each step is a 64-bit add of a compile-time constant
            auto issue_s = [&](int t, int ks) {
                const uint64_t a0 = sdesc_sw128(sQ + t * L::kQTile, 16, 1024);
                const uint64_t b0 = sdesc_sw128(sK + ks * L::kKV, 16, 1024);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t koff = static_cast<uint64_t>(((kk >> 2) * 16384 + (kk & 3) * 32) >> 4);
                    mma_ss(tmem + t * 128, a0 + koff, b0 + koff, idesc_s, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int vs, bool acc) {
                const uint64_t b0 = sdesc_sw128(sV + vs * L::kKV, kTileRows * 128, 1024);
#pragma unroll
                for (int kk = 0; kk < kTileRows / 16; ++kk)
                    mma_ts(tmem + 256 + t * D, tmem + t * 128 + kk * 8, b0 + static_cast<uint64_t>((kk * 16 * 128) >> 4),
                           idesc_o, (acc || kk > 0) ? 1u : 0u);
            };
            bool ok = E > 0 && mbar_wait(q_full, 0, abort, p.status) && mbar_wait(k_full(0), 0, abort, p.status);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                mma_commit(s_full(0));
                issue_s(1, 0);
                mma_commit(s_full(1));
                mma_commit(k_empty(0));
            }
            for (int j = 0; ok && j < E; ++j) {
                const int vs = j % kVS, ks = (j + 1) % kKS;
                if (!(ok = mbar_wait(v_full(vs), (j / kVS) & 1, abort, p.status))) break;
                if (!(ok = mbar_wait(p_full(0), j & 1, abort, p.status))) break;
                tc_fence_after();
                issue_pv(0, vs, j > 0);
                if (j + 1 < E) {
                    if (!(ok = mbar_wait(k_full(ks), ((j + 1) / kKS) & 1, abort, p.status))) break;
                    tc_fence_after();
                    issue_s(0, ks);
                    mma_commit(s_full(0));
                }
                if (!(ok = mbar_wait(p_full(1), j & 1, abort, p.status))) break;
                tc_fence_after();
                issue_pv(1, vs, j > 0);
                mma_commit(v_empty(vs));
                if (j + 1 < E) {
                    issue_s(1, ks);
                    mma_commit(s_full(1));
                    mma_commit(k_empty(ks));
                }
            }
            mma_commit(o_full);                               // all MMAs issued above are done
            mbar_wait(o_full, 0, nullptr, p.status);          // drain before TMEM is released
        }
    } else {
        // ------------------------------------------------------------------ softmax (warps 0-7)
        const int t = warp >> 2, q4 = warp & 3;
        const int m_flat = 128 * t + 32 * q4 + lane;
        const int hl = m_flat / p.R, rl = m_flat % p.R;
        const int r_abs = q_row0 + rl;
        const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
        const uint32_t tS = tmem + lane_off + t * 128;
        const uint32_t tO = tmem + lane_off + 256 + t * D;
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        WarpPackRecords recs;
        for (int j = 0; j < E; ++j) {
            int4 ra, rb;
            recs.get(tiles, j, E, lane, ra, rb);
            ok = __all_sync(0xffffffffu, mbar_wait(s_full(t), j & 1, abort, p.status));
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
            if (j == 0) {
                if (need) m_used = m_new;
            } else if (__any_sync(0xffffffffu, need)) {
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
            const float mref = m_used == -INFINITY ? 0.f : m_used;
            // p = 2^(s scale log2e - m): the arguments two at a time, four independent row sums
            const uint64_t sc2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mref, -mref);
            uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
            uint32_t pk[kTileRows / 2];
#pragma unroll
            for (int c = 0; c < kTileRows / 2; ++c) {
                float xa, xb;
                f2_unpack(f2_fma(f2_pack(s[2 * c], s[2 * c + 1]), sc2, nm2), xa, xb);
                const float a = ex2(xa), b = ex2(xb);
                acc[c & 3] = f2_add(acc[c & 3], f2_pack(a, b));
                pk[c] = pack_bf16(a, b);
            }
            float rs;
            {
                float r0, r1, r2, r3, r4, r5, r6, r7;
                f2_unpack(acc[0], r0, r1);
                f2_unpack(acc[1], r2, r3);
                f2_unpack(acc[2], r4, r5);
                f2_unpack(acc[3], r6, r7);
                rs = ((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7));
            }
            l += rs;
            tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
            tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();                            // the whole warp's P is in TMEM
            if (lane == 0) mbar_arrive(p_full(t));
        }
        ok = __all_sync(0xffffffffu, ok && mbar_wait(o_full, 0, abort, p.status));
        if (ok) {
            tc_fence_after();
            const bool valid = rl < n_rows && debug_in_range(r_abs, 0, p.N, p.status) &&
                               (slot < 0 || debug_in_range(slot, 0, p.n_slots, p.status));
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float lse = (m_used + log2f(l)) * 0.69314718055994531f;
            if (slot < 0)
                store_o_row<D>(tO, valid, inv, p.o + (static_cast<size_t>(r_abs) * p.Hq + g * p.G + hl) * D,
                               p.lse + static_cast<size_t>(g * p.G + hl) * p.N + r_abs, lse);
            else
                store_partial_row<D>(tO, valid, inv, p, slot, g, m_flat, lse);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Merge of a split block's parts (split-KV; the same rows' softmax over disjoint key sets):
//   lse = ln sum_k exp(lse_k),   O = sum_k exp(lse_k - lse) O_k
// with O_k the part's normalised output.  Grid (split blocks, KV heads, 8): a CTA takes 32 of
// the block's 256 MMA rows, a warp 4 of them.  Per row the lanes first run across the parts
// (max and sum of exp(lse_k - max)), then across the head dim, with the parts' loads unrolled
// so that several are in flight: the kernel is bound by the latency of those loads, not by
// their bytes (each part is read once).
template <int D>
__global__ void __launch_bounds__(256) fwd_combine_kernel(const FwdParams p) {
    constexpr int kPer = D / 32;                      // columns per lane: 2 or 4
    const int4 cb = __ldg(reinterpret_cast<const int4 *>(p.combine) + blockIdx.x);
    const int qb = cb.x, slot0 = cb.y, parts = cb.z;
    const int g = blockIdx.y;
    const int q_row0 = __ldg(p.blocks + 4 * qb), n_rows = __ldg(p.blocks + 4 * qb + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (!debug_in_range(slot0, 0, p.n_slots, p.status) || !debug_in_range(slot0 + parts, slot0 + 1, p.n_slots + 1, p.status))
        return;
    const size_t stride = static_cast<size_t>(p.Hkv) * 256;          // rows between consecutive slots
    const float *lse_part = p.partial + static_cast<size_t>(p.n_slots) * stride * D +
                            (static_cast<size_t>(slot0) * p.Hkv + g) * 256;
    const float *o_part = p.partial + (static_cast<size_t>(slot0) * p.Hkv + g) * 256 * D + kPer * lane;
    for (int i = 0; i < 4; ++i) {
        const int m = 32 * blockIdx.z + 4 * warp + i;
        const int hl = m / p.R, rl = m % p.R;
        if (rl >= n_rows) continue;                   // warp-uniform
        const int r_abs = q_row0 + rl, h = g * p.G + hl;
        if (!debug_in_range(r_abs, 0, p.N, p.status)) continue;
        float mx = -INFINITY;
        for (int k = lane; k < parts; k += 32) mx = fmaxf(mx, __ldcg(lse_part + k * stride + m));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float den = 0.f;
        if (mx > -INFINITY)
            for (int k = lane; k < parts; k += 32) den += expf(__ldcg(lse_part + k * stride + m) - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
        float acc[kPer];
#pragma unroll
        for (int c = 0; c < kPer; ++c) acc[c] = 0.f;
        if (mx > -INFINITY) {
#pragma unroll 4
            for (int k = 0; k < parts; ++k) {
                const float w = expf(__ldcg(lse_part + k * stride + m) - mx);
                const float *src = o_part + (k * stride + m) * D;
                if constexpr (kPer == 4) {
                    const float4 x = __ldcg(reinterpret_cast<const float4 *>(src));
                    acc[0] += w * x.x; acc[1] += w * x.y; acc[2] += w * x.z; acc[3] += w * x.w;
                } else {
                    const float2 x = __ldcg(reinterpret_cast<const float2 *>(src));
                    acc[0] += w * x.x; acc[1] += w * x.y;
                }
            }
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        __nv_bfloat16 *dst = p.o + (static_cast<size_t>(r_abs) * p.Hq + h) * D + kPer * lane;
        if constexpr (kPer == 4) {
            uint2 w;
            w.x = pack_bf16(acc[0] * inv, acc[1] * inv);
            w.y = pack_bf16(acc[2] * inv, acc[3] * inv);
            *reinterpret_cast<uint2 *>(dst) = w;
        } else {
            *reinterpret_cast<uint32_t *>(dst) = pack_bf16(acc[0] * inv, acc[1] * inv);
        }
        if (lane == 0) p.lse[static_cast<size_t>(h) * p.N + r_abs] = den > 0.f ? mx + logf(den) : -INFINITY;
    }
}

}  // namespace

cudaError_t launch_fwd(int D, const CUtensorMap &tm_q, const KvMaps &kv, const FwdParams &p, int n_items,
                       int n_split, cudaStream_t stream, void *const *trace) {
    trace_record(trace, 0, stream);
    cudaError_t err = cudaSuccess;
    if (D == 64) {
        constexpr int smem = FwdLayout<64>::bytes;
        err = cudaFuncSetAttribute(fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        fwd_kernel<64><<<n_items * p.Hkv, kThreads, smem, stream>>>(tm_q, kv.k_piece, kv.v_piece, kv.k_half,
                                                                   kv.v_half, p);
        err = cudaGetLastError();
    } else {
        err = launch_fwd_pair(tm_q, kv, p, n_items, stream);
    }
    if (err == cudaSuccess && n_split > 0) {
        const dim3 grid(n_split, p.Hkv, 8);
        if (D == 64) fwd_combine_kernel<64><<<grid, 256, 0, stream>>>(p);
        else fwd_combine_kernel<128><<<grid, 256, 0, stream>>>(p);
        err = cudaGetLastError();
    }
    trace_record(trace, 1, stream);
    return err;
}

}  // namespace treeattn
