// Forward epilogues shared by the single-SM and the CTA-pair forward: one thread writes its
// query row (one TMEM lane) of O, read from TMEM 32 columns at a time.
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace treeattn {

// A whole block: O scaled by inv = 1 / l, in bf16, and lse.
template <int D>
__device__ __forceinline__ void store_o_row(uint32_t tO, bool valid, float inv, __nv_bfloat16 *orow, float *lse_dst,
                                            float lse) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + c * 32, v);
        tmem_wait_ld();
        if (valid) {
            uint4 w[4];
            uint32_t *wp = reinterpret_cast<uint32_t *>(w);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                wp[i] = pack_bf16(__uint_as_float(v[2 * i]) * inv, __uint_as_float(v[2 * i + 1]) * inv);
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = w[i];
        }
    }
    if (valid) *lse_dst = lse;
}

// One part of a split block (split-KV): the part's normalised O in fp32 and its lse, at MMA row
// m_flat of partial slot `slot` (layout of FwdParams::partial).
template <int D>
__device__ __forceinline__ void store_partial_row(uint32_t tO, bool valid, float inv, const FwdParams &p, int slot,
                                                  int g, int m_flat, float lse) {
    const size_t row = (static_cast<size_t>(slot) * p.Hkv + g) * 256 + m_flat;
    float4 *dst = reinterpret_cast<float4 *>(p.partial + row * D);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tO + c * 32, v);
        tmem_wait_ld();
        if (valid) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                dst[8 * c + i] = make_float4(__uint_as_float(v[4 * i]) * inv, __uint_as_float(v[4 * i + 1]) * inv,
                                             __uint_as_float(v[4 * i + 2]) * inv, __uint_as_float(v[4 * i + 3]) * inv);
        }
    }
    if (valid) p.partial[static_cast<size_t>(p.n_slots) * p.Hkv * 256 * D + row] = lse;
}

}  // namespace treeattn
