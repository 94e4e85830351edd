// Compact-to-semantic log-probabilities and their gradient.
//
// HARTS (arXiv 2608.28158) Section 4: the LM-head logit row z_c of a compact row c serves every
// semantic position s with m(s) = c.  Eq. 17: lambda_s = z_{m(s), y_s} - log sum_v exp z_{m(s), v},
// with the vocabulary-wide maximum and sum-exp formed once per compact row; Eq. 19-20: backward
// accumulates the contributions of all positions of a row into that row,
//   dz_c = sum_{s: m(s) = c} g_s (e_{y_s} - softmax(z_c)) = -G_c softmax(z_c) + sum_s g_s e_{y_s},
// G_c = sum_{s: m(s) = c} g_s.  Nothing of size S x V is formed.
//
// HBM-bound (every logit read once forward, read once and written once backward): one CTA per
// compact row streams the row in 16-byte vectors; the exponentials use base 2 and the paired
// fp32 instructions, so the instruction and MUFU work stays well under the memory time.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

constexpr int kLpThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void unpack8(const uint4 &x, float (&t)[8]) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        t[2 * k] = __uint_as_float(w[k] << 16);
        t[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
}

// (m, s): s = sum of 2^(t - m) over the values seen, m their maximum (base-2 scaled logits)
__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
    const float mm = fmaxf(m, m2);
    if (mm == -INFINITY) return;
    s = (m == -INFINITY ? 0.f : s * ex2(m - mm)) + (m2 == -INFINITY ? 0.f : s2 * ex2(m2 - mm));
    m = mm;
}

// One CTA per compact row: lse_c = ln sum_v exp z_{c,v}.
__global__ void __launch_bounds__(kLpThreads) lse_kernel(const __nv_bfloat16 *__restrict__ z, int64_t V,
                                                         float *__restrict__ lse) {
    const int64_t c = blockIdx.x;
    const uint4 *row = reinterpret_cast<const uint4 *>(z + c * V);
    const int64_t n8 = V / 8;
    const uint64_t l2 = f2_pack(kLog2e, kLog2e);
    float m = -INFINITY, s = 0.f;
    for (int64_t i = threadIdx.x; i < n8; i += kLpThreads) {
        float t[8];
        unpack8(__ldcs(row + i), t);                  // read once: streaming
        float u[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) f2_unpack(f2_mul(f2_pack(t[2 * k], t[2 * k + 1]), l2), u[2 * k], u[2 * k + 1]);
        const float cm = fmaxf(max3(u[0], u[1], u[2]), max3(max3(u[3], u[4], u[5]), u[6], u[7]));
        const float mm = fmaxf(m, cm);
        const uint64_t nm = f2_pack(-mm, -mm);
        uint64_t acc = 0ull;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float a, b;
            f2_unpack(f2_add(f2_pack(u[2 * k], u[2 * k + 1]), nm), a, b);
            acc = f2_add(acc, f2_pack(ex2(a), ex2(b)));
        }
        float a0, a1;
        f2_unpack(acc, a0, a1);
        s = (m == -INFINITY ? 0.f : s * ex2(m - mm)) + (a0 + a1);
        m = mm;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
    __shared__ float sm[kLpThreads / 32], ss[kLpThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) { sm[warp] = m; ss[warp] = s; }
    __syncthreads();
    if (warp == 0) {
        m = lane < kLpThreads / 32 ? sm[lane] : -INFINITY;
        s = lane < kLpThreads / 32 ? ss[lane] : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) lse_merge(m, s, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, s, o));
        if (lane == 0) lse[c] = (m + log2f(s)) * 0.69314718055994531f;
    }
}

// lambda_s = z[m(s), y_s] - lse[m(s)] for every semantic position, in the caller's order;
// a row or target out of range gives NaN.
__global__ void __launch_bounds__(kLpThreads) gather_kernel(const __nv_bfloat16 *__restrict__ z, int64_t C, int64_t V,
                                                            const float *__restrict__ lse, const int64_t *__restrict__ pos_row,
                                                            const int32_t *__restrict__ pos_target, int64_t S,
                                                            float *__restrict__ out) {
    const int64_t s = static_cast<int64_t>(blockIdx.x) * kLpThreads + threadIdx.x;
    if (s >= S) return;
    const int64_t r = pos_row[s];
    const int32_t y = pos_target[s];
    if (r < 0 || r >= C || y < 0 || y >= V) {
        out[s] = __int_as_float(0x7FC00000);
        return;
    }
    out[s] = __bfloat162float(z[r * V + y]) - lse[r];
}

// One CTA per compact row: dz_c = -G_c softmax(z_c) everywhere, then every distinct target y of
// the row recomputed as -G_c p_y + (sum of g over the row's positions with target y) -- one
// rounding to bf16 per element, summation order fixed (deterministic).
// row_ptr / row_pos: the row's positions, sorted by target (tree_attn_logprob_index).
__global__ void __launch_bounds__(kLpThreads) dlogits_kernel(const __nv_bfloat16 *__restrict__ z, int64_t V,
                                                             const float *__restrict__ lse,
                                                             const int64_t *__restrict__ row_ptr,
                                                             const int64_t *__restrict__ row_pos,
                                                             const int32_t *__restrict__ pos_target,
                                                             const float *__restrict__ g,
                                                             __nv_bfloat16 *__restrict__ dz) {
    const int64_t c = blockIdx.x;
    const int64_t p0 = row_ptr[c], p1 = row_ptr[c + 1];
    // G_c: fixed-order block sum
    float part = 0.f;
    for (int64_t i = p0 + threadIdx.x; i < p1; i += kLpThreads) part += g[row_pos[i]];
#pragma unroll
    for (int o = 16; o; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    __shared__ float red[kLpThreads / 32];
    __shared__ float Gs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < kLpThreads / 32; ++w) t += red[w];
        Gs = t;
    }
    __syncthreads();
    const float G = Gs;
    const float lse2 = lse[c] * kLog2e;
    const uint4 *row = reinterpret_cast<const uint4 *>(z + c * V);
    uint4 *drow = reinterpret_cast<uint4 *>(dz + c * V);
    const int64_t n8 = V / 8;
    const uint64_t l2 = f2_pack(kLog2e, kLog2e), nl = f2_pack(-lse2, -lse2), ng = f2_pack(-G, -G);
    for (int64_t i = threadIdx.x; i < n8; i += kLpThreads) {
        float t[8];
        unpack8(__ldcs(row + i), t);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float a, b;
            f2_unpack(f2_fma(f2_pack(t[2 * k], t[2 * k + 1]), l2, nl), a, b);
            f2_unpack(f2_mul(f2_pack(ex2(a), ex2(b)), ng), a, b);
            w[k] = pack_bf16(a, b);
        }
        __stcs(drow + i, make_uint4(w[0], w[1], w[2], w[3]));
    }
    if (p1 == p0) return;
    __syncthreads();                                   // the dense values are written
    for (int64_t i = p0 + threadIdx.x; i < p1; i += kLpThreads) {
        const int32_t y = pos_target[row_pos[i]];
        if (i > p0 && pos_target[row_pos[i - 1]] == y) continue;     // not the first of its run
        float gy = 0.f;
        for (int64_t k = i; k < p1 && pos_target[row_pos[k]] == y; ++k) gy += g[row_pos[k]];
        const float py = ex2(fmaf(__bfloat162float(z[c * V + y]), kLog2e, -lse2));
        dz[c * V + y] = __float2bfloat16_rn(fmaf(-G, py, gy));
    }
}

}  // namespace

cudaError_t launch_logprob_fwd(const __nv_bfloat16 *z, int64_t C, int64_t V, const int64_t *pos_row,
                               const int32_t *pos_target, int64_t S, float *lse, float *logprob, cudaStream_t stream) {
    if (C > 0) {
        lse_kernel<<<static_cast<unsigned>(C), kLpThreads, 0, stream>>>(z, V, lse);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (S > 0) gather_kernel<<<static_cast<unsigned>((S + kLpThreads - 1) / kLpThreads), kLpThreads, 0, stream>>>(
        z, C, V, lse, pos_row, pos_target, S, logprob);
    return cudaGetLastError();
}

cudaError_t launch_logprob_bwd(const __nv_bfloat16 *z, int64_t C, int64_t V, const float *lse, const int64_t *row_ptr,
                               const int64_t *row_pos, const int32_t *pos_target, const float *g, __nv_bfloat16 *dz,
                               cudaStream_t stream) {
    if (C == 0) return cudaSuccess;
    dlogits_kernel<<<static_cast<unsigned>(C), kLpThreads, 0, stream>>>(z, V, lse, row_ptr, row_pos, pos_target, g, dz);
    return cudaGetLastError();
}

}  // namespace treeattn
