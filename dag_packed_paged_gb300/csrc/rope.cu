// Rotary position embedding on the compact rows, from the Eq. 2 position ids.
//
// Octopus (arXiv 2611.06956) Section 3.2: attention scores depend on positions only through
// the rotary phase relation <R_p q, R_s k> = <q, R_{s-p} k> (Eq. 1), so a mounted span keeps
// the positions it was computed at and the reader continues after it (Eq. 2); HARTS
// (arXiv 2608.28158) Section 4.2 applies RoPE once per compact row, before attention.  Here
// x is rotated pairwise -- (x_i, x_{i+D/2}) by the angle p * theta_i with
// theta_i = base^(-2i/D) -- in Q and in the K pool (through the page table), in place.
//
// HBM-bound: every element is read and written once.  One warp per compact row: the D/2
// angles depend on the row's position only, so they are formed once per row and shared by
// all Hq + Hkv heads.  The angle is formed and reduced mod 2 pi in fp64 (positions reach 2^18
// and beyond, where an fp32 product would be off by ~1e-2 rad), the sine and cosine in fp32.
#include "kernels.h"
#include "ptx.cuh"

namespace treeattn {

namespace {

template <int D>
__global__ void __launch_bounds__(256) rope_kernel(const RopeParams p) {
    constexpr int kPairs = D / 2;           // rotation pairs (i, i + D/2)
    constexpr int kTph = kPairs / 2;        // threads per head; each rotates pairs 2j and 2j + 1
    constexpr int kHpw = 32 / kTph;         // heads per warp pass
    const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (r >= p.N) return;                   // uniform per warp
    const int lane = threadIdx.x & 31, j = lane % kTph, hsub = lane / kTph;
    const double pos = static_cast<double>(__ldg(p.pos_ids + r));
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    float c[2], s[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        double a = pos * p.inv_freq[2 * j + u];
        a -= kTwoPi * rint(a * (1.0 / kTwoPi));
        sincosf(static_cast<float>(a), &s[u], &c[u]);
    }
    auto rotate = [&](__nv_bfloat16 *x) {
        __nv_bfloat162 *lo = reinterpret_cast<__nv_bfloat162 *>(x + 2 * j);
        __nv_bfloat162 *hi = reinterpret_cast<__nv_bfloat162 *>(x + kPairs + 2 * j);
        const float2 a = __bfloat1622float2(*lo), b = __bfloat1622float2(*hi);
        *lo = __floats2bfloat162_rn(a.x * c[0] - b.x * s[0], a.y * c[1] - b.y * s[1]);
        *hi = __floats2bfloat162_rn(b.x * c[0] + a.x * s[0], b.y * c[1] + a.y * s[1]);
    };
    __nv_bfloat16 *qrow = p.q + r * p.Hq * D;
    for (int h = hsub; h < p.Hq; h += kHpw) rotate(qrow + h * D);
    if (!debug_in_range(r / p.page_size, 0, p.n_logical_pages, p.status)) return;
    const int pg = __ldg(p.page_table + r / p.page_size);
    if (!debug_in_range(pg, 0, p.num_pages, p.status)) return;
    const int64_t prow = static_cast<int64_t>(pg) * p.page_size + r % p.page_size;
    __nv_bfloat16 *krow = p.k_pool + prow * p.Hkv * D;
    for (int h = hsub; h < p.Hkv; h += kHpw) rotate(krow + h * D);
}

}  // namespace

cudaError_t launch_rope(int D, const RopeParams &p, cudaStream_t stream) {
    if (p.N == 0) return cudaSuccess;
    const int64_t threads = p.N * 32;
    const unsigned grid = static_cast<unsigned>((threads + 255) / 256);
    if (D == 64)
        rope_kernel<64><<<grid, 256, 0, stream>>>(p);
    else
        rope_kernel<128><<<grid, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace treeattn
