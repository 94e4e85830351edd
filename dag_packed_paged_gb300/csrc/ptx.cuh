// Thin inline-PTX wrappers for sm_103a: mbarrier, TMA (cp.async.bulk.tensor), tcgen05
// (TMEM allocation, MMA, commit, loads/stores, fences).  Every wait is bounded: it gives up
// after kWaitNs of wall time (read from %globaltimer), raises the CTA's abort flag and
// records a status bit, so that a lost arrival can never hang the GPU.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>

#include "plan.h"

namespace treeattn {

constexpr unsigned long long kWaitNs = 2000000000ull;   // 2 s per wait, then give up

// status bits (device word, read by tree_attn_check)
constexpr int kStatusTimeout = 1;
constexpr int kStatusMisaligned = 2;   // dynamic shared memory not 1024-byte aligned: kernel did nothing
constexpr int kStatusBounds = 4;       // TA_DEBUG builds: a plan index or TMA row was out of range (access skipped)

// TA_DEBUG builds check every plan-derived page index, pool row and output row on the device
// before using it: an index out of [lo, hi) raises kStatusBounds and the caller skips the access
// (a load reads the zero-filled row past the pool instead).  Release builds compile the checks
// away and always return true.
__device__ __forceinline__ bool debug_in_range(long long v, long long lo, long long hi, int *status) {
#ifdef TA_DEBUG
    if (v < lo || v >= hi) {
        atomicOr(status, kStatusBounds);
        return false;
    }
#else
    (void)v;
    (void)lo;
    (void)hi;
    (void)status;
#endif
    return true;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false (and sets
// *abort and the status word) if it did not complete in kWaitNs, or -- when `abort` is not
// NULL -- as soon as another thread of the CTA has aborted.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, volatile int *abort, int *status,
                                              unsigned long long limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (abort != nullptr && *abort) return false;
            if (globaltimer() - t0 > limit_ns) {
                if (abort != nullptr) *abort = 1;
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort, int *status) {
    return mbar_wait_for(bar, parity, abort, status, kWaitNs);
}

// ------------------------------------------------------------------------------ CTA pairs
// A cluster of two CTAs on neighbouring SMs sharing one tcgen05 MMA (cta_group::2).  Barrier
// addresses of the other CTA are shared::cluster addresses obtained with mapa.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the variable at shared::cta address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier of any CTA of the cluster (default release semantics at CTA scope).
// The barriers carry the pair's hand-offs of TMEM and of TMA-written shared memory, whose
// ordering comes from the tcgen05 fences and the transaction counts; a cluster-scope release
// here costs over a thousand cycles per arrival on the critical path (measured) and orders
// nothing the kernels need.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// All threads of both CTAs: arrive and wait (orders shared-memory and barrier initialisation
// before any access from the other CTA, and keeps a CTA resident until its peer is done).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2D tiled load of one box into shared memory; completion is signalled on `bar` as
// transaction bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int32_t x, int32_t y,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 4D tiled load of one box into shared memory; completion is signalled on `bar` as
// transaction bytes.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, int32_t x, int32_t y, int32_t z,
                                            int32_t w, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

// Untiled bulk copy global -> shared (addresses 16-byte aligned, size a multiple of 16),
// completion signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// 2D tiled load into this CTA's shared memory whose completion is signalled on an mbarrier of
// either CTA of the pair (`bar_cluster`, a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const void *tmap, int32_t x, int32_t y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// ------------------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Pair forms (cta_group::2): one warp of each CTA allocates and frees together; one thread of
// the pair issues an MMA of M = 256 whose A rows, D lanes and half of B come from each CTA (the
// same shared-memory and TMEM addresses in both).
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_ss_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive (once) on the mbarrier at shared::cluster address `bar_cluster` (this CTA's or the
// peer's) when every pair MMA issued so far by this thread is done.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar_cluster) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar_cluster)
                 : "memory");
}

// Warp-wide forms: every lane of the issuing warp executes them (so addresses and descriptors
// stay warp-uniform), but only the lane with `issue` set issues the instruction.
__device__ __forceinline__ void mma_ss_if(uint32_t issue, uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
        : "memory");
}

__device__ __forceinline__ void mma_ts_if(uint32_t issue, uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "setp.ne.b32 q, %5, 0;\n\t"
        "@q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(issue)
        : "memory");
}

__device__ __forceinline__ void mma_commit_if(uint32_t issue, uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t"
        "setp.ne.b32 q, %1, 0;\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar),
        "r"(issue)
        : "memory");
}

// Bounded wait executed by a whole warp; the result is the same in every lane.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort, int *status) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, status));
}

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// tcgen05.wait::ld that also names the 32 loaded registers, so that no use of them can be
// placed above the wait by the compiler (the load writes them asynchronously)
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane (base lane + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
        "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
        "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading / stride byte offsets,
// descriptor version 1, 128-byte swizzle.  Tiles are stored as 128-byte rows in 8-row
// (1024-byte) swizzle atoms, each atom 1024-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;     // version
    d |= static_cast<uint64_t>(2) << 61;     // 128B swizzle
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
// a_mn / b_mn: operand stored MN-major (1) or K-major (0).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4)                        // D format: f32
           | (1u << 7)                      // A format: bf16
           | (1u << 10)                     // B format: bf16
           | (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
           (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Warp-cooperative prefetch of key-tile entries: lane i holds entry (base + i) of the list and
// the pool rows of its tile's pages, so one round trip serves 32 entries; the producer loop
// reads them with shuffles.  pages_per_tile <= 8.
struct EntryFeed {
    int4 e;
    int y[8];
};

__device__ __forceinline__ void feed_fill(EntryFeed &f, int base, int n, const int4 *entries,
                                          const int32_t *tile_rows, int ppt, int lane) {
    const int j = base + lane;
    if (j < n) {
        f.e = __ldg(entries + j);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (i < ppt) f.y[i] = __ldg(tile_rows + f.e.x * ppt + i);
    }
}

// TMA loads of one key tile (128 rows, `ppt` pages) of KV head g into a 128-row smem tile:
// page i goes to rows [i*P, (i+1)*P), each 64-column chunk c to its own 16 KB half.
__device__ __forceinline__ void tma_kv_tile(uint32_t dst, const void *tm, const int (&y)[8], int ppt, int P, int g,
                                            int D, uint32_t bar) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
        if (i < ppt)
            for (int c = 0; c < D / 64; ++c)
                tma_load_2d(dst + c * (128 * 128) + i * P * 128, tm, g * D + c * 64, y[i], bar);
}

// Warp-cooperative prefetch of packed key tiles (the forward's and dQ's tile lists): lane i
// holds the record of tile (base + i) and the TMA row of every box it loads, so one round trip
// serves 32 tiles.  A tile has 4 slots of 32 key rows; slot k's rows are box y[2k] (and, for
// 16-row pages, y[2k + 1]).  An empty slot, or the second 16-row half of a piece past the last
// logical page, reads row `oob_row` (past the pool: TMA fills zeros).
struct PackFeed {
    int4 a;      // slot pieces (first row / 32), -1 empty
    int4 b;      // slot row ranges and flags
    int y[8];
};

__device__ __forceinline__ void pack_feed_fill(PackFeed &f, int base, int n, const int4 *tiles,
                                               const int32_t *page_table, int n_logical, int P, int oob_row,
                                               int lane, int *status) {
    const int j = base + lane;
    if (j < n) {
        f.a = __ldg(tiles + 2 * j);
        f.b = __ldg(tiles + 2 * j + 1);
        const int pc[4] = {f.a.x, f.a.y, f.a.z, f.a.w};
#ifdef TA_DEBUG
        // a piece's logical page must exist and map into the pool; otherwise its rows read zeros
        const int num_pages = oob_row / P;
        auto row_of = [&](int li, int off) {
            if (!debug_in_range(li, 0, n_logical, status)) return oob_row;
            const int pg = __ldg(page_table + li);
            return debug_in_range(pg, 0, num_pages, status) ? pg * P + off : oob_row;
        };
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int p = pc[k];
            if (P >= 32) {
                f.y[2 * k] = p >= 0 ? row_of((32 * p) / P, (32 * p) % P) : oob_row;
                f.y[2 * k + 1] = oob_row;
            } else {
                f.y[2 * k] = p >= 0 ? row_of(2 * p, 0) : oob_row;
                f.y[2 * k + 1] = (p >= 0 && 2 * p + 1 < n_logical) ? row_of(2 * p + 1, 0) : oob_row;
            }
        }
#else
        (void)status;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int p = pc[k];
            if (P >= 32) {
                f.y[2 * k] = p >= 0 ? __ldg(page_table + (32 * p) / P) * P + (32 * p) % P : oob_row;
                f.y[2 * k + 1] = oob_row;
            } else {   // 16-row pages: a piece is two pages
                f.y[2 * k] = p >= 0 ? __ldg(page_table + 2 * p) * P : oob_row;
                f.y[2 * k + 1] = (p >= 0 && 2 * p + 1 < n_logical) ? __ldg(page_table + 2 * p + 1) * P : oob_row;
            }
        }
#endif
    }
}

// TMA loads of one packed key tile of KV head g into a 128-row smem tile (slot k at rows
// [32k, 32k + 32), each 64-column chunk c in its own 16 KB part).  `tm_s`: boxes of
// min(P, 32) rows; `tm_h`: boxes of 64 rows, used for a half whose two slots are one
// 64-row-aligned run (flag bit kPackHalf64 << h; pages of >= 64 rows).  Always 128 * D * 2
// bytes in total.
__device__ __forceinline__ void tma_packed_tile(uint32_t dst, const void *tm_s, const void *tm_h, const int (&y)[8],
                                                int flags, int P, int g, int D, uint32_t bar) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        if (flags & (kPackHalf64 << h)) {
            for (int c = 0; c < D / 64; ++c)
                tma_load_2d(dst + c * (128 * 128) + h * 64 * 128, tm_h, g * D + c * 64, y[4 * h], bar);
        } else {
#pragma unroll
            for (int s = 0; s < 2; ++s) {
                const int k = 2 * h + s;
                for (int c = 0; c < D / 64; ++c) {
                    tma_load_2d(dst + c * (128 * 128) + k * 32 * 128, tm_s, g * D + c * 64, y[2 * k], bar);
                    if (P < 32)
                        tma_load_2d(dst + c * (128 * 128) + k * 32 * 128 + 16 * 128, tm_s, g * D + c * 64,
                                    y[2 * k + 1], bar);
                }
            }
        }
    }
}

// Visible columns [lo, hi) of slot k of a packed tile for query row r: the slot's row range,
// cut above r when the slot is causal.  rec_a: slot pieces, rec_b: ranges and flags.
__device__ __forceinline__ void pack_slot_range(const int4 &rec_a, const int4 &rec_b, int k, int r, int &lo,
                                                int &hi) {
    const uint32_t w = static_cast<uint32_t>(k < 2 ? rec_b.x : rec_b.y) >> (12 * (k & 1));
    lo = static_cast<int>(w & 63u);
    hi = static_cast<int>((w >> 6) & 63u);
    if (rec_b.z & (kPackCausal << k)) {
        const int p = k == 0 ? rec_a.x : k == 1 ? rec_a.y : k == 2 ? rec_a.z : rec_a.w;
        hi = min(hi, r + 1 - 32 * p);
    }
}

// Per-warp broadcast of a list of int4 records (plan entries): lane i holds record (base + i);
// one coalesced load serves 32 iterations and every iteration reads its record by shuffle,
// so no global-memory latency sits on the per-iteration critical path.
struct WarpRecords {
    int4 mine = make_int4(0, 0, 0, 0);
    __device__ __forceinline__ int4 get(const int4 *recs, int i, int n, int lane) {
        if ((i & 31) == 0 && i + lane < n) mine = __ldg(recs + i + lane);
        const int src = i & 31;
        return make_int4(__shfl_sync(0xffffffffu, mine.x, src), __shfl_sync(0xffffffffu, mine.y, src),
                         __shfl_sync(0xffffffffu, mine.z, src), __shfl_sync(0xffffffffu, mine.w, src));
    }
};

// The same for packed key tiles (two int4 per record).
struct WarpPackRecords {
    int4 a = make_int4(0, 0, 0, 0), b = make_int4(0, 0, 0, 0);
    __device__ __forceinline__ void get(const int4 *tiles, int i, int n, int lane, int4 &ra, int4 &rb) {
        if ((i & 31) == 0 && i + lane < n) {
            a = __ldg(tiles + 2 * (i + lane));
            b = __ldg(tiles + 2 * (i + lane) + 1);
        }
        const int src = i & 31;
        ra = make_int4(__shfl_sync(0xffffffffu, a.x, src), __shfl_sync(0xffffffffu, a.y, src),
                       __shfl_sync(0xffffffffu, a.z, src), __shfl_sync(0xffffffffu, a.w, src));
        rb = make_int4(__shfl_sync(0xffffffffu, b.x, src), __shfl_sync(0xffffffffu, b.y, src),
                       __shfl_sync(0xffffffffu, b.z, src), 0);
    }
};

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two-lane fp32 arithmetic: each lane is rounded exactly like the scalar instruction.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace treeattn
