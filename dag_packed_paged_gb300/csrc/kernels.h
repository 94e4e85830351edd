// Internal: kernel parameter blocks and launchers (implemented in the .cu files).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace treeattn {

struct FwdParams {
    const int32_t *blocks;      // 4 per query block: first row, rows, entry begin, entry end
    const int32_t *ftiles;      // packed key tiles, kPackInts each (plan.h)
    const int32_t *items;       // forward work items, 4 each: block, first tile, end tile, slot (-1: whole block)
    const int32_t *combine;     // split blocks, 4 each: block, first slot, parts, 0
    float *partial;             // split parts' O [slots][Hkv][256][D], then lse [slots][Hkv][256]
    int32_t n_slots;
    const int32_t *page_table;  // logical page -> pool page
    const int32_t *tile_rows;   // per key tile, per page: pool row of the page (TMA y)
    int32_t n_logical_pages;
    int32_t num_pages;
    int32_t page_size;
    int32_t N;
    int32_t Hq, Hkv, G, R;      // R = query rows per block
    float scale_log2;           // softmax scale * log2(e)
    __nv_bfloat16 *o;           // [N, Hq, D]
    float *lse;                 // [Hq, N]
    int *status;
};

struct BwdParams {
    const int32_t *blocks;
    const int32_t *ftiles;      // packed key tiles of the dQ kernel (as the forward's)
    const int32_t *fblk;
    const int32_t *t_entries;   // 4 per entry, key-tile-major: block, lo, hi, flags
    const int32_t *chunks;      // 4 per chunk: tile, t_entry begin, end, partial slot
    const int32_t *reduce;      // 4 per split tile: tile, first slot, slots, 0
    const int32_t *order;
    const int32_t *page_table;
    const int32_t *tile_rows;
    const int32_t *t_info;      // per tile-major entry: block << 2 | flags, first row, lo, hi
    int32_t n_logical_pages;
    int32_t num_pages;
    int32_t page_size;
    int32_t N;
    int32_t Hq, Hkv, G, R;
    float scale;                // softmax scale
    float scale_log2;
    const __nv_bfloat16 *q;     // [N, Hq, D]
    const __nv_bfloat16 *k_pool;  // [num_pages, P, Hkv, D]
    const __nv_bfloat16 *v_pool;
    const __nv_bfloat16 *o;     // [N, Hq, D]
    const __nv_bfloat16 *d_o;   // [N, Hq, D]
    const float *lse;           // [Hq, N]
    float *utab;                // [Hkv][n_blocks][2 query tiles][128 lse*log2e | 128 delta] (workspace)
    int32_t n_blocks;
    float *dq;                  // [N, Hq, D]
    float *dk_pool;             // [num_pages, P, Hkv, D]
    float *dv_pool;
    float *partials;            // [slots, Hkv, 2, 128, D] (workspace)
    int *status;
};

// `trace`: NULL, or cudaEvent_t handles (entries may be NULL) recorded around the launches.
// Rotary position embedding of Q and the K pool in place (see rope.cu).
struct RopeParams {
    __nv_bfloat16 *q;           // [N, Hq, D]
    __nv_bfloat16 *k_pool;      // [num_pages * P, Hkv, D]
    const int32_t *pos_ids;     // [N] Eq. 2 positions
    const int32_t *page_table;  // logical page -> pool page
    int64_t N;
    int32_t Hq, Hkv, page_size;
    int64_t n_logical_pages, num_pages;   // bounds of the page table and the pool (TA_DEBUG checks)
    int *status;                // status word of the plan (TA_DEBUG checks)
    double inv_freq[64];        // theta_base^(-2i/D), i < D/2
};

cudaError_t launch_rope(int D, const RopeParams &p, cudaStream_t stream);

// Compact-to-semantic log-probabilities (see logprob.cu).
cudaError_t launch_logprob_fwd(const __nv_bfloat16 *z, int64_t C, int64_t V, const int64_t *pos_row,
                               const int32_t *pos_target, int64_t S, float *lse, float *logprob, cudaStream_t stream);
cudaError_t launch_logprob_bwd(const __nv_bfloat16 *z, int64_t C, int64_t V, const float *lse, const int64_t *row_ptr,
                               const int64_t *row_pos, const int32_t *pos_target, const float *g, __nv_bfloat16 *dz,
                               cudaStream_t stream);

// Tensor maps of the K/V pools: `page` boxes of one page (the dK/dV kernel's aligned tiles),
// `piece` boxes of min(page, 32) rows and `half` boxes of 64 rows (packed tiles of the forward
// and dQ; `half` is only used when pages hold >= 64 rows).
struct KvMaps {
    CUtensorMap k_page, v_page, k_piece, v_piece, k_half, v_half;
};

// The forward over n_items work items, then (n_split > 0) the combine of the split blocks.
cudaError_t launch_fwd(int D, const CUtensorMap &tm_q, const KvMaps &kv, const FwdParams &p, int n_items,
                       int n_split, cudaStream_t stream, void *const *trace);

// The forward on CTA pairs (head dim 128; see fwd_pair.cu); launch_fwd dispatches to it.
cudaError_t launch_fwd_pair(const CUtensorMap &tm_q, const KvMaps &kv, const FwdParams &p, int n_items,
                            cudaStream_t stream);

cudaError_t launch_bwd(int D, const CUtensorMap &tm_q, const KvMaps &kv, const CUtensorMap &tm_do,
                       const BwdParams &p, int n_blocks, int n_chunks, int n_reduce, cudaStream_t stream,
                       void *const *trace);

inline void trace_record(void *const *trace, int i, cudaStream_t s) {
    if (trace && trace[i]) cudaEventRecord(static_cast<cudaEvent_t>(trace[i]), s);
}

}  // namespace treeattn
