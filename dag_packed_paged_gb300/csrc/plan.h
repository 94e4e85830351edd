// Internal: the plan object shared by the host planner (plan.cpp) and the launch code.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/treeattn.h"

namespace treeattn {

// Names one call of the library on a profiler's timeline (Nsight Systems, ncu's NVTX filter).
// NVTX v3 is header-only: with no tool attached a push/pop costs a few nanoseconds.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

constexpr int kTileRows = 128;       // key rows per tile (the N of S = Q K^T, the K of O = P V)
constexpr int kBlockMRows = 256;     // query (row, head) pairs per query block: two 128-lane tiles

constexpr int32_t kEntryCausal = 1;  // mask key rows above the query row
constexpr int32_t kEntryPartial = 2; // the entry covers only part of its tile

// Packed key tiles of the query-major kernels (forward, dQ): a tile is 4 slots of 32 key rows,
// each slot one 32-row-aligned piece of the strip that the block sees in part or in full, so
// that the pieces of several visible intervals share one 128-row tile.  Record (8 x int32):
//   [0..3] piece index (first row / 32) of slot k, -1 for an empty slot
//   [4]    slots 0, 1: lo | hi << 6 | lo << 12 | hi << 18   (visible rows [lo, hi) of the piece)
//   [5]    slots 2, 3, the same
//   [6]    flags: kPackMask (some slot needs masking), kPackCausal << k (slot k: mask rows
//          above the query row), kPackHalf64 << h (slots 2h, 2h+1 are one 64-row-aligned run,
//          loaded as one box)
//   [7]    0
constexpr int kPieceRows = 32;
constexpr int kPackInts = 8;
constexpr int32_t kPackMask = 1;
constexpr int32_t kPackCausal = 2;    // bits 1..4
constexpr int32_t kPackHalf64 = 32;   // bits 5..6

void set_error(const std::string &msg);

struct HostPlan {
    ta_config cfg{};
    int G = 1;               // query heads per KV head
    int block_rows = 0;      // query rows per block = 256 / G
    float scale = 0.f;
    int64_t N = 0;
    int64_t n_logical_pages = 0;

    std::vector<int32_t> pos_ids;
    std::vector<int32_t> blocks;      // 4 per block: first row, rows, entry begin, entry end
    std::vector<int64_t> blk_iv_ptr;  // n_blocks + 1
    std::vector<int32_t> iv_lo, iv_hi;
    std::vector<int32_t> diag;        // 2 per block
    std::vector<int32_t> entries;     // 4 per entry: tile, lo, hi, flags
    std::vector<int32_t> t_entries;   // 4 per entry: block, lo, hi, flags (tile-major)
    std::vector<int32_t> chunks;      // 4 per chunk: tile, t_entry begin, end, slot (-1: direct)
    std::vector<int32_t> fwd_order;   // block ids, longest first
    std::vector<int32_t> reduce;      // 4 per split tile: tile, first slot, slots, 0
    std::vector<int32_t> page_table;
    std::vector<int32_t> tile_rows;   // per key tile, per page: TMA row of the page in the pool
                                      // (pool rows; num_pages * P past the strip: zero fill)
    std::vector<int32_t> t_info;      // per tile-major entry: block << 2 | flags, first row, lo, hi
    std::vector<int32_t> ftiles;      // packed key tiles of the query-major kernels (kPackInts each)
    std::vector<int64_t> fblk_ptr;    // n_blocks + 1: block b's packed tiles [fblk_ptr[b], fblk_ptr[b+1])
    // forward work items (split-KV): 4 per item, longest first: block, first packed tile, end
    // tile, partial slot (-1: the item is the whole block and writes O and lse itself)
    std::vector<int32_t> fwd_items;
    std::vector<int32_t> fwd_combine; // 4 per split block: block, first slot, parts, 0
    int64_t n_fwd_slots = 0;          // partial results of split blocks (one per part)
    int64_t fwd_split_cap = 0;        // packed tiles per forward item at most
    int64_t n_segments = 0;
    int64_t n_partial_slots = 0;
    int64_t chunk_cap = 0;            // entries per dK/dV chunk at most
    int32_t num_sms = 0;              // SM count the cap was derived from
    int64_t pairs = 0;
    double plan_ms = 0.0;
};

constexpr int kDefaultSms = 152;     // GB300; used when neither the config nor a device gives one

// Builds the host plan; returns TA_OK or an error code (message via set_error).  device_sms:
// the SM count of the device the plan is for (0: none, e.g. a host-only plan).
int build_host_plan(const ta_branch *branches, int32_t n_branches, const ta_mount *mounts,
                    int32_t n_mounts, const int32_t *page_table, int64_t n_logical_pages,
                    const ta_config *config, int device_sms, HostPlan &out);

}  // namespace treeattn

struct ta_plan {
    treeattn::HostPlan host;
    // device copies (one allocation)
    void *d_buf = nullptr;
    size_t d_bytes = 0;
    const int32_t *d_blocks = nullptr;
    const int32_t *d_entries = nullptr;
    const int32_t *d_t_entries = nullptr;
    const int32_t *d_chunks = nullptr;
    const int32_t *d_fwd_order = nullptr;
    const int32_t *d_reduce = nullptr;
    const int32_t *d_page_table = nullptr;
    const int32_t *d_tile_rows = nullptr;
    const int32_t *d_t_info = nullptr;
    const int32_t *d_fwd_items = nullptr;
    const int32_t *d_fwd_combine = nullptr;
    float *d_fwd_partial = nullptr;   // [slots][Hkv][256][D] O then [slots][Hkv][256] lse (own allocation)
    const int32_t *d_pos_ids = nullptr;   // Eq. 2 position of every compact row
    const int32_t *d_ftiles = nullptr;    // packed key tiles (forward, dQ)
    const int32_t *d_fblk = nullptr;      // per block: first packed tile, end (2 x int32)
    int32_t *d_status = nullptr;      // bounded-wait status words (zeroed at plan time)
    size_t ws_table_bytes = 0;        // workspace: per (KV head, block, query tile) 128 lse*log2e + 128 delta
    size_t ws_bytes = 0;              // total bwd workspace
    int device = -1;                  // -1: host-only plan
    bool stream_ordered = false;      // TA_PLAN_STREAM_ORDERED: d_buf is freed with cudaFreeAsync on `stream`
    void *stream = nullptr;           // cudaStream_t given to tree_attn_plan
    void *trace[7] = {nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr};  // cudaEvent_t
};
