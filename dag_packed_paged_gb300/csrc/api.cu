// C ABI of libtreeattn: plan construction and upload, TMA descriptors, kernel launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "kernels.h"
#include "plan.h"
#include "ptx.cuh"

namespace treeattn {

static thread_local std::string g_last_error;

void set_error(const std::string &msg) { g_last_error = msg; }

namespace {

int cuda_fail(cudaError_t e, const char *what) {
    set_error(std::string(what) + ": " + cudaGetErrorString(e));
    return TA_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A 2D bf16 view [rows][inner] with a row stride, boxes of box_inner x box_rows elements,
// 128-byte swizzle (box_inner * 2 == 128), zero fill out of bounds.
int make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows, uint64_t row_stride_bytes,
             uint32_t box_inner, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return TA_ERR_CUDA;
    }
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {row_stride_bytes};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled failed with code " + std::to_string(int(r)));
        return TA_ERR_CUDA;
    }
    return TA_OK;
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Rank-4 view {64 elements, rows, heads, 64-element chunks} of a bf16 [N, H, D] tensor whose
// box is one 128-lane query tile of the backward: QB rows x 128 / QB consecutive heads x all
// D / 64 chunks (QB = min(rows per block, 128)), 128-byte swizzle, zero fill past row N.
int make_qtile_map(CUtensorMap *m, const void *base, uint64_t N, uint32_t H, uint32_t D, uint32_t qb) {
    auto fn = encode_fn();
    if (!fn) {
        set_error("cuTensorMapEncodeTiled is not available from the driver");
        return TA_ERR_CUDA;
    }
    cuuint64_t dims[4] = {64, N, H, D / 64};
    cuuint64_t strides[3] = {uint64_t(H) * D * 2, uint64_t(D) * 2, 128};
    cuuint32_t box[4] = {64, qb, 128 / qb, D / 64};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        set_error("cuTensorMapEncodeTiled (query tile) failed with code " + std::to_string(int(r)));
        return TA_ERR_CUDA;
    }
    return TA_OK;
}

// Tensor maps for Q-like [N, H, D] and the K/V pools: boxes of one page (the dK/dV kernel's
// aligned key tiles), of min(page, 32) rows (one slot of a packed key tile) and of 64 rows (two
// slots that are one aligned run; pages of >= 64 rows only -- otherwise the 32-row map again,
// which is then never used for a 64-row half).
int make_maps(const ta_plan *plan, const void *q, const void *k_pool, const void *v_pool, CUtensorMap *tm_q,
              KvMaps *kv) {
    const HostPlan &h = plan->host;
    const ta_config &c = h.cfg;
    const uint32_t qb = std::min(h.block_rows, 128);
    int rc = make_map(tm_q, q, uint64_t(c.num_q_heads) * c.head_dim, uint64_t(h.N),
                      uint64_t(c.num_q_heads) * c.head_dim * 2, 64, qb);
    if (rc) return rc;
    const uint64_t pool_rows = uint64_t(c.num_pages) * c.page_size;
    const uint64_t inner = uint64_t(c.num_kv_heads) * c.head_dim;
    const uint32_t P = uint32_t(c.page_size), piece = std::min<uint32_t>(P, kPieceRows), half = P >= 64 ? 64 : piece;
    if ((rc = make_map(&kv->k_page, k_pool, inner, pool_rows, inner * 2, 64, P)) ||
        (rc = make_map(&kv->v_page, v_pool, inner, pool_rows, inner * 2, 64, P)) ||
        (rc = make_map(&kv->k_piece, k_pool, inner, pool_rows, inner * 2, 64, piece)) ||
        (rc = make_map(&kv->v_piece, v_pool, inner, pool_rows, inner * 2, 64, piece)) ||
        (rc = make_map(&kv->k_half, k_pool, inner, pool_rows, inner * 2, 64, half)))
        return rc;
    return make_map(&kv->v_half, v_pool, inner, pool_rows, inner * 2, 64, half);
}

// Stream-ordered plan upload (TA_PLAN_STREAM_ORDERED).  A copy from pageable memory is staged
// by the driver in chunks whose DMA is queued on the copy's stream, so on a stream still busy
// with earlier kernels the call blocks the host until they finish.  The upload therefore runs
// on an internal stream that nothing else uses, from pinned staging buffers, and the caller's
// stream waits for it through an event: the host never waits for the caller's earlier work.
// The staging buffers form a ring of kUploadSlots, each with the event of its last copy: a
// copy engine busy with the caller's own large transfers delays a plan's upload, and with a
// single buffer the next plan would wait on the host for it.
constexpr int kUploadSlots = 4;
struct UploadSlot {
    cudaEvent_t done = nullptr;   // recorded after the last copy out of `pinned`
    void *pinned = nullptr;
    size_t cap = 0;
};
struct Uploader {
    std::mutex mu;
    cudaStream_t stream = nullptr;
    UploadSlot slot[kUploadSlots];
    int next = 0;
};
constexpr int kMaxUploadDevices = 64;
Uploader g_uploader[kMaxUploadDevices];

struct Part {
    const void *src;
    size_t bytes;
    size_t off;
};

// Allocates *dst (stream-ordered) and fills it with `parts` (each at its offset, `total` bytes in
// all); work enqueued on `user` after this call is ordered after the copy.
int upload_stream_ordered(int dev, void **dst, const Part *parts, int n_parts, size_t total, cudaStream_t user) {
    if (dev < 0 || dev >= kMaxUploadDevices) {
        set_error("device index beyond the supported range");
        return TA_ERR_UNSUPPORTED;
    }
    Uploader &u = g_uploader[dev];
    std::lock_guard<std::mutex> lock(u.mu);
    cudaError_t e = cudaSuccess;
    if (!u.stream) e = cudaStreamCreateWithFlags(&u.stream, cudaStreamNonBlocking);
    UploadSlot &sl = u.slot[u.next];
    u.next = (u.next + 1) % kUploadSlots;
    if (e == cudaSuccess && !sl.done) e = cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventSynchronize(sl.done);   // this slot's previous copy has left it
    if (e == cudaSuccess && sl.cap < total) {
        if (sl.pinned) cudaFreeHost(sl.pinned);
        sl.pinned = nullptr;
        sl.cap = 0;
        e = cudaMallocHost(&sl.pinned, total);
        if (e == cudaSuccess) sl.cap = total;
    }
    if (e != cudaSuccess) return cuda_fail(e, "plan upload (staging)");
    uint8_t *stage = static_cast<uint8_t *>(sl.pinned);
    for (int i = 0; i < n_parts; ++i) {   // a part without a source (the status words) starts zeroed
        if (parts[i].src && parts[i].bytes) std::memcpy(stage + parts[i].off, parts[i].src, parts[i].bytes);
        else if (!parts[i].src) std::memset(stage + parts[i].off, 0, parts[i].bytes);
    }
    *dst = nullptr;
    e = cudaMallocAsync(dst, total, u.stream);
    if (e != cudaSuccess) {
        *dst = nullptr;
        if (e == cudaErrorMemoryAllocation) {
            set_error("device allocation failed");
            return TA_ERR_NOMEM;
        }
        return cuda_fail(e, "plan upload (allocation)");
    }
    e = cudaMemcpyAsync(*dst, stage, total, cudaMemcpyHostToDevice, u.stream);
    if (e == cudaSuccess) e = cudaEventRecord(sl.done, u.stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(user, sl.done, 0);
    if (e != cudaSuccess) {
        cudaFreeAsync(*dst, u.stream);
        *dst = nullptr;
        return cuda_fail(e, "plan upload");
    }
    return TA_OK;
}

}  // namespace
}  // namespace treeattn

using namespace treeattn;

extern "C" {

const char *tree_attn_last_error(void) { return g_last_error.c_str(); }

int tree_attn_plan(const ta_branch *branches, int32_t n_branches, const ta_mount *mounts, int32_t n_mounts,
                   const int32_t *page_table, int64_t n_logical_pages, const ta_config *config,
                   int32_t *pos_ids_out, void *stream, ta_plan **out) {
    NvtxRange nvtx_range("tree_attn_plan");
    if (!out) {
        set_error("out is NULL");
        return TA_ERR_INVALID;
    }
    *out = nullptr;
    ta_plan *plan = new (std::nothrow) ta_plan();
    if (!plan) {
        set_error("host allocation failed");
        return TA_ERR_NOMEM;
    }
    int device_sms = 0;
    if (config && !(config->flags & TA_PLAN_HOST_ONLY)) {
        cudaError_t e = cudaGetDevice(&plan->device);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&device_sms, cudaDevAttrMultiProcessorCount, plan->device);
        if (e != cudaSuccess) {
            delete plan;
            return cuda_fail(e, "tree_attn_plan: device query");
        }
    }
    int rc;
    try {
        rc = build_host_plan(branches, n_branches, mounts, n_mounts, page_table, n_logical_pages, config,
                             device_sms, plan->host);
    } catch (const std::bad_alloc &) {
        set_error("host allocation failed while planning");
        rc = TA_ERR_NOMEM;
    }
    if (rc) {
        delete plan;
        return rc;
    }
    HostPlan &h = plan->host;
    if (pos_ids_out && h.N > 0) std::memcpy(pos_ids_out, h.pos_ids.data(), sizeof(int32_t) * h.N);
    {
        const ta_config &c = h.cfg;
        plan->ws_table_bytes = align_up(sizeof(float) * 256 * 2 * size_t(c.num_kv_heads) * (h.blocks.size() / 4), 256);
        plan->ws_bytes = plan->ws_table_bytes +
                         sizeof(float) * size_t(h.n_partial_slots) * c.num_kv_heads * 2 * kTileRows * c.head_dim;
    }
    if (h.cfg.flags & TA_PLAN_HOST_ONLY) {
        *out = plan;
        return TA_OK;
    }

    // one device buffer for every array the kernels read, plus status words
    std::vector<int32_t> fblk(2 * (h.fblk_ptr.size() - 1));
    for (size_t b = 0; b + 1 < h.fblk_ptr.size(); ++b) {
        fblk[2 * b] = int32_t(h.fblk_ptr[b]);
        fblk[2 * b + 1] = int32_t(h.fblk_ptr[b + 1]);
    }
    Part parts[15] = {
        {h.blocks.data(), h.blocks.size() * 4, 0},   {h.entries.data(), h.entries.size() * 4, 0},
        {h.t_entries.data(), h.t_entries.size() * 4, 0}, {h.chunks.data(), h.chunks.size() * 4, 0},
        {h.fwd_order.data(), h.fwd_order.size() * 4, 0}, {h.reduce.data(), h.reduce.size() * 4, 0},
        {h.page_table.data(), h.page_table.size() * 4, 0}, {nullptr, 64, 0},
        {h.tile_rows.data(), h.tile_rows.size() * 4, 0}, {h.t_info.data(), h.t_info.size() * 4, 0},
        {h.pos_ids.data(), h.pos_ids.size() * 4, 0},
        {h.ftiles.data(), h.ftiles.size() * 4, 0},     {fblk.data(), fblk.size() * 4, 0},
        {h.fwd_items.data(), h.fwd_items.size() * 4, 0}, {h.fwd_combine.data(), h.fwd_combine.size() * 4, 0},
    };
    size_t total = 0;
    for (Part &p : parts) {
        p.off = total;
        total = align_up(total + std::max<size_t>(p.bytes, 16), 256);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    plan->stream_ordered = (h.cfg.flags & TA_PLAN_STREAM_ORDERED) != 0;
    plan->stream = stream;
    cudaError_t e = cudaSuccess;
    if (plan->stream_ordered) {
        if ((rc = upload_stream_ordered(plan->device, &plan->d_buf, parts, 15, total, s))) {
            delete plan;
            return rc;
        }
    } else {
        std::vector<uint8_t> staging(total, 0);
        for (Part &p : parts)
            if (p.src && p.bytes) std::memcpy(staging.data() + p.off, p.src, p.bytes);
        e = cudaMalloc(&plan->d_buf, total);
        if (e != cudaSuccess) {
            delete plan;
            return e == cudaErrorMemoryAllocation ? (set_error("device allocation failed"), TA_ERR_NOMEM)
                                                  : cuda_fail(e, "plan upload");
        }
        e = cudaMemcpyAsync(plan->d_buf, staging.data(), total, cudaMemcpyHostToDevice, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) {
            cudaFree(plan->d_buf);
            delete plan;
            return cuda_fail(e, "plan upload");
        }
    }
    uint8_t *d = static_cast<uint8_t *>(plan->d_buf);
    plan->d_buf = d;
    plan->d_bytes = total;
    plan->d_blocks = reinterpret_cast<const int32_t *>(d + parts[0].off);
    plan->d_entries = reinterpret_cast<const int32_t *>(d + parts[1].off);
    plan->d_t_entries = reinterpret_cast<const int32_t *>(d + parts[2].off);
    plan->d_chunks = reinterpret_cast<const int32_t *>(d + parts[3].off);
    plan->d_fwd_order = reinterpret_cast<const int32_t *>(d + parts[4].off);
    plan->d_reduce = reinterpret_cast<const int32_t *>(d + parts[5].off);
    plan->d_page_table = reinterpret_cast<const int32_t *>(d + parts[6].off);
    plan->d_status = reinterpret_cast<int32_t *>(d + parts[7].off);
    plan->d_tile_rows = reinterpret_cast<const int32_t *>(d + parts[8].off);
    plan->d_t_info = reinterpret_cast<const int32_t *>(d + parts[9].off);
    plan->d_pos_ids = reinterpret_cast<const int32_t *>(d + parts[10].off);
    plan->d_ftiles = reinterpret_cast<const int32_t *>(d + parts[11].off);
    plan->d_fblk = reinterpret_cast<const int32_t *>(d + parts[12].off);
    plan->d_fwd_items = reinterpret_cast<const int32_t *>(d + parts[13].off);
    plan->d_fwd_combine = reinterpret_cast<const int32_t *>(d + parts[14].off);
    // partial results of split forward blocks: written by the forward, read by the combine,
    // never uploaded (an allocation of its own, in stream order like d_buf)
    if (h.n_fwd_slots > 0) {
        const size_t bytes = sizeof(float) * size_t(h.n_fwd_slots) * h.cfg.num_kv_heads * 256 * (h.cfg.head_dim + 1);
        void *buf = nullptr;
        e = plan->stream_ordered ? cudaMallocAsync(&buf, bytes, s) : cudaMalloc(&buf, bytes);
        if (e != cudaSuccess) {
            if (plan->stream_ordered) cudaFreeAsync(plan->d_buf, s);
            else cudaFree(plan->d_buf);
            delete plan;
            return e == cudaErrorMemoryAllocation ? (set_error("device allocation failed"), TA_ERR_NOMEM)
                                                  : cuda_fail(e, "plan allocation (split forward)");
        }
        plan->d_fwd_partial = static_cast<float *>(buf);
    }
    *out = plan;
    return TA_OK;
}

void tree_attn_plan_destroy(ta_plan *plan) {
    if (!plan) return;
    if (plan->d_buf) {
        if (plan->stream_ordered) cudaFreeAsync(plan->d_buf, static_cast<cudaStream_t>(plan->stream));
        else cudaFree(plan->d_buf);
    }
    if (plan->d_fwd_partial) {
        if (plan->stream_ordered) cudaFreeAsync(plan->d_fwd_partial, static_cast<cudaStream_t>(plan->stream));
        else cudaFree(plan->d_fwd_partial);
    }
    delete plan;
}

size_t tree_attn_bwd_workspace_size(const ta_plan *plan) { return plan ? plan->ws_bytes : 0; }

int tree_attn_set_trace_events(ta_plan *plan, void *const *events, int n_events) {
    if (!plan || (events && n_events != 7)) {
        set_error("tree_attn_set_trace_events: NULL plan or n_events != 7");
        return TA_ERR_INVALID;
    }
    for (int i = 0; i < 7; ++i) plan->trace[i] = events ? events[i] : nullptr;
    return TA_OK;
}

int tree_attn_plan_stats(const ta_plan *plan, ta_plan_stats *out) {
    if (!plan || !out) {
        set_error("NULL argument");
        return TA_ERR_INVALID;
    }
    const HostPlan &h = plan->host;
    std::memset(out, 0, sizeof(*out));
    out->n_rows = h.N;
    out->pairs = h.pairs;
    out->fwd_flops = 4.0 * h.cfg.head_dim * h.cfg.num_q_heads * double(h.pairs);
    out->bwd_flops = 10.0 * h.cfg.head_dim * h.cfg.num_q_heads * double(h.pairs);
    out->n_segments = h.n_segments;
    out->n_blocks = int64_t(h.blocks.size() / 4);
    out->n_intervals = int64_t(h.iv_lo.size());
    out->n_entries = int64_t(h.entries.size() / 4);
    out->n_kv_tiles = (h.N + kTileRows - 1) / kTileRows;
    out->n_chunks = int64_t(h.chunks.size() / 4);
    out->n_partial_slots = h.n_partial_slots;
    out->block_rows = h.block_rows;
    out->tile_rows = kTileRows;
    out->bwd_workspace_bytes = plan->ws_bytes;
    out->plan_ms = h.plan_ms;
    out->n_ftiles = int64_t(h.ftiles.size() / kPackInts);
    out->chunk_cap = h.chunk_cap;
    out->num_sms = h.num_sms;
    out->device = plan->device;
    out->n_fwd_items = int64_t(h.fwd_items.size() / 4);
    out->n_fwd_split = int64_t(h.fwd_combine.size() / 4);
    out->fwd_split_cap = h.fwd_split_cap;
    return TA_OK;
}

int tree_attn_plan_export(const ta_plan *plan, ta_plan_arrays *out) {
    if (!plan || !out) {
        set_error("NULL argument");
        return TA_ERR_INVALID;
    }
    const HostPlan &h = plan->host;
    out->n_rows = h.N;
    out->n_blocks = int64_t(h.blocks.size() / 4);
    out->n_intervals = int64_t(h.iv_lo.size());
    out->n_entries = int64_t(h.entries.size() / 4);
    out->n_chunks = int64_t(h.chunks.size() / 4);
    out->pos_ids = h.pos_ids.data();
    out->blocks = h.blocks.data();
    out->blk_iv_ptr = h.blk_iv_ptr.data();
    out->iv_lo = h.iv_lo.data();
    out->iv_hi = h.iv_hi.data();
    out->diag = h.diag.data();
    out->entries = h.entries.data();
    out->t_entries = h.t_entries.data();
    out->chunks = h.chunks.data();
    out->fwd_order = h.fwd_order.data();
    out->n_ftiles = int64_t(h.ftiles.size() / kPackInts);
    out->fblk_ptr = h.fblk_ptr.data();
    out->ftiles = h.ftiles.data();
    out->n_fwd_items = int64_t(h.fwd_items.size() / 4);
    out->n_fwd_split = int64_t(h.fwd_combine.size() / 4);
    out->fwd_items = h.fwd_items.data();
    out->fwd_combine = h.fwd_combine.data();
    return TA_OK;
}

static bool host_only(const ta_plan *plan) {
    if (plan->d_buf) return false;
    set_error("the plan was built with TA_PLAN_HOST_ONLY");
    return true;
}

// The plan's arrays live on the device it was built on: launching with another device current
// would read them through the wrong GPU.  TA_OK, or TA_ERR_INVALID / TA_ERR_CUDA with a message.
static int check_device(const ta_plan *plan, const char *who) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, who);
    if (dev != plan->device) {
        set_error(std::string(who) + ": the plan was built on device " + std::to_string(plan->device) +
                  " but device " + std::to_string(dev) + " is current");
        return TA_ERR_INVALID;
    }
    return TA_OK;
}

int tree_attn_check(const ta_plan *plan, void *stream) {
    NvtxRange nvtx_range("tree_attn_check");
    if (!plan) {
        set_error("plan is NULL");
        return TA_ERR_INVALID;
    }
    if (host_only(plan)) return TA_ERR_INVALID;
    if (int rc = check_device(plan, "tree_attn_check")) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int32_t st[4] = {0, 0, 0, 0};
    e = cudaMemcpyAsync(st, plan->d_status, sizeof(st), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    const int32_t any = st[0] | st[1] | st[2] | st[3];
    if (any) {
        // clear on the same stream; only this stream waits for it
        e = cudaMemsetAsync(plan->d_status, 0, sizeof(st), s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "status clear");
        if (any & kStatusTimeout) {
            set_error("a bounded device-side wait expired; outputs of the affected launches are invalid");
            return TA_ERR_DEVICE_TIMEOUT;
        }
        if (any & kStatusBounds) {
            set_error("a device-side bounds check (TA_DEBUG build) found a page index, pool row or output row "
                      "out of range; the access was skipped and the outputs are invalid");
            return TA_ERR_DEVICE_BOUNDS;
        }
        set_error("a kernel found its dynamic shared memory misaligned and did nothing; outputs are invalid");
        return TA_ERR_CUDA;
    }
    return TA_OK;
}

int tree_attn_logprob_fwd(const void *logits, int64_t n_rows, int64_t vocab, const int64_t *pos_row,
                          const int32_t *pos_target, int64_t n_pos, float *row_lse, float *logprob, void *stream) {
    NvtxRange nvtx_range("tree_attn_logprob_fwd");
    if (n_rows < 0 || n_pos < 0 || vocab <= 0 || vocab > INT32_MAX) {
        set_error("tree_attn_logprob_fwd: bad sizes");
        return TA_ERR_INVALID;
    }
    if (vocab % 8) {
        set_error("tree_attn_logprob_fwd: vocab must be a multiple of 8");
        return TA_ERR_UNSUPPORTED;
    }
    if ((n_rows > 0 && (!aligned16(logits) || !row_lse)) || (n_pos > 0 && (!pos_row || !pos_target || !logprob))) {
        set_error("tree_attn_logprob_fwd: NULL or misaligned (16-byte) pointer");
        return TA_ERR_INVALID;
    }
    cudaError_t e = launch_logprob_fwd(static_cast<const __nv_bfloat16 *>(logits), n_rows, vocab, pos_row, pos_target,
                                       n_pos, row_lse, logprob, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TA_OK : cuda_fail(e, "logprob forward launch");
}

int tree_attn_logprob_bwd(const void *logits, int64_t n_rows, int64_t vocab, const float *row_lse,
                          const int64_t *row_ptr, const int64_t *row_pos, const int32_t *pos_target,
                          const float *dlogprob, void *dlogits, void *stream) {
    NvtxRange nvtx_range("tree_attn_logprob_bwd");
    if (n_rows < 0 || vocab <= 0 || vocab > INT32_MAX) {
        set_error("tree_attn_logprob_bwd: bad sizes");
        return TA_ERR_INVALID;
    }
    if (vocab % 8) {
        set_error("tree_attn_logprob_bwd: vocab must be a multiple of 8");
        return TA_ERR_UNSUPPORTED;
    }
    if (n_rows > 0 && (!aligned16(logits) || !aligned16(dlogits) || !row_lse || !row_ptr || !row_pos ||
                       !pos_target || !dlogprob)) {
        set_error("tree_attn_logprob_bwd: NULL or misaligned (16-byte) pointer");
        return TA_ERR_INVALID;
    }
    cudaError_t e = launch_logprob_bwd(static_cast<const __nv_bfloat16 *>(logits), n_rows, vocab, row_lse, row_ptr,
                                       row_pos, pos_target, dlogprob, static_cast<__nv_bfloat16 *>(dlogits),
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TA_OK : cuda_fail(e, "logprob backward launch");
}

int tree_attn_rope(const ta_plan *plan, void *q, void *k_pool, double theta_base, void *stream) {
    NvtxRange nvtx_range("tree_attn_rope");
    if (!plan) {
        set_error("plan is NULL");
        return TA_ERR_INVALID;
    }
    const HostPlan &h = plan->host;
    if (!(theta_base > 1.0) || !std::isfinite(theta_base)) {
        set_error("tree_attn_rope: theta_base must be a finite number > 1");
        return TA_ERR_INVALID;
    }
    if (h.N == 0) return TA_OK;
    if (host_only(plan)) return TA_ERR_INVALID;
    if (int rc = check_device(plan, "tree_attn_rope")) return rc;
    if (!aligned16(q) || !aligned16(k_pool)) {
        set_error("tree_attn_rope: NULL or misaligned (16-byte) pointer");
        return TA_ERR_INVALID;
    }
    const int D = h.cfg.head_dim;
    RopeParams p{};
    p.q = static_cast<__nv_bfloat16 *>(q);
    p.k_pool = static_cast<__nv_bfloat16 *>(k_pool);
    p.pos_ids = plan->d_pos_ids;
    p.page_table = plan->d_page_table;
    p.N = h.N;
    p.Hq = h.cfg.num_q_heads;
    p.Hkv = h.cfg.num_kv_heads;
    p.page_size = h.cfg.page_size;
    p.n_logical_pages = h.n_logical_pages;
    p.num_pages = h.cfg.num_pages;
    p.status = plan->d_status + 2;
    for (int i = 0; i < D / 2; ++i) p.inv_freq[i] = std::pow(theta_base, -2.0 * i / D);
    cudaError_t e = launch_rope(D, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TA_OK : cuda_fail(e, "rope launch");
}

int tree_attn_fwd(const ta_plan *plan, const void *q, const void *k_pool, const void *v_pool, void *o,
                  float *lse, void *stream) {
    NvtxRange nvtx_range("tree_attn_fwd");
    if (!plan) {
        set_error("plan is NULL");
        return TA_ERR_INVALID;
    }
    const HostPlan &h = plan->host;
    if (h.N == 0) return TA_OK;
    if (host_only(plan)) return TA_ERR_INVALID;
    if (int rc = check_device(plan, "tree_attn_fwd")) return rc;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o) || !aligned16(lse)) {
        set_error("tree_attn_fwd: NULL or misaligned (16-byte) pointer");
        return TA_ERR_INVALID;
    }
    CUtensorMap tm_q;
    KvMaps kv;
    int rc = make_maps(plan, q, k_pool, v_pool, &tm_q, &kv);
    if (rc) return rc;
    FwdParams p{};
    p.blocks = plan->d_blocks;
    p.ftiles = plan->d_ftiles;
    p.items = plan->d_fwd_items;
    p.combine = plan->d_fwd_combine;
    p.partial = plan->d_fwd_partial;
    p.n_slots = int32_t(h.n_fwd_slots);
    p.page_table = plan->d_page_table;
    p.tile_rows = plan->d_tile_rows;
    p.n_logical_pages = int32_t(h.n_logical_pages);
    p.num_pages = int32_t(h.cfg.num_pages);
    p.page_size = h.cfg.page_size;
    p.N = int32_t(h.N);
    p.Hq = h.cfg.num_q_heads;
    p.Hkv = h.cfg.num_kv_heads;
    p.G = h.G;
    p.R = h.block_rows;
    p.scale_log2 = h.scale * 1.4426950408889634f;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.lse = lse;
    p.status = plan->d_status;
    cudaError_t e = launch_fwd(h.cfg.head_dim, tm_q, kv, p, int(h.fwd_items.size() / 4),
                               int(h.fwd_combine.size() / 4), static_cast<cudaStream_t>(stream), plan->trace);
    if (e != cudaSuccess) return cuda_fail(e, "tree_attn_fwd launch");
    return TA_OK;
}

int tree_attn_bwd(const ta_plan *plan, const void *q, const void *k_pool, const void *v_pool, const void *o,
                  const float *lse, const void *d_o, float *dq, float *dk_pool, float *dv_pool, void *workspace,
                  size_t ws_bytes, void *stream) {
    NvtxRange nvtx_range("tree_attn_bwd");
    if (!plan) {
        set_error("plan is NULL");
        return TA_ERR_INVALID;
    }
    const HostPlan &h = plan->host;
    if (h.N == 0) return TA_OK;
    if (host_only(plan)) return TA_ERR_INVALID;
    if (int rc = check_device(plan, "tree_attn_bwd")) return rc;
    if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o) || !aligned16(lse) ||
        !aligned16(d_o) || !aligned16(dq) || !aligned16(dk_pool) || !aligned16(dv_pool)) {
        set_error("tree_attn_bwd: NULL or misaligned (16-byte) pointer");
        return TA_ERR_INVALID;
    }
    if (ws_bytes < plan->ws_bytes || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)) {
        set_error("tree_attn_bwd: workspace too small or not 256-byte aligned");
        return TA_ERR_INVALID;
    }
    CUtensorMap tm_q, tm_do;
    KvMaps kv;
    int rc = make_maps(plan, q, k_pool, v_pool, &tm_q, &kv);
    if (rc) return rc;
    const ta_config &c = h.cfg;
    // the backward loads Q and dO a whole 128-lane tile per box
    const uint32_t qb = uint32_t(std::min(h.block_rows, 128));
    if ((rc = make_qtile_map(&tm_q, q, uint64_t(h.N), uint32_t(c.num_q_heads), uint32_t(c.head_dim), qb)) ||
        (rc = make_qtile_map(&tm_do, d_o, uint64_t(h.N), uint32_t(c.num_q_heads), uint32_t(c.head_dim), qb)))
        return rc;
    BwdParams p{};
    p.blocks = plan->d_blocks;
    p.ftiles = plan->d_ftiles;
    p.fblk = plan->d_fblk;
    p.t_entries = plan->d_t_entries;
    p.chunks = plan->d_chunks;
    p.reduce = plan->d_reduce;
    p.order = plan->d_fwd_order;
    p.page_table = plan->d_page_table;
    p.tile_rows = plan->d_tile_rows;
    p.t_info = plan->d_t_info;
    p.n_logical_pages = int32_t(h.n_logical_pages);
    p.num_pages = int32_t(c.num_pages);
    p.page_size = c.page_size;
    p.N = int32_t(h.N);
    p.Hq = c.num_q_heads;
    p.Hkv = c.num_kv_heads;
    p.G = h.G;
    p.R = h.block_rows;
    p.scale = h.scale;
    p.scale_log2 = h.scale * 1.4426950408889634f;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_pool = static_cast<const __nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<const __nv_bfloat16 *>(v_pool);
    p.o = static_cast<const __nv_bfloat16 *>(o);
    p.d_o = static_cast<const __nv_bfloat16 *>(d_o);
    p.lse = lse;
    p.utab = static_cast<float *>(workspace);
    p.n_blocks = int32_t(h.blocks.size() / 4);
    p.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + plan->ws_table_bytes);
    p.dq = dq;
    p.dk_pool = dk_pool;
    p.dv_pool = dv_pool;
    p.status = plan->d_status + 1;
    cudaError_t e = launch_bwd(c.head_dim, tm_q, kv, tm_do, p, int(h.blocks.size() / 4),
                               int(h.chunks.size() / 4), int(h.reduce.size() / 4), static_cast<cudaStream_t>(stream),
                               plan->trace);
    if (e != cudaSuccess) return cuda_fail(e, "tree_attn_bwd launch");
    return TA_OK;
}

}  // extern "C"
