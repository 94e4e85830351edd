/*
 * treeattn -- tree/DAG-packed paged attention, forward and backward, for sm_103a (GB300).
 *
 * The problem (Octopus, arXiv 2611.06956, Section 3 and Section 3.3; HARTS, arXiv
 * 2608.28158, Section 2.1 and Section 4.2): an agentic episode is a DAG of branches.  Tree
 * edges are forks -- a child branch continues its parent after `fork_offset` rows, sharing
 * that prefix (HARTS Section 2.2 defines the fork position as the number of shared prefix
 * tokens).  Mount edges (Octopus Section 3.1 Table 2, read_thread; Section 3.2) lend a
 * completed span of a sibling's rows to a reader from one of the reader's rows onwards.
 * Every token is stored once, as one row of a compact row strip (Octopus Section 3.3 item 2:
 * nodes concatenated topologically into one unpadded strip), and its keys/values live in a
 * paged pool (Octopus Section 3.1 Figure 2: cursor-addressed page translation).
 *
 * Row r (offset i of branch b) attends exactly to its visible set vis(r): b's rows 0..i,
 * the rows of every mount of b whose reader offset is <= i, and everything b inherited from
 * its ancestors (the parent's rows before the fork offset, the parent's mounts active at the
 * row before the fork, and the parent's own inheritance) -- the gather of Octopus Eq. 4
 * [mounts || ancestors || self] with the causal triangle on the own rows (HARTS Eq. 21-22:
 * query i sees KV entry j iff j <= h + i).  vis(r) is a set: a row reachable twice counts
 * once.  Mounts are not transitive.
 *
 * All functions return 0 (TA_OK) or a negative TA_ERR_* code; tree_attn_last_error()
 * returns a message for the calling thread's most recent failure.  No function calls
 * exit(), abort() or traps on the GPU.
 */
#ifndef TREEATTN_H
#define TREEATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TA_OK 0
#define TA_ERR_INVALID (-1)         /* malformed DAG, page table or arguments */
#define TA_ERR_UNSUPPORTED (-2)     /* a shape the library does not implement */
#define TA_ERR_NOMEM (-3)           /* host or device allocation failed (planner only) */
#define TA_ERR_CUDA (-4)            /* a CUDA runtime/driver call failed */
#define TA_ERR_DEVICE_TIMEOUT (-5)  /* a bounded device-side wait expired; outputs are invalid */
#define TA_ERR_DEVICE_BOUNDS (-6)   /* a device-side bounds check of the TA_DEBUG build failed (a
                                       page index, pool row or output row out of range; the
                                       access was skipped); outputs are invalid */

/* Flags (ta_config.flags). */
#define TA_CLAMP_MOUNTS 0x1u  /* clamp a mount span to the source's rows instead of rejecting it
                                 (Octopus Appendix A clamps spans to the valid range) */
#define TA_NO_MOUNTS 0x2u     /* the mount-free view of the same episode, for layers that do
                                 not mount (Octopus Section 3.2, layer-selective mounting, and
                                 Appendix C Table 8, the mounted / unmounted dual pass): rows see
                                 their ancestor path and own earlier rows only.  Mounts are still
                                 validated and still set the Eq. 2 positions, so pos_ids and the
                                 row layout equal those of the mounted plan. */
#define TA_TRANSITIVE_MOUNTS 0x4u /* active mounts "including transitive mounts" (Octopus
                                 Section 3.3 item 1): a mounted span [s, e) of source A also
                                 brings, recursively, the mounts in effect at A's row e-1 (A's
                                 own mounts with reader offset <= e-1 and those A inherits through
                                 its fork points).  Positions are unchanged.  Excludes
                                 TA_NO_MOUNTS (TA_ERR_INVALID if both are set). */
#define TA_PLAN_HOST_ONLY 0x100u /* build the plan on the host only (no device upload, no GPU
                                    needed): for inspection with tree_attn_plan_export/_stats;
                                    tree_attn_fwd/_bwd reject such a plan */
#define TA_PLAN_STREAM_ORDERED 0x200u /* build and destroy the plan without waiting for the
                                    GPU: the device arrays are allocated (cudaMallocAsync) and
                                    uploaded from a pinned staging buffer on an internal stream
                                    of the library, `stream` is made to wait for that upload
                                    (an event), and tree_attn_plan_destroy frees them with
                                    cudaFreeAsync on `stream`.  Without the flag tree_attn_plan
                                    synchronises `stream` before returning and destroy uses
                                    cudaFree, which waits for the whole device.  With it the
                                    plan may be used on `stream` right away, or on another
                                    stream after an event recorded on `stream` after the plan
                                    call; every use on other streams must be ordered before
                                    work enqueued on `stream` after destroy, and `stream` must
                                    still exist then. */

/* A branch: `length` rows stored at compact rows [row_start, row_start + length).
 * parent = -1 for a root (fork_offset must be 0); otherwise the child shares the parent's
 * first `fork_offset` rows (0 <= fork_offset <= parent length). */
typedef struct {
    int32_t parent;
    int32_t fork_offset;
    int32_t length;
    int64_t row_start;
} ta_branch;

/* A mount edge (Octopus Section 3.1 Table 2 read_thread, Section 3.2): from row
 * `reader_offset` of branch `reader` on, the reader also sees rows [src_begin, src_end) of
 * branch `source` (offsets within the source).  The span must be complete before the reader
 * reads it: no mounted row may depend, through any chain of visibility, on a reader row at
 * or after reader_offset.  A span with src_begin == src_end is ignored. */
typedef struct {
    int32_t reader;
    int32_t reader_offset;
    int32_t source;
    int32_t src_begin;
    int32_t src_end;
} ta_mount;

/* Attention shape.  Supported: head_dim 64 or 128; page_size 16, 32, 64 or 128;
 * num_q_heads / num_kv_heads (query heads per KV head, consecutive grouping: query head h
 * uses KV head h / G) in {1, 2, 4, 8, 16}.  softmax_scale <= 0 selects 1/sqrt(head_dim).
 * num_pages is the number of pages in the K/V pools (>= the logical pages of the strip).
 *
 * Work balance of the dK/dV kernel (no effect on results beyond fp32 summation order): the
 * readers of a key tile are split into chunks of at most `dkdv_chunk_entries` (query block,
 * key tile) entries, each chunk one CTA, whose partial sums a fixed-order reduction adds.
 * dkdv_chunk_entries <= 0 selects max(8, entries * num_kv_heads / (4 * SMs)): no chunk longer
 * than about a quarter of an SM's average share.  SMs = num_sms if > 0, else the SM count of
 * the current device (152 on GB300) -- or 152 for a TA_PLAN_HOST_ONLY plan, which has no device.
 *
 * Split-KV forward (results equal up to fp32 summation order): a query block whose list of
 * packed key tiles is longer than fwd_split_tiles is cut into parts of at most that many tiles;
 * each part runs as its own work item and writes a partial O and lse to plan-owned device
 * memory, and a combine kernel merges the parts of each split block (O = sum_k w_k O_k with
 * w_k = exp(lse_k - lse), lse = ln sum_k exp(lse_k)).  fwd_split_tiles == 0 (automatic)
 * splits only when the longest block is more than 1.5x, and at least 32 tiles above, one
 * worker's share of the forward's tile work (share = packed tiles x num_kv_heads / workers;
 * workers: SM pairs for head_dim 128, SMs for 64), and then into parts of at most
 * max(16, share) tiles; < 0 never splits.
 * Forwards of a plan that has split blocks share its partial buffer: such forwards must not
 * run at the same time on different streams. */
typedef struct {
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t page_size;
    float softmax_scale;
    uint32_t flags;
    int64_t num_pages;
    int32_t num_sms;             /* 0: the device's (see above) */
    int32_t dkdv_chunk_entries;  /* 0: derived from the SM count (see above) */
    int32_t fwd_split_tiles;     /* 0: automatic, < 0: never (see above) */
} ta_config;

typedef struct ta_plan ta_plan; /* opaque; owned by the library */

/* Counts describing a plan. */
typedef struct {
    int64_t n_rows;          /* N: compact rows */
    int64_t pairs;           /* sum over rows of |vis(r)| (visible query-key row pairs) */
    double fwd_flops;        /* useful forward FLOPs: 4 * head_dim * num_q_heads * pairs */
    double bwd_flops;        /* useful backward FLOPs: 10 * head_dim * num_q_heads * pairs */
    int64_t n_segments;      /* query segments (branches split at mount offsets) */
    int64_t n_blocks;        /* query blocks */
    int64_t n_intervals;     /* visible intervals over all blocks (diagonal excluded) */
    int64_t n_entries;       /* (query block, key tile) work entries */
    int64_t n_kv_tiles;      /* 128-row key tiles of the strip */
    int64_t n_chunks;        /* dK/dV work chunks (key tile x entry range) */
    int64_t n_partial_slots; /* dK/dV partial accumulators for split key tiles */
    int32_t block_rows;      /* query rows per block (256 / G) */
    int32_t tile_rows;       /* key rows per tile (128) */
    size_t bwd_workspace_bytes;
    double plan_ms;          /* host time spent in tree_attn_plan */
    int64_t n_ftiles;        /* packed key tiles of the forward and dQ kernels */
    int64_t chunk_cap;       /* entries per dK/dV chunk at most (see ta_config) */
    int32_t num_sms;         /* SM count the chunk cap was derived from */
    int32_t device;          /* CUDA device the plan was uploaded to (-1: host-only plan) */
    int64_t n_fwd_items;     /* forward work items (blocks, or parts of split blocks) */
    int64_t n_fwd_split;     /* query blocks whose forward is split into parts */
    int64_t fwd_split_cap;   /* packed key tiles per forward work item at most (the longest
                                block's when nothing is split) */
} ta_plan_stats;

/* Host views of the plan's arrays, for inspection and bit-exact tests.  All pointers are
 * owned by the plan and stay valid until tree_attn_plan_destroy.
 *   pos_ids[n_rows]                    Eq. 2 position of every compact row
 *   blocks[4*n_blocks]                 {first row, rows, first entry, end entry}
 *   blk_iv_ptr[n_blocks+1], iv_lo/iv_hi[n_intervals]
 *                                      per block: sorted disjoint maximal intervals of rows
 *                                      visible to every row of the block
 *   diag[2*n_blocks]                   per block: own rows [lo, hi) seen causally (j <= r)
 *   entries[4*n_entries]               query-major {key tile, lo, hi, flags}
 *   t_entries[4*n_entries]             key-tile-major {block, lo, hi, flags}
 *   chunks[4*n_chunks]                 {key tile, first t_entry, end t_entry, partial slot or -1}
 *   fwd_order[n_blocks]                query blocks, longest first: the dQ kernel's launch
 *                                      order (the forward's items follow it, see fwd_items)
 *   fblk_ptr[n_blocks+1], ftiles[8*n_ftiles]
 *                                      per block: the packed key tiles the forward and dQ
 *                                      kernels visit -- 4 slots of 32 key rows each:
 *                                      {piece[4] (first row / 32, -1 empty), lo/hi of slots 0-1,
 *                                      lo/hi of slots 2-3 (lo | hi << 6 | lo' << 12 | hi' << 18:
 *                                      visible rows [lo, hi) of the piece), flags, 0}; flags bit
 *                                      0 = some slot needs masking, bit 1+k = slot k causal
 *                                      (mask j > r), bit 5+h = slots 2h, 2h+1 are one 64-row run
 *   fwd_items[4*n_fwd_items]           forward work items in launch order: {block, first packed
 *                                      tile, end tile, partial slot or -1 (whole block)}
 *   fwd_combine[4*n_fwd_split]         split blocks: {block, first slot, parts, 0}
 * flags (entries): bit 0 = causal (mask j > r), bit 1 = the entry does not cover its whole tile. */
typedef struct {
    int64_t n_rows, n_blocks, n_intervals, n_entries, n_chunks;
    const int32_t *pos_ids;
    const int32_t *blocks;
    const int64_t *blk_iv_ptr;
    const int32_t *iv_lo, *iv_hi;
    const int32_t *diag;
    const int32_t *entries;
    const int32_t *t_entries;
    const int32_t *chunks;
    const int32_t *fwd_order;
    int64_t n_ftiles;
    const int64_t *fblk_ptr;
    const int32_t *ftiles;
    int64_t n_fwd_items, n_fwd_split;
    const int32_t *fwd_items;
    const int32_t *fwd_combine;
} ta_plan_arrays;

/* Build the compact prefix-tree episode of a set of token trajectories.
 *
 * HARTS (arXiv 2608.28158) Section 2.1: one compact row per distinct token prefix and a map
 * m: S -> C from every semantic position (trajectory, offset) to its compact row (Eq. 3);
 * Section 3.2, Eq. 5: with the trajectories in lexicographic order, the row count is
 * |x_1| + sum_i (|x_i| - LCP(x_{i-1}, x_i)).  The result has exactly that many rows: each
 * trajectory forks from the branch of its predecessor's path holding its last shared token,
 * and its unshared suffix becomes a new branch.  Rows are laid out in creation order (a depth-
 * first order of the tree).  The branches need no mounts; tree_attn_plan accepts them as is,
 * and the plan's position ids equal the trajectory offsets.
 *
 *   tokens        host, int32[offsets[n_traj]]: the trajectories concatenated
 *   offsets       host, int64[n_traj + 1]: trajectory i is tokens[offsets[i], offsets[i+1]),
 *                 non-decreasing from offsets[0] = 0 (empty trajectories allowed)
 *   branches      host, out, capacity max_branches (n_traj always suffices); may be NULL to
 *                 query *n_branches only when max_branches >= the count
 *   row_tokens    host, out, int32[max_rows] (offsets[n_traj] always suffices): the token of
 *                 every compact row; may be NULL
 *   n_rows        out: the compact row count (Eq. 5)
 *   row_of        host, out, int64[offsets[n_traj]]: m, the compact row of every position,
 *                 in the layout of `tokens`
 *   row_owner     host, out, int32[max_rows], may be NULL: the trajectory (input index) whose
 *                 insertion created each compact row
 * Returns TA_OK, or TA_ERR_INVALID (bad offsets, NULL arrays, capacity too small).  Pure host
 * code: no GPU, no allocation visible to the caller. */
int tree_attn_ingest(const int32_t *tokens, const int64_t *offsets, int32_t n_traj,
                     ta_branch *branches, int32_t max_branches, int32_t *n_branches,
                     int32_t *row_tokens, int64_t max_rows, int64_t *n_rows, int64_t *row_of,
                     int32_t *row_owner);

/* Prefix-deduplicating loss mask (Octopus, arXiv 2611.06956, Section 3.4, Eq. 6): every
 * generated token of the packed strip is counted once, at the trajectory owning its node, so
 * that the masked sum of token log-probabilities over all trajectories is the episode's score
 * function (Eq. 7).  Position k = offsets[l] + t predicts token t + 1 of trajectory l; mask[k]
 * = 1 iff l owns the compact row of that token (row_owner from tree_attn_ingest) and
 * generated[k + 1] (NULL: every token counts); the last position of each trajectory is 0.
 * All arrays host, in the layout of `tokens` (row_owner: per compact row).  Returns TA_OK or
 * TA_ERR_INVALID.  (The pages do not say which trajectory owns a shared node; here it is the
 * one whose insertion created the row: the lexicographically first, input order on ties.) */
int tree_attn_owner_mask(const int64_t *offsets, int32_t n_traj, const int64_t *row_of,
                         const int32_t *row_owner, const uint8_t *generated, uint8_t *mask);

/* Compact-work microbatch planning across data-parallel replicas (HARTS, arXiv 2608.28158,
 * Section 3.2).  Complete trajectories (the smallest scheduling unit) are grouped into K
 * microbatches of at most `capacity` compact rows each -- a microbatch's work is the row count of
 * the compact trie of its trajectories (Eq. 5) -- with K a multiple of `replicas` (D), and each
 * microbatch is given a replica and a slot.  Plans are ranked lexicographically by Eq. 4: total
 * compact work, then the sum over slots of the slot's heaviest microbatch, then the heaviest
 * replica's cumulative work.  Candidate groupings (mode 0 uses both kinds, 1 only the first, 2
 * only the second):
 *   - partitions contiguous in lexicographic order for every K of Eq. 8, K from K_min of Eq. 7
 *     (D max(1, ceil(G / (T D))), G the work of all trajectories in one trie) to K_max (from the
 *     natural partition, which splits every interval heavier than T at its lowest adjacent-LCP
 *     valley): the exact dynamic program of Eq. 9 for up to `exact_max_traj` trajectories (0:
 *     512), else the natural partition evolved by merging the adjacent pair that saves the most
 *     and splitting at the lowest valley, over at most 32 sampled K;
 *   - greedy insertion by the exact compact-work increase of Eq. 10, in four processing orders
 *     (ascending and descending lexicographic, descending length, descending unique-suffix score)
 *     under two policies (best fit: the largest work after insertion; max shared: the largest
 *     |x| - increase), K raised to a multiple of D by splitting off the single trajectories that
 *     cost the least; of the eight, the one with the fewest microbatches, then the least work.
 * Every candidate gets the DP-replica assignment of the section: microbatches sorted by work,
 * each consecutive block of D one slot, the heavier ones to the replicas with less work so far.
 * Not built (they refine a candidate without changing what the planner guarantees): boundary
 * refinement and sparse repair.
 *
 *   tokens, offsets, n_traj   host: trajectory i is tokens[offsets[i] .. offsets[i+1]),
 *                             non-empty, no longer than capacity; n_traj >= replicas
 *   microbatch_of             host, out, int32[n_traj]: microbatch of each trajectory
 *   replica_of, slot_of       host, out, int32[n_traj] (capacity; the first K are written):
 *                             replica and slot of each microbatch; every replica gets exactly
 *                             one microbatch per slot
 *   mb_work                   host, out, int64[n_traj] or NULL: compact rows of each microbatch
 * Returns TA_OK, or TA_ERR_INVALID (arguments, a trajectory longer than the capacity, no
 * feasible plan), TA_ERR_NOMEM.  Pure host code. */
typedef struct {
    int32_t replicas;        /* D >= 1 */
    int32_t mode;            /* 0: contiguous and greedy candidates; 1: contiguous only; 2: greedy only */
    int64_t capacity;        /* T: compact rows per microbatch at most */
    int32_t exact_max_traj;  /* exact dynamic program up to this many trajectories (0: 512) */
    int32_t reserved;
} ta_place_config;

typedef struct {
    int64_t total_work;          /* Eq. 4, first term: sum of the microbatches' compact rows */
    int64_t slot_critical_work;  /* Eq. 4, second term: sum over slots of the heaviest microbatch */
    int64_t max_replica_work;    /* Eq. 4, third term: the heaviest replica's cumulative work */
    int64_t merged_work;         /* G: compact rows of all trajectories in one trie */
    int32_t n_microbatches;      /* K */
    int32_t n_slots;             /* K / D */
    int32_t n_candidates;        /* candidate plans compared */
    int32_t source;              /* the chosen plan's generator: 0 contiguous, 1 greedy */
    int32_t k_min, k_max;        /* Eq. 7-8 */
    int32_t k_natural;           /* microbatches of the natural partition */
    int32_t reserved;
} ta_place_stats;

int tree_attn_place(const int32_t *tokens, const int64_t *offsets, int32_t n_traj, const ta_place_config *cfg,
                    int32_t *microbatch_of, int32_t *replica_of, int32_t *slot_of, int64_t *mb_work,
                    ta_place_stats *stats);

/* The DP-replica assignment of tree_attn_place for units that are already grouped -- e.g. the
 * independent DAGs of a batch of episodes, whose attention shares no rows across units, so that
 * each replica runs its units with no collective: units sorted by work, each consecutive block of
 * `replicas` one slot (the last one may be short), the heavier units of a slot to the replicas
 * with less work so far.  work: host int64[n_units] (compact rows, or any additive cost);
 * replica_of, slot_of: host out int32[n_units]; stats as tree_attn_place (n_microbatches =
 * n_units).  Returns TA_OK or TA_ERR_INVALID. */
int tree_attn_place_units(const int64_t *work, int32_t n_units, int32_t replicas, int32_t *replica_of,
                          int32_t *slot_of, ta_place_stats *stats);

/*
 * tree_attn_plan -- validate an episode DAG and build the work plan (host C++).
 *
 * Splits branches into query segments at mount offsets (Octopus Section 3.3 item 1, node
 * splitting at read_thread boundaries; forks do not change a branch's own rows), computes
 * Eq. 2 position ids (Octopus Section 3.2), tiles each segment into query blocks, lists
 * per block the visible key-row intervals (Eq. 4 gather, expressed as row intervals rather
 * than copied), translates them into 128-row key tiles, builds the key-tile-major transpose
 * used by the dK/dV reduction, and uploads everything to the device on `stream`
 * (synchronising once, or not at all with TA_PLAN_STREAM_ORDERED).
 *
 *   branches[n_branches], mounts[n_mounts]   host arrays, read during the call only
 *   page_table[n_logical_pages]             host: logical page l of the strip (rows
 *                                           [l*page_size, (l+1)*page_size)) is pool page
 *                                           page_table[l]; entries distinct, < num_pages;
 *                                           n_logical_pages >= ceil(N / page_size)
 *   config                                  attention shape (see ta_config)
 *   pos_ids_out                             host int32[N] or NULL: receives the positions
 *   stream                                  cudaStream_t (may be NULL: the default stream)
 *   out                                     receives the plan; *out is NULL on failure
 *
 * Errors: TA_ERR_INVALID for a bad parent or a parent cycle, a root with a fork offset, a
 * fork offset beyond its parent, negative lengths, branch row ranges that overlap or leave
 * gaps in [0, N), N beyond 2^31-1, a mount with an index or offset out of range or a span
 * outside its source (unless TA_CLAMP_MOUNTS), a non-causal mount, a short page table, a
 * duplicate or out-of-range page; TA_ERR_UNSUPPORTED for shapes outside ta_config's list;
 * TA_ERR_NOMEM, TA_ERR_CUDA.  An empty DAG (N = 0) gives a valid plan on which fwd and
 * bwd do nothing.
 */
int tree_attn_plan(const ta_branch *branches, int32_t n_branches, const ta_mount *mounts,
                   int32_t n_mounts, const int32_t *page_table, int64_t n_logical_pages,
                   const ta_config *config, int32_t *pos_ids_out, void *stream, ta_plan **out);

/* Rotary position embedding of Q and the K pool, in place, at the plan's Eq. 2 positions.
 *
 * Octopus (arXiv 2611.06956) Section 3.2: scores see positions only through the rotary phase
 * relation <R_p q, R_s k> = <q, R_{s-p} k> (Eq. 1), which is why mounted spans keep their own
 * positions and readers continue after them (Eq. 2); HARTS (arXiv 2608.28158) Section 4.2
 * applies RoPE once per compact row before attention.  Pair layout (a reading: the pages give
 * only Eq. 1): element i and i + D/2 of every head vector are rotated by p * theta_i,
 * theta_i = theta_base^(-2i/D), i < D/2, p = pos_ids[row].
 *
 *   q       device, bf16 [N, num_q_heads, head_dim], compact rows; rotated in place
 *   k_pool  device, bf16 [num_pages, page_size, num_kv_heads, head_dim]; the rows the page
 *           table maps are rotated in place, spare pages are not touched (V is not rotated)
 *   theta_base  > 1 (10000 in the original RoPE; model-specific)
 * One kernel on `stream`, HBM-bound; TA_ERR_INVALID for bad arguments or a host-only plan. */
int tree_attn_rope(const ta_plan *plan, void *q, void *k_pool, double theta_base, void *stream);

/* Compact-to-semantic log-probabilities (HARTS, arXiv 2608.28158, Section 4).
 *
 * A compact row c's LM-head logits z_c serve every semantic position s with m(s) = c (the map
 * of tree_attn_ingest).  Eq. 17: lambda_s = z_{m(s), y_s} - log sum_v exp z_{m(s), v}, the
 * vocabulary-wide maximum and sum-exp formed once per compact row; Eq. 19-20: the backward
 * accumulates every position's gradient into its row, dz_c = sum_{m(s)=c} g_s (e_{y_s} -
 * softmax(z_c)).  Nothing of size positions x vocab is formed.
 *
 *   logits     device, bf16 [n_rows, vocab] row-major, 16-byte aligned; vocab a multiple of 8
 *              (TA_ERR_UNSUPPORTED otherwise)
 *   pos_row    device, int64 [n_pos]: m(s), the compact row of position s
 *   pos_target device, int32 [n_pos]: y_s, the next token of position s
 *   row_lse    device, fp32 [n_rows], out (fwd) / in (bwd): natural-log sum-exp of every row
 *   logprob    device, fp32 [n_pos], out: lambda_s in the caller's order (NaN for a position
 *              whose row or target is out of range)
 *   row_ptr, row_pos  device, int64 [n_rows + 1], [n_pos]: the positions of each row, ordered by
 *              target, as built by tree_attn_logprob_index (host)
 *   dlogprob   device, fp32 [n_pos]: g_s = dL/dlambda_s (0 for positions outside the action mask)
 *   dlogits    device, bf16 [n_rows, vocab], out, 16-byte aligned; every element written once
 *              (rows no position reads are 0); deterministic
 * Each call enqueues its kernels on `stream` (forward: 2, backward: 1); HBM-bound.  Returns
 * TA_OK, TA_ERR_INVALID or TA_ERR_UNSUPPORTED (arguments), TA_ERR_CUDA (launch). */
int tree_attn_logprob_fwd(const void *logits, int64_t n_rows, int64_t vocab, const int64_t *pos_row,
                          const int32_t *pos_target, int64_t n_pos, float *row_lse, float *logprob, void *stream);
int tree_attn_logprob_bwd(const void *logits, int64_t n_rows, int64_t vocab, const float *row_lse,
                          const int64_t *row_ptr, const int64_t *row_pos, const int32_t *pos_target,
                          const float *dlogprob, void *dlogits, void *stream);
/* Host: the CSR row_ptr[n_rows + 1] / row_pos[n_pos] that tree_attn_logprob_bwd reads, from
 * host copies of pos_row and pos_target; TA_ERR_INVALID if a row or target is out of range. */
int tree_attn_logprob_index(const int64_t *pos_row, const int32_t *pos_target, int64_t n_pos,
                            int64_t n_rows, int64_t vocab, int64_t *row_ptr, int64_t *row_pos);

/*
 * tree_attn_fwd -- O and logsumexp of every compact row (device, sm_103a).
 *
 *   O[r,h]   = sum_{j in vis(r)} softmax_j(scale <q[r,h], k[j,g]>) v[j,g],  g = h / G
 *   lse[h,r] = ln sum_{j in vis(r)} exp(scale <q[r,h], k[j,g]>)
 * (Octopus Section 3.3 Eq. 4 and the rectangular causal attention that follows it; HARTS
 * Section 4.2 Eq. 21-22.)
 *
 *   q       device bf16 [N, Hq, D], compact rows, contiguous; 16-byte aligned
 *   k_pool  device bf16 [num_pages, page_size, Hkv, D]; 16-byte aligned.  Rows of the last
 *   v_pool  logical page at or beyond N are read as part of whole tiles and must be finite
 *           (pages not listed in the page table are never read)
 *   o       device bf16 [N, Hq, D] (written)
 *   lse     device fp32 [Hq, N] (written), natural log
 * Everything is enqueued on `stream`; no allocation, no synchronisation.  Caller owns every
 * buffer.  Returns TA_ERR_INVALID for NULL/misaligned pointers, a host-only plan, or a plan
 * built while another device was current (the plan's arrays live on that device; the same
 * check guards tree_attn_bwd, tree_attn_rope and tree_attn_check), and TA_ERR_CUDA for a
 * launch failure.  A bounded device-side wait that expires inside the
 * launched kernels is not seen by this call: it is recorded in the plan's status words and
 * reported by the next tree_attn_check on the plan (TA_ERR_DEVICE_TIMEOUT).
 * Because the call only enqueues kernels, it can be recorded by CUDA stream capture: a graph
 * holding several layers' tree_attn_fwd and tree_attn_bwd calls on one plan replays them with
 * one launch, as long as the plan, the tensors and the workspace stay alive (tree_attn_check
 * synchronises and belongs outside the capture).
 */
int tree_attn_fwd(const ta_plan *plan, const void *q, const void *k_pool, const void *v_pool,
                  void *o, float *lse, void *stream);

/*
 * tree_attn_bwd -- gradients of sum <dO, O> w.r.t. q, k_pool and v_pool (device, sm_103a).
 *
 *   delta[h,r] = <dO[r,h], O[r,h]>
 *   dS         = P * (<dO[r,h], v[j,g]> - delta),  P recomputed from lse
 *   dq[r,h]    = scale sum_{j in vis(r)} dS k[j,g]
 *   dk[j,g]    = scale sum over every (r, h in g) with j in vis(r) of dS q[r,h]
 *   dv[j,g]    = sum over the same readers of P dO[r,h]
 * Gradients of a shared prefix row or a mounted row are summed over all of its readers --
 * tree descendants and mount readers -- and written exactly once (Octopus Section 3.4,
 * differentiable mount edges; HARTS Section 3.4, gather backward accumulates every consumer
 * into the unique compact row).
 *
 *   q, k_pool, v_pool, o, lse   as in tree_attn_fwd (o, lse: that call's outputs)
 *   d_o     device bf16 [N, Hq, D]: upstream gradient per compact row (a caller with several
 *           semantic positions per row sums their gradients first)
 *   dq      device fp32 [N, Hq, D] (written)
 *   dk_pool device fp32 [num_pages, page_size, Hkv, D]: rows of the strip's logical pages are
 *   dv_pool written; other pages are left untouched
 *   workspace, ws_bytes   device scratch of at least tree_attn_bwd_workspace_size(plan)
 *           bytes, 256-byte aligned, owned by the caller; contents need not be initialised
 * Returns as tree_attn_fwd, plus TA_ERR_INVALID for a short workspace.
 */
int tree_attn_bwd(const ta_plan *plan, const void *q, const void *k_pool, const void *v_pool,
                  const void *o, const float *lse, const void *d_o, float *dq, float *dk_pool,
                  float *dv_pool, void *workspace, size_t ws_bytes, void *stream);

/*
 * tree_attn_bwd_noalloc -- tree_attn_bwd without a caller-provided workspace.  The pages have
 * no counterpart to this; it exists for callers that cannot give the library device scratch:
 * plugin-style hosts that pass a kernel only its input and output buffers, and loops that
 * forbid device allocation while running (cudaMalloc can synchronise the device and may fail
 * or fragment a sized pool).  It allocates nothing.  The scratch (the lse/delta table and the
 * dK/dV partials) is a fixed 64 MiB array inside the library that every GPU loading the
 * library holds until the process exits; plans needing more (tree_attn_bwd_workspace_size(plan) > 64 MiB) are
 * rejected with TA_ERR_UNSUPPORTED and a message naming the size.  Every call looks up the
 * array's device address (cudaGetSymbolAddress) with the current device, which must be the
 * plan's (TA_ERR_INVALID otherwise), so the address stays right after a context reset; the
 * first call on a device may load the library's module there, so make that first call before
 * any stream capture.  All calls share the array and nothing in it
 * needs clearing between calls, so calls whose kernels overlap on the GPU (other streams or
 * host threads) race on it: serialise them.  Arguments, outputs and other errors are those of
 * tree_attn_bwd.
 */
int tree_attn_bwd_noalloc(const ta_plan *plan, const void *q, const void *k_pool, const void *v_pool,
                          const void *o, const float *lse, const void *d_o, float *dq, float *dk_pool,
                          float *dv_pool, void *stream);

/* Bytes of device scratch tree_attn_bwd needs for this plan: a 1 KB table per (KV head, query
 * block, 128-lane query tile) holding -lse * log2(e) and -delta, plus dK/dV partial slots. */
size_t tree_attn_bwd_workspace_size(const ta_plan *plan);

/* Synchronises `stream` and reports whether any bounded device wait of this plan's kernels
 * expired since the last check (TA_ERR_DEVICE_TIMEOUT), a device-side bounds check failed
 * (TA_ERR_DEVICE_BOUNDS; only the library built with TA_DEBUG, libtreeattn_debug.so, checks:
 * every page-table lookup, TMA pool row and output row of its kernels, skipping the access and
 * setting a status bit instead of faulting) or a CUDA error is pending (TA_ERR_CUDA); clears
 * the status with a copy on `stream` (other streams are not waited for). */
int tree_attn_check(const ta_plan *plan, void *stream);

/* Diagnostic: runs the bounded-wait error path on purpose.  Launches one kernel on `stream`
 * in which a single thread waits, for limit_us microseconds (100 .. 1,000,000), on a
 * shared-memory mbarrier that nothing arrives on; the wait expires, the kernel sets this
 * plan's timeout status bit exactly as the attention kernels do when a wait of theirs runs
 * out, and returns normally.  The next tree_attn_check on the plan returns
 * TA_ERR_DEVICE_TIMEOUT and clears the status; the CUDA context stays usable.  Returns
 * TA_ERR_INVALID for a NULL or host-only plan or a limit outside the range, TA_ERR_CUDA for a
 * launch failure. */
int tree_attn_selftest_timeout(const ta_plan *plan, int64_t limit_us, void *stream);

/* Optional per-kernel tracing.  With events set, tree_attn_fwd records events[0] before and
 * events[1] after its kernels (the forward and, for a plan with split blocks, the combine);
 * tree_attn_bwd records events[2], [3], [4], [5] before its
 * delta, dQ, dK/dV and reduce kernels and events[6] after the last one -- all on the call's
 * stream (cudaEvent_t handles created and owned by the caller; entries may be NULL).  Pass
 * events = NULL to stop.  n_events must be 7 unless events is NULL. */
int tree_attn_set_trace_events(ta_plan *plan, void *const *events, int n_events);

int tree_attn_plan_stats(const ta_plan *plan, ta_plan_stats *out);
int tree_attn_plan_export(const ta_plan *plan, ta_plan_arrays *out);
void tree_attn_plan_destroy(ta_plan *plan);
const char *tree_attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TREEATTN_H */
