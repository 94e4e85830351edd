// Host planner: episode DAG -> query blocks, visible key intervals, key tiles, transpose.
//
// Follows Octopus (arXiv 2611.06956) Section 3.3 item 1 (split the episode into maximal
// contiguous nodes at fork / read_thread boundaries, record parent, active mounts and start
// position), Eq. 2 (monotonic position continuation after a mount), Eq. 4 (a node's keys
// are [mounted spans || ancestor prefix || own rows], the causal triangle on the own rows),
// and HARTS (arXiv 2608.28158) Section 4.2 Eq. 21-22 (query i of a branch with h ancestor
// rows sees key j iff j <= h + i).  Instead of materialising Eq. 4's gathered K/V per node,
// the plan lists the visible compact-row intervals and the kernels read the pages in place.
#include <algorithm>
#include <array>
#include <chrono>
#include <climits>
#include <cmath>
#include <cstring>
#include <functional>
#include <numeric>

#include "plan.h"

namespace treeattn {

namespace {

struct Mount {
    int32_t reader, t, source, lo, hi;
};

struct Interval {
    int64_t lo, hi;
};

void merge_intervals(std::vector<Interval> &iv) {
    std::sort(iv.begin(), iv.end(), [](const Interval &a, const Interval &b) {
        return a.lo < b.lo || (a.lo == b.lo && a.hi < b.hi);
    });
    size_t w = 0;
    for (size_t i = 0; i < iv.size(); ++i) {
        if (iv[i].hi <= iv[i].lo) continue;
        if (w > 0 && iv[i].lo <= iv[w - 1].hi) {
            iv[w - 1].hi = std::max(iv[w - 1].hi, iv[i].hi);
        } else {
            iv[w++] = iv[i];
        }
    }
    iv.resize(w);
}

int fail(int code, const std::string &msg) {
    set_error(msg);
    return code;
}

// Packs one query block's visible key rows into tiles of 4 slots x 32 rows (see plan.h).
// `items`: the block's visible intervals, the own-rows run flagged causal; r0: its first row.
// Every interval is cut into 32-row-aligned pieces; an even piece followed by the next one
// forms a 64-row half (one TMA box when pages hold >= 64 rows), the other pieces pair up into
// halves of two single boxes; halves fill tiles in order.  Rows outside the block's visible
// set occupy only the uncovered ends of pieces and the empty slot of a last half or tile.
// Streams the pieces (no per-block allocation: the planner calls this once per block).
struct Piece {
    int64_t q;
    int32_t lo, hi;
    bool causal;
};

struct Packer {
    std::vector<std::pair<Interval, bool>> its;
    Piece half[2][2];
    bool joined[2];
    int n_halves = 0;
    Piece single{-1, 0, 0, false}, even{-1, 0, 0, false};
    bool have_single = false, have_even = false, half_boxes = false;
    std::vector<int32_t> *out = nullptr;

    void emit_tile() {
        const Piece none{-1, 0, 0, false};
        Piece s[4] = {half[0][0], half[0][1], n_halves > 1 ? half[1][0] : none, n_halves > 1 ? half[1][1] : none};
        int32_t flags = (joined[0] ? kPackHalf64 : 0) | (n_halves > 1 && joined[1] ? kPackHalf64 << 1 : 0);
        for (int k = 0; k < 4; ++k) {
            if (s[k].causal) flags |= kPackCausal << k;
            if (s[k].q < 0 || s[k].lo != 0 || s[k].hi != kPieceRows || s[k].causal) flags |= kPackMask;
        }
        const int32_t rec[kPackInts] = {int32_t(s[0].q), int32_t(s[1].q), int32_t(s[2].q), int32_t(s[3].q),
                                        s[0].lo | s[0].hi << 6 | s[1].lo << 12 | s[1].hi << 18,
                                        s[2].lo | s[2].hi << 6 | s[3].lo << 12 | s[3].hi << 18, flags, 0};
        out->insert(out->end(), rec, rec + kPackInts);
        n_halves = 0;
    }
    void push_half(const Piece &a, const Piece &b, bool j) {
        half[n_halves][0] = a;
        half[n_halves][1] = b;
        joined[n_halves] = j;
        if (++n_halves == 2) emit_tile();
    }
    void push_single(const Piece &p) {
        if (have_single) {
            push_half(single, p, false);
            have_single = false;
        } else {
            single = p;
            have_single = true;
        }
    }
    // pieces arrive in (q, lo) order; an even piece waits to see whether the next one is q + 1
    void add(const Piece &p) {
        if (have_even) {
            have_even = false;
            if (p.q == even.q + 1) {
                push_half(even, p, half_boxes);
                return;
            }
            push_single(even);
        }
        if (p.q % 2 == 0) {
            even = p;
            have_even = true;
        } else {
            push_single(p);
        }
    }

    void run(const std::vector<std::pair<Interval, bool>> &items, int64_t r0, bool hb, std::vector<int32_t> &dst) {
        out = &dst;
        half_boxes = hb;
        its.assign(items.begin(), items.end());
        std::sort(its.begin(), its.end(), [](const std::pair<Interval, bool> &a, const std::pair<Interval, bool> &b) {
            return a.first.lo < b.first.lo;
        });
        n_halves = 0;
        have_single = have_even = false;
        for (const auto &it : its) {
            const Interval x = it.first;
            for (int64_t q = x.lo / kPieceRows; q * kPieceRows < x.hi; ++q) {
                const int64_t a = std::max<int64_t>(x.lo, q * kPieceRows), z = std::min<int64_t>(x.hi, (q + 1) * kPieceRows);
                add({q, int32_t(a - q * kPieceRows), int32_t(z - q * kPieceRows), it.second && z - 1 > r0});
            }
        }
        if (have_even) push_single(even);
        if (have_single) push_half(single, Piece{-1, 0, 0, false}, false);
        if (n_halves == 1) emit_tile();
    }
};

}  // namespace

int build_host_plan(const ta_branch *branches, int32_t n_branches, const ta_mount *mounts,
                    int32_t n_mounts, const int32_t *page_table, int64_t n_logical_pages,
                    const ta_config *config, int device_sms, HostPlan &P) {
    auto t_start = std::chrono::steady_clock::now();
    if (!config) return fail(TA_ERR_INVALID, "config is NULL");
    if (n_branches < 0 || n_mounts < 0) return fail(TA_ERR_INVALID, "negative count");
    if ((n_branches > 0 && !branches) || (n_mounts > 0 && !mounts))
        return fail(TA_ERR_INVALID, "NULL branch or mount array");
    const ta_config &c = *config;
    if (c.num_q_heads <= 0 || c.num_kv_heads <= 0 || c.num_q_heads % c.num_kv_heads != 0)
        return fail(TA_ERR_UNSUPPORTED, "num_q_heads must be a positive multiple of num_kv_heads");
    const int G = c.num_q_heads / c.num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16)
        return fail(TA_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4, 8 or 16");
    if (c.head_dim != 64 && c.head_dim != 128)
        return fail(TA_ERR_UNSUPPORTED, "head_dim must be 64 or 128");
    if (c.page_size != 16 && c.page_size != 32 && c.page_size != 64 && c.page_size != 128)
        return fail(TA_ERR_UNSUPPORTED, "page_size must be 16, 32, 64 or 128");
    if (c.num_pages <= 0 || c.num_pages > (int64_t(1) << 31) / c.page_size)
        return fail(TA_ERR_INVALID, "num_pages out of range");
    P.cfg = c;
    P.G = G;
    P.block_rows = kBlockMRows / G;
    P.scale = c.softmax_scale > 0.f ? c.softmax_scale : 1.0f / std::sqrt(float(c.head_dim));

    // ------------------------------------------------------------------ branches
    const int nb = n_branches;
    std::vector<int32_t> par(nb), fork(nb), len(nb);
    std::vector<int64_t> rs(nb);
    int64_t N = 0;
    for (int b = 0; b < nb; ++b) {
        par[b] = branches[b].parent;
        fork[b] = branches[b].fork_offset;
        len[b] = branches[b].length;
        rs[b] = branches[b].row_start;
        if (par[b] < -1 || par[b] >= nb || par[b] == b)
            return fail(TA_ERR_INVALID, "branch " + std::to_string(b) + ": bad parent");
        if (len[b] < 0) return fail(TA_ERR_INVALID, "branch " + std::to_string(b) + ": negative length");
        if (rs[b] < 0) return fail(TA_ERR_INVALID, "branch " + std::to_string(b) + ": negative row_start");
        N += len[b];
    }
    if (N > INT32_MAX - 2 * kTileRows) return fail(TA_ERR_INVALID, "too many rows (N >= 2^31)");
    for (int b = 0; b < nb; ++b) {
        if (par[b] < 0) {
            if (fork[b] != 0) return fail(TA_ERR_INVALID, "branch " + std::to_string(b) + ": root with a fork offset");
        } else if (fork[b] < 0 || fork[b] > len[par[b]]) {
            return fail(TA_ERR_INVALID, "branch " + std::to_string(b) + ": fork offset outside its parent");
        }
        int steps = 0;   // parent chain must reach a root
        for (int x = b; x >= 0; x = par[x])
            if (++steps > nb + 1) return fail(TA_ERR_INVALID, "cycle in parent links at branch " + std::to_string(b));
    }
    {   // row ranges must tile [0, N) exactly
        std::vector<int> order(nb);
        std::iota(order.begin(), order.end(), 0);
        std::sort(order.begin(), order.end(), [&](int a, int b) { return rs[a] < rs[b] || (rs[a] == rs[b] && len[a] < len[b]); });
        int64_t cur = 0;
        for (int b : order) {
            if (len[b] == 0) {
                if (rs[b] > N) return fail(TA_ERR_INVALID, "empty branch row_start beyond the strip");
                continue;
            }
            if (rs[b] != cur)
                return fail(TA_ERR_INVALID, rs[b] < cur ? "branch row ranges overlap" : "branch row ranges leave a gap");
            cur = rs[b] + len[b];
        }
    }
    P.N = N;

    // ------------------------------------------------------------------ mounts
    const bool no_mounts = (c.flags & TA_NO_MOUNTS) != 0;
    const bool transitive = (c.flags & TA_TRANSITIVE_MOUNTS) != 0;
    if (no_mounts && transitive) return fail(TA_ERR_INVALID, "TA_NO_MOUNTS and TA_TRANSITIVE_MOUNTS exclude each other");
    std::vector<Mount> mt;
    for (int i = 0; i < n_mounts; ++i) {
        Mount m{mounts[i].reader, mounts[i].reader_offset, mounts[i].source, mounts[i].src_begin, mounts[i].src_end};
        if (m.reader < 0 || m.reader >= nb || m.source < 0 || m.source >= nb)
            return fail(TA_ERR_INVALID, "mount " + std::to_string(i) + ": branch index out of range");
        if (c.flags & TA_CLAMP_MOUNTS) {
            m.lo = std::max(m.lo, 0);
            m.hi = std::min(m.hi, len[m.source]);
        }
        if (m.hi <= m.lo) {
            if (m.hi < m.lo && !(c.flags & TA_CLAMP_MOUNTS))
                return fail(TA_ERR_INVALID, "mount " + std::to_string(i) + ": span end before begin");
            continue;  // empty span: no rows, no position jump
        }
        if (m.lo < 0 || m.hi > len[m.source])
            return fail(TA_ERR_INVALID, "mount " + std::to_string(i) + ": span outside the source branch");
        if (m.t < 0 || m.t >= len[m.reader])
            return fail(TA_ERR_INVALID, "mount " + std::to_string(i) + ": reader offset outside the reader");
        mt.push_back(m);
    }
    std::vector<std::vector<int>> mounts_of(nb);   // non-empty mounts per reader, by offset
    for (int i = 0; i < (int)mt.size(); ++i) mounts_of[mt[i].reader].push_back(i);
    for (auto &v : mounts_of)
        std::stable_sort(v.begin(), v.end(), [&](int a, int b) { return mt[a].t < mt[b].t; });

    // Causality: the rows a span depends on (transitively through visibility) must not
    // include the reader's row at its mount offset.  reach[x] = number of leading rows of
    // branch x the span depends on; need[x] = x's inherited rows are depended on.
    {
        std::vector<int64_t> reach(nb);
        std::vector<char> need(nb);
        for (size_t mi = 0; mi < mt.size(); ++mi) {
            const Mount &m = mt[mi];
            std::fill(reach.begin(), reach.end(), 0);
            std::fill(need.begin(), need.end(), 0);
            reach[m.source] = m.hi;
            need[m.source] = 1;
            bool changed = true;
            while (changed) {
                changed = false;
                for (int x = 0; x < nb; ++x) {
                    if (!need[x] && reach[x] == 0) continue;
                    if (reach[x] > 0) need[x] = 1;
                    int p = par[x];
                    if (p >= 0) {
                        if (fork[x] > reach[p]) { reach[p] = fork[x]; changed = true; }
                        if (!need[p]) { need[p] = 1; changed = true; }
                    }
                    for (int k : mounts_of[x]) {
                        if (mt[k].t < reach[x] && mt[k].hi > reach[mt[k].source]) {
                            reach[mt[k].source] = mt[k].hi;
                            changed = true;
                        }
                        if (mt[k].t < reach[x] && !need[mt[k].source]) { need[mt[k].source] = 1; changed = true; }
                    }
                }
            }
            if (reach[m.reader] > m.t)
                return fail(TA_ERR_INVALID, "mount " + std::to_string(mi) + ": mounted span depends on the reader's own rows at or after the mount offset");
        }
    }

    // ------------------------------------------------------------------ page table
    const int Pg = c.page_size;
    const int64_t need_pages = (N + Pg - 1) / Pg;
    if (n_logical_pages < need_pages) return fail(TA_ERR_INVALID, "page table shorter than the strip");
    if (need_pages > 0 && !page_table) return fail(TA_ERR_INVALID, "page table is NULL");
    P.n_logical_pages = need_pages;
    P.page_table.assign(page_table, page_table + need_pages);
    {
        std::vector<char> used(c.num_pages, 0);
        for (int64_t l = 0; l < need_pages; ++l) {
            int32_t pp = P.page_table[l];
            if (pp < 0 || pp >= c.num_pages) return fail(TA_ERR_INVALID, "page table entry out of range");
            if (used[pp]) return fail(TA_ERR_INVALID, "page table maps two logical pages to one physical page");
            used[pp] = 1;
        }
    }

    // ------------------------------------------------------------------ positions (Eq. 2)
    {
        std::vector<std::vector<int64_t>> pos(nb);
        for (int b = 0; b < nb; ++b) pos[b].resize(len[b]);
        std::vector<int32_t> done(nb, 0);
        std::vector<size_t> mcur(nb, 0);
        std::vector<char> busy(nb, 0);
        bool ok = true;
        std::function<bool(int, int)> ensure;
        std::function<int64_t(int)> start_next = [&](int b) -> int64_t {
            int p = par[b];
            if (p < 0) return 0;
            if (fork[b] == 0) return start_next(p);
            if (!ensure(p, fork[b] - 1)) return -1;
            return pos[p][fork[b] - 1] + 1;
        };
        ensure = [&](int b, int i) -> bool {
            if (done[b] > i) return true;
            if (busy[b]) return false;
            busy[b] = 1;
            while (done[b] <= i) {
                const int j = done[b];
                int64_t nxt = j == 0 ? start_next(b) : pos[b][j - 1] + 1;
                if (nxt < 0) return false;
                while (mcur[b] < mounts_of[b].size() && mt[mounts_of[b][mcur[b]]].t == j) {
                    const Mount &m = mt[mounts_of[b][mcur[b]]];
                    if (!ensure(m.source, m.hi - 1)) return false;
                    nxt = std::max(nxt, pos[m.source][m.hi - 1] + 1);
                    ++mcur[b];
                }
                pos[b][j] = nxt;
                ++done[b];
            }
            busy[b] = 0;
            return true;
        };
        P.pos_ids.assign(N, 0);
        for (int b = 0; b < nb && ok; ++b) {
            if (len[b] == 0) continue;
            ok = ensure(b, len[b] - 1);
            if (!ok) break;
            for (int i = 0; i < len[b]; ++i) {
                if (pos[b][i] > INT32_MAX) return fail(TA_ERR_INVALID, "position id beyond 2^31");
                P.pos_ids[rs[b] + i] = (int32_t)pos[b][i];
            }
        }
        if (!ok) return fail(TA_ERR_INVALID, "cyclic position dependency (non-causal mount)");
    }

    // ------------------------------------------------------------------ visible mounted spans
    // Per mount, the compact-row intervals it makes visible: its own span; with
    // TA_TRANSITIVE_MOUNTS also, recursively, the spans of the mounts in effect at the source's
    // last mounted row (the source's own mounts up to that row and those it inherits through
    // its fork points).  With TA_NO_MOUNTS nothing (positions above keep the mounts).
    std::vector<std::vector<Interval>> span_of(mt.size());
    {
        // mounts in effect at row (x, r): x's own with t <= r, then inherited along the parents
        auto in_effect = [&](int x, int32_t r, std::vector<int> &out) {
            for (int k : mounts_of[x])
                if (mt[k].t <= r) out.push_back(k);
            for (int y = x; par[y] >= 0; y = par[y])
                if (fork[y] > 0)
                    for (int k : mounts_of[par[y]])
                        if (mt[k].t <= fork[y] - 1) out.push_back(k);
        };
        std::vector<char> state(mt.size(), 0);   // 0 new, 1 on the stack, 2 done
        std::function<bool(int)> close = [&](int k) -> bool {
            if (state[k] == 2) return true;
            if (state[k] == 1) return false;     // a cycle: impossible for causal mounts
            state[k] = 1;
            std::vector<Interval> &v = span_of[k];
            v.push_back({rs[mt[k].source] + mt[k].lo, rs[mt[k].source] + mt[k].hi});
            if (transitive) {
                std::vector<int> eff;
                in_effect(mt[k].source, mt[k].hi - 1, eff);
                for (int k2 : eff) {
                    if (!close(k2)) return false;
                    v.insert(v.end(), span_of[k2].begin(), span_of[k2].end());
                }
                merge_intervals(v);
            }
            state[k] = 2;
            return true;
        };
        if (!no_mounts)
            for (int k = 0; k < (int)mt.size(); ++k)
                if (!close(k)) return fail(TA_ERR_INVALID, "cyclic transitive mounts");
    }

    // ------------------------------------------------------------------ segments and blocks
    const int R = P.block_rows;
    const int T = kTileRows;
    std::vector<int32_t> &blocks = P.blocks;
    std::vector<int64_t> &ivp = P.blk_iv_ptr;
    ivp.assign(1, 0);
    std::vector<int64_t> block_pairs;
    for (int b = 0; b < nb; ++b) {
        if (len[b] == 0) continue;
        // rows inherited from the ancestors (same for every row of b)
        std::vector<Interval> inh;
        for (int x = b; par[x] >= 0; x = par[x]) {
            int p = par[x], f = fork[x];
            if (f > 0) {
                inh.push_back({rs[p], rs[p] + f});
                if (!no_mounts)
                    for (int k : mounts_of[p])
                        if (mt[k].t <= f - 1) inh.insert(inh.end(), span_of[k].begin(), span_of[k].end());
            }
        }
        std::vector<int32_t> cuts{0, len[b]};
        if (!no_mounts)
            for (int k : mounts_of[b]) cuts.push_back(mt[k].t);
        std::sort(cuts.begin(), cuts.end());
        cuts.erase(std::unique(cuts.begin(), cuts.end()), cuts.end());
        for (size_t s = 0; s + 1 < cuts.size(); ++s) {
            const int32_t slo = cuts[s], shi = cuts[s + 1];
            ++P.n_segments;
            std::vector<Interval> base = inh;
            if (!no_mounts)
                for (int k : mounts_of[b])
                    if (mt[k].t <= slo) base.insert(base.end(), span_of[k].begin(), span_of[k].end());
            for (int32_t qs = slo; qs < shi; qs += R) {
                const int32_t qe = std::min<int32_t>(qs + R, shi);
                std::vector<Interval> iv = base;
                iv.push_back({rs[b], rs[b] + qs});
                merge_intervals(iv);
                const int64_t dlo = rs[b] + qs, dhi = rs[b] + qe;
                for (const Interval &x : iv)
                    if (x.lo < dhi && x.hi > dlo)
                        return fail(TA_ERR_INVALID, "internal: a visible interval overlaps the diagonal");
                int64_t vis = 0;
                for (const Interval &x : iv) {
                    P.iv_lo.push_back((int32_t)x.lo);
                    P.iv_hi.push_back((int32_t)x.hi);
                    vis += x.hi - x.lo;
                }
                ivp.push_back((int64_t)P.iv_lo.size());
                P.diag.push_back((int32_t)dlo);
                P.diag.push_back((int32_t)dhi);
                const int64_t n = qe - qs;
                block_pairs.push_back(n * vis + n * (n + 1) / 2);
                P.pairs += n * vis + n * (n + 1) / 2;
                blocks.push_back((int32_t)dlo);
                blocks.push_back((int32_t)n);
                blocks.push_back(0);
                blocks.push_back(0);
            }
        }
    }
    const int64_t n_blocks = (int64_t)blocks.size() / 4;

    // ------------------------------------------------------------------ key-tile entries
    P.fblk_ptr.assign(1, 0);
    Packer packer;
    P.ftiles.reserve(size_t(n_blocks) * 64 * kPackInts);
    for (int64_t qb = 0; qb < n_blocks; ++qb) {
        const int64_t r0 = blocks[4 * qb];
        blocks[4 * qb + 2] = (int32_t)(P.entries.size() / 4);
        std::vector<std::pair<Interval, bool>> items;
        for (int64_t e = ivp[qb]; e < ivp[qb + 1]; ++e) items.push_back({{P.iv_lo[e], P.iv_hi[e]}, false});
        Interval d{P.diag[2 * qb], P.diag[2 * qb + 1]};
        bool merged = false;
        for (auto &it : items)
            if (it.first.hi == d.lo) {         // own earlier rows + diagonal as one causal run
                it.first.hi = d.hi;
                it.second = true;
                merged = true;
            }
        if (!merged) items.push_back({d, true});
        for (auto &it : items) {
            const Interval x = it.first;
            for (int64_t k = x.lo / T; k * T < x.hi; ++k) {
                const int64_t lo = std::max<int64_t>(x.lo, k * T), hi = std::min<int64_t>(x.hi, (k + 1) * T);
                int32_t flags = 0;
                if (it.second && hi - 1 > r0) flags |= kEntryCausal;
                if (lo != k * T || hi != (k + 1) * T) flags |= kEntryPartial;
                P.entries.insert(P.entries.end(), {(int32_t)k, (int32_t)lo, (int32_t)hi, flags});
            }
        }
        blocks[4 * qb + 3] = (int32_t)(P.entries.size() / 4);
        packer.run(items, r0, Pg >= 64, P.ftiles);
        P.fblk_ptr.push_back((int64_t)(P.ftiles.size() / kPackInts));
    }
    const int64_t n_entries = (int64_t)P.entries.size() / 4;

    // launch order for query-major kernels: most packed tiles first (LPT)
    P.fwd_order.resize(n_blocks);
    std::iota(P.fwd_order.begin(), P.fwd_order.end(), 0);
    std::stable_sort(P.fwd_order.begin(), P.fwd_order.end(), [&](int32_t a, int32_t b) {
        return P.fblk_ptr[a + 1] - P.fblk_ptr[a] > P.fblk_ptr[b + 1] - P.fblk_ptr[b];
    });

    // ------------------------------------------------------------------ transpose (tile-major)
    const int64_t n_tiles = (N + T - 1) / T;
    std::vector<int64_t> tptr(n_tiles + 1, 0);
    for (int64_t e = 0; e < n_entries; ++e) ++tptr[P.entries[4 * e] + 1];
    for (int64_t k = 0; k < n_tiles; ++k) tptr[k + 1] += tptr[k];
    P.t_entries.assign(4 * n_entries, 0);
    {
        std::vector<int64_t> fill(tptr.begin(), tptr.end() - 1);
        for (int64_t qb = 0; qb < n_blocks; ++qb)
            for (int32_t e = blocks[4 * qb + 2]; e < blocks[4 * qb + 3]; ++e) {
                const int64_t k = P.entries[4 * e];
                const int64_t w = fill[k]++;
                P.t_entries[4 * w] = (int32_t)qb;
                P.t_entries[4 * w + 1] = P.entries[4 * e + 1];
                P.t_entries[4 * w + 2] = P.entries[4 * e + 2];
                P.t_entries[4 * w + 3] = P.entries[4 * e + 3];
            }
    }
    // chunks: bound the entries per dK/dV work item so that no item is much longer than a
    // quarter of the average per-SM share (the work per entry is about constant)
    P.num_sms = c.num_sms > 0 ? c.num_sms : (device_sms > 0 ? device_sms : kDefaultSms);
    const int64_t work = n_entries * c.num_kv_heads;
    const int64_t cap = c.dkdv_chunk_entries > 0 ? int64_t(c.dkdv_chunk_entries)
                                                 : std::max<int64_t>(8, work / (int64_t(P.num_sms) * 4));
    P.chunk_cap = cap;

    // forward work items (split-KV): a query block whose packed-tile list is long against one
    // worker's share of the forward is cut into parts of at most fwd_split_cap tiles; each part
    // is a work item writing a partial O and lse that a combine step merges.  Workers are SM
    // pairs for head dim 128 (the forward on CTA pairs) and SMs for 64.  The (block, KV head)
    // items run longest first, so the forward's span is about max(share, longest block): only
    // a longest block well above the share (1.5x, and by 32 tiles: the combine and the parts'
    // partial O cost about as much as 8 tiles) is worth splitting, and then the automatic cap
    // is the share (at least 16 tiles).  Otherwise the cap is the longest block (no split).
    {
        int64_t longest = 0;
        for (size_t b = 0; b + 1 < P.fblk_ptr.size(); ++b) longest = std::max(longest, P.fblk_ptr[b + 1] - P.fblk_ptr[b]);
        const int64_t workers = std::max<int64_t>(1, c.head_dim == 128 ? P.num_sms / 2 : P.num_sms);
        const int64_t share = (P.fblk_ptr.back() * c.num_kv_heads + workers - 1) / workers;
        int64_t split_cap = longest;
        if (c.fwd_split_tiles > 0) split_cap = c.fwd_split_tiles;
        else if (c.fwd_split_tiles == 0 && 2 * longest > 3 * share && longest - share >= 32)
            split_cap = std::max<int64_t>(16, share);
        P.fwd_split_cap = split_cap;
        std::vector<std::array<int32_t, 4>> items;
        for (int32_t qb : P.fwd_order) {
            const int64_t a = P.fblk_ptr[qb], z = P.fblk_ptr[qb + 1];
            if (z - a <= split_cap) {
                items.push_back({qb, (int32_t)a, (int32_t)z, -1});
                continue;
            }
            // parts of floor or ceil of (z - a) / parts tiles: none empty, none above the cap
            const int64_t n = z - a, parts = (n + split_cap - 1) / split_cap;
            P.fwd_combine.insert(P.fwd_combine.end(), {qb, (int32_t)P.n_fwd_slots, (int32_t)parts, 0});
            for (int64_t k = 0; k < parts; ++k)
                items.push_back({qb, (int32_t)(a + k * n / parts), (int32_t)(a + (k + 1) * n / parts),
                                 (int32_t)P.n_fwd_slots++});
        }
        // longest first (stable: the block order breaks ties)
        std::stable_sort(items.begin(), items.end(),
                         [](const std::array<int32_t, 4> &x, const std::array<int32_t, 4> &y) {
                             return x[2] - x[1] > y[2] - y[1];
                         });
        P.fwd_items.reserve(items.size() * 4);
        for (auto &it : items) P.fwd_items.insert(P.fwd_items.end(), it.begin(), it.end());
    }
    std::vector<std::array<int64_t, 4>> ch;
    for (int64_t k = 0; k < n_tiles; ++k) {
        const int64_t a = tptr[k], z = tptr[k + 1];
        if (z == a) continue;
        const int64_t pieces = (z - a + cap - 1) / cap;
        const int64_t first_slot = pieces > 1 ? P.n_partial_slots : -1;
        for (int64_t i = 0; i < pieces; ++i) {
            const int64_t lo = a + (z - a) * i / pieces, hi = a + (z - a) * (i + 1) / pieces;
            ch.push_back({k, lo, hi, pieces > 1 ? first_slot + i : -1});
        }
        if (pieces > 1) {
            P.reduce.insert(P.reduce.end(), {(int32_t)k, (int32_t)first_slot, (int32_t)pieces, 0});
            P.n_partial_slots += pieces;
        }
    }
    std::stable_sort(ch.begin(), ch.end(), [](const std::array<int64_t, 4> &a, const std::array<int64_t, 4> &b) {
        return a[2] - a[1] > b[2] - b[1];
    });
    for (auto &x : ch) P.chunks.insert(P.chunks.end(), {(int32_t)x[0], (int32_t)x[1], (int32_t)x[2], (int32_t)x[3]});

    // device-side helpers: TMA rows of every tile's pages; reader info per tile-major entry
    {
        const int ppt = T / Pg;
        P.tile_rows.assign(n_tiles * ppt, 0);
        for (int64_t k = 0; k < n_tiles; ++k)
            for (int i = 0; i < ppt; ++i) {
                const int64_t l = k * ppt + i;
                P.tile_rows[k * ppt + i] = l < need_pages ? P.page_table[l] * Pg : int32_t(c.num_pages * Pg);
            }
        P.t_info.assign(4 * n_entries, 0);
        for (int64_t e = 0; e < n_entries; ++e) {
            const int32_t b = P.t_entries[4 * e];
            P.t_info[4 * e] = (b << 2) | P.t_entries[4 * e + 3];
            P.t_info[4 * e + 1] = blocks[4 * b];
            P.t_info[4 * e + 2] = P.t_entries[4 * e + 1];
            P.t_info[4 * e + 3] = P.t_entries[4 * e + 2];
        }
    }

    P.plan_ms = std::chrono::duration<double, std::milli>(std::chrono::steady_clock::now() - t_start).count();
    return TA_OK;
}

}  // namespace treeattn
