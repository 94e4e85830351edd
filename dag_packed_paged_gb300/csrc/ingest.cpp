// Trajectory ingestion: raw token trajectories -> the compact prefix-tree DAG.
//
// HARTS (arXiv 2608.28158) Section 2.1 keeps one compact row per distinct token prefix and a
// map m: S -> C from every semantic position s = (trajectory, offset) to its compact row
// (Eq. 3); Section 3.2 counts the rows of a trajectory set as
//   C(M) = |x_1| + sum_{i >= 2} (|x_i| - LCP(x_{i-1}, x_i))        (Eq. 5)
// over the trajectories in lexicographic order, where the immediate predecessor gives the
// longest prefix shared with any trajectory already inserted.  Building the tree in that order
// gives exactly C(M) rows: each trajectory forks from the branch of its predecessor's path
// that holds its last shared token, at that token's offset within the branch, and its
// unshared suffix becomes a new branch.  Branches are laid out in creation order, which is a
// depth-first order of the prefix tree (every subtree's rows are contiguous).
#include <algorithm>
#include <cstring>
#include <numeric>
#include <string>
#include <vector>

#include "plan.h"

namespace treeattn {
void set_error(const std::string &msg);
}

using treeattn::set_error;

extern "C" int tree_attn_ingest(const int32_t *tokens, const int64_t *offsets, int32_t n_traj,
                                ta_branch *branches, int32_t max_branches, int32_t *n_branches,
                                int32_t *row_tokens, int64_t max_rows, int64_t *n_rows, int64_t *row_of,
                                int32_t *row_owner) {
    treeattn::NvtxRange nvtx_range("tree_attn_ingest");
    if (n_traj < 0 || !offsets || !n_branches || !n_rows || (n_traj > 0 && !row_of)) {
        set_error("tree_attn_ingest: bad arguments");
        return TA_ERR_INVALID;
    }
    for (int32_t i = 0; i < n_traj; ++i)
        if (offsets[i + 1] < offsets[i] || offsets[i] < 0) {
            set_error("tree_attn_ingest: offsets must be non-decreasing from 0");
            return TA_ERR_INVALID;
        }
    const int64_t total = n_traj > 0 ? offsets[n_traj] : 0;
    if (total > 0 && !tokens) {
        set_error("tree_attn_ingest: tokens is NULL");
        return TA_ERR_INVALID;
    }
    auto len = [&](int32_t i) { return offsets[i + 1] - offsets[i]; };
    auto tok = [&](int32_t i) { return tokens + offsets[i]; };

    // lexicographic order (ties keep the input order)
    std::vector<int32_t> order(n_traj);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
        return std::lexicographical_compare(tok(a), tok(a) + len(a), tok(b), tok(b) + len(b));
    });

    struct Seg { int32_t branch; int64_t start; };   // a branch on the current path, from offset start
    std::vector<Seg> path;                           // path of the previous trajectory
    std::vector<ta_branch> out;
    int64_t rows = 0;
    int32_t prev = -1;
    for (int32_t i : order) {
        const int64_t n = len(i);
        int64_t lcp = 0;
        if (prev >= 0) {
            const int64_t m = std::min(n, len(prev));
            const int32_t *a = tok(prev), *b = tok(i);
            while (lcp < m && a[lcp] == b[lcp]) ++lcp;
        }
        // keep the path's branches that hold offsets < lcp; the last one is the fork parent
        while (!path.empty() && path.back().start >= lcp) path.pop_back();
        if (n > lcp) {
            ta_branch br;
            if (path.empty()) {
                br.parent = -1;
                br.fork_offset = 0;
            } else {
                br.parent = path.back().branch;
                br.fork_offset = static_cast<int32_t>(lcp - path.back().start);
            }
            br.length = static_cast<int32_t>(n - lcp);
            br.row_start = rows;
            if ((int64_t)out.size() >= max_branches || rows + (n - lcp) > max_rows) {
                set_error("tree_attn_ingest: output capacity too small");
                return TA_ERR_INVALID;
            }
            if (row_tokens) std::memcpy(row_tokens + rows, tok(i) + lcp, sizeof(int32_t) * (n - lcp));
            if (row_owner) std::fill(row_owner + rows, row_owner + rows + (n - lcp), i);
            rows += n - lcp;
            out.push_back(br);
            path.push_back({static_cast<int32_t>(out.size() - 1), lcp});
        }
        // the compact row of every offset of trajectory i, along its path
        for (size_t k = 0; k < path.size(); ++k) {
            const int64_t a = path[k].start;
            const int64_t z = k + 1 < path.size() ? path[k + 1].start : n;
            const ta_branch &b = out[path[k].branch];
            for (int64_t t = a; t < z && t < n; ++t) row_of[offsets[i] + t] = b.row_start + (t - a);
        }
        prev = i;
    }
    if (branches) std::copy(out.begin(), out.end(), branches);
    *n_branches = static_cast<int32_t>(out.size());
    *n_rows = rows;
    return TA_OK;
}

// The positions of every compact row, for the backward of the compact log-probabilities: a
// CSR (row_ptr[C + 1], row_pos[S]) of the semantic positions grouped by compact row and, within
// a row, ordered by target token (then by position), so that positions sharing a target are
// adjacent and the kernel sums their gradients in a fixed order.
extern "C" int tree_attn_logprob_index(const int64_t *pos_row, const int32_t *pos_target, int64_t n_pos,
                                       int64_t n_rows, int64_t vocab, int64_t *row_ptr, int64_t *row_pos) {
    if (n_pos < 0 || n_rows < 0 || vocab <= 0 || !row_ptr || (n_pos > 0 && (!pos_row || !pos_target || !row_pos))) {
        set_error("tree_attn_logprob_index: bad arguments");
        return TA_ERR_INVALID;
    }
    std::fill(row_ptr, row_ptr + n_rows + 1, 0);
    for (int64_t s = 0; s < n_pos; ++s) {
        if (pos_row[s] < 0 || pos_row[s] >= n_rows || pos_target[s] < 0 || pos_target[s] >= vocab) {
            set_error("tree_attn_logprob_index: position " + std::to_string(s) + " has a row or target out of range");
            return TA_ERR_INVALID;
        }
        ++row_ptr[pos_row[s] + 1];
    }
    for (int64_t c = 0; c < n_rows; ++c) row_ptr[c + 1] += row_ptr[c];
    std::vector<int64_t> fill(row_ptr, row_ptr + n_rows);
    for (int64_t s = 0; s < n_pos; ++s) row_pos[fill[pos_row[s]]++] = s;
    for (int64_t c = 0; c < n_rows; ++c)
        std::stable_sort(row_pos + row_ptr[c], row_pos + row_ptr[c + 1],
                         [&](int64_t a, int64_t b) { return pos_target[a] < pos_target[b]; });
    return TA_OK;
}

// Octopus (arXiv 2611.06956) Section 3.4, Eq. 6: a prefix-deduplicating loss mask that counts
// every generated token of the packed strip once, at the trajectory that owns its node, so that
// summing masked token log-probabilities over all trajectories gives the episode's score
// function (Eq. 7).  Position (l, t) of trajectory l (t < |l| - 1) predicts token t + 1 from the
// prefix ending at t; two positions predict the same thing exactly when their predicted tokens
// share a compact row, so the mask is 1 iff l owns that row (row_owner, from tree_attn_ingest:
// the trajectory whose insertion created the row) and the predicted token is generated.
// mask has the layout of `tokens`; the last entry of every trajectory is 0 (no next token).
extern "C" int tree_attn_owner_mask(const int64_t *offsets, int32_t n_traj, const int64_t *row_of,
                                    const int32_t *row_owner, const uint8_t *generated, uint8_t *mask) {
    if (n_traj < 0 || !offsets || (n_traj > 0 && (!row_of || !row_owner || !mask))) {
        set_error("tree_attn_owner_mask: bad arguments");
        return TA_ERR_INVALID;
    }
    for (int32_t l = 0; l < n_traj; ++l) {
        const int64_t a = offsets[l], z = offsets[l + 1];
        if (z < a) {
            set_error("tree_attn_owner_mask: offsets must be non-decreasing");
            return TA_ERR_INVALID;
        }
        for (int64_t k = a; k < z; ++k) {
            const bool has_next = k + 1 < z;
            mask[k] = has_next && row_owner[row_of[k + 1]] == l && (!generated || generated[k + 1]) ? 1 : 0;
        }
    }
    return TA_OK;
}
