// Compact-work microbatch planning across data-parallel replicas (host C++).
//
// Follows HARTS (arXiv 2608.28158) Section 3.2, "Prefix-aware microbatch planning and schedule
// construction": complete root-to-leaf trajectories are grouped into K microbatches of at most
// T compact rows each (a microbatch's work is the row count of the compact trie of its
// trajectories, Eq. 5), K a multiple of the replica count D, and the microbatches are assigned
// to replicas and slots.  Plans are ranked lexicographically by Eq. 4: total compact work, then
// the sum over slots of the slot's heaviest microbatch, then the heaviest replica's cumulative
// work.  Candidates come from
//   - the exact dynamic program of Eq. 9 over partitions contiguous in lexicographic order, for
//     every K of the range of Eq. 7-8 (up to N0 trajectories; above that, the natural partition
//     evolved by merges and splits to sampled K);
//   - trie-aware greedy insertion by the exact increase of Eq. 10, under four processing orders
//     and two placement policies, with K raised to a multiple of D by singleton splits.
// Every candidate then gets the DP-replica assignment of the section (microbatches sorted by
// work, consecutive blocks of D form a slot, heavier ones go to replicas with less work so far).
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <numeric>
#include <string>
#include <vector>

#include "plan.h"

namespace treeattn {

namespace {

using i64 = int64_t;

struct Traj {
    const int32_t *t;
    i64 n;
};

i64 lcp(const Traj &a, const Traj &b) {
    const i64 m = std::min(a.n, b.n);
    i64 i = 0;
    while (i < m && a.t[i] == b.t[i]) ++i;
    return i;
}

bool lex_less(const Traj &a, const Traj &b) {
    const i64 m = std::min(a.n, b.n);
    for (i64 i = 0; i < m; ++i)
        if (a.t[i] != b.t[i]) return a.t[i] < b.t[i];
    return a.n < b.n;
}

// A plan: membership (microbatch per trajectory, by input index), plus its assignment.
struct Plan {
    std::vector<int32_t> mb_of;      // per trajectory
    std::vector<i64> work;           // per microbatch
    std::vector<int32_t> replica, slot;
    i64 j1 = 0, j2 = 0, j3 = 0;      // Eq. 4
    int source = 0;                  // 0 exact / evolved contiguous, 1 greedy
};

// DP-replica assignment and the Eq. 4 objective.  K must be a multiple of D.
void assign(Plan &p, int D) {
    const int K = int(p.work.size());
    std::vector<int32_t> order(K);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return p.work[a] > p.work[b]; });
    p.replica.assign(K, 0);
    p.slot.assign(K, 0);
    std::vector<i64> load(D, 0);
    p.j1 = p.j2 = 0;
    for (int s = 0; s * D < K; ++s) {
        // replicas by cumulative work so far, least first; the slot's microbatches heaviest first
        std::vector<int32_t> reps(D);
        std::iota(reps.begin(), reps.end(), 0);
        std::stable_sort(reps.begin(), reps.end(), [&](int32_t a, int32_t b) { return load[a] < load[b]; });
        i64 heaviest = 0;
        for (int i = 0; i < D && s * D + i < K; ++i) {
            const int32_t m = order[s * D + i];
            p.replica[m] = reps[i];
            p.slot[m] = s;
            load[reps[i]] += p.work[m];
            heaviest = std::max(heaviest, p.work[m]);
        }
        p.j2 += heaviest;
    }
    for (i64 w : p.work) p.j1 += w;
    p.j3 = *std::max_element(load.begin(), load.end());
}

bool better(const Plan &a, const Plan &b) {
    if (a.j1 != b.j1) return a.j1 < b.j1;
    if (a.j2 != b.j2) return a.j2 < b.j2;
    return a.j3 < b.j3;
}

struct Planner {
    std::vector<Traj> X;
    int D = 1;
    i64 T = 0;
    int N = 0;
    std::vector<int32_t> sorted;     // trajectory indices in lexicographic order
    std::vector<i64> L;              // L[i] = LCP(sorted[i-1], sorted[i]), L[0] = 0
    std::vector<i64> A, Lp;          // prefix sums of lengths and of L

    // compact work of the contiguous run sorted[s..e] (inclusive, 0-based)
    i64 W(int s, int e) const { return (A[e + 1] - A[s]) - (Lp[e + 1] - Lp[s + 1]); }

    std::vector<std::vector<i64>> rmq;   // sparse table of minima of L

    void init() {
        N = int(X.size());
        sorted.resize(N);
        std::iota(sorted.begin(), sorted.end(), 0);
        std::stable_sort(sorted.begin(), sorted.end(), [&](int32_t a, int32_t b) { return lex_less(X[a], X[b]); });
        L.assign(N, 0);
        for (int i = 1; i < N; ++i) L[i] = lcp(X[sorted[i - 1]], X[sorted[i]]);
        A.assign(N + 1, 0);
        Lp.assign(N + 1, 0);
        for (int i = 0; i < N; ++i) {
            A[i + 1] = A[i] + X[sorted[i]].n;
            Lp[i + 1] = Lp[i] + L[i];
        }
        rmq.assign(1, L);
        for (int h = 1; (1 << h) <= N; ++h) {
            const auto &prev = rmq.back();
            std::vector<i64> cur(N, 0);
            for (int i = 0; i + (1 << h) <= N; ++i) cur[i] = std::min(prev[i], prev[i + (1 << (h - 1))]);
            rmq.push_back(std::move(cur));
        }
    }

    // LCP of the trajectories of lexicographic ranks a != b: the minimum adjacent LCP between
    // them (sorted strings share with a later one exactly what every step in between shares).
    i64 lcp_r(int a, int b) const {
        if (a > b) std::swap(a, b);
        const int lo = a + 1, n = b - a;                       // L[lo .. b]
        int h = 0;
        while ((2 << h) <= n) ++h;
        return std::min(rmq[h][lo], rmq[h][b - (1 << h) + 1]);
    }

    Plan from_cuts(const std::vector<int> &starts) const {    // contiguous microbatches
        Plan p;
        p.mb_of.assign(N, 0);
        for (size_t k = 0; k < starts.size(); ++k) {
            const int s = starts[k], e = (k + 1 < starts.size() ? starts[k + 1] : N) - 1;
            p.work.push_back(W(s, e));
            for (int i = s; i <= e; ++i) p.mb_of[sorted[i]] = int32_t(k);
        }
        return p;
    }

    // Natural partition: split every interval heavier than T at its lowest adjacent-LCP valley
    // (ties: the smaller heavier side, then the smaller difference).
    void natural(int s, int e, std::vector<int> &starts) const {
        if (W(s, e) <= T || s == e) {
            starts.push_back(s);
            return;
        }
        int best = -1;
        for (int i = s + 1; i <= e; ++i) {
            if (best < 0) {
                best = i;
                continue;
            }
            const i64 hb = std::max(W(s, best - 1), W(best, e)), hi = std::max(W(s, i - 1), W(i, e));
            const i64 db = std::llabs(W(s, best - 1) - W(best, e)), di = std::llabs(W(s, i - 1) - W(i, e));
            if (L[i] < L[best] || (L[i] == L[best] && (hi < hb || (hi == hb && di < db)))) best = i;
        }
        natural(s, best - 1, starts);
        natural(best, e, starts);
    }

    // Eq. 9: F[k][e] = minimum total work of sorted[0..e) in k contiguous capacity-feasible
    // microbatches, ties broken by the smaller heaviest microbatch; one pass serves every K up
    // to kmax.  exact_cuts(K) reads off the partition (empty if infeasible).
    std::vector<std::vector<i64>> F, H;
    std::vector<std::vector<int>> arg;
    void exact_dp(int kmax) {
        const i64 INF = std::numeric_limits<i64>::max() / 4;
        F.assign(kmax + 1, std::vector<i64>(N + 1, INF));
        H.assign(kmax + 1, std::vector<i64>(N + 1, INF));
        arg.assign(kmax + 1, std::vector<int>(N + 1, -1));
        F[0][0] = 0;
        H[0][0] = 0;
        for (int k = 1; k <= kmax; ++k)
            for (int e = k; e <= N; ++e)
                for (int s = e - 1; s >= k - 1; --s) {            // last microbatch sorted[s..e-1]
                    const i64 w = W(s, e - 1);
                    if (w > T) break;                             // W only grows as s moves left
                    if (F[k - 1][s] >= INF) continue;
                    const i64 f = F[k - 1][s] + w, h = std::max(H[k - 1][s], w);
                    if (f < F[k][e] || (f == F[k][e] && h < H[k][e])) {
                        F[k][e] = f;
                        H[k][e] = h;
                        arg[k][e] = s;
                    }
                }
    }
    std::vector<int> exact_cuts(int K) const {
        if (K >= int(F.size()) || arg[K][N] < 0) return {};
        std::vector<int> starts(K);
        for (int k = K, e = N; k >= 1; --k) {
            starts[k - 1] = arg[k][e];
            e = arg[k][e];
        }
        return starts;
    }

    // Natural partition evolved to K microbatches: merge the adjacent pair with the largest
    // saving (the LCP at their boundary) or split at the lowest valley, capacity permitting.
    std::vector<int> evolve(std::vector<int> starts, int K) const {
        while (int(starts.size()) > K) {
            int best = -1;
            for (size_t k = 1; k < starts.size(); ++k) {
                const int s = starts[k - 1], e = (k + 1 < starts.size() ? starts[k + 1] : N) - 1;
                if (W(s, e) > T) continue;
                if (best < 0 || L[starts[k]] > L[starts[best]]) best = int(k);
            }
            if (best < 0) return {};
            starts.erase(starts.begin() + best);
        }
        while (int(starts.size()) < K) {
            int bi = -1;
            for (size_t k = 0; k < starts.size(); ++k) {
                const int s = starts[k], e = (k + 1 < starts.size() ? starts[k + 1] : N) - 1;
                for (int i = s + 1; i <= e; ++i)
                    if (bi < 0 || L[i] < L[bi]) bi = i;
            }
            if (bi < 0) return {};
            starts.insert(std::upper_bound(starts.begin(), starts.end(), bi), bi);
        }
        return starts;
    }

    // Greedy trie-aware insertion (Eq. 10) in one processing order with one policy.
    Plan greedy(const std::vector<int32_t> &order, bool max_shared) const {
        std::vector<int> rank(N);
        for (int i = 0; i < N; ++i) rank[sorted[i]] = i;
        std::vector<std::vector<int32_t>> mbs;    // members by global lexicographic rank
        std::vector<i64> work;
        for (int32_t x : order) {
            const int r = rank[x];
            int best = -1;
            i64 best_key = 0, best_dc = 0;
            for (size_t m = 0; m < mbs.size(); ++m) {
                auto it = std::lower_bound(mbs[m].begin(), mbs[m].end(), r);
                const bool hp = it != mbs[m].begin(), hq = it != mbs[m].end();
                const int p = hp ? *(it - 1) : -1, q = hq ? *it : -1;
                i64 dc = X[x].n;                                   // Eq. 10
                if (hp) dc -= lcp_r(p, r);
                if (hq) dc -= lcp_r(r, q);
                if (hp && hq) dc += lcp_r(p, q);
                if (work[m] + dc > T) continue;
                const i64 key = max_shared ? X[x].n - dc : work[m] + dc;
                if (best < 0 || key > best_key) {
                    best = int(m);
                    best_key = key;
                    best_dc = dc;
                }
            }
            if (best < 0) {
                mbs.push_back({r});
                work.push_back(X[x].n);
            } else {
                mbs[best].insert(std::lower_bound(mbs[best].begin(), mbs[best].end(), r), r);
                work[best] += best_dc;
            }
        }
        // raise K to a multiple of D: split off single trajectories, each time the one whose
        // removal and singleton cost the least extra compact work
        while (mbs.size() % size_t(D) != 0) {
            int bm = -1, bi = -1;
            i64 bd = 0;
            for (size_t m = 0; m < mbs.size(); ++m) {
                if (mbs[m].size() < 2) continue;
                for (size_t i = 0; i < mbs[m].size(); ++i) {
                    const int r = mbs[m][i], x = sorted[r];
                    const bool hp = i > 0, hq = i + 1 < mbs[m].size();
                    i64 dc = X[x].n;                              // what x adds to its microbatch
                    if (hp) dc -= lcp_r(mbs[m][i - 1], r);
                    if (hq) dc -= lcp_r(r, mbs[m][i + 1]);
                    if (hp && hq) dc += lcp_r(mbs[m][i - 1], mbs[m][i + 1]);
                    const i64 inc = X[x].n - dc;                  // singleton minus the saving
                    if (bm < 0 || inc < bd) {
                        bm = int(m);
                        bi = int(i);
                        bd = inc;
                    }
                }
            }
            if (bm < 0) break;                                    // fewer trajectories than D
            const int r = mbs[bm][bi];
            mbs[bm].erase(mbs[bm].begin() + bi);
            work[bm] = trie_of_ranks(mbs[bm]);
            mbs.push_back({r});
            work.push_back(X[sorted[r]].n);
        }
        Plan p;
        p.source = 1;
        p.mb_of.assign(N, 0);
        for (size_t m = 0; m < mbs.size(); ++m)
            for (int r : mbs[m]) p.mb_of[sorted[r]] = int32_t(m);
        p.work = work;
        return p;
    }

    i64 trie_of_ranks(const std::vector<int32_t> &ranks) const {   // ranks sorted ascending (Eq. 5)
        if (ranks.empty()) return 0;
        i64 w = X[sorted[ranks[0]]].n;
        for (size_t i = 1; i < ranks.size(); ++i) w += X[sorted[ranks[i]]].n - lcp_r(ranks[i - 1], ranks[i]);
        return w;
    }
};

}  // namespace

}  // namespace treeattn

using namespace treeattn;

extern "C" int tree_attn_place(const int32_t *tokens, const int64_t *offsets, int32_t n_traj, const ta_place_config *cfg,
                               int32_t *microbatch_of, int32_t *replica_of, int32_t *slot_of, int64_t *mb_work,
                               ta_place_stats *stats) {
    treeattn::NvtxRange nvtx_range("tree_attn_place");
    if (!cfg || !offsets || n_traj <= 0 || !microbatch_of || !replica_of || !slot_of || !stats) {
        set_error("tree_attn_place: NULL argument or no trajectories");
        return TA_ERR_INVALID;
    }
    if (cfg->replicas < 1 || cfg->capacity < 1 || cfg->mode < 0 || cfg->mode > 2) {
        set_error("tree_attn_place: replicas and capacity must be >= 1, mode 0, 1 or 2");
        return TA_ERR_INVALID;
    }
    if (offsets[0] != 0) {
        set_error("tree_attn_place: offsets[0] must be 0");
        return TA_ERR_INVALID;
    }
    try {
        Planner P;
        P.D = cfg->replicas;
        P.T = cfg->capacity;
        P.X.resize(n_traj);
        for (int i = 0; i < n_traj; ++i) {
            const int64_t n = offsets[i + 1] - offsets[i];
            if (n < 1 || (n > 0 && !tokens)) {
                set_error("tree_attn_place: trajectory " + std::to_string(i) + " is empty or offsets decrease");
                return TA_ERR_INVALID;
            }
            if (n > P.T) {
                set_error("tree_attn_place: trajectory " + std::to_string(i) + " is longer than the capacity");
                return TA_ERR_INVALID;
            }
            P.X[i] = {tokens + offsets[i], n};
        }
        P.init();
        const int N = P.N, D = P.D;
        const i64 G = P.W(0, N - 1);
        // Eq. 7-8: K_min = D max(1, ceil(G / (T D))); K_max = max(K_min, min(D ceil(K0 / D), D floor(N / D)))
        const i64 kmin = i64(D) * std::max<i64>(1, (G + P.T * D - 1) / (P.T * D));
        std::vector<int> nat;
        P.natural(0, N - 1, nat);
        const i64 K0 = i64(nat.size());
        const i64 kmax = std::max(kmin, std::min(i64(D) * ((K0 + D - 1) / D), i64(D) * (N / D)));
        const int exact_max = cfg->exact_max_traj > 0 ? cfg->exact_max_traj : 512;

        std::vector<Plan> cands;
        if (cfg->mode != 2) {
            std::vector<i64> ks;
            for (i64 k = kmin; k <= kmax; k += D) ks.push_back(k);
            if (N > exact_max && ks.size() > 32) {     // sampled K: both ends, dense small, sparse span
                std::vector<i64> s;
                for (size_t i = 0; i < ks.size() && s.size() < 16; ++i) s.push_back(ks[i]);
                for (int j = 1; j <= 15; ++j) s.push_back(ks[(ks.size() - 1) * j / 15]);
                std::sort(s.begin(), s.end());
                s.erase(std::unique(s.begin(), s.end()), s.end());
                ks = s;
            }
            while (!ks.empty() && ks.back() > N) ks.pop_back();
            if (N <= exact_max && !ks.empty()) P.exact_dp(int(ks.back()));
            for (i64 k : ks) {
                std::vector<int> st = N <= exact_max ? P.exact_cuts(int(k)) : P.evolve(nat, int(k));
                if (st.empty()) continue;
                Plan p = P.from_cuts(st);
                bool ok = true;
                for (i64 w : p.work) ok = ok && w <= P.T;
                if (ok) cands.push_back(std::move(p));
            }
        }
        if (cfg->mode != 1) {
            // four processing orders x two policies; keep the one with the fewest microbatches,
            // then the least total work
            std::vector<std::vector<int32_t>> orders(4);
            orders[0] = P.sorted;
            orders[1].assign(P.sorted.rbegin(), P.sorted.rend());
            orders[2] = P.sorted;
            std::stable_sort(orders[2].begin(), orders[2].end(), [&](int32_t a, int32_t b) { return P.X[a].n > P.X[b].n; });
            std::vector<i64> u(N);
            for (int r = 0; r < N; ++r) {
                const i64 lp = r > 0 ? P.L[r] : 0, lq = r + 1 < N ? P.L[r + 1] : 0;
                u[P.sorted[r]] = P.X[P.sorted[r]].n - std::max(lp, lq);
            }
            orders[3] = P.sorted;
            std::stable_sort(orders[3].begin(), orders[3].end(), [&](int32_t a, int32_t b) { return u[a] > u[b]; });
            Plan best;
            bool have = false;
            for (const auto &o : orders)
                for (int pol = 0; pol < 2; ++pol) {
                    Plan g = P.greedy(o, pol == 1);
                    if (g.work.size() % size_t(D) != 0) continue;
                    i64 tw = 0;
                    for (i64 w : g.work) tw += w;
                    i64 bw = 0;
                    for (i64 w : best.work) bw += w;
                    if (!have || g.work.size() < best.work.size() || (g.work.size() == best.work.size() && tw < bw)) {
                        best = std::move(g);
                        have = true;
                    }
                }
            if (have) cands.push_back(std::move(best));
        }
        if (cands.empty()) {
            set_error("tree_attn_place: no plan with a multiple of the replica count of microbatches within capacity "
                      "(fewer trajectories than replicas?)");
            return TA_ERR_INVALID;
        }
        int bi = -1;
        for (size_t c = 0; c < cands.size(); ++c) {
            assign(cands[c], D);
            if (bi < 0 || better(cands[c], cands[bi])) bi = int(c);
        }
        const Plan &p = cands[bi];
        const int K = int(p.work.size());
        std::memcpy(microbatch_of, p.mb_of.data(), sizeof(int32_t) * N);
        std::memcpy(replica_of, p.replica.data(), sizeof(int32_t) * K);
        std::memcpy(slot_of, p.slot.data(), sizeof(int32_t) * K);
        if (mb_work) std::memcpy(mb_work, p.work.data(), sizeof(int64_t) * K);
        std::memset(stats, 0, sizeof(*stats));
        stats->total_work = p.j1;
        stats->slot_critical_work = p.j2;
        stats->max_replica_work = p.j3;
        stats->merged_work = G;
        stats->n_microbatches = K;
        stats->n_slots = K / D;
        stats->n_candidates = int32_t(cands.size());
        stats->source = p.source;
        stats->k_min = int32_t(kmin);
        stats->k_max = int32_t(kmax);
        stats->k_natural = int32_t(K0);
    } catch (const std::bad_alloc &) {
        set_error("tree_attn_place: host allocation failed");
        return TA_ERR_NOMEM;
    }
    return TA_OK;
}

extern "C" int tree_attn_place_units(const int64_t *work, int32_t n_units, int32_t replicas, int32_t *replica_of,
                                     int32_t *slot_of, ta_place_stats *stats) {
    if (!work || n_units <= 0 || replicas < 1 || !replica_of || !slot_of || !stats) {
        set_error("tree_attn_place_units: NULL argument, no units or replicas < 1");
        return TA_ERR_INVALID;
    }
    Plan p;
    p.work.assign(work, work + n_units);
    for (i64 w : p.work)
        if (w < 0) {
            set_error("tree_attn_place_units: negative work");
            return TA_ERR_INVALID;
        }
    assign(p, replicas);
    std::memcpy(replica_of, p.replica.data(), sizeof(int32_t) * n_units);
    std::memcpy(slot_of, p.slot.data(), sizeof(int32_t) * n_units);
    std::memset(stats, 0, sizeof(*stats));
    stats->total_work = p.j1;
    stats->slot_critical_work = p.j2;
    stats->max_replica_work = p.j3;
    stats->merged_work = p.j1;
    stats->n_microbatches = n_units;
    stats->n_slots = (n_units + replicas - 1) / replicas;
    stats->n_candidates = 1;
    return TA_OK;
}
