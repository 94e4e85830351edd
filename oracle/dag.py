"""Oracle: DAG semantics of tree/DAG-packed attention, written from the definitions.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this module; only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use it.  It shares no
code with the CUDA path or its planner.

Every function follows a passage of the pages:

* visible set of a row -- Octopus (arXiv 2611.06956) Section 3.3, Eq. 4: a node's query
  rows see ``[mounted spans || ancestor prefix || own rows]``, with the causal triangle
  aligned to the rightmost (own) keys; HARTS (arXiv 2608.28158) Section 4.2, Eq. 21-22:
  query i of a branch with h ancestor rows sees KV entries j <= h + i.  The fork position is
  the number of shared prefix tokens (HARTS Section 2.2).  A mount lends a completed span
  ``[s, e)`` of a sibling to the reader from its row ``t`` on (Octopus Section 3.1 Table 2,
  read_thread; Section 3.2).
* positions -- Octopus Section 3.2, Eq. 2: after a mount the reader continues at
  ``max(pos_next, max_m pos_end(m) + 1)``; mounted rows keep their own positions.
* trajectories and compact rows -- HARTS Section 2.1 (semantic positions s = (x, i) and the
  compact map m: S -> C) and Section 3.2, Eq. 5 (compact row count of a trajectory set).

Readings where the pages are silent (each listed in the design notes):
* visibility is a *set*: a row reachable by two routes counts once;
* mounts are not transitive: a reader sees the mounted rows only, not the source's own
  ancestors or mounts;
* a child forking at offset f inherits its parent's rows [0, f), the parent's mounts active
  at row f-1, and everything the parent inherited (for f = 0 only the latter);
* a zero-length mount contributes no rows and no position jump.

Two further views of the same episode (same rows, same Eq. 2 positions):
* ``view="no_mounts"`` -- layers that do not mount (Octopus Section 3.2, layer-selective
  mounting; Appendix C Table 8, the mounted / unmounted dual pass) see the ancestor path and
  their own rows only;
* ``view="transitive"`` -- a node's active mounted segments "including transitive mounts"
  (Octopus Section 3.3 item 1): a mounted span [s, e) of source A also brings the mounts in
  effect at A's row e-1 (A's own with reader offset <= e-1 and those A inherits), and so on
  recursively.
"""
from __future__ import annotations

import numpy as np


def _br(branches):
    return [(int(b["parent"]), int(b["fork_offset"]), int(b["length"]), int(b["row_start"]))
            for b in branches]


def _mt(mounts):
    return [(int(m["reader"]), int(m["reader_offset"]), int(m["source"]),
             int(m["src_begin"]), int(m["src_end"])) for m in mounts]


def n_rows(branches) -> int:
    return max((rs + ln for _, _, ln, rs in _br(branches)), default=0)


def row_owner(branches):
    """compact row -> (branch, offset), from the row layout."""
    out = {}
    for b, (_, _, ln, rs) in enumerate(_br(branches)):
        for i in range(ln):
            out[rs + i] = (b, i)
    return out


VIEWS = ("mounted", "no_mounts", "transitive")


def mounts_in_effect(branches, mounts, b, i):
    """Non-empty mounted spans (source, lo_off, hi_off) in effect at row (b, i): b's own
    mounts with reader offset <= i, and the mounts b inherits (those of an ancestor p that are
    active at the fork row f-1 of the edge into p's subtree)."""
    B, M = _br(branches), _mt(mounts)
    out = [(s, lo, hi) for (r, t, s, lo, hi) in M if r == b and t <= i and hi > lo]
    x = b
    while B[x][0] >= 0:
        p, f = B[x][0], B[x][1]
        if f > 0:
            out += [(s, lo, hi) for (r, t, s, lo, hi) in M if r == p and t <= f - 1 and hi > lo]
        x = p
    return out


def _closure(branches, mounts, spans):
    """The spans plus, recursively, the spans in effect at each span's last source row."""
    out, seen, stack = [], set(), list(spans)
    while stack:
        sp = stack.pop()
        if sp in seen:
            continue
        seen.add(sp)
        out.append(sp)
        s, lo, hi = sp
        stack.extend(mounts_in_effect(branches, mounts, s, hi - 1))
    return out


def _spans(branches, mounts, spans, view):
    if view == "no_mounts":
        return []
    if view == "transitive":
        return _closure(branches, mounts, spans)
    assert view == "mounted", view
    return list(spans)


def inherited_pieces(branches, mounts, b, view="mounted"):
    """Rows a branch shares with its ancestors, as (branch, lo_off, hi_off) pieces.

    inh(root) = {};  inh(b) = rows [0, f) of the parent p  +  rows of p's mounts that are
    active at p's row f-1  +  inh(p)."""
    B, M = _br(branches), _mt(mounts)
    out = []
    while B[b][0] >= 0:
        p, f = B[b][0], B[b][1]
        if f > 0:
            out.append((p, 0, f))
            out += _spans(branches, mounts, [(s, lo, hi) for (r, t, s, lo, hi) in M
                                             if r == p and t <= f - 1 and hi > lo], view)
        b = p
    return out


def visible_pieces(branches, mounts, b, i, view="mounted"):
    """Visible rows of the row at offset i of branch b, as (branch, lo_off, hi_off) pieces:
    own rows 0..i, every non-empty mount of b with reader offset <= i, and inh(b)."""
    M = _mt(mounts)
    out = [(b, 0, i + 1)]
    out += _spans(branches, mounts, [(s, lo, hi) for (r, t, s, lo, hi) in M
                                     if r == b and t <= i and hi > lo], view)
    out += inherited_pieces(branches, mounts, b) if view == "mounted" else \
        inherited_pieces(branches, mounts, b, view=view)
    return out


def visible_set(branches, mounts, row, view="mounted") -> set:
    """The visible compact rows of ``row`` as an explicit Python set (small cases)."""
    B = _br(branches)
    b, i = row_owner(branches)[row]
    out = set()
    for (x, lo, hi) in visible_pieces(branches, mounts, b, i, view=view):
        rs = B[x][3]
        out.update(range(rs + lo, rs + hi))
    return out


def visible_intervals_of(branches, mounts, b, i):
    """Visible compact rows of (b, i) as sorted, disjoint, maximal [lo, hi) intervals."""
    B = _br(branches)
    iv = sorted((B[x][3] + lo, B[x][3] + hi) for (x, lo, hi) in visible_pieces(branches, mounts, b, i))
    merged = []
    for lo, hi in iv:
        if merged and lo <= merged[-1][1]:
            merged[-1][1] = max(merged[-1][1], hi)
        else:
            merged.append([lo, hi])
    return [(lo, hi) for lo, hi in merged]


def visible_intervals(branches, mounts, rows=None, view="mounted"):
    """CSR of visible intervals for the given compact rows (default: all rows, in order).

    Returns (rows int64[n], ptr int64[n+1], lo int64[nnz], hi int64[nnz])."""
    B = _br(branches)
    N = n_rows(branches)
    if rows is None:
        rows = np.arange(N, dtype=np.int64)
    rows = np.asarray(rows, dtype=np.int64)
    starts = np.array([rs for (_, _, _, rs) in B], dtype=np.int64)
    ends = np.array([rs + ln for (_, _, ln, rs) in B], dtype=np.int64)
    ptr = [0]
    lo_all, hi_all = [], []
    cache = {}
    mlist = _mt(mounts)
    offsets_of = {}
    for (rr, t, s, lo, hi) in mlist:
        offsets_of.setdefault(rr, []).append(t)
    order = np.argsort(starts, kind="stable")
    sorted_starts = starts[order]
    for r in rows:
        b = int(order[np.searchsorted(sorted_starts, r, side="right") - 1])
        assert starts[b] <= r < ends[b]
        i = int(r - starts[b])
        # everything except the own-row piece depends only on (b, number of mount offsets <= i)
        key = (b, sum(1 for t in offsets_of.get(b, ()) if t <= i))
        if key not in cache:
            vp = visible_pieces(branches, mounts, b, i) if view == "mounted" else \
                visible_pieces(branches, mounts, b, i, view=view)
            cache[key] = vp[1:]
        pieces = [(b, 0, i + 1)] + cache[key]
        iv = sorted((B[x][3] + lo, B[x][3] + hi) for (x, lo, hi) in pieces)
        merged = []
        for lo, hi in iv:
            if merged and lo <= merged[-1][1]:
                merged[-1][1] = max(merged[-1][1], hi)
            else:
                merged.append([lo, hi])
        for lo, hi in merged:
            lo_all.append(lo)
            hi_all.append(hi)
        ptr.append(len(lo_all))
    return (rows, np.array(ptr, dtype=np.int64), np.array(lo_all, dtype=np.int64),
            np.array(hi_all, dtype=np.int64))


def count_pairs(branches, mounts, view="mounted") -> int:
    """Sum over rows of the size of the visible set."""
    _, ptr, lo, hi = visible_intervals(branches, mounts, view=view)
    return int((hi - lo).sum())


# ----------------------------------------------------------------------------------------
# positions: Octopus Eq. 2
# ----------------------------------------------------------------------------------------

def positions(branches, mounts) -> np.ndarray:
    """Position id of every compact row.

    A root's row k has position k.  A child forked at f starts at pos(p, f-1) + 1 (at f = 0,
    at the position its parent started from).  Every later row continues at pos(prev) + 1,
    except that at a reader offset t with non-empty mounts starting there the row jumps to
    max(pos_next, max over those mounts of pos(source, e-1) + 1).  Mounted rows keep their
    own positions."""
    B, M = _br(branches), _mt(mounts)
    n = len(B)
    pos = [[None] * B[b][2] for b in range(n)]
    busy = set()
    starting_at = {}
    for (r, t, s, lo, hi) in M:
        if hi > lo:
            starting_at.setdefault((r, t), []).append((s, hi))

    def start_next(b):
        p, f = B[b][0], B[b][1]
        if p < 0:
            return 0
        if f == 0:
            return start_next(p)
        return get(p, f - 1) + 1

    def get(b, i):
        if pos[b][i] is not None:
            return pos[b][i]
        if (b, i) in busy:
            raise ValueError("cyclic position dependency (non-causal mount)")
        busy.add((b, i))
        # walk forward from the last computed row of this branch
        k = i
        while k > 0 and pos[b][k - 1] is None:
            k -= 1
        for j in range(k, i + 1):
            nxt = start_next(b) if j == 0 else pos[b][j - 1] + 1
            for (s, hi) in starting_at.get((b, j), ()):
                nxt = max(nxt, get(s, hi - 1) + 1)
            pos[b][j] = nxt
        busy.discard((b, i))
        return pos[b][i]

    out = np.zeros(n_rows(branches), dtype=np.int64)
    for b in range(n):
        for i in range(B[b][2]):
            out[B[b][3] + i] = get(b, i)
    return out


# ----------------------------------------------------------------------------------------
# trajectories (semantic positions) -- used to pin the packed definition
# ----------------------------------------------------------------------------------------

def trajectories(branches, mounts):
    """One expanded trajectory per branch: the root-to-branch-end path.

    Each trajectory is a list of (compact_row, is_query) entries in sequence order: the path's
    own rows in order (is_query=True) and, for every mount whose reader row lies on the path,
    the mounted span inserted as key/value-only entries (is_query=False) just before the
    reader row (the order of Octopus Eq. 4: mounted keys, then ancestors, then own rows).
    Under ordinary causal attention each query row of a trajectory then sees exactly the
    entries before it and itself."""
    B, M = _br(branches), _mt(mounts)
    out = []
    for leaf in range(len(B)):
        path = [leaf]
        while B[path[-1]][0] >= 0:
            path.append(B[path[-1]][0])
        path.reverse()
        seq = []
        for k, x in enumerate(path):
            hi_x = B[path[k + 1]][1] if k + 1 < len(path) else B[x][2]
            for i in range(hi_x):
                for (r, t, s, lo, hi) in M:
                    if r == x and t == i and hi > lo:
                        seq.extend((B[s][3] + j, False) for j in range(lo, hi))
                seq.append((B[x][3] + i, True))
        out.append(seq)
    return out


def compact_rows_eq5(traj_tokens):
    """HARTS Eq. 5: C(M) = |x_1| + sum_{i>=2} (|x_i| - LCP(x_{i-1}, x_i)) over the
    trajectories sorted lexicographically."""
    xs = sorted(tuple(t) for t in traj_tokens)
    if not xs:
        return 0
    total = len(xs[0])
    for a, b in zip(xs, xs[1:]):
        lcp = 0
        while lcp < min(len(a), len(b)) and a[lcp] == b[lcp]:
            lcp += 1
        total += len(b) - lcp
    return total
