"""ctypes binding of libtreeattn (the C ABI in include/treeattn.h): argument marshalling only.

Every step of the hot path runs in the library's kernels.  There is no fallback: if the
shared library has not been built, importing the functions raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np

from .build import LIB as _LIB_RELEASE, LIB_DEBUG, INCLUDE

# TREEATTN_DEBUG=1 selects the TA_DEBUG build (device-side bounds checks; build it with
# dag_packed_paged_gb300.build.build(debug=True)).
LIB = LIB_DEBUG if os.environ.get("TREEATTN_DEBUG") == "1" else _LIB_RELEASE

# numpy view of ta_branch (int32 parent, fork_offset, length; int64 row_start; C alignment)
BRANCH_DTYPE = np.dtype(
    [("parent", "<i4"), ("fork_offset", "<i4"), ("length", "<i4"), ("row_start", "<i8")], align=True)

TA_OK = 0
TA_ERR_INVALID = -1
TA_ERR_UNSUPPORTED = -2
TA_ERR_NOMEM = -3
TA_ERR_CUDA = -4
TA_ERR_DEVICE_TIMEOUT = -5
TA_ERR_DEVICE_BOUNDS = -6
TA_CLAMP_MOUNTS = 0x1
TA_NO_MOUNTS = 0x2
TA_TRANSITIVE_MOUNTS = 0x4
TA_PLAN_HOST_ONLY = 0x100
TA_PLAN_STREAM_ORDERED = 0x200

HEADER = os.path.join(INCLUDE, "treeattn.h")


class TreeAttnError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"treeattn error {code}: {msg}")
        self.code = code


class ta_branch(ctypes.Structure):
    _fields_ = [("parent", ctypes.c_int32), ("fork_offset", ctypes.c_int32),
                ("length", ctypes.c_int32), ("row_start", ctypes.c_int64)]


class ta_mount(ctypes.Structure):
    _fields_ = [("reader", ctypes.c_int32), ("reader_offset", ctypes.c_int32),
                ("source", ctypes.c_int32), ("src_begin", ctypes.c_int32),
                ("src_end", ctypes.c_int32)]


class ta_config(ctypes.Structure):
    _fields_ = [("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("softmax_scale", ctypes.c_float), ("flags", ctypes.c_uint32),
                ("num_pages", ctypes.c_int64), ("num_sms", ctypes.c_int32),
                ("dkdv_chunk_entries", ctypes.c_int32), ("fwd_split_tiles", ctypes.c_int32)]


class ta_plan_stats(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int64), ("pairs", ctypes.c_int64),
                ("fwd_flops", ctypes.c_double), ("bwd_flops", ctypes.c_double),
                ("n_segments", ctypes.c_int64), ("n_blocks", ctypes.c_int64),
                ("n_intervals", ctypes.c_int64), ("n_entries", ctypes.c_int64),
                ("n_kv_tiles", ctypes.c_int64), ("n_chunks", ctypes.c_int64),
                ("n_partial_slots", ctypes.c_int64), ("block_rows", ctypes.c_int32),
                ("tile_rows", ctypes.c_int32), ("bwd_workspace_bytes", ctypes.c_size_t),
                ("plan_ms", ctypes.c_double), ("n_ftiles", ctypes.c_int64), ("chunk_cap", ctypes.c_int64),
                ("num_sms", ctypes.c_int32),
                ("device", ctypes.c_int32), ("n_fwd_items", ctypes.c_int64), ("n_fwd_split", ctypes.c_int64),
                ("fwd_split_cap", ctypes.c_int64)]


class ta_place_config(ctypes.Structure):
    _fields_ = [("replicas", ctypes.c_int32), ("mode", ctypes.c_int32), ("capacity", ctypes.c_int64),
                ("exact_max_traj", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class ta_place_stats(ctypes.Structure):
    _fields_ = [("total_work", ctypes.c_int64), ("slot_critical_work", ctypes.c_int64),
                ("max_replica_work", ctypes.c_int64), ("merged_work", ctypes.c_int64),
                ("n_microbatches", ctypes.c_int32), ("n_slots", ctypes.c_int32), ("n_candidates", ctypes.c_int32),
                ("source", ctypes.c_int32), ("k_min", ctypes.c_int32), ("k_max", ctypes.c_int32),
                ("k_natural", ctypes.c_int32), ("reserved", ctypes.c_int32)]


_P32 = ctypes.POINTER(ctypes.c_int32)
_P64 = ctypes.POINTER(ctypes.c_int64)


class ta_plan_arrays(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_int64), ("n_blocks", ctypes.c_int64),
                ("n_intervals", ctypes.c_int64), ("n_entries", ctypes.c_int64),
                ("n_chunks", ctypes.c_int64), ("pos_ids", _P32), ("blocks", _P32),
                ("blk_iv_ptr", _P64), ("iv_lo", _P32), ("iv_hi", _P32), ("diag", _P32),
                ("entries", _P32), ("t_entries", _P32), ("chunks", _P32), ("fwd_order", _P32),
                ("n_ftiles", ctypes.c_int64), ("fblk_ptr", _P64), ("ftiles", _P32),
                ("n_fwd_items", ctypes.c_int64), ("n_fwd_split", ctypes.c_int64),
                ("fwd_items", _P32), ("fwd_combine", _P32)]


_lib = None


def header_functions() -> list[str]:
    """Names of the functions declared in include/treeattn.h."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return re.findall(r"\b(tree_attn_\w+)\s*\(", txt)


def lib():
    """Load libtreeattn.so (built by dag_packed_paged_gb300.build / __graft_entry__.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise ImportError(f"{LIB} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    L.tree_attn_plan.argtypes = [vp, i32, vp, i32, vp, i64, ctypes.POINTER(ta_config), vp, vp,
                                 ctypes.POINTER(vp)]
    L.tree_attn_plan.restype = ctypes.c_int
    L.tree_attn_fwd.argtypes = [vp, vp, vp, vp, vp, vp, vp]
    L.tree_attn_fwd.restype = ctypes.c_int
    L.tree_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.tree_attn_bwd.restype = ctypes.c_int
    L.tree_attn_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.tree_attn_bwd_noalloc.restype = ctypes.c_int
    L.tree_attn_bwd_workspace_size.argtypes = [vp]
    L.tree_attn_bwd_workspace_size.restype = sz
    L.tree_attn_check.argtypes = [vp, vp]
    L.tree_attn_check.restype = ctypes.c_int
    L.tree_attn_selftest_timeout.argtypes = [vp, i64, vp]
    L.tree_attn_selftest_timeout.restype = ctypes.c_int
    L.tree_attn_plan_stats.argtypes = [vp, ctypes.POINTER(ta_plan_stats)]
    L.tree_attn_plan_stats.restype = ctypes.c_int
    L.tree_attn_plan_export.argtypes = [vp, ctypes.POINTER(ta_plan_arrays)]
    L.tree_attn_plan_export.restype = ctypes.c_int
    L.tree_attn_plan_destroy.argtypes = [vp]
    L.tree_attn_plan_destroy.restype = None
    L.tree_attn_set_trace_events.argtypes = [vp, ctypes.POINTER(vp), ctypes.c_int]
    L.tree_attn_set_trace_events.restype = ctypes.c_int
    L.tree_attn_logprob_fwd.argtypes = [vp, i64, i64, vp, vp, i64, vp, vp, vp]
    L.tree_attn_logprob_fwd.restype = ctypes.c_int
    L.tree_attn_logprob_bwd.argtypes = [vp, i64, i64, vp, vp, vp, vp, vp, vp, vp]
    L.tree_attn_logprob_bwd.restype = ctypes.c_int
    L.tree_attn_logprob_index.argtypes = [vp, vp, i64, i64, i64, vp, vp]
    L.tree_attn_logprob_index.restype = ctypes.c_int
    L.tree_attn_rope.argtypes = [vp, vp, vp, ctypes.c_double, vp]
    L.tree_attn_rope.restype = ctypes.c_int
    L.tree_attn_ingest.argtypes = [vp, vp, i32, vp, i32, ctypes.POINTER(i32), vp, i64, ctypes.POINTER(i64), vp, vp]
    L.tree_attn_owner_mask.argtypes = [vp, i32, vp, vp, vp, vp]
    L.tree_attn_owner_mask.restype = ctypes.c_int
    L.tree_attn_ingest.restype = ctypes.c_int
    L.tree_attn_place.argtypes = [vp, vp, i32, ctypes.POINTER(ta_place_config), vp, vp, vp, vp,
                                  ctypes.POINTER(ta_place_stats)]
    L.tree_attn_place.restype = ctypes.c_int
    L.tree_attn_place_units.argtypes = [vp, i32, i32, vp, vp, ctypes.POINTER(ta_place_stats)]
    L.tree_attn_place_units.restype = ctypes.c_int
    L.tree_attn_last_error.argtypes = []
    L.tree_attn_last_error.restype = ctypes.c_char_p
    _lib = L
    return L


def tree_attn_last_error() -> str:
    return lib().tree_attn_last_error().decode()


def _check(rc):
    if rc != TA_OK:
        raise TreeAttnError(rc, tree_attn_last_error())


def _ptr(x):
    """Device or host address of a torch tensor, numpy array, int or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available() and torch.cuda.is_initialized():
                return torch.cuda.current_stream().cuda_stream
        except Exception:  # pragma: no cover
            pass
        return None
    return stream if isinstance(stream, int) else stream.cuda_stream


class Plan:
    """Owns a ta_plan*; destroyed with tree_attn_plan_destroy."""

    def __init__(self, handle, n_rows, pos_ids):
        self.handle = handle
        self.n_rows = n_rows
        self.pos_ids = pos_ids

    def __del__(self):
        h, self.handle = getattr(self, "handle", None), None
        if h and _lib is not None:
            _lib.tree_attn_plan_destroy(h)


def tree_attn_plan(branches: np.ndarray, mounts: np.ndarray, page_table: np.ndarray, *,
                   num_q_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                   num_pages: int, softmax_scale: float = 0.0, flags: int = 0,
                   stream=None, num_sms: int = 0, dkdv_chunk_entries: int = 0,
                   fwd_split_tiles: int = 0) -> Plan:
    """branches: structured array with fields parent, fork_offset, length, row_start (the
    ta_branch layout); mounts: reader, reader_offset, source, src_begin, src_end.
    num_sms / dkdv_chunk_entries / fwd_split_tiles: the work-balance knobs of ta_config
    (0: defaults; fwd_split_tiles < 0 never splits a forward block)."""
    br = np.ascontiguousarray(branches)
    mt = np.ascontiguousarray(mounts)
    assert br.dtype.itemsize == ctypes.sizeof(ta_branch) and mt.dtype.itemsize == ctypes.sizeof(ta_mount)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    cfg = ta_config(num_q_heads, num_kv_heads, head_dim, page_size, softmax_scale, flags, num_pages,
                    num_sms, dkdv_chunk_entries, fwd_split_tiles)
    n_rows = int((br["row_start"] + br["length"]).max()) if len(br) else 0
    pos = np.zeros(max(n_rows, 1), dtype=np.int32)
    h = ctypes.c_void_p()
    rc = lib().tree_attn_plan(br.ctypes.data if len(br) else None, len(br),
                              mt.ctypes.data if len(mt) else None, len(mt),
                              pt.ctypes.data if len(pt) else None, len(pt), ctypes.byref(cfg),
                              pos.ctypes.data, _stream(stream) if not (flags & TA_PLAN_HOST_ONLY) else None,
                              ctypes.byref(h))
    _check(rc)
    return Plan(h.value, n_rows, pos[:n_rows])


def tree_attn_fwd(plan: Plan, q, k_pool, v_pool, o, lse, stream=None) -> None:
    _check(lib().tree_attn_fwd(plan.handle, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(o), _ptr(lse),
                               _stream(stream)))


def tree_attn_bwd(plan: Plan, q, k_pool, v_pool, o, lse, d_o, dq, dk_pool, dv_pool, workspace,
                  ws_bytes=None, stream=None) -> None:
    if ws_bytes is None:
        ws_bytes = workspace.numel() * workspace.element_size()
    _check(lib().tree_attn_bwd(plan.handle, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(o), _ptr(lse),
                               _ptr(d_o), _ptr(dq), _ptr(dk_pool), _ptr(dv_pool), _ptr(workspace),
                               int(ws_bytes), _stream(stream)))


def tree_attn_bwd_noalloc(plan: Plan, q, k_pool, v_pool, o, lse, d_o, dq, dk_pool, dv_pool,
                          stream=None) -> None:
    """tree_attn_bwd using the library's fixed scratch array instead of a workspace (for
    callers that cannot allocate device memory; see include/treeattn.h)."""
    _check(lib().tree_attn_bwd_noalloc(plan.handle, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(o), _ptr(lse),
                                       _ptr(d_o), _ptr(dq), _ptr(dk_pool), _ptr(dv_pool), _stream(stream)))


def tree_attn_bwd_workspace_size(plan: Plan) -> int:
    return int(lib().tree_attn_bwd_workspace_size(plan.handle))


def tree_attn_check(plan: Plan, stream=None) -> None:
    _check(lib().tree_attn_check(plan.handle, _stream(stream)))


def tree_attn_selftest_timeout(plan: Plan, limit_us: int = 1000, stream=None) -> None:
    """Launch the kernel whose bounded wait always expires (see include/treeattn.h); the next
    tree_attn_check on `plan` raises with TA_ERR_DEVICE_TIMEOUT."""
    _check(lib().tree_attn_selftest_timeout(plan.handle, int(limit_us), _stream(stream)))


def tree_attn_set_trace_events(plan: Plan, events) -> None:
    """events: None, or 7 torch.cuda.Event objects (or None entries) -- see the header."""
    if events is None:
        _check(lib().tree_attn_set_trace_events(plan.handle, None, 0))
        return
    arr = (ctypes.c_void_p * 7)(*[None if e is None else e.cuda_event for e in events])
    plan._trace_keepalive = events
    _check(lib().tree_attn_set_trace_events(plan.handle, arr, 7))


def tree_attn_plan_stats(plan: Plan) -> dict:
    st = ta_plan_stats()
    _check(lib().tree_attn_plan_stats(plan.handle, ctypes.byref(st)))
    return {f: getattr(st, f) for f, _ in ta_plan_stats._fields_}


def tree_attn_plan_export(plan: Plan) -> dict:
    """Copies of the plan's host arrays (see ta_plan_arrays)."""
    a = ta_plan_arrays()
    _check(lib().tree_attn_plan_export(plan.handle, ctypes.byref(a)))

    def arr(p, n, dt=np.int32):
        if n == 0:
            return np.zeros(0, dtype=dt)
        return np.ctypeslib.as_array(p, shape=(n,)).copy()

    nb, ne = a.n_blocks, a.n_entries
    return {
        "n_rows": a.n_rows,
        "pos_ids": arr(a.pos_ids, a.n_rows),
        "blocks": arr(a.blocks, 4 * nb).reshape(nb, 4),
        "blk_iv_ptr": arr(a.blk_iv_ptr, nb + 1, np.int64),
        "iv_lo": arr(a.iv_lo, a.n_intervals),
        "iv_hi": arr(a.iv_hi, a.n_intervals),
        "diag": arr(a.diag, 2 * nb).reshape(nb, 2),
        "entries": arr(a.entries, 4 * ne).reshape(ne, 4),
        "t_entries": arr(a.t_entries, 4 * ne).reshape(ne, 4),
        "chunks": arr(a.chunks, 4 * a.n_chunks).reshape(a.n_chunks, 4),
        "fwd_order": arr(a.fwd_order, nb),
        "fblk_ptr": arr(a.fblk_ptr, nb + 1, np.int64),
        "ftiles": arr(a.ftiles, 8 * a.n_ftiles).reshape(a.n_ftiles, 8),
        "fwd_items": arr(a.fwd_items, 4 * a.n_fwd_items).reshape(a.n_fwd_items, 4),
        "fwd_combine": arr(a.fwd_combine, 4 * a.n_fwd_split).reshape(a.n_fwd_split, 4),
    }


def tree_attn_plan_destroy(plan: Plan) -> None:
    h, plan.handle = plan.handle, None
    if h:
        lib().tree_attn_plan_destroy(h)


def tree_attn_ingest(trajectories, with_owner=False):
    """Compact prefix-tree episode of a list of token trajectories (1-D int arrays).

    Returns (branches, row_tokens, row_of): the ta_branch structured array, the token of every
    compact row, and for each trajectory the int64 array of compact rows of its positions;
    with_owner=True appends row_owner (the trajectory whose insertion created each row)."""
    trajs = [np.ascontiguousarray(t, dtype=np.int32).ravel() for t in trajectories]
    offsets = np.zeros(len(trajs) + 1, dtype=np.int64)
    for i, t in enumerate(trajs):
        offsets[i + 1] = offsets[i] + len(t)
    tokens = np.concatenate(trajs) if trajs and offsets[-1] > 0 else np.zeros(1, dtype=np.int32)
    total = int(offsets[-1])
    br = np.zeros(max(len(trajs), 1), dtype=BRANCH_DTYPE)
    row_tokens = np.zeros(max(total, 1), dtype=np.int32)
    row_of = np.zeros(max(total, 1), dtype=np.int64)
    row_owner = np.zeros(max(total, 1), dtype=np.int32)
    nb, nr = ctypes.c_int32(0), ctypes.c_int64(0)
    _check(lib().tree_attn_ingest(tokens.ctypes.data, offsets.ctypes.data, len(trajs), br.ctypes.data, len(br),
                                  ctypes.byref(nb), row_tokens.ctypes.data, len(row_tokens), ctypes.byref(nr),
                                  row_of.ctypes.data, row_owner.ctypes.data))
    out = (br[:nb.value].copy(), row_tokens[:nr.value].copy(), [row_of[offsets[i]:offsets[i + 1]].copy()
                                                                 for i in range(len(trajs))])
    return out + (row_owner[:nr.value].copy(),) if with_owner else out


def tree_attn_owner_mask(row_of, row_owner, generated=None) -> list:
    """Octopus Eq. 6 loss mask per trajectory position (list of uint8 arrays, the layout of
    tree_attn_ingest's row_of): 1 where the position's predicted token is generated and its
    compact row is owned by this trajectory."""
    lens = [len(r) for r in row_of]
    offsets = np.zeros(len(lens) + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(lens)
    flat = np.concatenate(row_of).astype(np.int64) if offsets[-1] else np.zeros(1, np.int64)
    own = np.ascontiguousarray(row_owner, dtype=np.int32)
    gen = None
    if generated is not None:
        gen = np.concatenate([np.asarray(g, dtype=np.uint8) for g in generated]) if offsets[-1] else np.zeros(1, np.uint8)
    mask = np.zeros(max(int(offsets[-1]), 1), dtype=np.uint8)
    _check(lib().tree_attn_owner_mask(offsets.ctypes.data, len(lens), flat.ctypes.data,
                                      own.ctypes.data if len(own) else None,
                                      gen.ctypes.data if gen is not None else None, mask.ctypes.data))
    return [mask[offsets[i]:offsets[i + 1]].copy() for i in range(len(lens))]


def tree_attn_rope(plan: Plan, q, k_pool, theta_base: float = 10000.0, stream=None) -> None:
    """Rotate Q [N, Hq, D] and the K pool in place at the plan's Eq. 2 positions."""
    _check(lib().tree_attn_rope(plan.handle, _ptr(q), _ptr(k_pool), float(theta_base), _stream(stream)))


def tree_attn_logprob_fwd(logits, pos_row, pos_target, row_lse, logprob, stream=None) -> None:
    """logits bf16 [C, V]; pos_row int64 [S]; pos_target int32 [S] (device tensors) ->
    row_lse fp32 [C], logprob fp32 [S]."""
    C, V = logits.shape
    _check(lib().tree_attn_logprob_fwd(_ptr(logits), C, V, _ptr(pos_row), _ptr(pos_target), pos_row.shape[0],
                                       _ptr(row_lse), _ptr(logprob), _stream(stream)))


def tree_attn_logprob_index(pos_row: np.ndarray, pos_target: np.ndarray, n_rows: int, vocab: int):
    """Host CSR of the positions of every compact row, ordered by target: (row_ptr, row_pos)."""
    pr = np.ascontiguousarray(pos_row, dtype=np.int64)
    pt = np.ascontiguousarray(pos_target, dtype=np.int32)
    row_ptr = np.zeros(n_rows + 1, dtype=np.int64)
    row_pos = np.zeros(max(len(pr), 1), dtype=np.int64)
    _check(lib().tree_attn_logprob_index(pr.ctypes.data if len(pr) else None, pt.ctypes.data if len(pt) else None,
                                         len(pr), n_rows, vocab, row_ptr.ctypes.data, row_pos.ctypes.data))
    return row_ptr, row_pos[: len(pr)]


def tree_attn_logprob_bwd(logits, row_lse, row_ptr, row_pos, pos_target, dlogprob, dlogits, stream=None) -> None:
    """dlogits bf16 [C, V] from dlogprob fp32 [S] (device tensors; row_ptr / row_pos from
    tree_attn_logprob_index, moved to the device)."""
    C, V = logits.shape
    _check(lib().tree_attn_logprob_bwd(_ptr(logits), C, V, _ptr(row_lse), _ptr(row_ptr), _ptr(row_pos),
                                       _ptr(pos_target), _ptr(dlogprob), _ptr(dlogits), _stream(stream)))


def _place_stats(st):
    return {f: getattr(st, f) for f, _ in ta_place_stats._fields_ if f != "reserved"}


def tree_attn_place(trajectories, replicas: int, capacity: int, mode: int = 0, exact_max_traj: int = 0) -> dict:
    """Compact-work microbatch plan of a list of token trajectories over `replicas` data-parallel
    replicas (see include/treeattn.h): microbatch of every trajectory, replica / slot / compact
    rows of every microbatch, and the Eq. 4 objective terms."""
    trajs = [np.ascontiguousarray(t, dtype=np.int32).ravel() for t in trajectories]
    n = len(trajs)
    offsets = np.zeros(n + 1, dtype=np.int64)
    for i, t in enumerate(trajs):
        offsets[i + 1] = offsets[i] + len(t)
    tokens = np.concatenate(trajs) if n and offsets[-1] else np.zeros(1, dtype=np.int32)
    mb = np.zeros(max(n, 1), dtype=np.int32)
    rep = np.zeros(max(n, 1), dtype=np.int32)
    slot = np.zeros(max(n, 1), dtype=np.int32)
    work = np.zeros(max(n, 1), dtype=np.int64)
    cfg = ta_place_config(replicas, mode, capacity, exact_max_traj, 0)
    st = ta_place_stats()
    _check(lib().tree_attn_place(tokens.ctypes.data, offsets.ctypes.data, n, ctypes.byref(cfg), mb.ctypes.data,
                                 rep.ctypes.data, slot.ctypes.data, work.ctypes.data, ctypes.byref(st)))
    K = st.n_microbatches
    return {"microbatch_of": mb[:n].copy(), "replica_of": rep[:K].copy(), "slot_of": slot[:K].copy(),
            "work": work[:K].copy(), **_place_stats(st)}


def tree_attn_place_units(work, replicas: int) -> dict:
    """Replica and slot of already-grouped units (e.g. independent DAGs) by the DP-replica
    assignment of tree_attn_place; work: compact rows (or any additive cost) per unit."""
    w = np.ascontiguousarray(work, dtype=np.int64)
    n = len(w)
    rep = np.zeros(max(n, 1), dtype=np.int32)
    slot = np.zeros(max(n, 1), dtype=np.int32)
    st = ta_place_stats()
    _check(lib().tree_attn_place_units(w.ctypes.data if n else None, n, replicas, rep.ctypes.data,
                                       slot.ctypes.data, ctypes.byref(st)))
    return {"replica_of": rep[:n].copy(), "slot_of": slot[:n].copy(), **_place_stats(st)}
