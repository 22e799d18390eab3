"""CPU oracle for the topology-aware expert-routing plan (test infrastructure).

This package is the plain, slow, single-threaded statement of what the GPU
path computes.  It exists to check the CUDA library bit for bit and to give
the benchmark a CPU baseline.  Only the tests, the smoke check and the
benchmark's CPU-baseline leg may import it; the product path never does.

The arithmetic lives in ``oracle.c`` (plain C, built with gcc into
``oracle/_build/liboracle.so``); this module only builds, loads and
marshals numpy arrays.  It shares no code with the CUDA library.

Sources: "TopoEP: Topology-Aware Load Balancing for Expert-Parallel MoE
Training" (§4.1 Eqs. 3-4, §4.2 C1-C5 and Eqs. 5-8, §4.3 Eqs. 9-10 and Fig. 9,
§5) and "Expert Coupling in MoE Pretraining" (within-layer co-selection,
cross-layer routing correlation).

Parity status per function (what pins each one is in ``tests/test_oracle_*``):
  hist      pinned (closed form: per-block bincount; sum = T*k)
  cooccur   pinned (closed form: indicator-matrix products; hand case)
  plan      pinned (hand-worked cases incl. the Fig. 9 shape, Fig. 3
            arithmetic, constraint invariants, brute-force optimum bound,
            special cases); tie-break orders beyond the hand cases follow
            the stated readings
  reroute   pinned (hand case; per-(source, instance) counts equal q)
  layout    pinned (stable argsort; bijection; count identities)
  permute   pinned (hand case; every token row lands k times, in its pairs'
            positions; row sums)
  combine   pinned (hand cases incl. round-to-nearest-even ties and the slot
            summation order; exact round trip combine(permute(x)) == x with
            dyadic weights; one-hot weights select a slot)
  dedup     pinned (hand case; every pair covered by exactly one row; k = 1
            keeps one row per pair; the pages' printed top-2 / top-6 row
            savings against the closed-form expectation)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ERANGE = 0, -1, -2
STAT_NAMES = ("L_max", "L_max_static", "n_replicas", "n_stage1", "refine_iters",
              "T_token", "T_replica", "sum_L")
LAYOUT_STAT_NAMES = ("pairs_local", "pairs_intra", "pairs_inter", "bytes_local",
                     "bytes_intra", "bytes_inter", "pairs_replica", "reserved")


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, -O2, portable flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-Wall", "-Wextra", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i32p = np.ctypeslib.ndpointer(np.int32, flags="C_CONTIGUOUS")
            i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
            ci, cl = ctypes.c_int, ctypes.c_int64
            vp = ctypes.c_void_p
            lib.oracle_hist.argtypes = [ci, ci, ci, ci, ci, vp, i32p, i32p]
            lib.oracle_cooccur.argtypes = [ci, ci, ci, ci, i32p, i64p, ctypes.c_void_p]
            lib.oracle_plan.argtypes = [ci, ci, ci, ci, ci, ci, cl, cl, cl, cl, ci,
                                        ctypes.c_void_p, ci, i32p, i32p, i32p, i32p,
                                        i32p, i64p]
            lib.oracle_reroute.argtypes = [ci, ci, ci, ci, ci, ci, vp, vp, ci,
                                           i32p, i32p, i32p, i32p]
            lib.oracle_layout.argtypes = [ci, ci, ci, ci, ci, ci, cl, vp, ci, i32p, i32p,
                                          i32p, i64p, i64p]
            u16p = np.ctypeslib.ndpointer(np.uint16, flags="C_CONTIGUOUS")
            f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
            lib.oracle_permute.argtypes = [ci, ci, ci, ci, u16p, i32p, u16p]
            lib.oracle_combine.argtypes = [ci, ci, ci, ci, u16p, i32p, f32p, u16p]
            u64p = np.ctypeslib.ndpointer(np.uint64, flags="C_CONTIGUOUS")
            lib.oracle_dedup.argtypes = [ci, ci, ci, ci, vp, ci, i32p, i32p, i32p, u64p, u64p, i64p, i64p]
            lib.oracle_gate.argtypes = [ci, ci, ci, ci, ci, vp, ci, vp, vp, i32p, f32p, i32p]
            lib.oracle_shuffle.argtypes = [ci, ci, ci, ci, ci, i32p, i64p, vp, vp, i32p, i64p]
            lib.oracle_place.argtypes = [ci, ci, ci, ci, i64p, i32p, i64p]
            for f in ("oracle_place", "oracle_shuffle", "oracle_gate", "oracle_hist", "oracle_cooccur", "oracle_plan", "oracle_reroute",
                      "oracle_layout", "oracle_permute", "oracle_combine", "oracle_dedup"):
                getattr(lib, f).restype = ci
            _lib = lib
    return _lib


class OracleError(RuntimeError):
    def __init__(self, fn: str, rc: int):
        super().__init__(f"{fn} returned {rc}")
        self.rc = rc


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def _offsets(rank_offsets):
    """(keep-alive array, pointer) for int64 [R+1] source offsets, or (None, None)."""
    if rank_offsets is None:
        return None, None
    o = np.ascontiguousarray(rank_offsets, dtype=np.int64)
    return o, o.ctypes.data_as(ctypes.c_void_p)


def _check(fn, rc, allow=(OK,)):
    if rc not in allow:
        raise OracleError(fn, rc)
    return rc


def gate(logits, k: int, R: int, bias=None, rank_offsets=None):
    """Top-k gating and Omega [TopoEP §2.1, §6.4; O1].

    logits: float32 [L, T, E] (or [T, E]), or uint16 bf16 patterns of that
    shape.  bias: float32 [E] or None.  Returns dict with ids int32 [L, T, k],
    scores float32 [L, T, k] (raw logits of the selected experts) and hist
    int32 [L, R, E] (without the leading L for a 2-D input)."""
    a = np.asarray(logits)
    if a.dtype not in (np.float32, np.uint16):
        raise TypeError("logits must be float32 or uint16 bf16 patterns")
    a = np.ascontiguousarray(a)
    squeeze = a.ndim == 2
    if squeeze:
        a = a[None]
    L, T, E = a.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    if b is not None and b.shape != (E,):
        raise ValueError("bias must be float32 [E]")
    out = dict(ids=np.zeros((L, T, k), np.int32), scores=np.zeros((L, T, k), np.float32),
               hist=np.zeros((L, R, E), np.int32))
    keep, op = _offsets(rank_offsets)
    _check("oracle_gate", _load().oracle_gate(
        T, E, k, R, L, op, int(a.dtype == np.uint16), a.ctypes.data_as(ctypes.c_void_p),
        None if b is None else b.ctypes.data_as(ctypes.c_void_p), out["ids"].reshape(-1),
        out["scores"].reshape(-1), out["hist"].reshape(-1)))
    if squeeze:
        out = {key: v[0] for key, v in out.items()}
    return out


PLACE_STAT_NAMES = ("within_contiguous", "within_greedy", "within_final", "swaps")


def place(co, R: int, max_iters: int = 0):
    """Correlated expert placement [Zyphra, "Moving Correlated Experts Together"].

    co int64 [L, E, E] (or [E, E]).  Returns (main_rank int32 [L, E], stats
    int64 [L, 4]) (without the leading L for a 2-D input)."""
    c = np.ascontiguousarray(co, dtype=np.int64)
    squeeze = c.ndim == 2
    if squeeze:
        c = c[None]
    L, E, _ = c.shape
    mr = np.zeros((L, E), np.int32)
    st = np.zeros((L, 4), np.int64)
    _check("oracle_place", _load().oracle_place(L, E, R, max_iters, c.reshape(-1), mr.reshape(-1),
                                                st.reshape(-1)))
    return (mr[0], st[0]) if squeeze else (mr, st)


SHUFFLE_STAT_NAMES = ("next_pairs_on_target", "next_pairs_on_source", "tokens_moved", "next_pairs")


def shuffle(ids, tr, R: int, main_rank=None, rank_offsets=None):
    """Token-shuffle targets [Zyphra, "Moving Tokens Toward Their Next Experts"].

    ids int32 [L, T, k]; tr int64 [L-1, E, E] (cooccur's transitions); main_rank
    int32 [E] or None; rank_offsets int64 [R+1] or None (equal blocks).
    Returns (target int32 [L-1, T], stats int64 [L-1, 4])."""
    a = _i32(ids)
    L, T, k = a.shape
    t = np.ascontiguousarray(tr, dtype=np.int64)
    E = t.shape[-1] if t.size else int(a.max()) + 1
    if L > 1 and t.shape != (L - 1, E, E):
        raise ValueError("tr must be int64 [L-1, E, E]")
    mr = None if main_rank is None else _i32(main_rank)
    target = np.zeros((max(L - 1, 0), T), np.int32)
    stats = np.zeros((max(L - 1, 0), 4), np.int64)
    keep, op = _offsets(rank_offsets)
    _check("oracle_shuffle", _load().oracle_shuffle(
        L, T, E, k, R, a.reshape(-1), t.reshape(-1) if t.size else np.zeros(1, np.int64),
        None if mr is None else mr.ctypes.data_as(ctypes.c_void_p), op, target.reshape(-1),
        stats.reshape(-1)))
    return target, stats


def hist(ids, R: int, E: int, rank_offsets=None):
    """Routing matrix Omega [TopoEP §4.1, Eq. 3].

    ids: int32 [L, T, k] or [T, k]; rank_offsets: int64 [R+1] token offsets of
    the sources, or None for equal blocks.  Returns int32 [L, R, E] (or [R, E])."""
    a = _i32(ids)
    squeeze = a.ndim == 2
    if squeeze:
        a = a[None]
    L, T, k = a.shape
    out = np.zeros((L, R, E), np.int32)
    keep, op = _offsets(rank_offsets)
    _check("oracle_hist", _load().oracle_hist(T, E, k, R, L, op, a.reshape(-1), out.reshape(-1)))
    return out[0] if squeeze else out


def cooccur(ids, E: int, transitions: bool = True):
    """Co-selection co[L,E,E] and transitions tr[L-1,E,E] (int64), ids [L,T,k]."""
    a = _i32(ids)
    L, T, k = a.shape
    co = np.zeros((L, E, E), np.int64)
    tr = np.zeros((max(L - 1, 0), E, E), np.int64)
    trp = tr.ctypes.data_as(ctypes.c_void_p) if (transitions and L > 1) else None
    _check("oracle_cooccur", _load().oracle_cooccur(L, T, E, k, a.reshape(-1), co.reshape(-1), trp))
    return (co, tr) if transitions else co


def _main_ptr(main_rank):
    if main_rank is None:
        return None, None
    m = _i32(main_rank)
    return m, m.ctypes.data_as(ctypes.c_void_p)


def plan(cfg: dict, hist_arr, max_refine_iters: int | None = None):
    """Two-stage plan [TopoEP §4.3] for each layer of hist int32 [L, R, E].

    cfg keys: T, E, k, R, ranks_per_node, n_slot, tok_bytes, expert_bytes,
    c_intra, c_inter, optional max_refine_iters, optional main_rank (the
    plan reads only Omega, so rank_offsets plays no part here).
    Returns dict of numpy arrays: slot_expert [L,R,n_slot], route_cnt
    [L,R,R,n_local], inst_load [L,R,n_local], rank_load [L,R], stats [L,8]."""
    h = _i32(hist_arr)
    squeeze = h.ndim == 2
    if squeeze:
        h = h[None]
    L = h.shape[0]
    T, E, k, R = cfg["T"], cfg["E"], cfg["k"], cfg["R"]
    rpn, ns = cfg["ranks_per_node"], cfg["n_slot"]
    nl = E // R + ns
    it = cfg.get("max_refine_iters", 0) if max_refine_iters is None else max_refine_iters
    keep, mp = _main_ptr(cfg.get("main_rank"))
    out = dict(slot_expert=np.zeros((L, R, ns), np.int32),
               route_cnt=np.zeros((L, R, R, nl), np.int32),
               inst_load=np.zeros((L, R, nl), np.int32),
               rank_load=np.zeros((L, R), np.int32),
               stats=np.zeros((L, 8), np.int64))
    rc = _load().oracle_plan(T, E, k, R, rpn, ns, cfg["tok_bytes"], cfg["expert_bytes"],
                             cfg.get("c_intra", 1), cfg.get("c_inter", 4), it, mp, L,
                             h.reshape(-1), out["slot_expert"].reshape(-1),
                             out["route_cnt"].reshape(-1), out["inst_load"].reshape(-1),
                             out["rank_load"].reshape(-1), out["stats"].reshape(-1))
    del keep
    _check("oracle_plan", rc)
    if squeeze:
        out = {key: v[0] for key, v in out.items()}
    return out


def reroute(cfg: dict, ids, plan_out: dict):
    """dst_inst int32 [L, T*k] for ids [L, T, k] under the plan: within a source the
    pairs of expert e, in pair order, fill e's instances in ascending (rank,
    slot) order, each up to its routed count q (oracle.c, section O7)."""
    a = _i32(ids)
    squeeze = a.ndim == 2
    if squeeze:
        a = a[None]
    L, T, k = a.shape
    se = _i32(plan_out["slot_expert"]).reshape(L, -1)
    q = _i32(plan_out["route_cnt"]).reshape(L, -1)
    keep, mp = _main_ptr(cfg.get("main_rank"))
    keep_o, op = _offsets(cfg.get("rank_offsets"))
    dst = np.zeros((L, T * k), np.int32)
    rc = _load().oracle_reroute(T, cfg["E"], k, cfg["R"], cfg["ranks_per_node"], cfg["n_slot"],
                                mp, op, L, a.reshape(-1), se.reshape(-1), q.reshape(-1),
                                dst.reshape(-1))
    del keep, keep_o
    _check("oracle_reroute", rc)
    return dst[0] if squeeze else dst


def layout(cfg: dict, dst_inst, n_layers: int | None = None):
    """Dispatch layout for dst_inst int32 [L, T*k]: (sorted_pairs, seg_off,
    send_counts [L,R,R] int64, layout_stats [L,8] int64)."""
    d = _i32(dst_inst)
    squeeze = d.ndim == 1
    if squeeze:
        d = d[None]
    L = d.shape[0]
    T, E, k, R = cfg["T"], cfg["E"], cfg["k"], cfg["R"]
    nl = E // R + cfg["n_slot"]
    sp = np.zeros((L, T * k), np.int32)
    so = np.zeros((L, R * nl + 1), np.int32)
    sc = np.zeros((L, R, R), np.int64)
    st = np.zeros((L, 8), np.int64)
    keep, op = _offsets(cfg.get("rank_offsets"))
    _check("oracle_layout", _load().oracle_layout(T, E, k, R, cfg["ranks_per_node"], cfg["n_slot"],
                                                  cfg["tok_bytes"], op, L, d.reshape(-1),
                                                  sp.reshape(-1), so.reshape(-1),
                                                  sc.reshape(-1), st.reshape(-1)))
    if squeeze:
        return sp[0], so[0], sc[0], st[0]
    return sp, so, sc, st


def permute(x, sorted_pairs, k: int):
    """Dispatch pack: y[l][pos] = x[l][sorted_pairs[l][pos] // k] (bf16 rows as
    uint16).  x: uint16 [L, T, H]; sorted_pairs: int32 [L, T*k].  Returns
    uint16 [L, T*k, H]."""
    xa = np.ascontiguousarray(x, dtype=np.uint16)
    sp = _i32(sorted_pairs)
    L, T, H = xa.shape
    y = np.zeros((L, T * k, H), np.uint16)
    _check("oracle_permute", _load().oracle_permute(L, T, k, H, xa.reshape(-1), sp.reshape(-1),
                                                    y.reshape(-1)))
    return y


def combine(y, sorted_pairs, w, k: int):
    """Combine: out[l][t] = bf16(sum_j w[l][t][j] * y[l][pos(t, j)]) in float,
    slot order, one rounding.  y: uint16 [L, T*k, H]; w: float32 [L, T, k].
    Returns uint16 [L, T, H]."""
    ya = np.ascontiguousarray(y, dtype=np.uint16)
    sp = _i32(sorted_pairs)
    wa = np.ascontiguousarray(w, dtype=np.float32)
    L, n, H = ya.shape
    T = n // k
    out = np.zeros((L, T, H), np.uint16)
    _check("oracle_combine", _load().oracle_combine(L, T, k, H, ya.reshape(-1), sp.reshape(-1),
                                                    wa.reshape(-1), out.reshape(-1)))
    return out


DEDUP_STAT_NAMES = ("rows", "pairs", "rows_remote", "pairs_remote")


def dedup(cfg: dict, dst_inst):
    """Deduplicated dispatch layout for dst_inst int32 [L, T*k]: dict with
    seg [L, R+1], row_token [L, T*k], row_slots uint64 [L, T*k] (first seg[R]
    rows used), tok_dst uint64 [L, T, ceil(R/64)], send [L, R, R] int64,
    stats [L, 4] int64."""
    d = _i32(dst_inst)
    if d.ndim == 1:
        d = d[None]
    L = d.shape[0]
    T, E, k, R = cfg["T"], cfg["E"], cfg["k"], cfg["R"]
    nl = E // R + cfg["n_slot"]
    RW = (R + 63) // 64
    out = dict(seg=np.zeros((L, R + 1), np.int32), row_token=np.zeros((L, T * k), np.int32),
               row_slots=np.zeros((L, T * k), np.uint64), tok_dst=np.zeros((L, T, RW), np.uint64),
               send=np.zeros((L, R, R), np.int64), stats=np.zeros((L, 4), np.int64))
    keep, op = _offsets(cfg.get("rank_offsets"))
    _check("oracle_dedup", _load().oracle_dedup(T, k, R, nl, op, L, d.reshape(-1),
                                                out["seg"].reshape(-1), out["row_token"].reshape(-1),
                                                out["row_slots"].reshape(-1), out["tok_dst"].reshape(-1),
                                                out["send"].reshape(-1), out["stats"].reshape(-1)))
    return out
