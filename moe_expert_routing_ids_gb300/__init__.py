"""Python binding of libtopoep (GB300, sm_103a): the topology-aware
expert-routing plan of "TopoEP: Topology-Aware Load Balancing for
Expert-Parallel MoE Training" (§4) plus the expert co-selection statistics of
"Expert Coupling in MoE Pretraining".

This module only marshals arguments into the C ABI declared in
``include/topo.h``; every step runs in the library's CUDA kernels.  The
functions carry the C names and take device pointers as Python ints or as
objects with ``data_ptr()`` (torch tensors), and CUDA streams as raw handles
(``torch.cuda.current_stream().cuda_stream``) or objects with ``cuda_stream``.
A nonzero return code raises :class:`TopoError`.  If the shared library has
not been built, every call raises -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libtopoep.so")

TOPO_OK, TOPO_EINVAL, TOPO_ENOSPC, TOPO_ECUDA = 0, -1, -2, -3
TOPO_ERANGE, TOPO_ESTATE, TOPO_EMAP, TOPO_EOFFSETS, TOPO_ETIMEOUT = -4, -5, -6, -7, -8
TOPO_CALL_HIST, TOPO_CALL_PLAN, TOPO_CALL_REROUTE, TOPO_CALL_LAYOUT = 0, 1, 2, 3
TOPO_CALL_COOCCUR, TOPO_CALL_CHAIN, TOPO_CALL_REROUTE_LAYOUT = 4, 5, 6
TOPO_CALL_PACK = 7
TOPO_CALL_DEDUP = 8
TOPO_CALL_GATE = 9
TOPO_DTYPE_F32 = 0
TOPO_DTYPE_BF16 = 1
TOPO_GATE_MAX_E = 1024
TOPO_SHUFFLE_STATS = 4
TOPO_SHUFFLE_MAX_RANKS = 256
TOPO_PLACE_STATS = 4
TOPO_DEDUP_STATS = 4
TOPO_STATS = 8
TOPO_LAYOUT_STATS = 8
EXPORTS = ("topo_workspace_bytes", "topo_ws_reset", "topo_hist", "topo_cooccur", "topo_plan",
           "topo_reroute", "topo_dispatch_layout", "topo_reroute_layout", "topo_read_error",
           "topo_strerror", "topo_hist_noalloc", "topo_permute", "topo_combine",
           "topo_dedup_layout", "topo_gate_hist", "topo_shuffle_workspace_bytes",
           "topo_shuffle_targets", "topo_place_experts", "topo_cooccur_workspace_bytes")
TOPO_HIST_NOALLOC_SCRATCH_BYTES = 16 << 20


class TopoError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {code} ({strerror(code)})")
        self.code = code


class TopoCfg(ctypes.Structure):
    """Mirror of topo_cfg."""
    _fields_ = [("T", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("R", ctypes.c_int32), ("ranks_per_node", ctypes.c_int32),
                ("n_slot", ctypes.c_int32), ("tok_bytes", ctypes.c_int64),
                ("expert_bytes", ctypes.c_int64), ("c_intra", ctypes.c_int32),
                ("c_inter", ctypes.c_int32), ("max_refine_iters", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("main_rank", ctypes.c_void_p),
                ("rank_offsets", ctypes.c_void_p)]


class TopoPlan(ctypes.Structure):
    """Mirror of topo_plan_t (device pointers)."""
    _fields_ = [("slot_expert", ctypes.c_void_p), ("route_cnt", ctypes.c_void_p),
                ("inst_load", ctypes.c_void_p), ("rank_load", ctypes.c_void_p),
                ("stats", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded shared library; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libtopoep.so not built ({LIB_PATH}); run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            vp, sz, i32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32
            cfgp, planp = ctypes.POINTER(TopoCfg), ctypes.POINTER(TopoPlan)
            L.topo_workspace_bytes.argtypes = [cfgp, i32, i32]
            L.topo_workspace_bytes.restype = sz
            L.topo_ws_reset.argtypes = [vp, sz, vp]
            L.topo_hist.argtypes = [cfgp, i32, vp, vp, vp, sz, vp]
            L.topo_cooccur.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, sz, vp]
            L.topo_plan.argtypes = [cfgp, i32, vp, planp, vp, sz, vp]
            L.topo_reroute.argtypes = [cfgp, i32, vp, planp, vp, vp, sz, vp]
            L.topo_dispatch_layout.argtypes = [cfgp, i32, vp, planp, vp, vp, vp, vp, vp, sz, vp]
            L.topo_reroute_layout.argtypes = [cfgp, i32, vp, planp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.topo_hist_noalloc.argtypes = [cfgp, i32, vp, vp, vp, vp]
            L.topo_permute.argtypes = [cfgp, i32, i32, vp, vp, vp, vp, sz, vp]
            L.topo_dedup_layout.argtypes = [cfgp, i32, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.topo_gate_hist.argtypes = [cfgp, i32, vp, i32, vp, vp, vp, vp, vp, sz, vp]
            L.topo_cooccur_workspace_bytes.argtypes = [i32, i32, i32, i32]
            L.topo_cooccur_workspace_bytes.restype = sz
            L.topo_shuffle_workspace_bytes.argtypes = [i32, i32, i32]
            L.topo_shuffle_workspace_bytes.restype = sz
            L.topo_shuffle_targets.argtypes = [i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.topo_place_experts.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp]
            L.topo_combine.argtypes = [cfgp, i32, i32, vp, vp, vp, vp, vp, sz, vp]
            L.topo_read_error.argtypes = [vp]
            L.topo_strerror.argtypes = [ctypes.c_int]
            L.topo_strerror.restype = ctypes.c_char_p
            for f in ("topo_ws_reset", "topo_hist", "topo_cooccur", "topo_plan", "topo_reroute",
                      "topo_dispatch_layout", "topo_reroute_layout", "topo_read_error",
                      "topo_hist_noalloc", "topo_permute", "topo_combine", "topo_dedup_layout", "topo_gate_hist", "topo_shuffle_targets", "topo_place_experts"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def _p(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr() or None
    return int(x) or None


def _s(stream):
    if stream is None:
        return None
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream or None
    return int(stream) or None


def _chk(fn, rc):
    if rc != TOPO_OK:
        raise TopoError(fn, rc)
    return rc


def make_cfg(T, E, k, R, ranks_per_node, n_slot, tok_bytes=0, expert_bytes=0, c_intra=1,
             c_inter=4, max_refine_iters=0, main_rank=None, rank_offsets=None, **_ignored) -> TopoCfg:
    """topo_cfg from plain values; main_rank (int32 [E]) and rank_offsets
    (int64 [R+1]) are device pointers/tensors or None."""
    return TopoCfg(T, E, k, R, ranks_per_node, n_slot, tok_bytes, expert_bytes, c_intra, c_inter,
                   max_refine_iters, 0, _p(main_rank), _p(rank_offsets))


def make_plan(slot_expert, route_cnt, inst_load, rank_load, stats) -> TopoPlan:
    return TopoPlan(_p(slot_expert), _p(route_cnt), _p(inst_load), _p(rank_load), _p(stats))


def strerror(code: int) -> str:
    try:
        return lib().topo_strerror(code).decode()
    except RuntimeError:
        return "library not loaded"


def topo_workspace_bytes(cfg: TopoCfg | None, n_layers: int, which_call: int) -> int:
    return lib().topo_workspace_bytes(ctypes.byref(cfg) if cfg is not None else None, n_layers,
                                      which_call)


def topo_ws_reset(ws, ws_bytes: int, stream=None) -> int:
    return _chk("topo_ws_reset", lib().topo_ws_reset(_p(ws), ws_bytes, _s(stream)))


def topo_hist(cfg: TopoCfg, n_layers: int, ids, hist, ws, ws_bytes: int, stream=None) -> int:
    return _chk("topo_hist", lib().topo_hist(ctypes.byref(cfg), n_layers, _p(ids), _p(hist), _p(ws),
                                             ws_bytes, _s(stream)))


def topo_cooccur(L: int, T: int, E: int, k: int, ids, co, tr, ws, ws_bytes: int, stream=None) -> int:
    return _chk("topo_cooccur", lib().topo_cooccur(L, T, E, k, _p(ids), _p(co), _p(tr), _p(ws),
                                                   ws_bytes, _s(stream)))


def topo_plan(cfg: TopoCfg, n_layers: int, hist, plan: TopoPlan, ws, ws_bytes: int,
              stream=None) -> int:
    return _chk("topo_plan", lib().topo_plan(ctypes.byref(cfg), n_layers, _p(hist),
                                             ctypes.byref(plan), _p(ws), ws_bytes, _s(stream)))


def topo_reroute(cfg: TopoCfg, n_layers: int, ids, plan: TopoPlan, dst_inst, ws, ws_bytes: int,
                 stream=None) -> int:
    return _chk("topo_reroute", lib().topo_reroute(ctypes.byref(cfg), n_layers, _p(ids),
                                                   ctypes.byref(plan), _p(dst_inst), _p(ws),
                                                   ws_bytes, _s(stream)))


def topo_dispatch_layout(cfg: TopoCfg, n_layers: int, dst_inst, plan: TopoPlan, sorted_pairs,
                         seg_off, send_counts, layout_stats, ws, ws_bytes: int,
                         stream=None) -> int:
    return _chk("topo_dispatch_layout",
                lib().topo_dispatch_layout(ctypes.byref(cfg), n_layers, _p(dst_inst),
                                           ctypes.byref(plan), _p(sorted_pairs), _p(seg_off),
                                           _p(send_counts), _p(layout_stats), _p(ws), ws_bytes,
                                           _s(stream)))


def topo_reroute_layout(cfg: TopoCfg, n_layers: int, ids, plan: TopoPlan, dst_inst, sorted_pairs,
                        seg_off, send_counts, layout_stats, ws, ws_bytes: int, stream=None) -> int:
    return _chk("topo_reroute_layout",
                lib().topo_reroute_layout(ctypes.byref(cfg), n_layers, _p(ids), ctypes.byref(plan),
                                          _p(dst_inst), _p(sorted_pairs), _p(seg_off),
                                          _p(send_counts), _p(layout_stats), _p(ws), ws_bytes,
                                          _s(stream)))


def topo_hist_noalloc(cfg: TopoCfg, n_layers: int, ids, hist, err=None, stream=None) -> int:
    """topo_hist with the library's fixed scratch array instead of a workspace;
    err: optional device int32 that receives the device error word."""
    return _chk("topo_hist_noalloc", lib().topo_hist_noalloc(ctypes.byref(cfg), n_layers, _p(ids),
                                                             _p(hist), _p(err), _s(stream)))


def topo_place_experts(L: int, E: int, R: int, max_iters: int, co, main_rank, stats, stream=None) -> int:
    """Correlated expert placement from co-selection counts into a main-rank map."""
    return _chk("topo_place_experts",
                lib().topo_place_experts(L, E, R, max_iters, _p(co), _p(main_rank), _p(stats), _s(stream)))


def topo_shuffle_workspace_bytes(L: int, E: int, R: int) -> int:
    return int(lib().topo_shuffle_workspace_bytes(L, E, R))


def topo_cooccur_workspace_bytes(L: int, T: int, E: int, k: int) -> int:
    """Workspace bytes that let topo_cooccur use the tensor cores."""
    return int(lib().topo_cooccur_workspace_bytes(L, T, E, k))


def topo_shuffle_targets(L: int, T: int, E: int, k: int, R: int, ids, tr, main_rank, rank_offsets, target,
                         stats, ws, ws_bytes: int, stream=None) -> int:
    """Token-shuffle targets from cross-layer transition counts."""
    return _chk("topo_shuffle_targets",
                lib().topo_shuffle_targets(L, T, E, k, R, _p(ids), _p(tr), _p(main_rank), _p(rank_offsets),
                                           _p(target), _p(stats), _p(ws), ws_bytes, _s(stream)))


def topo_gate_hist(cfg: TopoCfg, n_layers: int, logits, logits_dtype: int, bias, ids, scores, hist,
                   ws, ws_bytes: int, stream=None) -> int:
    """Top-k gating of router logits (plus an optional expert bias) and Omega."""
    return _chk("topo_gate_hist",
                lib().topo_gate_hist(ctypes.byref(cfg), n_layers, _p(logits), logits_dtype, _p(bias),
                                     _p(ids), _p(scores), _p(hist), _p(ws), ws_bytes, _s(stream)))


def topo_dedup_layout(cfg: TopoCfg, n_layers: int, dst_inst, seg, row_token, row_slots, tok_dst,
                      send, stats, ws, ws_bytes: int, stream=None) -> int:
    """Deduplicated dispatch layout: one row per (token, destination rank)."""
    return _chk("topo_dedup_layout",
                lib().topo_dedup_layout(ctypes.byref(cfg), n_layers, _p(dst_inst), _p(seg),
                                        _p(row_token), _p(row_slots), _p(tok_dst), _p(send),
                                        _p(stats), _p(ws), ws_bytes, _s(stream)))


def topo_permute(cfg: TopoCfg, n_layers: int, H: int, x, sorted_pairs, y, ws, ws_bytes: int,
                 stream=None) -> int:
    """Dispatch pack: y[l][pos] = x[l][sorted_pairs[l][pos] // k] (bf16 rows)."""
    return _chk("topo_permute", lib().topo_permute(ctypes.byref(cfg), n_layers, H, _p(x),
                                                   _p(sorted_pairs), _p(y), _p(ws), ws_bytes,
                                                   _s(stream)))


def topo_combine(cfg: TopoCfg, n_layers: int, H: int, y, sorted_pairs, w, out, ws, ws_bytes: int,
                 stream=None) -> int:
    """Combine: out[l][t] = bf16(sum_j w[l][t][j] * y[l][pos(t, j)]), float, slot order."""
    return _chk("topo_combine", lib().topo_combine(ctypes.byref(cfg), n_layers, H, _p(y),
                                                   _p(sorted_pairs), _p(w), _p(out), _p(ws),
                                                   ws_bytes, _s(stream)))


def topo_read_error(ws) -> int:
    return lib().topo_read_error(_p(ws))


def topo_strerror(code: int) -> str:
    return strerror(code)
