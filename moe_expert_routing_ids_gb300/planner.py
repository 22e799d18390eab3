"""Device buffers and the call chain hist -> plan -> reroute -> dispatch layout.

Allocation uses torch (device memory and streams only); every computation is
a call into libtopoep through the same-named binding functions.
"""
from __future__ import annotations

import dataclasses

import torch

from . import (TOPO_CALL_CHAIN, TOPO_CALL_COOCCUR, TOPO_DTYPE_BF16, TOPO_DTYPE_F32, TOPO_LAYOUT_STATS,
               TOPO_STATS, make_cfg, make_plan, topo_cooccur, topo_cooccur_workspace_bytes,
               topo_dispatch_layout, topo_gate_hist,
               topo_hist, topo_plan, topo_read_error, topo_reroute, topo_reroute_layout,
               topo_workspace_bytes, topo_ws_reset)


@dataclasses.dataclass
class PlanBuffers:
    hist: torch.Tensor          # int32 [L, R, E]
    slot_expert: torch.Tensor   # int32 [L, R, n_slot]
    route_cnt: torch.Tensor     # int32 [L, R, R, n_local]
    inst_load: torch.Tensor     # int32 [L, R, n_local]
    rank_load: torch.Tensor     # int32 [L, R]
    stats: torch.Tensor         # int64 [L, 8]
    dst_inst: torch.Tensor      # int32 [L, T*k]
    sorted_pairs: torch.Tensor  # int32 [L, T*k]
    seg_off: torch.Tensor       # int32 [L, R*n_local + 1]
    send_counts: torch.Tensor   # int64 [L, R, R]
    layout_stats: torch.Tensor  # int64 [L, 8]


class Planner:
    """Owns the workspace and output buffers of one problem shape.

    cfg: dict with T, E, k, R, ranks_per_node, n_slot, tok_bytes, expert_bytes,
    c_intra, c_inter, optional max_refine_iters, rank_offsets (int64 [R+1]
    token offsets of the sources, device tensor or array, or None) and main_rank (device int32
    tensor or None)."""

    def __init__(self, cfg: dict, n_layers: int, device="cuda", stream=None):
        self.cfg_dict = dict(cfg)
        self.L = n_layers
        self.device = torch.device(device)
        self.main_rank = cfg.get("main_rank")
        if self.main_rank is not None and not isinstance(self.main_rank, torch.Tensor):
            self.main_rank = torch.as_tensor(self.main_rank, dtype=torch.int32, device=self.device)
        self.rank_offsets = cfg.get("rank_offsets")
        if self.rank_offsets is not None and not isinstance(self.rank_offsets, torch.Tensor):
            self.rank_offsets = torch.as_tensor(self.rank_offsets, dtype=torch.int64, device=self.device)
        self.cfg = make_cfg(**{**cfg, "main_rank": self.main_rank, "rank_offsets": self.rank_offsets})
        self.stream = stream
        T, E, k, R, ns = cfg["T"], cfg["E"], cfg["k"], cfg["R"], cfg["n_slot"]
        nl = E // R + ns
        self.n_local = nl
        self.ws_bytes = topo_workspace_bytes(self.cfg, n_layers, TOPO_CALL_CHAIN)
        if self.ws_bytes == 0:
            raise ValueError("invalid configuration for libtopoep")
        dev, i32, i64 = self.device, torch.int32, torch.int64
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        L = n_layers
        self.buf = PlanBuffers(
            hist=torch.empty((L, R, E), dtype=i32, device=dev),
            slot_expert=torch.empty((L, R, ns), dtype=i32, device=dev),
            route_cnt=torch.empty((L, R, R, nl), dtype=i32, device=dev),
            inst_load=torch.empty((L, R, nl), dtype=i32, device=dev),
            rank_load=torch.empty((L, R), dtype=i32, device=dev),
            stats=torch.empty((L, TOPO_STATS), dtype=i64, device=dev),
            dst_inst=torch.empty((L, T * k), dtype=i32, device=dev),
            sorted_pairs=torch.empty((L, T * k), dtype=i32, device=dev),
            seg_off=torch.empty((L, R * nl + 1), dtype=i32, device=dev),
            send_counts=torch.empty((L, R, R), dtype=i64, device=dev),
            layout_stats=torch.empty((L, TOPO_LAYOUT_STATS), dtype=i64, device=dev))
        b = self.buf
        self.plan = make_plan(b.slot_expert, b.route_cnt, b.inst_load, b.rank_load, b.stats)
        topo_ws_reset(self.ws, self.ws_bytes, self._stream())

    def _stream(self):
        return self.stream if self.stream is not None else torch.cuda.current_stream(self.device)

    def hist(self, ids: torch.Tensor):
        topo_hist(self.cfg, self.L, ids, self.buf.hist, self.ws, self.ws_bytes, self._stream())

    def gate_hist(self, logits: torch.Tensor, ids: torch.Tensor, bias: torch.Tensor | None = None,
                  scores: torch.Tensor | None = None):
        """Top-k gating of router logits (float32 or bfloat16 [L, T, E]) plus an
        optional float32 expert bias into ids (int32 [L, T, k]), the selected
        raw logits (float32 [L, T, k], optional) and the histogram; leaves the
        tile index so that make_plan / reroute_layout(ids) can follow."""
        if logits.dtype == torch.float32:
            dt = TOPO_DTYPE_F32
        elif logits.dtype == torch.bfloat16:
            dt = TOPO_DTYPE_BF16
        else:
            raise TypeError("logits must be float32 or bfloat16")
        topo_gate_hist(self.cfg, self.L, logits, dt, bias, ids, scores, self.buf.hist, self.ws,
                       self.ws_bytes, self._stream())

    def make_plan(self, hist: torch.Tensor | None = None):
        h = self.buf.hist if hist is None else hist
        topo_plan(self.cfg, self.L, h, self.plan, self.ws, self.ws_bytes, self._stream())

    def reroute(self, ids: torch.Tensor):
        topo_reroute(self.cfg, self.L, ids, self.plan, self.buf.dst_inst, self.ws, self.ws_bytes,
                     self._stream())

    def layout(self):
        b = self.buf
        topo_dispatch_layout(self.cfg, self.L, b.dst_inst, self.plan, b.sorted_pairs, b.seg_off,
                             b.send_counts, b.layout_stats, self.ws, self.ws_bytes, self._stream())

    def reroute_layout(self, ids: torch.Tensor):
        b = self.buf
        topo_reroute_layout(self.cfg, self.L, ids, self.plan, b.dst_inst, b.sorted_pairs, b.seg_off,
                            b.send_counts, b.layout_stats, self.ws, self.ws_bytes, self._stream())

    def run(self, ids: torch.Tensor, fused: bool = True):
        """The whole hot path on one batch of ids (device int32 [L, T, k]):
        histogram, plan, rerouting and dispatch layout (fused into one pass
        over the pairs unless fused=False)."""
        self.hist(ids)
        self.make_plan()
        if fused:
            self.reroute_layout(ids)
        else:
            self.reroute(ids)
            self.layout()

    def run_from_logits(self, logits: torch.Tensor, ids: torch.Tensor, bias: torch.Tensor | None = None,
                        scores: torch.Tensor | None = None):
        """Gating, plan, rerouting and dispatch layout from router logits."""
        self.gate_hist(logits, ids, bias, scores)
        self.make_plan()
        self.reroute_layout(ids)

    def error(self) -> int:
        """Device error word (synchronises the device)."""
        torch.cuda.synchronize(self.device)
        return topo_read_error(self.ws)

    def reset_error(self):
        topo_ws_reset(self.ws, self.ws_bytes, self._stream())

    def numpy(self) -> dict:
        return {f.name: getattr(self.buf, f.name).cpu().numpy() for f in dataclasses.fields(PlanBuffers)}


class Cooccur:
    """Buffers for topo_cooccur on [L, T, k] ids.  tensor_cores: give the call
    the workspace of its tensor-core path (used when E <= 128 and k <= 16);
    False keeps the header-only workspace and the shared-atomic kernels."""

    def __init__(self, L: int, T: int, E: int, k: int, device="cuda", transitions=True, tensor_cores=True):
        self.L, self.T, self.E, self.k = L, T, E, k
        dev = torch.device(device)
        self.device = dev
        self.ws_bytes = (topo_cooccur_workspace_bytes(L, T, E, k) if tensor_cores
                         else topo_workspace_bytes(None, 0, TOPO_CALL_COOCCUR))
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.co = torch.empty((L, E, E), dtype=torch.int64, device=dev)
        self.tr = torch.empty((max(L - 1, 0), E, E), dtype=torch.int64, device=dev) if transitions else None

    def run(self, ids: torch.Tensor, stream=None):
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        topo_cooccur(self.L, self.T, self.E, self.k, ids, self.co,
                     self.tr if (self.tr is not None and self.L > 1) else None, self.ws,
                     self.ws_bytes, s)

    def error(self) -> int:
        torch.cuda.synchronize(self.device)
        return topo_read_error(self.ws)
