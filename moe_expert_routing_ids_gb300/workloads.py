"""Seeded synthetic routing workloads (inputs only; none of the method's arithmetic).

The pages measure on real model routing over text corpora that are not
available here.  These generators stand in for them with the shapes and
structure of the pages' workloads:

* Biased-logit Top-k ("random logits with a fixed expert-specific bias",
  TopoEP §6.4): each token takes k distinct experts by successive sampling
  without replacement from a Zipf distribution over a seeded expert order.
  Successive sampling without replacement is the same distribution as
  Gumbel-top-k over log-probabilities (Plackett-Luce), drawn here by inverse
  CDF with redraw of repeats so that a million tokens take about a second.
* Cross-layer structure (Expert Coupling in MoE Pretraining, "Routing Is Also
  Correlated Across Layers"): a slot at layer l+1 keeps, with a fixed
  probability, an expert from a seeded neighbourhood of its layer-l expert.
* Within-layer grouping ("Experts Are Correlated Within a Layer"): experts
  fall in seeded groups; later slots stay in the first slot's group with a
  fixed probability.

Every array is produced by numpy ``Generator(PCG64(SeedSequence([seed,
layer])))`` so a workload is reproducible on any machine.

The five named workloads (``WORKLOADS``, by name; ``SMALL``, ``PLAN_LATENCY``,
``FOUR_LAYER``, ``COOCCUR``, ``STRESS``) carry the planner parameters the pages
fix or imply: S_tok = 2 * hidden (BF16 activations, TopoEP §2.3 / §4.1) and
||W|| = 3 * hidden * intermediate * 2 bytes (gate, up and down projections in
BF16; TopoEP §2.3 Fig. 3 and Table 1), with integer per-byte costs
c_intra = 1, c_inter = 4 (NVLink vs RDMA bandwidth ratio, TopoEP §6.1).
"""
from __future__ import annotations

import dataclasses

import numpy as np


def rng_for(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def zipf_probs(E: int, s: float, order: np.ndarray) -> np.ndarray:
    """p[order[i]] proportional to (i+1)^-s."""
    w = np.arange(1, E + 1, dtype=np.float64) ** (-float(s))
    p = np.empty(E, np.float64)
    p[order] = w / w.sum()
    return p


def _draw(rng, cdf: np.ndarray, n: int) -> np.ndarray:
    u = rng.random(n)
    return np.minimum(np.searchsorted(cdf, u, side="right"), len(cdf) - 1).astype(np.int32)


def topk_without_replacement(rng, p: np.ndarray, T: int, k: int) -> np.ndarray:
    """ids int32 [T, k]: k distinct experts per token, slot j = j-th draw of
    successive sampling without replacement proportional to p."""
    E = len(p)
    if k > int(np.count_nonzero(p)):
        raise ValueError("k exceeds the number of experts with nonzero probability")
    cdf = np.cumsum(p)
    ids = np.empty((T, k), np.int32)
    for j in range(k):
        cand = _draw(rng, cdf, T)
        rows = np.arange(T)
        while True:
            dup = np.zeros(len(rows), bool)
            for i in range(j):
                dup |= ids[rows, i] == cand
            ids[rows[~dup], j] = cand[~dup]
            rows = rows[dup]
            if len(rows) == 0:
                break
            cand = _draw(rng, cdf, len(rows))
    assert E > 0
    return ids


def neighbourhood_topk(rng, p: np.ndarray, prev: np.ndarray, nbr: np.ndarray,
                       keep: float) -> np.ndarray:
    """Next-layer ids: slot j keeps, with probability ``keep``, an expert drawn
    uniformly from nbr[prev[t, j]] (a seeded neighbourhood), else a draw from p;
    a repeat within the token is redrawn with the same mixture."""
    T, k = prev.shape
    cdf = np.cumsum(p)
    width = nbr.shape[1]
    ids = np.empty((T, k), np.int32)

    def mix(rows, j):
        near = rng.random(len(rows)) < keep
        pick = nbr[prev[rows, j], rng.integers(0, width, len(rows))]
        far = _draw(rng, cdf, len(rows))
        return np.where(near, pick, far).astype(np.int32)

    for j in range(k):
        rows = np.arange(T)
        cand = mix(rows, j)
        while True:
            dup = np.zeros(len(rows), bool)
            for i in range(j):
                dup |= ids[rows, i] == cand
            ids[rows[~dup], j] = cand[~dup]
            rows = rows[dup]
            if len(rows) == 0:
                break
            cand = mix(rows, j)
    return ids


def grouped_topk(rng, E: int, T: int, k: int, groups: np.ndarray, stay: float) -> np.ndarray:
    """Slot 0 uniform over E; later slots, with probability ``stay``, uniform in
    slot 0's group, else uniform over E; repeats redrawn with the same mixture.
    groups: int [G, g] expert ids."""
    gid = np.empty(E, np.int64)
    for g, members in enumerate(groups):
        gid[members] = g
    ids = np.empty((T, k), np.int32)
    ids[:, 0] = rng.integers(0, E, T)
    home = gid[ids[:, 0]]
    width = groups.shape[1]

    def mix(rows):
        near = rng.random(len(rows)) < stay
        pick = groups[home[rows], rng.integers(0, width, len(rows))]
        far = rng.integers(0, E, len(rows))
        return np.where(near, pick, far).astype(np.int32)

    for j in range(1, k):
        rows = np.arange(T)
        cand = mix(rows)
        while True:
            dup = np.zeros(len(rows), bool)
            for i in range(j):
                dup |= ids[rows, i] == cand
            ids[rows[~dup], j] = cand[~dup]
            rows = rows[dup]
            if len(rows) == 0:
                break
            cand = mix(rows)
    return ids


@dataclasses.dataclass(frozen=True)
class Workload:
    """One named workload.  ``plan_cfg`` is the planner's parameter set."""
    seed: int                 # first key of every layer's random stream
    name: str
    kind: str                 # "plan" (hist, plan, reroute, layout) or "cooccur"
    structure: str            # "zipf", "neighbourhood" or "grouped"
    T: int
    E: int
    k: int
    n_layers: int             # layers, or microbatches, planned per call
    R: int = 0
    ranks_per_node: int = 0
    n_slot: int = 0
    hidden: int = 0
    intermediate: int = 0
    c_intra: int = 1
    c_inter: int = 4
    zipf_s: float = 1.0

    @property
    def plan_cfg(self) -> dict:
        return dict(T=self.T, E=self.E, k=self.k, R=self.R,
                    ranks_per_node=self.ranks_per_node, n_slot=self.n_slot,
                    tok_bytes=2 * self.hidden,
                    expert_bytes=3 * self.hidden * self.intermediate * 2,
                    c_intra=self.c_intra, c_inter=self.c_inter,
                    max_refine_iters=0, main_rank=None)

    @property
    def pairs(self) -> int:
        return self.T * self.k * self.n_layers

    def ids(self, replica: int = 0, n_layers: int | None = None) -> np.ndarray:
        """int32 [n_layers, T, k].  ``replica`` > 0 draws an independent copy
        (another data-parallel replica); ``n_layers`` truncates the stack."""
        n = self.n_layers if n_layers is None else n_layers
        if self.structure == "zipf":
            return _gen_zipf(self, self.zipf_s, replica, n)
        if self.structure == "neighbourhood":
            return _gen_neighbourhood(self, replica, n)
        return _gen_grouped(self, replica, n)


def _seed(w: Workload, replica: int, l: int):
    return rng_for(w.seed, l) if replica == 0 else rng_for(w.seed, l, replica)


def _gen_zipf(w: Workload, s: float, replica: int, n_layers: int) -> np.ndarray:
    out = np.empty((n_layers, w.T, w.k), np.int32)
    for l in range(n_layers):
        rng = _seed(w, replica, l)
        order = rng.permutation(w.E)
        out[l] = topk_without_replacement(rng, zipf_probs(w.E, s, order), w.T, w.k)
    return out


def _gen_neighbourhood(w: Workload, replica: int, n_layers: int) -> np.ndarray:
    s_per_layer = (0.8, 1.2, 1.6, 1.2)
    out = np.empty((n_layers, w.T, w.k), np.int32)
    for l in range(n_layers):
        rng = _seed(w, replica, l)
        order = rng.permutation(w.E)
        p = zipf_probs(w.E, s_per_layer[l % len(s_per_layer)], order)
        if l == 0:
            out[l] = topk_without_replacement(rng, p, w.T, w.k)
        else:
            nbr = np.stack([rng.choice(w.E, 16, replace=False) for _ in range(w.E)]).astype(np.int32)
            out[l] = neighbourhood_topk(rng, p, out[l - 1], nbr, keep=0.6)
    return out


def _gen_grouped(w: Workload, replica: int, n_layers: int) -> np.ndarray:
    out = np.empty((n_layers, w.T, w.k), np.int32)
    for l in range(n_layers):
        rng = _seed(w, replica, l)
        groups = rng.permutation(w.E).reshape(16, w.E // 16)
        out[l] = grouped_topk(rng, w.E, w.T, w.k, groups, stay=0.7)
    return out


SMALL = Workload(1, "t4096_e8_k2_r8", "plan", "zipf", T=4096, E=8, k=2, n_layers=1, R=8,
                 ranks_per_node=4, n_slot=2, hidden=1024, intermediate=768, zipf_s=1.0)
PLAN_LATENCY = Workload(2, "t16384_e64_k6_r32", "plan", "zipf", T=16384, E=64, k=6, n_layers=1,
                        R=32, ranks_per_node=8, n_slot=8, hidden=4096, intermediate=1408,
                        zipf_s=1.2)
FOUR_LAYER = Workload(3, "t65536_e256_k8_r64_4layers", "plan", "neighbourhood", T=65536, E=256,
                      k=8, n_layers=4, R=64, ranks_per_node=8, n_slot=32, hidden=7168,
                      intermediate=1536)
COOCCUR = Workload(4, "cooccur_l8_t262144_e128_k8", "cooccur", "grouped", T=262144, E=128, k=8,
                   n_layers=8)
STRESS = Workload(5, "t1048576_e512_k10_r128_4mb", "plan", "zipf", T=1048576, E=512, k=10,
                  n_layers=4, R=128, ranks_per_node=8, n_slot=64, hidden=7168, intermediate=1536,
                  zipf_s=1.4)

WORKLOADS = {w.name: w for w in (SMALL, PLAN_LATENCY, FOUR_LAYER, COOCCUR, STRESS)}
PLAN_WORKLOADS = (SMALL, PLAN_LATENCY, FOUR_LAYER, STRESS)


def random_small(seed: int, T: int, E: int, k: int, n_layers: int = 1, s: float = 1.0) -> np.ndarray:
    """Small Zipf Top-k ids for tests, int32 [n_layers, T, k]."""
    out = np.empty((n_layers, T, k), np.int32)
    for l in range(n_layers):
        rng = rng_for(1000 + seed, l)
        out[l] = topk_without_replacement(rng, zipf_probs(E, s, rng.permutation(E)), T, k)
    return out


def gumbel_logits(seed: int, L: int, T: int, E: int, chunk: int = 1 << 16) -> np.ndarray:
    """Router logits float32 [L, T, E]: standard Gumbel noise (the "random
    logits" of TopoEP §6.4), drawn in token chunks so the float64 draw never
    holds more than `chunk` rows."""
    out = np.empty((L, T, E), np.float32)
    for l in range(L):
        rng = rng_for(seed, l)
        for a in range(0, T, chunk):
            b = min(T, a + chunk)
            out[l, a:b] = rng.gumbel(size=(b - a, E))
    return out


def zipf_bias(seed: int, E: int, s: float) -> np.ndarray:
    """Fixed expert-specific bias float32 [E]: log of Zipf(s) probabilities
    over a seeded expert order (TopoEP §6.4)."""
    rng = rng_for(seed, 1 << 20)
    return np.log(zipf_probs(E, s, rng.permutation(E))).astype(np.float32)


def _solver_point(seed: int, E: int, R: int) -> Workload:
    return Workload(seed, f"t{4096 * R}_e{E}_k8_r{R}", "plan", "zipf", T=4096 * R, E=E, k=8,
                    n_layers=1, R=R, ranks_per_node=8, n_slot=2, hidden=2048, intermediate=768,
                    zipf_s=1.2)


# Solver-latency sweeps shaped like TopoEP §6.3 Fig. 11: Top-8 routing with two
# replica slots per rank (the setting §6.2 adopts after Fig. 10), 4096 tokens
# per source rank, 8 ranks per node, Zipf(1.2) over a seeded expert order,
# hidden 2048 / intermediate 768 (the Qwen3-30B-A3B row of Table 1, whose
# expert is the 9 MiB of Fig. 3).  (a) E = 640 over EP 8..128; (b) EP 32 over
# a 16x range of expert counts.
SOLVER_RANKS = tuple(_solver_point(600 + i, 640, R) for i, R in enumerate((8, 16, 32, 64, 128)))
SOLVER_EXPERTS = tuple(_solver_point(700 + i, E, 32)
                       for i, E in enumerate((64, 128, 256, 512, 640, 1024)))


def random_cooccur(seed: int, L: int, E: int, hi: int = 1000) -> np.ndarray:
    """Co-selection counts int64 [L, E, E] with independent uniform entries in
    [0, hi): a graph without planted groups, on which the greedy placement
    leaves gainful swaps."""
    return np.stack([rng_for(seed, l).integers(0, hi, size=(E, E)) for l in range(L)]).astype(np.int64)
