"""Pins of the oracle's deduplicated dispatch layout."""
from math import comb

import numpy as np

import oracle
from moe_expert_routing_ids_gb300 import workloads as W


def test_dedup_hand_case(golden):
    g = golden("dedup_t4.json")
    o = oracle.dedup(g["cfg"], np.array([g["dst_inst"]], np.int32))
    ex = g["expected"]
    n = ex["seg"][-1]
    assert o["seg"][0].tolist() == ex["seg"]
    assert o["row_token"][0, :n].tolist() == ex["row_token"]
    assert o["row_slots"][0, :n].tolist() == ex["row_slots"]
    assert o["tok_dst"][0, :, 0].tolist() == ex["tok_dst"]
    assert o["send"][0].tolist() == ex["send"]
    assert o["stats"][0].tolist() == ex["stats"]


def _chain(cfg, ids):
    h = oracle.hist(ids, cfg["R"], cfg["E"])
    p = oracle.plan(cfg, h)
    return oracle.reroute(cfg, ids, p)


def _cfg(T, E, k, R, rpn, ns):
    return dict(T=T, E=E, k=k, R=R, ranks_per_node=rpn, n_slot=ns, tok_bytes=256,
                expert_bytes=1 << 20, c_intra=1, c_inter=4, max_refine_iters=0, main_rank=None)


def test_every_pair_is_covered_by_exactly_one_row():
    cfg = _cfg(T=512, E=32, k=4, R=8, rpn=4, ns=2)
    ids = W.random_small(5, 512, 32, 4, 2, s=1.3)
    d = _chain(cfg, ids)
    o = oracle.dedup(cfg, d)
    nl = 32 // 8 + 2
    for l in range(2):
        n = o["seg"][l, -1]
        covered = np.zeros((512, 4), np.int32)
        for row in range(n):
            t, m = o["row_token"][l, row], int(o["row_slots"][l, row])
            r = int(np.searchsorted(o["seg"][l], row, side="right")) - 1
            for j in range(4):
                if (m >> j) & 1:
                    covered[t, j] += 1
                    assert d[l, t * 4 + j] // nl == r
        assert np.all(covered == 1)
        # each token has one row per bit of its bitmap, rows are token-ordered in a rank
        bits = np.array([bin(int(x)).count("1") for x in o["tok_dst"][l, :, 0]])
        assert bits.sum() == n == o["stats"][l, 0]
        for r in range(8):
            seg = o["row_token"][l, o["seg"][l, r]:o["seg"][l, r + 1]]
            assert np.all(np.diff(seg) > 0)


def test_single_slot_keeps_one_row_per_pair():
    cfg = _cfg(T=256, E=16, k=1, R=4, rpn=2, ns=1)
    d = _chain(cfg, W.random_small(6, 256, 16, 1, 1))
    o = oracle.dedup(cfg, d)
    assert o["stats"][0, 0] == o["stats"][0, 1] == 256


def test_savings_match_the_printed_top2_and_top6_figures():
    # Expert Coupling in MoE Pretraining, "Moving Correlated Experts Together":
    # at EP8 deduplication alone removes about 6% of rows for top-2 and 25% for
    # top-6 routing.  With 64 experts on 8 ranks (8 each) and uniform distinct
    # Top-k, the expected fraction of rows saved is 1 - 8 * (1 - C(56,k)/C(64,k)) / k.
    rng = np.random.default_rng(0)
    for k, printed in ((2, 0.06), (6, 0.25)):
        T = 8 * 4096
        cfg = _cfg(T=T, E=64, k=k, R=8, rpn=8, ns=0)
        ids = np.stack([rng.permutation(64)[:k] for _ in range(T)]).astype(np.int32)[None]
        d = _chain(cfg, ids)
        st = oracle.dedup(cfg, d)["stats"][0]
        saved = 1 - st[0] / st[1]
        expect = 1 - 8 * (1 - comb(56, k) / comb(64, k)) / k
        assert abs(saved - expect) < 0.005, (k, saved, expect)
        assert abs(saved - printed) < 0.02, (k, saved, printed)
