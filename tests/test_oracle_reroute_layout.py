"""Pins for the oracle's rerouting and dispatch layout (CPU only).

Rerouting: a hand-worked case, and the identities every valid rerouting
satisfies (each pair assigned once, counts per (source, instance) equal q,
the instance holds the pair's expert, per-rank received pairs equal L_r),
plus the order property of the chosen reading (occurrences of (s, e) fill
e's instances in ascending rank order).
Layout: numpy's stable argsort, bijection and count identities.
"""
import numpy as np
import pytest

import oracle
from moe_expert_routing_ids_gb300 import workloads as W

from test_oracle_plan import instance_experts


def test_reroute_and_layout_hand_case(golden):
    g = golden("reroute_layout_t2.json")
    cfg = g["cfg"]
    ids = np.array(g["ids"], np.int32)
    plan = dict(slot_expert=np.array(g["slot_expert"], np.int32),
                route_cnt=np.array(g["route_cnt"], np.int32))
    dst = oracle.reroute(cfg, ids, plan)
    ex = g["expected"]
    assert dst.tolist() == ex["dst_inst"]
    sp, so, sc, st = oracle.layout(cfg, dst)
    assert sp.tolist() == ex["sorted_pairs"]
    assert so.tolist() == ex["seg_off"]
    assert sc.tolist() == ex["send_counts"]
    assert st.tolist() == ex["layout_stats"]


def test_reroute_t1_source0_expert0(golden):
    """Pair-to-instance order on the Fig. 9-shaped plan: a source's pairs for
    an expert fill that expert's instances in ascending rank order, each up
    to its routed count, so source 0's six e0 assignments go 2 to the main
    on r0, then 4 to r1's replica."""
    g = golden("plan_t1_fig9_shape.json")
    cfg = dict(g["cfg"])
    # ids consistent with the hist rows: 14 pairs per source would need equal
    # blocks, so use k = 14 slots per token with one token per source
    h = np.array(g["hist"], np.int32)
    cfg["T"], cfg["k"] = 4, 14
    ids = np.full((4, 14), -1, np.int32)
    for s in range(4):
        row = np.repeat(np.arange(4), h[s])
        ids[s, :len(row)] = row
    # pad sources with fewer than 14 assignments using their own main expert
    plan_h = h.copy()
    for s in range(4):
        n = h[s].sum()
        ids[s, n:] = s
        plan_h[s, s] += 14 - n
    p = oracle.plan(cfg, plan_h)
    dst = oracle.reroute(cfg, ids[None], p)[0]
    nl = cfg["E"] // cfg["R"] + cfg["n_slot"]
    e0_pairs = [j for j in range(14) if ids[0, j] == 0]
    got = [(int(dst[j]) // nl, int(dst[j]) % nl) for j in e0_pairs]
    want_r0 = int(p["route_cnt"][0, 0, 0])
    assert got == [(0, 0)] * want_r0 + [(1, 1)] * (len(e0_pairs) - want_r0)


def reroute_invariants(cfg, ids, p, dst):
    R, E, k, T = cfg["R"], cfg["E"], cfg["k"], cfg["T"]
    nl = E // R + cfg["n_slot"]
    inst, owner = instance_experts(cfg, p["slot_expert"])
    flat = ids.reshape(-1)
    assert dst.shape == flat.shape
    assert ((dst >= 0) & (dst < R * nl)).all()
    src = (np.arange(T * k) // k) // (T // R)
    # the instance holds the pair's expert
    assert np.array_equal(inst[dst // nl, dst % nl], flat)
    # per (source, instance) counts equal q
    cnt = np.zeros((R, R * nl), np.int64)
    np.add.at(cnt, (src, dst), 1)
    assert np.array_equal(cnt.reshape(R, R, nl), p["route_cnt"])
    # received pairs per rank = L_r
    assert np.array_equal(np.bincount(dst // nl, minlength=R), p["rank_load"])
    # reading: within (s, e), occurrences fill instances in ascending rank order
    for s in range(R):
        sel = src == s
        for e in np.unique(flat[sel]):
            ranks = (dst[sel][flat[sel] == e]) // nl
            assert (np.diff(ranks) >= 0).all()


@pytest.mark.parametrize("shape", [(8, 4, 8, 2, 512, 2, 1.0, 0.01), (8, 2, 16, 3, 800, 3, 1.4, 0.02),
                                   (16, 8, 32, 8, 1600, 6, 1.2, 0.03), (6, 3, 6, 1, 300, 2, 0.8, 0.001),
                                   (4, 4, 8, 0, 400, 2, 1.2, 1.0)])
def test_reroute_invariants_random(shape):
    from test_oracle_plan import _random_case
    R, rpn, E, ns, T, k, s, Wmul = shape
    cfg, ids, h = _random_case(11 + R, R, rpn, E, ns, T, k, s, Wmul)
    p = oracle.plan(cfg, h)
    dst = oracle.reroute(cfg, ids[0], p)
    reroute_invariants(cfg, ids[0], p, dst)


def layout_invariants(cfg, dst, sp, so, sc, st):
    R, E, k, T = cfg["R"], cfg["E"], cfg["k"], cfg["T"]
    nl = E // R + cfg["n_slot"]
    assert np.array_equal(sp, np.argsort(dst, kind="stable"))
    assert np.array_equal(np.sort(sp), np.arange(T * k))                  # bijection
    counts = np.bincount(dst, minlength=R * nl)
    assert np.array_equal(so, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(dst[sp], np.repeat(np.arange(R * nl), counts))
    src = (np.arange(T * k) // k) // (T // R)
    assert sc.sum() == T * k
    assert np.array_equal(sc.sum(axis=1), np.bincount(src, minlength=R))
    assert np.array_equal(sc.sum(axis=0), np.bincount(dst // nl, minlength=R))
    assert st[0] + st[1] + st[2] == T * k
    assert st[0] == np.trace(sc)
    assert list(st[3:6]) == [x * cfg["tok_bytes"] for x in st[0:3]]
    assert st[6] == int(((dst % nl) >= E // R).sum())


@pytest.mark.parametrize("shape", [(8, 4, 8, 2, 512, 2, 1.0, 0.01), (16, 8, 32, 8, 1600, 6, 1.2, 0.03),
                                   (6, 3, 6, 1, 300, 2, 0.8, 0.001)])
def test_layout_invariants_random(shape):
    from test_oracle_plan import _random_case
    R, rpn, E, ns, T, k, s, Wmul = shape
    cfg, ids, h = _random_case(21 + R, R, rpn, E, ns, T, k, s, Wmul)
    p = oracle.plan(cfg, h)
    dst = oracle.reroute(cfg, ids[0], p)
    sp, so, sc, st = oracle.layout(cfg, dst)
    layout_invariants(cfg, dst, sp, so, sc, st)


def test_layout_of_arbitrary_keys_is_stable_sort():
    cfg = dict(T=40, E=4, k=3, R=4, ranks_per_node=2, n_slot=2, tok_bytes=8)
    rng = W.rng_for(3, 3)
    dst = rng.integers(0, 4 * 3, 120).astype(np.int32)
    sp, so, sc, st = oracle.layout(cfg, dst)
    layout_invariants(cfg, dst, sp, so, sc, st)


def test_layout_rejects_bad_key():
    cfg = dict(T=4, E=4, k=1, R=4, ranks_per_node=2, n_slot=0, tok_bytes=8)
    with pytest.raises(oracle.OracleError):
        oracle.layout(cfg, np.array([0, 1, 2, 9], np.int32))


def test_reroute_out_of_range_id():
    cfg = dict(T=4, E=4, k=1, R=4, ranks_per_node=2, n_slot=0)
    p = dict(slot_expert=np.zeros((4, 0), np.int32), route_cnt=np.zeros((4, 4, 1), np.int32))
    with pytest.raises(oracle.OracleError) as ex:
        oracle.reroute(cfg, np.array([[0], [7], [2], [3]], np.int32), p)
    assert ex.value.rc == oracle.ERANGE
