"""Pins of the oracle's unequal source blocks (rank_offsets): each rank
routes its own local tokens (TopoEP §2.1), so the ranks' blocks may differ in
length or be empty."""
import numpy as np
import pytest

import oracle
from moe_expert_routing_ids_gb300 import workloads as W


def _cfg(c):
    return dict(T=c["T"], E=c["E"], k=c["k"], R=c["R"], ranks_per_node=c["ranks_per_node"],
                n_slot=c["n_slot"], tok_bytes=c["tok_bytes"], expert_bytes=1 << 20, c_intra=1,
                c_inter=4, max_refine_iters=0, main_rank=None, rank_offsets=c["rank_offsets"])


def test_hand_cases(golden):
    for c in golden("offsets_hand.json")["cases"]:
        cfg = _cfg(c)
        ids = np.array(c["ids"], np.int32)[None]
        h = oracle.hist(ids, c["R"], c["E"], rank_offsets=c["rank_offsets"])
        assert h[0].tolist() == c["hist"], c["name"]
        p = oracle.plan(cfg, h)
        d = oracle.reroute(cfg, ids, p)
        assert d[0].tolist() == c["dst_inst"], c["name"]
        sp, so, sc, st = oracle.layout(cfg, d)
        assert sp[0].tolist() == c["sorted_pairs"], c["name"]
        assert so[0].tolist() == c["seg_off"], c["name"]
        assert sc[0].tolist() == c["send_counts"], c["name"]
        assert st[0].tolist() == c["layout_stats"], c["name"]
        if "dedup" in c:
            dd = oracle.dedup(cfg, d)
            for key, want in c["dedup"].items():
                got = dd[key][0]
                if key == "tok_dst":
                    got = got[:, 0]
                if key in ("row_token", "row_slots"):
                    got = got[:dd["seg"][0][-1]]
                assert np.asarray(got).tolist() == want, (c["name"], key)
        if "ids_next" in c:
            both = np.stack([ids[0], np.array(c["ids_next"], np.int32)])
            _, tr = oracle.cooccur(both, c["E"])
            tg, sst = oracle.shuffle(both, tr, c["R"], rank_offsets=c["rank_offsets"])
            assert tg[0].tolist() == c["shuffle_target"]
            assert sst[0].tolist() == c["shuffle_stats"]


def _random_offsets(rng, T, R, empty=True):
    cuts = np.sort(rng.integers(0, T + 1, size=R - 1))
    off = np.concatenate([[0], cuts, [T]]).astype(np.int64)
    if not empty:
        assert np.all(np.diff(off) > 0)
    return off


def test_equal_offsets_reduce_to_equal_blocks():
    # offsets that spell out the equal blocks give the NULL-offsets results
    rng = np.random.default_rng(4)
    T, E, k, R, rpn, ns = 96, 16, 3, 8, 4, 2
    ids = W.random_small(5, T, E, k, n_layers=2, s=1.1)
    eq = np.arange(R + 1, dtype=np.int64) * (T // R)
    base = dict(T=T, E=E, k=k, R=R, ranks_per_node=rpn, n_slot=ns, tok_bytes=64,
                expert_bytes=4096, c_intra=1, c_inter=4, max_refine_iters=0, main_rank=None)
    h0 = oracle.hist(ids, R, E)
    assert np.array_equal(h0, oracle.hist(ids, R, E, rank_offsets=eq))
    p = oracle.plan(base, h0)
    d0 = oracle.reroute(base, ids, p)
    d1 = oracle.reroute({**base, "rank_offsets": eq}, ids, p)
    assert np.array_equal(d0, d1)
    for a, b in zip(oracle.layout(base, d0), oracle.layout({**base, "rank_offsets": eq}, d0)):
        assert np.array_equal(a, b)
    x0, x1 = oracle.dedup(base, d0), oracle.dedup({**base, "rank_offsets": eq}, d0)
    for key in x0:
        assert np.array_equal(x0[key], x1[key]), key
    _, tr = oracle.cooccur(ids, E)
    for a, b in zip(oracle.shuffle(ids, tr, R), oracle.shuffle(ids, tr, R, rank_offsets=eq)):
        assert np.array_equal(a, b)
    del rng


def test_hist_is_blockwise_bincount():
    rng = np.random.default_rng(7)
    for trial in range(6):
        T, E, k, R = 200 + trial, 12, 3, 4
        ids = W.random_small(20 + trial, T, E, k, n_layers=2)
        off = _random_offsets(rng, T, R)
        h = oracle.hist(ids, R, E, rank_offsets=off)
        for l in range(2):
            for s in range(R):
                blk = ids[l, off[s]:off[s + 1]].ravel()
                assert np.array_equal(h[l, s], np.bincount(blk, minlength=E))


def test_reroute_and_layout_follow_the_source_blocks():
    # every pair of source s (tokens off[s] .. off[s+1]) goes to an instance
    # of its expert, q[s] pairs to each instance; send counts are the blocks'
    # per-rank totals; locality counts classify by the pair's own source
    rng = np.random.default_rng(8)
    T, E, k, R, rpn, ns = 300, 16, 4, 8, 4, 3
    ids = W.random_small(31, T, E, k, n_layers=1, s=1.3)
    for trial in range(4):
        off = _random_offsets(rng, T, R)
        cfg = dict(T=T, E=E, k=k, R=R, ranks_per_node=rpn, n_slot=ns, tok_bytes=5, expert_bytes=64,
                   c_intra=1, c_inter=4, max_refine_iters=0, main_rank=None, rank_offsets=off)
        h = oracle.hist(ids, R, E, rank_offsets=off)
        p = oracle.plan(cfg, h)
        d = oracle.reroute(cfg, ids, p)[0]
        nl = E // R + ns
        q = p["route_cnt"][0]
        src = np.repeat(np.arange(R), np.diff(off))
        src_pair = np.repeat(src, k)
        got = np.zeros_like(q)
        for pair, inst in enumerate(d):
            got[src_pair[pair], inst // nl, inst % nl] += 1
        assert np.array_equal(got, q)
        sp, so, sc, st = oracle.layout(cfg, d[None])
        assert np.array_equal(sp[0], np.argsort(d, kind="stable"))
        want_sc = np.zeros((R, R), np.int64)
        np.add.at(want_sc, (src_pair, d // nl), 1)
        assert np.array_equal(sc[0], want_sc)
        r = d // nl
        assert st[0][0] == np.sum(src_pair == r)
        assert st[0][1] == np.sum((src_pair != r) & (src_pair // rpn == r // rpn))


def test_bad_offsets_are_rejected():
    ids = np.zeros((1, 8, 1), np.int32)
    for off in ([0, 3, 7], [1, 3, 8], [0, 5, 3, 8][:3], [0, 9, 8]):
        with pytest.raises(oracle.OracleError):
            oracle.hist(ids, 2, 4, rank_offsets=off)
    with pytest.raises(oracle.OracleError):
        oracle.hist(np.zeros((1, 9, 1), np.int32), 2, 4)          # 9 tokens, 2 equal blocks
