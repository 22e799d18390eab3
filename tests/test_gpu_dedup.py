"""Deduplicated dispatch layout (topo_dedup_layout) on the GPU against the
oracle, bit for bit: on layouts the library's own planner produced, and on
synthetic destination instances with many slots of one token on one rank."""
import numpy as np
import pytest

import moe_expert_routing_ids_gb300 as topo
import oracle
from moe_expert_routing_ids_gb300 import workloads as W


def _cfg(T, E, k, R, rpn, ns):
    return dict(T=T, E=E, k=k, R=R, ranks_per_node=rpn, n_slot=ns, tok_bytes=2048,
                expert_bytes=1 << 20, c_intra=1, c_inter=4, max_refine_iters=0, main_rank=None)


def test_dedup_arguments_are_checked_on_the_host():
    try:
        topo.lib()
    except RuntimeError:
        pytest.skip("library not built")
    c = topo.make_cfg(**_cfg(256, 8, 2, 4, 2, 1))
    need = topo.topo_workspace_bytes(c, 1, topo.TOPO_CALL_DEDUP)
    assert need >= 256 + 4 * 4 * 4
    a = 1 << 20                                             # never dereferenced
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_dedup_layout(c, 1, a, a, a, a, a, a, a, a, need - 1)
    assert ex.value.code == topo.TOPO_ENOSPC
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_dedup_layout(c, 1, a, a, None, a, a, a, a, a, need)
    assert ex.value.code == topo.TOPO_EINVAL
    for big in (_cfg(256, 64, 17, 4, 2, 1), _cfg(2048, 2048, 2, 2048, 32, 0)):
        cb = topo.make_cfg(**big)
        nb = max(topo.topo_workspace_bytes(cb, 1, topo.TOPO_CALL_DEDUP), 1 << 12)
        with pytest.raises(topo.TopoError) as ex:
            topo.topo_dedup_layout(cb, 1, a, a, a, a, a, a, a, a, nb)
        assert ex.value.code == topo.TOPO_EINVAL


torch = pytest.importorskip("torch")
gpu = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch.device("cuda:0")


def run_dedup(cfg, L, dst, dev):
    """dst: device int32 [L, T*k] -> dict of numpy arrays, plus the error word."""
    c = topo.make_cfg(**cfg)
    T, k, R = cfg["T"], cfg["k"], cfg["R"]
    RW = (R + 63) // 64
    nb = topo.topo_workspace_bytes(c, L, topo.TOPO_CALL_DEDUP)
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    o = dict(seg=torch.full((L, R + 1), -7, dtype=torch.int32, device=dev),
             row_token=torch.full((L, T * k), -7, dtype=torch.int32, device=dev),
             row_slots=torch.zeros((L, T * k), dtype=torch.int64, device=dev),
             tok_dst=torch.full((L, T, RW), -1, dtype=torch.int64, device=dev),
             send=torch.full((L, R, R), -7, dtype=torch.int64, device=dev),
             stats=torch.full((L, topo.TOPO_DEDUP_STATS), -7, dtype=torch.int64, device=dev))
    topo.topo_dedup_layout(c, L, dst, o["seg"], o["row_token"], o["row_slots"], o["tok_dst"],
                           o["send"], o["stats"], ws, nb)
    torch.cuda.synchronize()
    got = {key: v.cpu().numpy() for key, v in o.items()}
    got["row_slots"] = got["row_slots"].view(np.uint64)
    got["tok_dst"] = got["tok_dst"].view(np.uint64)
    return got, topo.topo_read_error(ws)


def assert_same(got, want):
    for key in ("seg", "send", "stats", "tok_dst"):
        assert np.array_equal(got[key], want[key]), key
    for l in range(want["seg"].shape[0]):
        n = int(want["seg"][l, -1])                          # rows past seg[R] are unused
        assert np.array_equal(got["row_token"][l, :n], want["row_token"][l, :n]), l
        assert np.array_equal(got["row_slots"][l, :n], want["row_slots"][l, :n]), l


PLANNED = {
    # name: (cfg, L); tokens per source chosen so that tiles of 256 end ragged
    "k8_r16_ragged": (_cfg(16 * 600, 64, 8, 16, 8, 4), 1),
    "k10_r32_two_layers": (_cfg(32 * 300, 64, 10, 32, 8, 4), 2),
    "k1_r8": (_cfg(8 * 64, 8, 1, 8, 4, 1), 1),
    "k16_r128": (_cfg(128 * 40, 256, 16, 128, 8, 2), 1),
    "k3_r4_generic": (_cfg(4 * 1000, 24, 3, 4, 2, 2), 1),
}


@gpu
@pytest.mark.parametrize("name", sorted(PLANNED))
def test_dedup_on_planned_layouts_matches_the_oracle(name):
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    cfg, L = PLANNED[name]
    ids = W.random_small(11, cfg["T"], cfg["E"], cfg["k"], L, s=1.2)
    P = Planner(cfg, L, dev)
    P.run(torch.as_tensor(ids, device=dev))
    assert P.error() == 0
    got, err = run_dedup(cfg, L, P.buf.dst_inst, dev)
    assert err == 0
    assert_same(got, oracle.dedup(cfg, P.buf.dst_inst.cpu().numpy()))


def _clustered_dst(seed, cfg, L):
    """Destination instances that put several slots of a token on one rank:
    each token draws a few ranks, then each slot picks one of them and a
    local instance there."""
    T, E, k, R, ns = cfg["T"], cfg["E"], cfg["k"], cfg["R"], cfg["n_slot"]
    nl = E // R + ns
    rng = np.random.default_rng(seed)
    home = rng.integers(0, R, size=(L, T, 3))
    pick = rng.integers(0, 3, size=(L, T, k))
    rank = np.take_along_axis(home, pick, axis=2)
    return (rank * nl + rng.integers(0, nl, size=(L, T, k))).astype(np.int32).reshape(L, T * k)


DIRECT = {
    "k16_r1024": (_cfg(1024 * 3, 1024, 16, 1024, 32, 1), 1),
    "k10_r128_three_layers": (_cfg(128 * 257, 512, 10, 128, 8, 4), 3),
    "k2_r64": (_cfg(64 * 513, 64, 2, 64, 8, 1), 1),
    "k5_r1": (_cfg(1000, 4, 5, 1, 1, 1), 1),
    "k4_r192_three_words": (_cfg(192 * 20, 192, 4, 192, 8, 1), 1),
    # the fill kernel keeps a row's rank in the row's 32-bit word while
    # R <= 2^(24 - k): at the limit (rank in the top 8 or 9 bits) and past it
    "k16_r256_rank_at_the_word_limit": (_cfg(256 * 12, 256, 16, 256, 8, 1), 1),
    "k15_r512_rank_at_the_word_limit": (_cfg(512 * 6, 512, 15, 512, 8, 1), 1),
    "k15_r1024_rank_apart": (_cfg(1024 * 3, 1024, 15, 1024, 32, 1), 1),
}


@gpu
@pytest.mark.parametrize("name", sorted(DIRECT))
def test_dedup_on_clustered_destinations_matches_the_oracle(name):
    dev = _dev()
    cfg, L = DIRECT[name]
    d = _clustered_dst(len(name), cfg, L)
    got, err = run_dedup(cfg, L, torch.as_tensor(d, device=dev), dev)
    assert err == 0
    want = oracle.dedup(cfg, d)
    assert want["stats"][:, 0].sum() < want["stats"][:, 1].sum() or cfg["k"] == 1
    assert_same(got, want)


@gpu
def test_dedup_of_an_empty_batch():
    dev = _dev()
    cfg = _cfg(0, 8, 2, 4, 2, 1)
    got, err = run_dedup(cfg, 2, torch.zeros((2, 0), dtype=torch.int32, device=dev), dev)
    assert err == 0
    assert not got["seg"].any() and not got["send"].any() and not got["stats"].any()


@gpu
def test_dedup_flags_an_instance_out_of_range():
    dev = _dev()
    cfg = _cfg(256, 8, 2, 4, 2, 1)                          # 4 ranks x 3 instances
    d = _clustered_dst(3, cfg, 1)
    d[0, 17] = 12
    got, err = run_dedup(cfg, 1, torch.as_tensor(d, device=dev), dev)
    assert err == topo.TOPO_ESTATE


@gpu
def test_dedup_full_size_stress_workload():
    # the T = 1048576, E = 512, k = 10, R = 128 workload, all 4 microbatches, as
    # bench.py times it: every output against the oracle
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    w = W.STRESS
    P = Planner(w.plan_cfg, w.n_layers, dev)
    P.run(torch.as_tensor(w.ids(), device=dev))
    assert P.error() == 0
    got, err = run_dedup(w.plan_cfg, w.n_layers, P.buf.dst_inst, dev)
    assert err == 0
    assert_same(got, oracle.dedup(w.plan_cfg, P.buf.dst_inst.cpu().numpy()))


@gpu
@pytest.mark.parametrize("lens", [[700, 0, 1300, 257, 0, 900, 1840, 3], [5000] + [0] * 7,
                                  [1, 2, 3, 4, 5, 6, 7, 4972]], ids=["ragged", "one_source", "tiny_heads"])
def test_dedup_with_unequal_source_blocks(lens):
    # destinations from the oracle chain over unequal blocks (TopoEP §2.1);
    # rows, send counts and remote counts are per source block
    dev = _dev()
    T, E, k, R = 5000, 64, 6, 8
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    cfg = dict(_cfg(T, E, k, R, 4, 3), rank_offsets=off)
    ids = W.random_small(61, T, E, k, 2, s=1.3)
    h = oracle.hist(ids, R, E, rank_offsets=off)
    d = oracle.reroute(cfg, ids, oracle.plan(cfg, h))
    want = oracle.dedup(cfg, d)
    gcfg = dict(cfg, rank_offsets=torch.as_tensor(off, device=dev))
    got, err = run_dedup(gcfg, 2, torch.as_tensor(d, device=dev), dev)
    assert err == 0
    assert_same(got, want)
