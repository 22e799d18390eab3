"""GPU parity: every output of the CUDA path equals the CPU oracle bit for bit.

All calls go through the C ABI (ctypes binding).  Integer work, so the bar is
exact equality.  Covers the five named workloads at full size and edge cases:
empty input, ragged and unaligned tiles, several tiles per source, one expert
per rank, no replica slots, one domain, all ids equal, free and prohibitive
replicas, a main-rank map, an iteration cap, the widest domain, k = 1.
"""
import numpy as np
import pytest

import oracle
from moe_expert_routing_ids_gb300 import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")


def gpu_chain(cfg, ids, fused=True):
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    L = ids.shape[0]
    mr = cfg.get("main_rank")
    ro = cfg.get("rank_offsets")
    gcfg = dict(cfg, main_rank=None if mr is None else torch.as_tensor(mr, dtype=torch.int32, device=dev),
                rank_offsets=None if ro is None else torch.as_tensor(ro, dtype=torch.int64, device=dev))
    P = Planner(gcfg, L, dev)
    d_ids = torch.as_tensor(ids, device=dev).contiguous()
    P.run(d_ids, fused=fused)
    err = P.error()
    out = P.numpy()
    return out, err


def oracle_chain(cfg, ids):
    L = ids.shape[0]
    h = oracle.hist(ids, cfg["R"], cfg["E"], rank_offsets=cfg.get("rank_offsets"))
    p = oracle.plan(cfg, h)
    d = oracle.reroute(cfg, ids, p)
    sp, so, sc, st = oracle.layout(cfg, d)
    return dict(hist=h, slot_expert=p["slot_expert"], route_cnt=p["route_cnt"],
                inst_load=p["inst_load"], rank_load=p["rank_load"], stats=p["stats"],
                dst_inst=d, sorted_pairs=sp, seg_off=so, send_counts=sc, layout_stats=st)


def assert_same(gpu, orc, keys=None):
    for key in keys or orc:
        a, b = np.asarray(gpu[key]), np.asarray(orc[key])
        assert a.shape == b.shape, (key, a.shape, b.shape)
        if not np.array_equal(a, b):
            idx = np.argwhere(a != b)
            first = tuple(idx[0])
            raise AssertionError(f"{key}: {len(idx)} mismatches, first at {first}: gpu {a[first]} "
                                 f"oracle {b[first]}")


def check(cfg, ids, both=True):
    """Both the fused reroute+layout call and the separate calls."""
    want = oracle_chain(cfg, ids)
    for fused in ((True, False) if both else (True,)):
        gpu, err = gpu_chain(cfg, ids, fused)
        assert err == 0, f"device error {err} (fused={fused})"
        assert_same(gpu, want)


@pytest.mark.parametrize("w", W.PLAN_WORKLOADS, ids=lambda w: w.name)
def test_named_workloads_full_size(w):
    check(w.plan_cfg, w.ids())


def _cfg(T, E, k, R, rpn, ns, S=2048, Wb=4_718_592, **kw):
    return dict(T=T, E=E, k=k, R=R, ranks_per_node=rpn, n_slot=ns, tok_bytes=S, expert_bytes=Wb,
                c_intra=1, c_inter=4, max_refine_iters=0, main_rank=None, **kw)


EDGE = {
    # name: (cfg, ids-maker)
    "unaligned_tiles": (_cfg(8 * 1001, 16, 3, 8, 4, 2, S=64, Wb=10_000),
                        lambda c: W.random_small(1, c["T"], c["E"], c["k"], 2, s=1.3)),
    "multi_tile_ragged": (_cfg(2 * 10001, 8, 4, 2, 2, 3, S=64, Wb=1000),
                          lambda c: W.random_small(2, c["T"], c["E"], c["k"], 1, s=1.5)),
    "many_tiles_per_source": (_cfg(8 * 20000, 32, 5, 8, 2, 4, S=128, Wb=50_000),
                              lambda c: W.random_small(3, c["T"], c["E"], c["k"], 2, s=1.2)),
    "empty": (_cfg(0, 8, 2, 4, 2, 1), lambda c: np.zeros((1, 0, 2), np.int32)),
    "one_expert_per_rank_k1": (_cfg(4000, 8, 1, 8, 4, 2, S=256, Wb=1000),
                               lambda c: W.random_small(4, c["T"], c["E"], c["k"], 1, s=1.1)),
    "no_slots": (_cfg(4000, 16, 3, 8, 4, 0, S=256, Wb=1000),
                 lambda c: W.random_small(5, c["T"], c["E"], c["k"], 1, s=1.3)),
    "single_domain": (_cfg(6000, 32, 4, 8, 8, 3, S=256, Wb=0),
                      lambda c: W.random_small(6, c["T"], c["E"], c["k"], 1, s=1.6)),
    "all_ids_equal": (_cfg(4096, 8, 1, 8, 2, 2, S=64, Wb=100),
                      lambda c: np.full((1, c["T"], 1), 5, np.int32)),
    "free_replicas": (_cfg(8000, 32, 4, 8, 2, 4, S=256, Wb=0),
                      lambda c: W.random_small(7, c["T"], c["E"], c["k"], 1, s=1.0)),
    "prohibitive_replicas": (_cfg(8000, 32, 4, 8, 2, 4, S=1, Wb=1 << 36),
                             lambda c: W.random_small(8, c["T"], c["E"], c["k"], 1, s=1.4)),
    "iteration_cap": (_cfg(8000, 32, 4, 16, 4, 4, S=256, Wb=10_000, ),
                      lambda c: W.random_small(9, c["T"], c["E"], c["k"], 1, s=1.4)),
    "widest_domain": (_cfg(64 * 300, 128, 6, 64, 32, 6, S=512, Wb=200_000),
                      lambda c: W.random_small(10, c["T"], c["E"], c["k"], 1, s=1.2)),
    "tiny": (_cfg(2, 2, 1, 2, 1, 1, S=1, Wb=1), lambda c: np.array([[[1], [1]]], np.int32)),
    "three_layers": (_cfg(16 * 700, 64, 6, 16, 8, 8, S=8192, Wb=34_603_008),
                     lambda c: W.random_small(11, c["T"], c["E"], c["k"], 3, s=1.2)),
    "k_above_fast_path": (_cfg(8 * 600, 64, 20, 8, 4, 4, S=256, Wb=20_000),
                          lambda c: W.random_small(13, c["T"], c["E"], c["k"], 1, s=1.1)),
    "k16_two_rounds": (_cfg(4 * 1100, 64, 16, 4, 2, 4, S=256, Wb=20_000),
                       lambda c: W.random_small(14, c["T"], c["E"], c["k"], 1, s=1.1)),
    "k3_odd": (_cfg(8 * 777, 24, 3, 8, 4, 3, S=256, Wb=5_000),
               lambda c: W.random_small(15, c["T"], c["E"], c["k"], 1, s=1.3)),
    # R = 256 with many slots: the refinement keeps only the domain's own
    # sources' rows of q in shared memory, fetching the busiest rank's rows
    "rows_in_global_memory": (_cfg(256 * 150, 512, 8, 256, 8, 48, S=1024, Wb=60_000),
                              lambda c: W.random_small(17, c["T"], c["E"], c["k"], 1, s=1.3)),
    # free replicas and 96 slots: about 47 used per rank, so several warps
    # evaluate and the rest fetch
    "rows_in_global_memory_many_slots": (_cfg(256 * 150, 512, 8, 256, 8, 96, S=1024, Wb=0),
                                         lambda c: W.random_small(18, c["T"], c["E"], c["k"], 1, s=1.6)),
    "repeated_ids_in_a_token": (_cfg(8 * 700, 16, 4, 8, 4, 2, S=256, Wb=5_000),
                                lambda c: _with_repeats(W.random_small(16, c["T"], c["E"], c["k"], 1, s=1.2))),
}


def _offsets(T, lens):
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    assert off[-1] == T
    return off


def _ragged(T, R, seed):
    """Unequal source blocks: random cut points (some sources may be empty)."""
    rng = np.random.default_rng(seed)
    return np.concatenate([[0], np.sort(rng.integers(0, T + 1, R - 1)), [T]]).astype(np.int64)


# Unequal source blocks (TopoEP §2.1: each rank routes its own local tokens).
OFFSETS = {
    # ragged cut points over several tiles per source, two layers
    "ragged_blocks": (_cfg(8 * 3001, 16, 3, 8, 4, 2, S=64, Wb=10_000),
                      lambda c: W.random_small(41, c["T"], c["E"], c["k"], 2, s=1.3),
                      lambda c: _ragged(c["T"], c["R"], 1)),
    # an empty source in the middle and one at the end
    "empty_sources": (_cfg(7000, 32, 4, 8, 2, 4, S=256, Wb=5_000),
                      lambda c: W.random_small(42, c["T"], c["E"], c["k"], 1, s=1.2),
                      lambda c: _offsets(c["T"], [900, 1100, 0, 1500, 1200, 1300, 1000, 0])),
    # one source holding most tokens (many tiles), the others a few each
    "one_heavy_source": (_cfg(40_000, 64, 6, 16, 8, 6, S=512, Wb=40_000),
                         lambda c: W.random_small(43, c["T"], c["E"], c["k"], 1, s=1.4),
                         lambda c: _offsets(c["T"], [3] * 7 + [40_000 - 3 * 15] + [3] * 8)),
    # k = 10 over E = 512, R = 128 (the stress kernel path), ragged blocks
    "ragged_k10_r128": (_cfg(128 * 1200 + 77, 512, 10, 128, 8, 16, S=14336, Wb=66_060_288),
                        lambda c: W.random_small(44, c["T"], c["E"], c["k"], 2, s=1.4),
                        lambda c: _ragged(c["T"], c["R"], 2)),
    # R = 256 with 48 slots (the refinement's q as 16-bit counts in shared
    # memory), ragged blocks with empty sources
    "ragged_q16": (_cfg(256 * 150, 512, 8, 256, 8, 48, S=1024, Wb=60_000),
                   lambda c: W.random_small(46, c["T"], c["E"], c["k"], 1, s=1.3),
                   lambda c: _ragged(c["T"], c["R"], 4)),
    # R = 256 with 96 slots and free replicas (q in global memory, rows fetched)
    "ragged_fetch": (_cfg(256 * 150, 512, 8, 256, 8, 96, S=1024, Wb=0),
                     lambda c: W.random_small(47, c["T"], c["E"], c["k"], 1, s=1.6),
                     lambda c: _ragged(c["T"], c["R"], 5)),
    # repeated ids inside a token with unequal blocks (the exact path)
    "ragged_repeats": (_cfg(8 * 700 + 5, 16, 4, 8, 4, 2, S=256, Wb=5_000),
                       lambda c: _with_repeats(W.random_small(45, c["T"], c["E"], c["k"], 1, s=1.2)),
                       lambda c: _ragged(c["T"], c["R"], 3)),
    "no_tokens": (_cfg(0, 8, 2, 4, 2, 1), lambda c: np.zeros((1, 0, 2), np.int32),
                  lambda c: np.zeros(5, np.int64)),
}


@pytest.mark.parametrize("name", sorted(OFFSETS))
def test_unequal_source_blocks(name):
    cfg, mk, mo = OFFSETS[name]
    cfg = dict(cfg, rank_offsets=mo(cfg))
    check(cfg, mk(cfg))


def test_bad_offsets_set_the_error_word():
    cfg = _cfg(800, 16, 2, 4, 2, 1, S=64, Wb=1000)
    ids = W.random_small(46, 800, 16, 2, 1)
    for bad in ([0, 300, 200, 500, 800], [0, 200, 400, 600, 799], [5, 200, 400, 600, 800]):
        gpu, err = gpu_chain(dict(cfg, rank_offsets=np.array(bad, np.int64)), ids)
        assert err == -7, (bad, err)


def _with_repeats(ids):
    """Plant a repeated expert inside some tokens (not Top-k, but the
    definitions use count vectors and the kernels must stay exact)."""
    ids = ids.copy()
    ids[0, 5, 1] = ids[0, 5, 0]
    ids[0, 1300, 3] = ids[0, 1300, 2]
    ids[0, -1, 2] = ids[0, -1, 0]
    return ids


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(name):
    cfg, mk = EDGE[name]
    cfg = dict(cfg)
    if name == "iteration_cap":
        cfg["max_refine_iters"] = 1
    check(cfg, mk(cfg))


def test_refinement_beyond_16_bit_counts():
    """Every token picks 8 of domain 0's 32 main experts and replicas cost too
    much to place elsewhere, so each source sends 72000 pairs into domain 0:
    that domain's refinement cannot keep q as 16-bit counts and keeps it in
    global memory, the other domains do; the plan is the oracle's either way."""
    R, rpn, E, k, ns = 64, 8, 256, 8, 100
    T = R * 9000
    cfg = _cfg(T, E, k, R, rpn, ns, S=1024, Wb=2_000_000_000)
    rng = W.rng_for(23, 0)
    ids = np.argsort(rng.random((T, 32)), axis=1)[:, :8].astype(np.int32)[None]
    want = oracle_chain(cfg, ids)
    share = want["route_cnt"][0][:, :rpn, :].sum(axis=(1, 2))   # kept by every move
    assert share.max() > 65535 and want["stats"][0, 4] > 0
    gpu, err = gpu_chain(cfg, ids)
    assert err == 0
    assert_same(gpu, want)


def test_main_rank_map():
    cfg = _cfg(8 * 900, 32, 4, 8, 4, 3, S=256, Wb=20_000)
    cfg["main_rank"] = (W.rng_for(21, 0).permutation(32) % 8).astype(np.int32)
    check(cfg, W.random_small(12, cfg["T"], cfg["E"], cfg["k"], 2, s=1.3))


def test_repeat_runs_are_byte_identical():
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    w = W.PLAN_LATENCY
    ids = torch.as_tensor(w.ids(), device=dev)
    P = Planner(w.plan_cfg, w.n_layers, dev)
    P.run(ids)
    ref = P.numpy()
    for _ in range(9):
        P.run(ids)
        again = P.numpy()
        for key in ref:
            assert np.array_equal(ref[key], again[key]), key
    assert P.error() == 0


# ---------------------------------------------------------------- co-occurrence

def gpu_cooccur(ids, E, transitions=True, tensor_cores=True):
    """tensor_cores: the workspace of the tcgen05 path (used for E <= 128,
    k <= 16); False: the shared-atomic kernels."""
    from moe_expert_routing_ids_gb300.planner import Cooccur
    dev = _dev()
    L, T, k = ids.shape
    C = Cooccur(L, T, E, k, dev, transitions, tensor_cores=tensor_cores)
    C.run(torch.as_tensor(ids, device=dev).contiguous())
    err = C.error()
    co = C.co.cpu().numpy()
    tr = C.tr.cpu().numpy() if C.tr is not None else None
    return co, tr, err


PATHS = pytest.mark.parametrize("tc", [True, False], ids=["tensor_cores", "atomics"])


@PATHS
def test_cooccur_full_size(tc):
    w = W.COOCCUR
    ids = w.ids()
    co, tr, err = gpu_cooccur(ids, w.E, tensor_cores=tc)
    assert err == 0
    oco, otr = oracle.cooccur(ids, w.E)
    assert np.array_equal(co, oco)
    assert np.array_equal(tr, otr)


@PATHS
@pytest.mark.parametrize("L,T,E,k", [(3, 5000, 16, 4), (1, 3000, 32, 8), (2, 1, 8, 2),
                                     (2, 777, 40, 20), (2, 900, 300, 6), (4, 2048, 128, 16),
                                     (3, 70_000, 128, 10), (2, 4096, 127, 3), (5, 257, 64, 1)])
def test_cooccur_shapes(L, T, E, k, tc):
    ids = W.random_small(T + E + k, T, E, k, L, s=1.1)
    co, tr, err = gpu_cooccur(ids, E, tensor_cores=tc)
    assert err == 0
    oco, otr = oracle.cooccur(ids, E)
    assert np.array_equal(co, oco)
    if L > 1:
        assert np.array_equal(tr, otr)


@PATHS
def test_cooccur_repeated_ids(tc):
    ids = np.array([[[1, 1, 2], [0, 0, 0]], [[0, 2, 2], [1, 2, 1]]], np.int32)
    co, tr, err = gpu_cooccur(ids, 3, tensor_cores=tc)
    oco, otr = oracle.cooccur(ids, 3)
    assert err == 0 and np.array_equal(co, oco) and np.array_equal(tr, otr)


def test_cooccur_tensor_core_sums_are_exact():
    # counts up to 16 per token (k = 16 over E = 8), products up to 256, and
    # each unit's float32 accumulator summing ~1800 tokens: cells far above
    # 2^14 with arbitrary low bits must come out exact
    rng = np.random.default_rng(5)
    ids = rng.integers(0, 8, size=(2, 131072, 16)).astype(np.int32)
    ids[:, ::3, :] = rng.integers(0, 2, size=(2, ids[:, ::3, :].shape[1], 16))
    co, tr, err = gpu_cooccur(ids, 8, tensor_cores=True)
    oco, otr = oracle.cooccur(ids, 8)
    assert err == 0 and oco.max() > (1 << 20)
    assert np.array_equal(co, oco) and np.array_equal(tr, otr)


@pytest.mark.parametrize("L,T,E,k", [(2, 3001, 159, 10), (2, 1500, 160, 8), (3, 2000, 64, 6),
                                     (2, 500, 100, 2)])
def test_cooccur_shapes_around_the_shared_memory_limit(L, T, E, k):
    # E <= 159 keeps both (E+1)^2 matrices of a CTA in shared memory; 160 does not
    ids = W.random_small(T + 3 * E + k, T, E, k, L, s=1.2)
    co, tr, err = gpu_cooccur(ids, E)
    assert err == 0
    oco, otr = oracle.cooccur(ids, E)
    assert np.array_equal(co, oco) and np.array_equal(tr, otr)


@PATHS
def test_cooccur_repeated_ids_exact_k(tc):
    rng = np.random.default_rng(3)
    ids = rng.integers(0, 5, size=(3, 700, 4)).astype(np.int32)   # many repeats per token
    co, tr, err = gpu_cooccur(ids, 5, tensor_cores=tc)
    oco, otr = oracle.cooccur(ids, 5)
    assert err == 0 and np.array_equal(co, oco) and np.array_equal(tr, otr)


@PATHS
@pytest.mark.parametrize("k", [8, 3])
def test_cooccur_out_of_range_id_is_dropped_and_flagged(k, tc):
    from moe_expert_routing_ids_gb300 import TOPO_ERANGE
    E = 32
    ids = W.random_small(9, 600, E, k, 2)
    ids[0, 17, 1] = E + 5
    ids[1, 40, k - 1] = -1
    co, tr, err = gpu_cooccur(ids, E, tensor_cores=tc)
    assert err == TOPO_ERANGE
    # the same counts as with the bad ids moved to a spare expert E and dropped
    spare = ids.copy()
    spare[(spare < 0) | (spare >= E)] = E
    oco, otr = oracle.cooccur(spare, E + 1)
    assert np.array_equal(co, oco[:, :E, :E]) and np.array_equal(tr, otr[:, :E, :E])


@PATHS
def test_cooccur_without_transitions(tc):
    ids = W.random_small(5, 1000, 16, 4, 3)
    co, tr, err = gpu_cooccur(ids, 16, transitions=False, tensor_cores=tc)
    assert err == 0 and tr is None
    assert np.array_equal(co, oracle.cooccur(ids, 16, transitions=False))


# ---------------------------------------------------------------- device errors

def test_out_of_range_id_sets_error_word():
    from moe_expert_routing_ids_gb300 import TOPO_ERANGE
    cfg = _cfg(400, 8, 2, 4, 2, 1, S=8, Wb=10)
    ids = W.random_small(1, 400, 8, 2, 1)
    ids[0, 17, 1] = 8
    _, err = gpu_chain(cfg, ids)
    assert err == TOPO_ERANGE


def test_reroute_without_hist_index_is_rejected():
    from moe_expert_routing_ids_gb300 import TOPO_ESTATE
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    cfg = _cfg(400, 8, 2, 4, 2, 1, S=8, Wb=10)
    ids = torch.as_tensor(W.random_small(2, 400, 8, 2, 1), device=dev)
    other = ids.clone()
    P = Planner(cfg, 1, dev)
    P.hist(ids)
    P.make_plan()
    P.reroute(other)             # index was built for `ids`, not `other`
    assert P.error() == TOPO_ESTATE
    P.reset_error()              # clears the error word and the indices' fingerprints
    P.reroute(ids)
    assert P.error() == TOPO_ESTATE
    P.reset_error()
    P.run(ids)                   # the chain restarts from topo_hist
    assert P.error() == 0


def test_expert_twice_on_a_rank_sets_estate():
    """A plan whose slots hold an expert the rank already hosts, or an id
    outside [0, E), is a bad state: the reroute's instance index says so."""
    from moe_expert_routing_ids_gb300 import TOPO_ESTATE
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    cfg = _cfg(400, 8, 2, 4, 2, 1, S=8, Wb=10)       # E_R = 2: rank 0 hosts experts 0 and 1
    ids = torch.as_tensor(W.random_small(4, 400, 8, 2, 1), device=dev)
    P = Planner(cfg, 1, dev)
    P.run(ids)
    assert P.error() == 0
    P.buf.slot_expert[0, 0, 0] = 0                   # rank 0's own main in its slot
    P.reroute_layout(ids)
    assert P.error() == TOPO_ESTATE
    P.reset_error()
    P.run(ids)
    assert P.error() == 0
    P.buf.slot_expert[0, 1, 0] = 99                  # not an expert
    P.reroute_layout(ids)
    assert P.error() == TOPO_ESTATE
    P.reset_error()
    P.run(ids)
    assert P.error() == 0


def test_layout_with_foreign_dst_is_rejected():
    from moe_expert_routing_ids_gb300 import TOPO_ESTATE
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    cfg = _cfg(400, 8, 2, 4, 2, 1, S=8, Wb=10)
    ids = torch.as_tensor(W.random_small(3, 400, 8, 2, 1), device=dev)
    P = Planner(cfg, 1, dev)
    P.run(ids, fused=False)
    assert P.error() == 0
    P.buf.dst_inst = P.buf.dst_inst.clone()   # not the buffer topo_reroute wrote
    P.layout()
    assert P.error() == TOPO_ESTATE


def test_unbalanced_main_rank_sets_error_word():
    from moe_expert_routing_ids_gb300 import TOPO_EMAP
    cfg = _cfg(400, 8, 2, 4, 2, 1, S=8, Wb=10)
    cfg["main_rank"] = np.array([0, 0, 0, 1, 2, 2, 3, 3], np.int32)
    _, err = gpu_chain(cfg, W.random_small(4, 400, 8, 2, 1))
    assert err == TOPO_EMAP
