"""Correlated expert placement (topo_place_experts) on the GPU against the
oracle, bit for bit, and the plan chain run on the map it produces."""
import json
import os

import numpy as np
import pytest

import moe_expert_routing_ids_gb300 as topo
import oracle


def test_place_arguments_are_checked_on_the_host():
    try:
        topo.lib()
    except RuntimeError:
        pytest.skip("library not built")
    a = 1 << 20                                             # never dereferenced
    for (L, E, R, it) in ((1, 18, 4, 0), (1, 2048, 8, 0), (1, 16, 4, -1), (-1, 16, 4, 0), (1, 1024, 1024, 0)):
        with pytest.raises(topo.TopoError) as ex:
            topo.topo_place_experts(L, E, R, it, a, a, a)
        assert ex.value.code == topo.TOPO_EINVAL
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_place_experts(1, 16, 4, 0, None, a, a)
    assert ex.value.code == topo.TOPO_EINVAL


torch = pytest.importorskip("torch")
gpu = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch.device("cuda:0")


def run_place(co, R, dev, max_iters=0):
    L, E, _ = co.shape
    d_co = co if isinstance(co, torch.Tensor) else torch.as_tensor(co, device=dev)
    mr = torch.full((L, E), -7, dtype=torch.int32, device=dev)
    st = torch.full((L, topo.TOPO_PLACE_STATS), -7, dtype=torch.int64, device=dev)
    topo.topo_place_experts(L, E, R, max_iters, d_co, mr, st)
    torch.cuda.synchronize()
    return mr.cpu().numpy(), st.cpu().numpy()


@gpu
def test_place_hand_cases():
    dev = _dev()
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "place_hand.json")))
    for c in g["cases"]:
        mr, st = run_place(np.array([c["co"]], np.int64), c["R"], dev)
        assert mr[0].tolist() == c["main_rank"] and st[0].tolist() == c["stats"], c["notes"]


CASES = {
    # name: (L, E, R, max_iters, kind)
    "e16_r4_random_three_layers": (3, 16, 4, 0, "random"),
    "e12_r3_random": (1, 12, 3, 0, "random"),
    "e64_r8_random": (2, 64, 8, 0, "random"),
    "e64_r8_capped": (1, 64, 8, 3, "random"),
    "e128_r16_planted": (1, 128, 16, 0, "planted"),
    "e256_r64_random": (1, 256, 64, 0, "random"),
    "e32_r1": (1, 32, 1, 0, "random"),
    "e32_r32": (1, 32, 32, 0, "random"),
}


@gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_place_matches_the_oracle(name):
    dev = _dev()
    L, E, R, it, kind = CASES[name]
    rng = np.random.default_rng(len(name))
    co = rng.integers(0, 50, size=(L, E, E)).astype(np.int64)
    if kind == "planted":
        group = rng.permutation(E) // 8
        co += 400 * (group[:, None] == group[None, :])
    mr, st = run_place(co, R, dev, it)
    emr, est = oracle.place(co, R, it)
    assert np.array_equal(mr, emr)
    assert np.array_equal(st, est)


@gpu
@pytest.mark.parametrize("kind", ["wide", "negative"])
def test_place_weights_outside_the_packed_key_range(kind):
    # pair weights >= 2^36 or < 0 take the general (value, index) key path
    dev = _dev()
    rng = np.random.default_rng(5)
    E, R = 64, 8
    if kind == "wide":
        co = rng.integers(0, 50, size=(1, E, E)).astype(np.int64)
        co += (1 << 40) * (rng.random((1, E, E)) < 0.05)
    else:
        co = rng.integers(-30, 50, size=(1, E, E)).astype(np.int64)
    mr, st = run_place(co, R, dev)
    emr, est = oracle.place(co, R)
    assert np.array_equal(mr, emr)
    assert np.array_equal(st, est)


@gpu
def test_placement_from_gpu_cooccurrence_feeds_the_plan_chain():
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Cooccur, Planner
    dev = _dev()
    w = W.COOCCUR
    L, T, E, k = 1, 16384, w.E, w.k
    ids = w.ids()[:1, :T]
    C = Cooccur(L, T, E, k, dev, transitions=False)
    C.run(torch.as_tensor(np.ascontiguousarray(ids), device=dev))
    assert C.error() == 0
    R = 16
    mr, st = run_place(C.co, R, dev)
    co = C.co.cpu().numpy()
    emr, est = oracle.place(co, R)
    assert np.array_equal(mr, emr) and np.array_equal(st, est)
    assert st[0, 2] > 2 * st[0, 0]                    # the planted groups come together
    cfg = dict(T=T, E=E, k=k, R=R, ranks_per_node=8, n_slot=2, tok_bytes=14336, expert_bytes=66060288,
               c_intra=1, c_inter=4, max_refine_iters=0, main_rank=mr[0])
    P = Planner(cfg, 1, dev)
    P.run(torch.as_tensor(np.ascontiguousarray(ids), device=dev))
    assert P.error() == 0
    h = oracle.hist(ids, R, E)
    p = oracle.plan(cfg, h)
    d = oracle.reroute(cfg, ids, p)
    got = P.numpy()
    assert np.array_equal(got["slot_expert"], p["slot_expert"])
    assert np.array_equal(got["dst_inst"], d)


@gpu
def test_place_of_no_layers_is_a_no_op():
    _dev()
    topo.topo_place_experts(0, 16, 4, 0, None, None, None)


@gpu
def test_place_full_size_cooccurrence_workload():
    # all 8 layers of the co-occurrence workload at EP8, as bench.py times it
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Cooccur
    dev = _dev()
    w = W.COOCCUR
    C = Cooccur(w.n_layers, w.T, w.E, w.k, dev, transitions=False)
    C.run(torch.as_tensor(w.ids(), device=dev))
    assert C.error() == 0
    mr, st = run_place(C.co, 8, dev)
    emr, est = oracle.place(C.co.cpu().numpy(), 8)
    assert np.array_equal(mr, emr) and np.array_equal(st, est)
