"""Top-k gating fused with Omega (topo_gate_hist) on the GPU against the
oracle, bit for bit: ids, the selected raw logits and the histogram, then the
plan chain fed from it."""
import numpy as np
import pytest

import moe_expert_routing_ids_gb300 as topo
import oracle


def _cfg(T, E, k, R, rpn, ns):
    return dict(T=T, E=E, k=k, R=R, ranks_per_node=rpn, n_slot=ns, tok_bytes=2048,
                expert_bytes=1 << 20, c_intra=1, c_inter=4, max_refine_iters=0, main_rank=None)


def test_gate_arguments_are_checked_on_the_host():
    try:
        topo.lib()
    except RuntimeError:
        pytest.skip("library not built")
    c = topo.make_cfg(**_cfg(256, 64, 6, 4, 2, 1))
    need = topo.topo_workspace_bytes(c, 1, topo.TOPO_CALL_GATE)
    assert need == topo.topo_workspace_bytes(c, 1, topo.TOPO_CALL_CHAIN)
    a = 1 << 20                                             # never dereferenced
    for dt in (2, -1):
        with pytest.raises(topo.TopoError) as ex:
            topo.topo_gate_hist(c, 1, a, dt, None, a, None, a, a, need)
        assert ex.value.code == topo.TOPO_EINVAL
    with pytest.raises(topo.TopoError) as ex:                      # logits not float-aligned
        topo.topo_gate_hist(c, 1, a + 2, topo.TOPO_DTYPE_F32, None, a, None, a, a, need)
    assert ex.value.code == topo.TOPO_EINVAL
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_gate_hist(c, 1, a, topo.TOPO_DTYPE_F32, None, a, None, a, a, need - 1)
    assert ex.value.code == topo.TOPO_ENOSPC
    for big in (_cfg(256, 8, 9, 4, 2, 1), _cfg(2048, 2048, 2, 8, 8, 0)):   # k > E, E > 1024
        cb = topo.make_cfg(**big)
        nb = max(topo.topo_workspace_bytes(cb, 1, topo.TOPO_CALL_GATE), 1 << 12)
        with pytest.raises(topo.TopoError) as ex:
            topo.topo_gate_hist(cb, 1, a, topo.TOPO_DTYPE_F32, None, a, None, a, a, nb)
        assert ex.value.code == topo.TOPO_EINVAL


torch = pytest.importorskip("torch")
gpu = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch.device("cuda:0")


def run_gate(cfg, L, logits, bias, dev, with_scores=True):
    """logits: numpy float32 or uint16 (bf16 patterns) [L, T, E]."""
    from moe_expert_routing_ids_gb300.planner import Planner
    T, k = cfg["T"], cfg["k"]
    P = Planner(cfg, L, dev)
    if logits.dtype == np.uint16:
        x = torch.as_tensor(logits.view(np.int16), device=dev).view(torch.bfloat16)
    else:
        x = torch.as_tensor(logits, device=dev)
    ids = torch.full((L, T, k), -7, dtype=torch.int32, device=dev)
    sc = torch.full((L, T, k), -7.0, dtype=torch.float32, device=dev) if with_scores else None
    b = None if bias is None else torch.as_tensor(bias, device=dev)
    P.gate_hist(x, ids, b, sc)
    assert P.error() == 0
    return P, ids, sc


def _check(cfg, L, logits, bias, dev, with_scores=True):
    P, ids, sc = run_gate(cfg, L, logits, bias, dev, with_scores)
    want = oracle.gate(logits, cfg["k"], cfg["R"], bias=bias, rank_offsets=cfg.get("rank_offsets"))
    assert np.array_equal(ids.cpu().numpy(), want["ids"])
    if with_scores:
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), want["scores"].view(np.uint32))
    assert np.array_equal(P.buf.hist.cpu().numpy(), want["hist"])
    return P, ids


def _gumbel(rng, shape):
    return (-np.log(-np.log(rng.random(shape)))).astype(np.float32)


def _bf16(f):
    return (f.view(np.uint32) >> 16).astype(np.uint16)


CASES = {
    # name: (cfg, L, dtype, bias); tokens per source chosen so that the tiles end ragged
    "e512_k10_f32_bias": (_cfg(8 * 600, 512, 10, 8, 8, 4), 1, "f32", True),
    "e512_k10_bf16_bias": (_cfg(8 * 600, 512, 10, 8, 8, 4), 1, "bf16", True),
    "e64_k6_f32_two_layers": (_cfg(32 * 100, 64, 6, 32, 8, 8), 2, "f32", False),
    "e8_k2_scalar": (_cfg(8 * 50, 8, 2, 8, 4, 2), 1, "f32", True),
    "e160_k8_bf16_scalar_rows": (_cfg(4 * 333, 160, 8, 4, 2, 2), 1, "bf16", False),
    "e1000_k16_f32": (_cfg(2 * 300, 1000, 16, 2, 2, 1), 1, "f32", True),
    "e1000_k16_bf16": (_cfg(2 * 300, 1000, 16, 2, 2, 1), 1, "bf16", False),
    "e37_k3_odd": (_cfg(4 * 77, 37, 3, 1, 1, 1), 1, "f32", True),
    "e100_k5_bf16_unaligned_rows": (_cfg(4 * 100, 100, 5, 4, 2, 1), 1, "bf16", True),
    "e64_k40_exact_path": (_cfg(2 * 64, 64, 40, 2, 2, 1), 1, "f32", True),
    "e256_k32": (_cfg(8 * 40, 256, 32, 8, 8, 1), 1, "f32", False),
    # 16 lanes per token (128 < E <= 512, k <= 16) at its edges, and k = 17 just past them
    "e129_k16_f32_unaligned_rows": (_cfg(3 * 150, 129, 16, 3, 3, 1), 1, "f32", True),
    "e130_k16_bf16_scalar_rows": (_cfg(2 * 150, 130, 16, 2, 2, 1), 1, "bf16", True),
    "e384_k17_f32": (_cfg(4 * 150, 384, 17, 4, 2, 1), 1, "f32", True),
    "e448_k1_bf16_three_layers": (_cfg(2 * 131, 448, 1, 2, 2, 1), 3, "bf16", False),
}


@gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_gate_matches_the_oracle(name):
    dev = _dev()
    cfg, L, dt, with_bias = CASES[name]
    rng = np.random.default_rng(len(name))
    E = cfg["E"]
    x = _gumbel(rng, (L, cfg["T"], E))
    bias = np.log(rng.dirichlet(np.ones(E) * 0.5) + 1e-9).astype(np.float32) if with_bias else None
    if dt == "bf16":
        x = _bf16(x)
    _check(cfg, L, x, bias, dev)


@gpu
def test_gate_without_scores_output():
    dev = _dev()
    cfg = _cfg(8 * 64, 128, 8, 8, 8, 2)
    x = _gumbel(np.random.default_rng(0), (1, 512, 128))
    _check(cfg, 1, x, None, dev, with_scores=False)


@gpu
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("E", [96, 200, 512])      # 32 lanes per token; 16 lanes, ragged; 16, full
def test_gate_ties_signed_zeros_and_nans(dt, E):
    dev = _dev()
    rng = np.random.default_rng(7)
    cfg = _cfg(4 * 256, E, 6, 4, 2, 1)
    x = rng.integers(-2, 3, size=(1, 1024, E)).astype(np.float32)    # > 64 candidates: exact path
    x[rng.random(x.shape) < 0.1] = -0.0
    x[rng.random(x.shape) < 0.05] = np.nan
    x[0, 5, :] = np.nan                                             # all NaN
    x[0, 9, :E - 6] = np.nan                                        # exactly k numbers left
    x[0, 10, E - 7:] = np.nan                                       # k + 1, all in the last lanes
    x[0, 11, 3] = np.inf
    x[0, 12, :] = -np.inf
    x[0, 100:200] = _gumbel(rng, (100, E))                          # fast path rows
    x[0, 300] = 0.0                                                 # all equal
    if dt == "bf16":
        x = _bf16(x)
    _check(cfg, 1, x, None, dev)
    _check(cfg, 1, x, np.zeros(E, np.float32), dev)                # +0 bias: -0 + 0 = +0


@gpu
def test_gate_feeds_the_plan_chain():
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    cfg = _cfg(64 * 256, 256, 8, 64, 8, 8)
    L = 2
    rng = np.random.default_rng(3)
    x = _gumbel(rng, (L, cfg["T"], 256))
    p = 1.0 / np.arange(1, 257) ** 1.2
    bias = np.log(p / p.sum())[rng.permutation(256)].astype(np.float32)
    P = Planner(cfg, L, dev)
    ids = torch.empty((L, cfg["T"], 8), dtype=torch.int32, device=dev)
    P.run_from_logits(torch.as_tensor(x, device=dev), ids, torch.as_tensor(bias, device=dev))
    assert P.error() == 0
    g = oracle.gate(x, 8, 64, bias=bias)
    assert np.array_equal(ids.cpu().numpy(), g["ids"])
    h = g["hist"]
    pl = oracle.plan(cfg, h)
    d = oracle.reroute(cfg, g["ids"], pl)
    sp, so, sc, st = oracle.layout(cfg, d)
    got = P.numpy()
    for key, v in dict(hist=h, slot_expert=pl["slot_expert"], route_cnt=pl["route_cnt"], dst_inst=d,
                       sorted_pairs=sp, seg_off=so, send_counts=sc, layout_stats=st).items():
        assert np.array_equal(got[key], v), key


@gpu
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_gate_full_size_every_token(dtype):
    # one whole microbatch of the T = 1048576, E = 512, k = 10, R = 128
    # workload (Gumbel logits plus a log-Zipf(1.4) bias): every token's ids and
    # selected logits, and Omega, against the oracle
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    w = W.STRESS
    cfg = dict(w.plan_cfg)
    T, E, k = w.T, w.E, w.k
    x = W.gumbel_logits(23, 1, T, E)
    if dtype == "bf16":
        x = (x.view(np.uint32) >> 16).astype(np.uint16)          # bf16 patterns of the logits
        xd = torch.as_tensor(x.view(np.int16), device=dev).view(torch.bfloat16)
    else:
        xd = torch.as_tensor(x, device=dev)
    bias = W.zipf_bias(23, E, w.zipf_s)
    P = Planner(cfg, 1, dev)
    ids = torch.empty((1, T, k), dtype=torch.int32, device=dev)
    sc = torch.empty((1, T, k), dtype=torch.float32, device=dev)
    P.gate_hist(xd, ids, torch.as_tensor(bias, device=dev), sc)
    assert P.error() == 0
    del xd
    want = oracle.gate(x, k, w.R, bias=bias)
    assert np.array_equal(ids.cpu().numpy(), want["ids"])
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), want["scores"].view(np.uint32))
    assert np.array_equal(P.buf.hist.cpu().numpy(), want["hist"])


@gpu
def test_gate_of_an_empty_batch_and_no_layers():
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    cfg = _cfg(0, 16, 2, 4, 2, 1)
    P = Planner(cfg, 2, dev)
    x = torch.zeros((2, 0, 16), dtype=torch.float32, device=dev)
    ids = torch.zeros((2, 0, 2), dtype=torch.int32, device=dev)
    P.gate_hist(x, ids)
    assert P.error() == 0
    assert not P.buf.hist.cpu().numpy().any()
    c = topo.make_cfg(**cfg)
    topo.topo_gate_hist(c, 0, None, topo.TOPO_DTYPE_F32, None, None, None, P.buf.hist, P.ws, P.ws_bytes)


@gpu
def test_gate_with_unequal_source_blocks():
    # Omega and the tile index over unequal blocks (one empty), then the
    # whole chain from the gated ids against the oracle
    from moe_expert_routing_ids_gb300.planner import Planner
    dev = _dev()
    T, E, k, R = 3000, 256, 8, 8
    off = np.array([0, 100, 100, 1700, 1701, 2200, 2900, 2999, 3000], np.int64)
    cfg = dict(_cfg(T, E, k, R, 4, 8), rank_offsets=off)
    rng = np.random.default_rng(12)
    x = _gumbel(rng, (2, T, E))
    bias = rng.standard_normal(E).astype(np.float32)
    P, ids = _check(cfg, 2, x, bias, dev)
    P.make_plan()
    P.reroute_layout(ids)
    assert P.error() == 0
    g = oracle.gate(x, k, R, bias=bias, rank_offsets=off)
    pl = oracle.plan(cfg, g["hist"])
    d = oracle.reroute(cfg, g["ids"], pl)
    sp, so, sc, st = oracle.layout(cfg, d)
    got = P.numpy()
    for key, v in dict(dst_inst=d, sorted_pairs=sp, seg_off=so, send_counts=sc, layout_stats=st).items():
        assert np.array_equal(got[key], v), key
