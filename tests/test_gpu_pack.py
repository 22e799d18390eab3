"""Dispatch pack (topo_permute) and combine (topo_combine) on the GPU against
the oracle, bit for bit, on layouts the library itself produced."""
import numpy as np
import pytest

import moe_expert_routing_ids_gb300 as topo
import oracle
from moe_expert_routing_ids_gb300 import workloads as W


def _cfg(T, E, k, R, rpn, ns):
    return dict(T=T, E=E, k=k, R=R, ranks_per_node=rpn, n_slot=ns, tok_bytes=2048,
                expert_bytes=1 << 20, c_intra=1, c_inter=4, max_refine_iters=0, main_rank=None)


def test_pack_arguments_are_checked_on_the_host():
    try:
        topo.lib()
    except RuntimeError:
        pytest.skip("library not built")
    cfg = topo.make_cfg(**_cfg(64, 8, 2, 4, 2, 1))
    need = topo.topo_workspace_bytes(cfg, 1, topo.TOPO_CALL_PACK)
    assert need >= 256 + 64 * 2 * 4
    a = 1 << 20                                             # never dereferenced
    for H in (0, 4, 12):
        with pytest.raises(topo.TopoError) as ex:
            topo.topo_permute(cfg, 1, H, a, a, a, a, need)
        assert ex.value.code == topo.TOPO_EINVAL
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_permute(cfg, 1, 16, a + 8, a, a, a, need)    # x not 16-byte aligned
    assert ex.value.code == topo.TOPO_EINVAL
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_combine(cfg, 1, 16, a, a, a, a, a, need - 1)
    assert ex.value.code == topo.TOPO_ENOSPC
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_combine(cfg, 1, 16, a, a, None, a, a, need)  # no weights
    assert ex.value.code == topo.TOPO_EINVAL


torch = pytest.importorskip("torch")
gpu = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch.device("cuda:0")


def _layout(cfg, ids, dev):
    from moe_expert_routing_ids_gb300.planner import Planner
    P = Planner(cfg, ids.shape[0], dev)
    P.run(torch.as_tensor(ids, device=dev))
    assert P.error() == 0
    return P.buf.sorted_pairs


def _bf16_bits(rng, shape, scale=4.0):
    f = (rng.standard_normal(shape) * scale).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)          # finite bf16 patterns


def _run_pack(cfg, L, H, sorted_pairs, x_bits, w, dev):
    c = topo.make_cfg(**cfg)
    ws_bytes = topo.topo_workspace_bytes(c, L, topo.TOPO_CALL_PACK)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    T, k = cfg["T"], cfg["k"]
    x = torch.as_tensor(x_bits.view(np.int16), device=dev)
    y = torch.empty((L, T * k, H), dtype=torch.int16, device=dev)
    topo.topo_permute(c, L, H, x, sorted_pairs, y, ws, ws_bytes)
    out = torch.empty((L, T, H), dtype=torch.int16, device=dev)
    wd = torch.as_tensor(w, device=dev)
    topo.topo_combine(c, L, H, y, sorted_pairs, wd, out, ws, ws_bytes)
    torch.cuda.synchronize()
    return (y.cpu().numpy().view(np.uint16), out.cpu().numpy().view(np.uint16),
            topo.topo_read_error(ws))


CASES = {
    # name: (cfg, L, H)
    "k8_h7168": (_cfg(2048, 64, 8, 16, 8, 4), 1, 7168),
    "k3_generic_h40_two_layers": (_cfg(1000, 24, 3, 8, 4, 2), 2, 40),
    "k1_h8": (_cfg(512, 8, 1, 8, 4, 1), 1, 8),
    "k10_h264": (_cfg(4096, 64, 10, 32, 8, 4), 1, 264),
    "k20_h16": (_cfg(640, 64, 20, 8, 4, 2), 1, 16),
}


@gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_permute_and_combine_match_the_oracle(name):
    dev = _dev()
    cfg, L, H = CASES[name]
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    rng = np.random.default_rng(len(name))
    ids = W.random_small(7, T, E, k, L, s=1.2)
    sp = _layout(cfg, ids, dev)
    x = _bf16_bits(rng, (L, T, H))
    w = rng.random((L, T, k)).astype(np.float32)
    y, out, err = _run_pack(cfg, L, H, sp, x, w, dev)
    assert err == 0
    spn = sp.cpu().numpy()
    assert np.array_equal(y, oracle.permute(x, spn, k))
    assert np.array_equal(out, oracle.combine(y, spn, w, k))


@gpu
def test_pack_flags_a_layout_that_is_not_a_permutation():
    dev = _dev()
    cfg, L, H = _cfg(256, 8, 2, 4, 2, 1), 1, 16
    sp = torch.arange(256 * 2, dtype=torch.int32, device=dev).view(1, -1).clone()
    sp[0, 5] = sp[0, 6]                                      # pair 5 missing, pair 6 twice
    rng = np.random.default_rng(0)
    _, _, err = _run_pack(cfg, L, H, sp, _bf16_bits(rng, (1, 256, H)),
                          np.ones((1, 256, 2), np.float32), dev)
    assert err == topo.TOPO_ESTATE


@gpu
def test_permute_and_combine_at_the_benchmarked_size():
    # the first layer of the T = 65536, E = 256, k = 8, R = 64 workload with
    # H = 7168 bf16 rows (x 0.94 GB, send buffer 7.5 GB), the size the
    # benchmark times.  The layout comes from the oracle chain; the GPU runs on
    # whole rows and every byte is compared, in blocks of columns (both
    # operations act on each column independently).
    from moe_expert_routing_ids_gb300 import workloads as W
    dev = _dev()
    w = W.FOUR_LAYER
    cfg = dict(w.plan_cfg)
    T, k, H = w.T, w.k, 7168
    ids = w.ids(n_layers=1)
    h = oracle.hist(ids, w.R, w.E)
    pl = oracle.plan(cfg, h)
    sp, _, _, _ = oracle.layout(cfg, oracle.reroute(cfg, ids, pl))
    sp = sp.reshape(1, T * k)
    rng = np.random.default_rng(71)
    x = _bf16_bits(rng, (1, T, H))
    wts = rng.random((1, T, k)).astype(np.float32)
    c = topo.make_cfg(**cfg)
    ws_bytes = topo.topo_workspace_bytes(c, 1, topo.TOPO_CALL_PACK)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    d_sp = torch.as_tensor(sp, device=dev)
    d_x = torch.as_tensor(x.view(np.int16), device=dev)
    y = torch.empty((1, T * k, H), dtype=torch.int16, device=dev)
    topo.topo_permute(c, 1, H, d_x, d_sp, y, ws, ws_bytes)
    out = torch.empty((1, T, H), dtype=torch.int16, device=dev)
    topo.topo_combine(c, 1, H, y, d_sp, torch.as_tensor(wts, device=dev), out, ws, ws_bytes)
    torch.cuda.synchronize()
    assert topo.topo_read_error(ws) == 0
    del d_x
    out_h = out.cpu().numpy().view(np.uint16)
    step = 512
    for a in range(0, H, step):
        xa = np.ascontiguousarray(x[:, :, a:a + step])
        ya = oracle.permute(xa, sp, k)
        got = y[:, :, a:a + step].contiguous().cpu().numpy().view(np.uint16)
        assert np.array_equal(got, ya), f"permute, columns {a}..{a + step}"
        oa = oracle.combine(ya, sp, wts, k)
        assert np.array_equal(out_h[:, :, a:a + step], oa), f"combine, columns {a}..{a + step}"
