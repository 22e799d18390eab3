"""topo_hist_noalloc: the histogram with the library's fixed scratch array
must give exactly what topo_hist gives with an allocated workspace, and what
the CPU oracle gives, call after call, and must refuse shapes whose scratch
does not fit."""
import numpy as np
import pytest

import moe_expert_routing_ids_gb300 as topo
import oracle
from moe_expert_routing_ids_gb300 import workloads as W


def _cfg(T, E, k, R, rpn, n_slot):
    return topo.make_cfg(T=T, E=E, k=k, R=R, ranks_per_node=rpn, n_slot=n_slot,
                         tok_bytes=4096, expert_bytes=1 << 20)


def test_shape_beyond_the_scratch_is_refused():
    try:
        topo.lib()
    except RuntimeError:
        pytest.skip("library not built")
    # 80 layers x 128 ranks x 1 tile x 512 experts x 4 B = 20 MiB of tile counts
    cfg = _cfg(T=128 * 64, E=512, k=2, R=128, rpn=8, n_slot=0)
    assert topo.TOPO_HIST_NOALLOC_SCRATCH_BYTES == 16 << 20
    assert topo.topo_workspace_bytes(cfg, 80, topo.TOPO_CALL_HIST) > 0     # a valid shape
    with pytest.raises(topo.TopoError) as exc:
        topo.topo_hist_noalloc(cfg, 80, 1 << 20, 1 << 20)
    assert exc.value.code == topo.TOPO_ENOSPC
    # 60 layers (15 MiB) fit: rejected only for the NULL hist below, not for size
    with pytest.raises(topo.TopoError) as exc:
        topo.topo_hist_noalloc(cfg, 60, 1 << 20, None)
    assert exc.value.code == topo.TOPO_EINVAL


def _hist_with_workspace(torch, cfg, L, d_ids, stream):
    R, E = cfg.R, cfg.E
    ws_bytes = topo.topo_workspace_bytes(cfg, L, topo.TOPO_CALL_HIST)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=d_ids.device)
    hist = torch.empty((L, R, E), dtype=torch.int32, device=d_ids.device)
    topo.topo_hist(cfg, L, d_ids, hist, ws, ws_bytes, stream)
    torch.cuda.synchronize()
    assert topo.topo_read_error(ws) == 0
    return hist.cpu().numpy()


@pytest.mark.gpu
def test_hist_noalloc_matches_topo_hist_twice_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    cases = []
    # the full-size 4-microbatch workloads (T = 1048576 with 8 tiles per
    # source, then T = 65536), then a small ragged one: no call may see the
    # previous call's counts or error word
    for w in (W.STRESS, W.FOUR_LAYER):
        cases.append((_cfg(w.T, w.E, w.k, w.R, w.ranks_per_node, w.n_slot), w.n_layers,
                      w.ids()))
    ids_small = W.random_small(seed=11, T=8 * 300, E=24, k=3, n_layers=2)
    cases.append((_cfg(8 * 300, 24, 3, 8, 4, 2), 2, ids_small))
    err = torch.full((1,), -99, dtype=torch.int32, device=dev)
    outs = []
    for cfg, L, ids in cases:
        d_ids = torch.as_tensor(np.ascontiguousarray(ids, dtype=np.int32), device=dev)
        hist = torch.full((L, cfg.R, cfg.E), -1, dtype=torch.int32, device=dev)
        topo.topo_hist_noalloc(cfg, L, d_ids, hist, err, stream)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        outs.append((hist.cpu().numpy(), _hist_with_workspace(torch, cfg, L, d_ids, stream)))
    for (got, want), (cfg, L, ids) in zip(outs, cases):
        np.testing.assert_array_equal(got, want)
        # and the oracle's Omega (Eq. 3), independently of both GPU paths
        np.testing.assert_array_equal(got, oracle.hist(ids, cfg.R, cfg.E))
    # the same shape once more, after the other: identical again
    cfg, L, ids = cases[0]
    d_ids = torch.as_tensor(np.ascontiguousarray(ids, dtype=np.int32), device=dev)
    hist = torch.empty((L, cfg.R, cfg.E), dtype=torch.int32, device=dev)
    topo.topo_hist_noalloc(cfg, L, d_ids, hist, err, stream)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    np.testing.assert_array_equal(hist.cpu().numpy(), outs[0][1])


@pytest.mark.gpu
def test_hist_noalloc_with_unequal_source_blocks():
    # the table of each source's first tile lives in the fixed array too
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    dev = torch.device("cuda:0")
    T, E, k, R = 9000, 32, 4, 8
    off = np.array([0, 3000, 3000, 3001, 6000, 6100, 8000, 8999, 9000], np.int64)
    d_off = torch.as_tensor(off, device=dev)
    cfg = topo.make_cfg(T=T, E=E, k=k, R=R, ranks_per_node=4, n_slot=1, tok_bytes=64,
                        expert_bytes=1 << 10, rank_offsets=d_off)
    ids = W.random_small(seed=12, T=T, E=E, k=k, n_layers=2)
    d_ids = torch.as_tensor(ids, device=dev)
    hist = torch.empty((2, R, E), dtype=torch.int32, device=dev)
    err = torch.full((1,), -99, dtype=torch.int32, device=dev)
    for _ in range(2):
        topo.topo_hist_noalloc(cfg, 2, d_ids, hist, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        np.testing.assert_array_equal(hist.cpu().numpy(), oracle.hist(ids, R, E, rank_offsets=off))


@pytest.mark.gpu
def test_hist_noalloc_reports_out_of_range_ids():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    dev = torch.device("cuda:0")
    cfg = _cfg(T=8 * 64, E=16, k=2, R=8, rpn=4, n_slot=1)
    ids = np.zeros((1, 8 * 64, 2), dtype=np.int32)
    ids[0, :, 1] = 1
    ids[0, 5, 1] = 16                                  # outside [0, E)
    d_ids = torch.as_tensor(ids, device=dev)
    hist = torch.empty((1, 8, 16), dtype=torch.int32, device=dev)
    err = torch.zeros((1,), dtype=torch.int32, device=dev)
    topo.topo_hist_noalloc(cfg, 1, d_ids, hist, err)
    torch.cuda.synchronize()
    assert int(err.item()) == topo.TOPO_ERANGE
    # the next call starts from a clear error word
    ids[0, 5, 1] = 1
    d_ids.copy_(torch.as_tensor(ids))
    topo.topo_hist_noalloc(cfg, 1, d_ids, hist, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    h = hist.cpu().numpy()
    assert h[0, :, 0].tolist() == [64] * 8 and h[0, :, 1].tolist() == [64] * 8
