"""Token-shuffle targets (topo_shuffle_targets) on the GPU against the
oracle, bit for bit: targets and statistics, with random and with GPU
co-occurrence transition counts."""
import numpy as np
import pytest

import moe_expert_routing_ids_gb300 as topo
import oracle


def test_shuffle_arguments_are_checked_on_the_host():
    try:
        topo.lib()
    except RuntimeError:
        pytest.skip("library not built")
    a = 1 << 20                                             # never dereferenced
    need = topo.topo_shuffle_workspace_bytes(2, 16, 4)
    assert need >= 256 + 16 * 4 * 8
    assert topo.topo_shuffle_workspace_bytes(2, 16, 257) == 0
    bad = [(2, 64, 16, 2, 257), (2, 66, 16, 2, 4), (2, 64, 18, 2, 4), (2, 64, 16, 0, 4), (2, 64, 16, 65, 4)]
    for (L, T, E, k, R) in bad:
        with pytest.raises(topo.TopoError) as ex:
            topo.topo_shuffle_targets(L, T, E, k, R, a, a, None, None, a, a, a, 1 << 20)
        assert ex.value.code == topo.TOPO_EINVAL
    with pytest.raises(topo.TopoError) as ex:
        topo.topo_shuffle_targets(2, 64, 16, 2, 4, a, a, None, None, a, a, a, need - 1)
    assert ex.value.code == topo.TOPO_ENOSPC


torch = pytest.importorskip("torch")
gpu = pytest.mark.gpu


def _dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return torch.device("cuda:0")


def run_shuffle(ids, tr, R, main_rank, dev, rank_offsets=None):
    L, T, k = ids.shape
    E = tr.shape[-1]
    nb = topo.topo_shuffle_workspace_bytes(L, E, R)
    ws = torch.zeros(nb, dtype=torch.uint8, device=dev)
    d_ids = torch.as_tensor(ids, device=dev)
    d_tr = tr if isinstance(tr, torch.Tensor) else torch.as_tensor(tr, device=dev)
    mr = None if main_rank is None else torch.as_tensor(main_rank, device=dev)
    roff = None if rank_offsets is None else torch.as_tensor(np.asarray(rank_offsets, np.int64), device=dev)
    target = torch.full((L - 1, T), -7, dtype=torch.int32, device=dev)
    stats = torch.full((L - 1, topo.TOPO_SHUFFLE_STATS), -7, dtype=torch.int64, device=dev)
    topo.topo_shuffle_targets(L, T, E, k, R, d_ids, d_tr, mr, roff, target, stats, ws, nb)
    torch.cuda.synchronize()
    return target.cpu().numpy(), stats.cpu().numpy(), topo.topo_read_error(ws)


def _ids(rng, L, T, E, k):
    return np.stack([np.argsort(rng.random((T, E)), axis=1)[:, :k] for _ in range(L)]).astype(np.int32)


CASES = {
    # name: (L, T, E, k, R, map)
    "r4_g4_map": (3, 96 * 4, 16, 2, 4, True),
    "r8_g8": (2, 1000 * 8, 64, 6, 8, False),
    "r16_g16_three_layers": (4, 2048, 128, 8, 16, False),
    "r32_smem_table": (2, 32 * 40, 256, 8, 32, True),
    "r64_global_table": (2, 64 * 20, 256, 8, 64, False),
    "r128_rpl4": (2, 128 * 8, 512, 10, 128, False),
    "r256_rpl8": (2, 256 * 4, 512, 4, 256, True),
    "r1": (2, 100, 12, 3, 1, False),
    "r3_unequal_map": (2, 3 * 50, 7, 2, 3, True),
}


@gpu
@pytest.mark.parametrize("name", sorted(CASES))
def test_shuffle_matches_the_oracle(name):
    dev = _dev()
    L, T, E, k, R, with_map = CASES[name]
    rng = np.random.default_rng(len(name))
    ids = _ids(rng, L, T, E, k)
    tr = rng.integers(0, 3, size=(L - 1, E, E)).astype(np.int64)       # many ties
    mr = rng.integers(0, R, size=E).astype(np.int32) if with_map else None
    t, st, err = run_shuffle(ids, tr, R, mr, dev)
    assert err == 0
    et, est = oracle.shuffle(ids, tr, R, main_rank=mr)
    assert np.array_equal(t, et)
    assert np.array_equal(st, est)


@gpu
def test_shuffle_from_gpu_cooccurrence_on_the_four_layer_workload():
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Cooccur
    dev = _dev()
    w = W.FOUR_LAYER
    ids = w.ids()
    C = Cooccur(w.n_layers, w.T, w.E, w.k, dev)
    C.run(torch.as_tensor(ids, device=dev))
    assert C.error() == 0
    t, st, err = run_shuffle(ids, C.tr, w.R, None, dev)
    assert err == 0
    et, est = oracle.shuffle(ids, C.tr.cpu().numpy(), w.R)
    assert np.array_equal(t, et) and np.array_equal(st, est)
    assert np.all(st[:, 0] > 4 * st[:, 1])           # the prediction beats staying on the source


@gpu
def test_shuffle_flags_bad_ids_and_maps():
    dev = _dev()
    rng = np.random.default_rng(9)
    ids = _ids(rng, 2, 64, 16, 2)
    tr = rng.integers(0, 3, size=(1, 16, 16)).astype(np.int64)
    bad = ids.copy()
    bad[0, 5, 1] = 16
    _, _, err = run_shuffle(bad, tr, 4, None, dev)
    assert err == topo.TOPO_ERANGE
    mr = np.repeat(np.arange(4), 4).astype(np.int32)
    mr[3] = 4
    _, _, err = run_shuffle(ids, tr, 4, mr, dev)
    assert err == topo.TOPO_EMAP


@gpu
def test_shuffle_with_one_layer_or_no_tokens_is_a_no_op():
    dev = _dev()
    nb = topo.topo_shuffle_workspace_bytes(1, 16, 4)
    ws = torch.zeros(max(nb, 256), dtype=torch.uint8, device=dev)
    topo.topo_shuffle_targets(1, 64, 16, 2, 4, None, None, None, None, None, None, ws, ws.numel())
    ids = np.zeros((3, 0, 2), np.int32)
    tr = np.zeros((2, 16, 16), np.int64)
    t, st, err = run_shuffle(ids, tr, 4, None, dev)
    assert err == 0 and t.shape == (2, 0) and not st.any()


@gpu
@pytest.mark.parametrize("R", [4, 16, 64])
def test_shuffle_with_counts_too_large_for_int32_scores(R):
    dev = _dev()
    rng = np.random.default_rng(R)
    L, T, E, k = 2, 64 * 16, 64, 6
    ids = _ids(rng, L, T, E, k)
    tr = rng.integers(0, 1 << 40, size=(L - 1, E, E)).astype(np.int64)
    t, st, err = run_shuffle(ids, tr, R, None, dev)
    assert err == 0
    et, est = oracle.shuffle(ids, tr, R)
    assert np.array_equal(t, et) and np.array_equal(st, est)


@gpu
def test_shuffle_full_size_cooccurrence_workload():
    # the 8-layer, 262144-token, E = 128, k = 8 workload as EP16, as bench.py
    # times it, with its own GPU transition counts
    from moe_expert_routing_ids_gb300 import workloads as W
    from moe_expert_routing_ids_gb300.planner import Cooccur
    dev = _dev()
    w = W.COOCCUR
    ids = w.ids()
    C = Cooccur(w.n_layers, w.T, w.E, w.k, dev)
    C.run(torch.as_tensor(ids, device=dev))
    assert C.error() == 0
    t, st, err = run_shuffle(ids, C.tr, 16, None, dev)
    assert err == 0
    et, est = oracle.shuffle(ids, C.tr.cpu().numpy(), 16)
    assert np.array_equal(t, et) and np.array_equal(st, est)


@gpu
def test_shuffle_with_unequal_source_blocks():
    # the tie rule and the statistics use each token's own source block
    dev = _dev()
    rng = np.random.default_rng(21)
    L, T, E, k = 3, 3000, 64, 4
    for R, lens in ((8, [10, 0, 1990, 300, 200, 0, 499, 1]), (64, None)):
        if lens is None:
            cuts = np.sort(rng.integers(0, T + 1, R - 1))
            off = np.concatenate([[0], cuts, [T]]).astype(np.int64)
        else:
            off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        ids = _ids(rng, L, T, E, k)
        tr = rng.integers(0, 3, size=(L - 1, E, E)).astype(np.int64)     # many ties
        tg, st, err = run_shuffle(ids, tr, R, None, dev, rank_offsets=off)
        assert err == 0
        want_t, want_s = oracle.shuffle(ids, tr, R, rank_offsets=off)
        assert np.array_equal(tg, want_t)
        assert np.array_equal(st, want_s)
