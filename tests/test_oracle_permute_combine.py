"""Pins of the oracle's dispatch pack (permute) and combine against hand cases
and properties that hold whatever the implementation."""
import numpy as np

import oracle
from moe_expert_routing_ids_gb300 import workloads as W


def _bf16_exact(values):
    """float32 values that are exact in bf16 -> their 16-bit patterns."""
    f = np.asarray(values, np.float32)
    u = f.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0)
    return (u >> 16).astype(np.uint16)


def _as_float(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def _small_layout(seed, T=64, E=8, k=3, R=4, rpn=2, ns=1):
    cfg = dict(T=T, E=E, k=k, R=R, ranks_per_node=rpn, n_slot=ns, tok_bytes=64,
               expert_bytes=1000, c_intra=1, c_inter=4, max_refine_iters=0, main_rank=None)
    ids = W.random_small(seed, T, E, k, 1)
    h = oracle.hist(ids, R, E)
    p = oracle.plan(cfg, h)
    d = oracle.reroute(cfg, ids, p)
    sp, _, _, _ = oracle.layout(cfg, d)
    return cfg, sp


def test_permute_hand_case(golden):
    g = golden("permute_combine_cases.json")["permute"]
    x = np.array([g["x"]], np.uint16)
    y = oracle.permute(x, np.array([g["sorted_pairs"]]), g["k"])
    assert y[0].tolist() == g["expected_y"]


def test_permute_puts_each_token_row_at_its_pairs_positions():
    cfg, sp = _small_layout(1)
    T, k, H = cfg["T"], cfg["k"], 5
    rng = np.random.default_rng(0)
    x = rng.integers(0, 1 << 16, size=(1, T, H)).astype(np.uint16)
    y = oracle.permute(x, sp, k)
    for t in range(T):
        where = np.nonzero(sp[0] // k == t)[0]
        assert len(where) == k
        assert np.all(y[0, where] == x[0, t])
    # every output row is a copy: the row sums (as integers) are k times the input's
    assert y.astype(np.int64).sum() == k * x.astype(np.int64).sum()


def test_combine_hand_cases(golden):
    cases = golden("permute_combine_cases.json")
    for name in ("combine_tie_to_even", "combine_slot_order", "combine_weights"):
        c = cases[name]
        y = np.array([c["y"]], np.uint16)
        out = oracle.combine(y, np.array([c["sorted_pairs"]]), np.array([c["w"]], np.float32), c["k"])
        assert out[0].tolist() == c["expected_out"], name


def test_combine_of_permute_is_identity_with_dyadic_weights():
    cfg, sp = _small_layout(2, k=4)
    T, k, H = cfg["T"], cfg["k"], 7
    rng = np.random.default_rng(1)
    xf = rng.integers(-64, 64, size=(1, T, H)).astype(np.float32)     # exact in bf16
    x = _bf16_exact(xf)
    w = np.tile(np.array([0.5, 0.25, 0.125, 0.125], np.float32), (1, T, 1))
    out = oracle.combine(oracle.permute(x, sp, k), sp, w, k)
    assert np.array_equal(out, x)


def test_combine_one_hot_weight_selects_that_slot():
    cfg, sp = _small_layout(3, k=3)
    T, k, H = cfg["T"], cfg["k"], 4
    rng = np.random.default_rng(2)
    y = _bf16_exact(rng.integers(-100, 100, size=(1, T * k, H)).astype(np.float32))
    pos_of = np.argsort(sp[0])                      # position of each pair
    for j in range(k):
        w = np.zeros((1, T, k), np.float32)
        w[..., j] = 1.0
        out = oracle.combine(y, sp, w, k)
        assert np.array_equal(out[0], y[0, pos_of[np.arange(T) * k + j]]), j


def test_combine_matches_float64_within_one_bf16_step():
    cfg, sp = _small_layout(4, k=3)
    T, k, H = cfg["T"], cfg["k"], 6
    rng = np.random.default_rng(3)
    y = _bf16_exact(np.ldexp(rng.integers(-255, 256, size=(1, T * k, H)), -4).astype(np.float32))
    w = rng.random((1, T, k)).astype(np.float32)
    out = _as_float(oracle.combine(y, sp, w, k))
    pos_of = np.argsort(sp[0])
    yy = _as_float(y[0]).astype(np.float64)
    want = sum(w[0, :, j, None].astype(np.float64) * yy[pos_of[np.arange(T) * k + j]] for j in range(k))
    # bf16 keeps 8 significant bits: within half a unit in the last place, plus float rounding
    assert np.all(np.abs(out[0] - want) <= np.abs(want) * 2.0 ** -8 + 1e-6)
