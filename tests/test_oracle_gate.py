"""Pins of the oracle's Top-k gating (TopoEP §2.1 Top-k gating; §6.4 synthetic
routing from random logits with a fixed expert-specific bias)."""
import numpy as np

import oracle


def _val(x):
    return {"nan": np.nan, "inf": np.inf, "-inf": -np.inf, "-0": -0.0}.get(x, x) if isinstance(x, str) else x


def _arr(rows):
    return np.array([[_val(v) for v in row] for row in rows], np.float32)


def _same_bits(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32), np.asarray(b, np.float32).view(np.uint32))


def test_gate_hand_case(golden):
    g = golden("gate_hand.json")
    c = g["cfg"]
    x = _arr(g["logits"])
    o = oracle.gate(x, c["k"], c["R"])
    ex = g["expected_no_bias"]
    assert o["ids"].tolist() == ex["ids"]
    assert _same_bits(o["scores"], _arr(ex["scores"]))
    assert o["hist"].tolist() == ex["hist"]
    b = np.array(g["bias_token1"], np.float32)
    o = oracle.gate(x[1:2], c["k"], 1, bias=b)
    assert o["ids"][0].tolist() == g["expected_token1_with_bias"]["ids"]
    assert o["scores"][0].tolist() == g["expected_token1_with_bias"]["scores"]


def _numpy_gate(x, k, bias):
    s = x if bias is None else (x + bias).astype(np.float32)
    ids = np.argsort(-s, axis=-1, kind="stable")[..., :k]       # NaN sorts last, ties by index
    return ids.astype(np.int32), np.take_along_axis(x, ids, axis=-1)


def test_gate_is_a_stable_descending_sort_of_the_biased_scores():
    rng = np.random.default_rng(1)
    for (L, T, E, k) in ((2, 64, 8, 2), (1, 96, 64, 6), (1, 40, 160, 8), (1, 16, 1000, 16)):
        x = rng.standard_normal((L, T, E)).astype(np.float32)
        for bias in (None, rng.standard_normal(E).astype(np.float32)):
            o = oracle.gate(x, k, 4 if T % 4 == 0 else 1, bias=bias)
            ids, sc = _numpy_gate(x, k, bias)
            assert np.array_equal(o["ids"], ids)
            assert _same_bits(o["scores"], sc)


def test_ties_signed_zeros_and_nans_follow_the_stable_sort():
    rng = np.random.default_rng(2)
    x = rng.integers(-3, 4, size=(1, 256, 32)).astype(np.float32)   # many equal scores
    x[rng.random(x.shape) < 0.1] = -0.0
    x[rng.random(x.shape) < 0.05] = np.nan
    x[0, 7, :] = np.nan
    o = oracle.gate(x, 5, 8)
    ids, sc = _numpy_gate(x, 5, None)
    assert np.array_equal(o["ids"], ids)
    assert _same_bits(o["scores"], sc)


def test_bf16_logits_are_the_widened_patterns():
    rng = np.random.default_rng(3)
    f = rng.standard_normal((2, 32, 48)).astype(np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    wide = (bits.astype(np.uint32) << 16).view(np.float32)
    b = rng.standard_normal(48).astype(np.float32)
    o16 = oracle.gate(bits, 4, 4, bias=b)
    o32 = oracle.gate(wide, 4, 4, bias=b)
    for key in ("ids", "hist"):
        assert np.array_equal(o16[key], o32[key])
    assert _same_bits(o16["scores"], o32["scores"])


def test_hist_counts_the_selected_ids_per_source():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((1, 120, 24)).astype(np.float32)
    o = oracle.gate(x, 3, 6)
    for s in range(6):
        blk = o["ids"][0, s * 20:(s + 1) * 20].reshape(-1)
        assert np.array_equal(o["hist"][0, s], np.bincount(blk, minlength=24))


def test_gumbel_logits_with_log_probability_bias_sample_the_top1_by_p():
    # The pages' synthetic routing adds a fixed expert bias to random logits.
    # With standard Gumbel logits and bias log p, the top-1 expert is a draw
    # from p (the Gumbel-max property), so its frequencies must match p.
    rng = np.random.default_rng(5)
    E, T = 8, 40000
    p = 1.0 / np.arange(1, E + 1) ** 1.2
    p /= p.sum()
    g = (-np.log(-np.log(rng.random((T, E))))).astype(np.float32)
    o = oracle.gate(g, 2, 1, bias=np.log(p).astype(np.float32))
    freq = np.bincount(o["ids"][:, 0], minlength=E) / T
    assert np.all(np.abs(freq - p) < 4 * np.sqrt(p * (1 - p) / T))
    assert np.all(o["ids"][:, 0] != o["ids"][:, 1])
