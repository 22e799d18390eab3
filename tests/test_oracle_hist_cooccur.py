"""Pins for the oracle's histogram and co-occurrence (CPU only).

Each check compares the oracle with something other than itself: a numpy
closed form, a hand-worked case from the pages' definitions, or an identity
that holds for every input.
"""
import numpy as np
import pytest

import oracle
from moe_expert_routing_ids_gb300 import workloads as W


def _bincount_blocks(ids, R, E):
    """Omega by numpy: bincount of each source's contiguous token block."""
    L, T, k = ids.shape
    out = np.zeros((L, R, E), np.int64)
    for l in range(L):
        for s, blk in enumerate(np.split(ids[l], R)):
            out[l, s] = np.bincount(blk.reshape(-1), minlength=E)
    return out


@pytest.mark.parametrize("T,E,k,R,L", [(64, 8, 2, 8, 1), (96, 16, 3, 4, 2), (1000, 40, 5, 10, 3),
                                       (0, 8, 2, 4, 1), (12, 1, 1, 3, 1)])
def test_hist_matches_blockwise_bincount(T, E, k, R, L):
    ids = W.random_small(T + E, T, E, k, L) if T else np.zeros((L, 0, k), np.int32)
    h = oracle.hist(ids, R, E)
    assert np.array_equal(h, _bincount_blocks(ids, R, E))
    assert h.sum() == T * k * L


def test_hist_duplicate_ids_are_counted_twice():
    ids = np.array([[[1, 1], [0, 2]]], np.int32)
    h = oracle.hist(ids, 2, 3)
    assert h[0].tolist() == [[0, 2, 0], [1, 0, 1]]


def test_hist_out_of_range_is_reported():
    ids = np.array([[[0, 5], [1, 2]]], np.int32)
    with pytest.raises(oracle.OracleError) as ex:
        oracle.hist(ids, 1, 4)
    assert ex.value.rc == oracle.ERANGE


def test_cooccur_hand_case(golden):
    g = golden("cooccur_t3.json")
    co, tr = oracle.cooccur(np.array(g["ids"], np.int32), g["E"])
    assert co.tolist() == g["expected_co"]
    assert tr.shape == (0, g["E"], g["E"])


def _count_matrix(ids_l, E):
    T, k = ids_l.shape
    C = np.zeros((T, E), np.int64)
    np.add.at(C, (np.repeat(np.arange(T), k), ids_l.reshape(-1)), 1)
    return C


@pytest.mark.parametrize("T,E,k,L", [(50, 8, 3, 3), (200, 16, 4, 2), (33, 5, 5, 4), (1, 4, 2, 2)])
def test_cooccur_closed_form(T, E, k, L):
    ids = W.random_small(7 * T + E, T, E, k, L)
    co, tr = oracle.cooccur(ids, E)
    for l in range(L):
        C = _count_matrix(ids[l], E)
        assert np.array_equal(co[l], C.T @ C)
        if l + 1 < L:
            assert np.array_equal(tr[l], C.T @ _count_matrix(ids[l + 1], E))
    # identities for distinct ids per token
    assert co.sum() == L * T * k * k
    for l in range(L):
        load = np.bincount(ids[l].reshape(-1), minlength=E)
        assert np.array_equal(np.diag(co[l]), load)
        assert np.array_equal(co[l], co[l].T)
        if l + 1 < L:
            assert np.array_equal(tr[l].sum(axis=1), k * load)
            assert np.array_equal(tr[l].sum(axis=0), k * np.bincount(ids[l + 1].reshape(-1), minlength=E))


def test_cooccur_with_repeated_ids_uses_count_vectors():
    # token selects expert 1 twice: n = [0, 2, 1] -> co = n n^T
    ids = np.array([[[1, 1, 2]], [[0, 2, 2]]], np.int32)
    co, tr = oracle.cooccur(ids, 3)
    n0, n1 = np.array([0, 2, 1]), np.array([1, 0, 2])
    assert np.array_equal(co[0], np.outer(n0, n0))
    assert np.array_equal(co[1], np.outer(n1, n1))
    assert np.array_equal(tr[0], np.outer(n0, n1))


def test_cooccur_grouped_generator_shows_structure():
    """Distributional sanity of the grouped generator only (not parity):
    a within-group expert pair is co-selected far more often than a
    cross-group pair."""
    rng = W.rng_for(99, 0)
    E = 32
    groups = rng.permutation(E).reshape(4, 8)
    ids = W.grouped_topk(rng, E, 4000, 4, groups, stay=0.7)[None]
    co = oracle.cooccur(ids, E, transitions=False)[0]
    gid = np.empty(E, int)
    for g, m in enumerate(groups):
        gid[m] = g
    same = gid[:, None] == gid[None, :]
    off = ~np.eye(E, dtype=bool)
    assert co[same & off].mean() > 3 * co[~same].mean()
