"""Pins of the oracle's token-shuffle targets ("Expert Coupling in MoE
Pretraining", "Moving Tokens Toward Their Next Experts")."""
import numpy as np

import oracle


def test_shuffle_hand_case(golden):
    g = golden("shuffle_hand.json")
    t, st = oracle.shuffle(np.array(g["ids"], np.int32), np.array(g["tr"], np.int64), g["cfg"]["R"])
    assert t.tolist() == g["expected_target"]
    assert st.tolist() == g["expected_stats"]


def _counts(ids, E):
    T, k = ids.shape
    C = np.zeros((T, E), np.int64)
    np.add.at(C, (np.repeat(np.arange(T), k), ids.reshape(-1)), 1)
    return C


def _numpy_shuffle(ids, tr, R, rank_of):
    L, T, k = ids.shape
    E = tr.shape[-1]
    P = np.zeros((E, R), np.int64)
    P[np.arange(E), rank_of] = 1
    src = np.arange(T) // (T // R)
    targets, stats = [], []
    for l in range(L - 1):
        S = _counts(ids[l], E) @ (tr[l] @ P)                       # scores [T, R]
        mx = S.max(axis=1)
        first = np.argmax(S == mx[:, None], axis=1)
        tgt = np.where(S[np.arange(T), src] == mx, src, first)
        nxt_rank = rank_of[ids[l + 1]]
        stats.append([(nxt_rank == tgt[:, None]).sum(), (nxt_rank == src[:, None]).sum(),
                      (tgt != src).sum(), T * k])
        targets.append(tgt)
    return np.array(targets, np.int32), np.array(stats, np.int64)


def test_shuffle_is_the_matrix_form_with_arbitrary_counts_and_maps():
    rng = np.random.default_rng(0)
    for (L, T, E, k, R) in ((3, 96, 16, 2, 4), (2, 64, 24, 5, 8), (4, 128, 32, 3, 2)):
        ids = np.stack([np.stack([rng.permutation(E)[:k] for _ in range(T)]) for _ in range(L)])
        ids = ids.astype(np.int32)
        tr = rng.integers(0, 4, size=(L - 1, E, E)).astype(np.int64)   # many ties
        rank_of = np.repeat(np.arange(R), E // R).astype(np.int32)
        mr = rng.permutation(rank_of).astype(np.int32)
        for m in (None, mr):
            ro = rank_of if m is None else m
            t, st = oracle.shuffle(ids, tr, R, main_rank=m)
            et, est = _numpy_shuffle(ids, tr, R, ro)
            assert np.array_equal(t, et)
            assert np.array_equal(st, est)


def test_transitions_from_cooccur_feed_the_same_form():
    rng = np.random.default_rng(1)
    L, T, E, k, R = 3, 80, 20, 3, 4
    ids = np.stack([np.stack([rng.permutation(E)[:k] for _ in range(T)]) for _ in range(L)]).astype(np.int32)
    _, tr = oracle.cooccur(ids, E)
    t, st = oracle.shuffle(ids, tr, R)
    et, est = _numpy_shuffle(ids, tr, R, np.arange(E) // (E // R))
    assert np.array_equal(t, et) and np.array_equal(st, est)


def test_no_information_keeps_every_token_home():
    ids = np.random.default_rng(2).integers(0, 8, size=(2, 32, 1)).astype(np.int32)
    t, st = oracle.shuffle(ids, np.zeros((1, 8, 8), np.int64), 4)
    assert np.array_equal(t[0], np.arange(32) // 8)
    assert st[0, 2] == 0 and st[0, 0] == st[0, 1]


def test_planted_transitions_are_predicted():
    # each expert hands its tokens to one fixed expert of the next layer 80% of
    # the time: the prediction must land most next-layer pairs on the target
    rng = np.random.default_rng(3)
    L, T, E, k, R = 2, 4096, 32, 1, 8
    pi = rng.permutation(E)
    a = rng.integers(0, E, size=T)
    b = np.where(rng.random(T) < 0.8, pi[a], rng.integers(0, E, size=T))
    ids = np.stack([a, b])[:, :, None].astype(np.int32)
    _, tr = oracle.cooccur(ids, E)
    t, st = oracle.shuffle(ids, tr, R)
    assert st[0, 0] / st[0, 3] > 0.75
    assert st[0, 1] / st[0, 3] < 0.25
