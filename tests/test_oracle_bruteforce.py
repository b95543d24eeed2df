"""Brute force over every routing of tiny batches: the oracle's sequential
(token, rank) capacity fill against an independent sort-based formulation.
CPU only.

Independent formulation ([MoE 模型原理 §4.2]: per expert, the earliest tokens
up to the capacity are kept): list every routed slot as (expert, token),
stable-sort by expert, and within each expert keep the first C entries.
"""

import itertools

import numpy as np
import pytest

import oracle


def sort_based_fill(ids, E, C):
    T, k = ids.shape
    slots = [(int(ids[t, r]), t, r) for t in range(T) for r in range(k)]
    slots.sort(key=lambda s: (s[0], s[1]))  # by expert, then token (a token holds an expert once)
    counts = np.zeros(E, np.int64)
    for e, _, _ in slots:
        counts[e] += 1
    kept = np.minimum(counts, C)
    offsets = np.concatenate([[0], np.cumsum(kept)])
    slot_row = np.full((T, k), -1, np.int64)
    row_token = np.full(int(offsets[-1]), -1, np.int64)
    seen = np.zeros(E, np.int64)
    for e, t, r in slots:
        if seen[e] < C:
            row = offsets[e] + seen[e]
            slot_row[t, r] = row
            row_token[row] = t
        seen[e] += 1
    return counts, kept, offsets, slot_row, row_token


CASES = [(3, 3, 1), (4, 4, 2), (5, 3, 1), (3, 4, 3), (6, 2, 1), (4, 3, 2)]


@pytest.mark.parametrize("T,E,k", CASES)
def test_fill_all_routings(T, E, k):
    per_token = list(itertools.permutations(range(E), k))
    caps = sorted({oracle.capacity(T, k, E, c) for c in (0.25, 0.5, 1.0, 1.5)} | {1, T})
    n = 0
    for routing in itertools.product(per_token, repeat=T):
        ids = np.array(routing, np.int32).reshape(T, k)
        for C in caps:
            fl = oracle.fill(ids, E, C)
            counts, kept, offsets, slot_row, row_token = sort_based_fill(ids, E, C)
            assert (fl["counts"] == counts).all()
            assert (fl["kept"] == kept).all()
            assert (fl["offsets"] == offsets).all()
            assert (fl["slot_row"] == slot_row).all()
            assert (fl["row_token"] == row_token).all()
            n += 1
    assert n == len(per_token) ** T * len(caps)


def test_fill_invariants_random():
    rng = np.random.default_rng(1)
    for trial in range(30):
        E = int(rng.integers(1, 40))
        k = int(rng.integers(1, min(E, 9) + 1))
        T = int(rng.integers(1, 400))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        C = oracle.capacity(T, k, E, float(rng.choice([0.3, 1.0, 1.25, 2.0])))
        fl = oracle.fill(ids, E, C)
        assert fl["counts"].sum() == T * k
        assert (fl["kept"] == np.minimum(fl["counts"], C)).all()
        n = fl["offsets"][E]
        assert n <= min(T * k, E * C)
        rows = fl["slot_row"][fl["slot_row"] >= 0]
        assert sorted(rows.tolist()) == list(range(n))          # injective onto [0, n)
        for e in range(E):
            grp = fl["row_token"][fl["offsets"][e]:fl["offsets"][e + 1]]
            assert (np.diff(grp) > 0).all()                      # ascending tokens
            assert (ids[grp] == e).any(axis=1).all()
