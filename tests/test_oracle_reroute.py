"""Pins for the oracle's overflow reroute ([MoE 模型原理 §4.3], second policy:
an overflowing slot goes to the next expert of the token's candidate list).

The expected values come from the §4.2 worked example worked by hand, from
the no-overflow special case (identical to the plain fill), from a stable
argsort (the candidate ranks), and from invariants that any correct reroute
must satisfy on random tiny batches.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def two_expert_logits(routing0):
    s = np.empty((len(routing0), 2), np.float32)
    for t, e in enumerate(routing0):
        s[t] = (math.log(0.6), math.log(0.4)) if e == 0 else (math.log(0.4), math.log(0.6))
    return s


def test_reroute_capacity_example_wrblog_s4_2():
    # §4.2: tokens 0-5 choose expert 1, tokens 6-7 expert 2 (0-based 0, 1).
    g = golden("wrblog_s4_2_capacity_example.json")
    routing0 = [r - 1 for r in g["routing_one_based"]]
    ids, _, _, _, cand = oracle.select(two_expert_logits(routing0), 1, True, want_cand=True)
    assert cand[:, 0].tolist() == [1 - e for e in routing0]  # the other expert
    # C = 4: tokens 4 and 5 overflow expert 0; expert 1 has 4 - 2 = 2 places
    # left, so both are served after expert 1's own tokens 6 and 7.
    fl = oracle.fill_reroute(ids, cand, 2, 4)
    assert fl["counts"].tolist() == [6, 2]
    assert fl["kept"].tolist() == [4, 4]
    assert fl["row_token"].tolist() == [0, 1, 2, 3, 6, 7, 4, 5]
    assert fl["slot_row"][:, 0].tolist() == [0, 1, 2, 3, 6, 7, 4, 5]
    assert fl["slot_expert"][:, 0].tolist() == [0, 0, 0, 0, 1, 1, 1, 1]
    # C = 3: tokens 3, 4, 5 overflow; one place is left on expert 1 and the
    # first offer (token 3) takes it; tokens 4 and 5 are dropped.
    fl = oracle.fill_reroute(ids, cand, 2, 3)
    assert fl["kept"].tolist() == [3, 3]
    assert fl["row_token"].tolist() == [0, 1, 2, 6, 7, 3]
    assert fl["slot_row"][:, 0].tolist() == [0, 1, 2, 5, -1, -1, 3, 4]


def test_reroute_without_overflow_is_the_plain_fill():
    rng = np.random.default_rng(1)
    s = rng.normal(size=(60, 8)).astype(np.float32)
    ids, _, _, _, cand = oracle.select(s, 3, True, want_cand=True)
    a = oracle.fill(ids, 8, 60)
    b = oracle.fill_reroute(ids, cand, 8, 60)
    for name in ["counts", "kept", "offsets", "slot_row", "row_token"]:
        np.testing.assert_array_equal(a[name], b[name], name)


@pytest.mark.parametrize("bias", [False, True])
def test_candidates_are_the_next_ranks(bias):
    rng = np.random.default_rng(2)
    T, E, k = 50, 11, 4
    s = rng.normal(size=(T, E)).astype(np.float32)
    sb = rng.normal(size=E).astype(np.float32) if bias else None
    ids, _, _, _, cand = oracle.select(s, k, True, sel_bias=sb, want_cand=True)
    key = s + sb[None, :] if bias else s
    order = np.argsort(-key.astype(np.float32), axis=1, kind="stable")
    np.testing.assert_array_equal(ids, order[:, :k])
    want = np.full((T, k), -1, np.int32)
    n = min(2 * k, E) - k
    want[:, :n] = order[:, k:k + n]
    np.testing.assert_array_equal(cand, want)


@pytest.mark.parametrize("seed", range(40))
def test_reroute_invariants_on_tiny_batches(seed):
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(1, 14))
    E = int(rng.integers(2, 6))
    k = int(rng.integers(1, min(3, E) + 1))
    C = int(rng.integers(0, 4))
    s = rng.normal(size=(T, E)).astype(np.float32)
    s[:, 0] += 1.5  # make expert 0 hot
    ids, _, _, _, cand = oracle.select(s, k, True, want_cand=True)
    plain = oracle.fill(ids, E, C)
    fl = oracle.fill_reroute(ids, cand, E, C)
    dest, rows = fl["slot_expert"], fl["slot_row"]
    off, kept = fl["offsets"], fl["kept"]
    np.testing.assert_array_equal(fl["counts"], plain["counts"])
    assert (kept <= C).all() and (kept >= plain["kept"]).all()
    # Slots kept by the plain fill keep their expert and position.
    first = plain["slot_row"] >= 0
    assert (dest[first] == ids[first]).all()
    np.testing.assert_array_equal(rows[first] - off[ids[first]],
                                  plain["slot_row"][first] - plain["offsets"][ids[first]])
    # Overflowing slots go to the token's m-th candidate, or are dropped.
    room = C - plain["kept"]
    served = np.zeros(E, np.int64)
    for t in range(T):
        m = 0
        for r in range(k):
            if first[t, r]:
                continue
            e2 = cand[t, m] if m < k else -1
            m += 1
            if e2 >= 0 and served[e2] < room[e2]:
                # served first come: its row follows the expert's first-fill rows
                assert dest[t, r] == e2
                assert rows[t, r] == off[e2] + plain["kept"][e2] + served[e2]
                served[e2] += 1
            else:
                assert dest[t, r] == -1 and rows[t, r] == -1
    # The buffer holds each kept slot once; row_token matches.
    kr = rows[rows >= 0]
    assert len(np.unique(kr)) == len(kr) == off[E]
    tok = np.repeat(np.arange(T), k).reshape(T, k)
    np.testing.assert_array_equal(fl["row_token"][kr], tok[rows >= 0])
