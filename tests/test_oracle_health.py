"""Pins for the oracle's expert-bias selection and routing-health indicators.

Sources: the ai-master.cc page on MoE expert-parallelism engineering
([EP 工程 ai-master]: 一、负载均衡 — an expert bias that replaces the auxiliary
loss and moves which experts are chosen; 追问 2 — the entropy of the expert
activation distribution and the variance of the tokens each expert
processes) and [MoE 模型原理 §10.4] (the overflow share).  Every expected value
here comes from a closed form, a worked example of the pages, or an
independent library routine, never from the oracle itself.
"""

import json
import math
import os

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --- selection bias --------------------------------------------------------------

def _logits(T, E, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(0, 1.5, (T, E)).astype(np.float32)


def test_zero_selection_bias_changes_nothing():
    s = _logits(64, 12, 1)
    a = oracle.select(s, 3, True)
    b = oracle.select(s, 3, True, sel_bias=np.zeros(12, np.float32))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    np.testing.assert_array_equal(a[2], b[2])


@pytest.mark.parametrize("renorm", [True, False])
def test_selection_bias_ranks_biased_scores_and_weights_unbiased_p(renorm):
    # Restated with library routines: ids = first k of a stable descending
    # sort of the float32 sums s + b (ties to the lower index); weights from
    # scipy's softmax of the unbiased scores.
    T, E, k = 80, 16, 4
    s = _logits(T, E, 2)
    b = np.random.default_rng(3).normal(0, 1.0, E).astype(np.float32)
    ids, w, psum, _ = oracle.select(s, k, renorm, sel_bias=b)
    key = (s + b[None, :]).astype(np.float32)
    want_ids = np.argsort(-key, axis=1, kind="stable")[:, :k]
    np.testing.assert_array_equal(ids, want_ids)
    p = scipy.special.softmax(s.astype(np.float64), axis=1)
    pk = np.take_along_axis(p, want_ids, axis=1)
    want_w = pk / pk.sum(axis=1, keepdims=True) if renorm else pk
    np.testing.assert_allclose(w, want_w, rtol=1e-12, atol=0)
    # Σ_t p is the unbiased softmax's column sum.
    np.testing.assert_allclose(psum, p.sum(axis=0), rtol=1e-12)


def test_large_selection_bias_forces_an_expert_without_changing_its_weight():
    T, E, k = 40, 8, 2
    s = _logits(T, E, 4)
    b = np.zeros(E, np.float32)
    b[5] = 1000.0
    ids, w, _, _ = oracle.select(s, k, True, sel_bias=b)
    assert (ids[:, 0] == 5).all()
    p = scipy.special.softmax(s.astype(np.float64), axis=1)
    other = ids[:, 1]
    want = p[np.arange(T), 5] / (p[np.arange(T), 5] + p[np.arange(T), other])
    np.testing.assert_allclose(w[:, 0], want, rtol=1e-12)
    # the second expert is the unbiased argmax among the rest
    rest = s.copy()
    rest[:, 5] = -np.inf
    np.testing.assert_array_equal(other, np.argmax(rest, axis=1))


def test_selection_bias_ties_go_to_the_lower_index():
    # Equal biased keys: s + b is the same for experts 1, 2 and 4.
    s = np.array([[0.0, 1.0, 0.5, -3.0, 0.0]], np.float32)
    b = np.array([0.0, 0.0, 0.5, 0.0, 1.0], np.float32)
    ids, *_ = oracle.select(s, 3, True, sel_bias=b)
    assert ids[0].tolist() == [1, 2, 4]


# --- routing health ------------------------------------------------------------

def test_health_uniform_load():
    E, T, k = 8, 64, 2
    counts = np.full(E, T * k // E, np.int32)
    h = oracle.routing_health(counts, counts, T, k)
    assert abs(h[0] - math.log(E)) < 1e-12
    assert h[1] == 0.0 and h[2] == 0.0 and h[3] == 0.0


def test_health_all_tokens_on_one_expert():
    E, T, k, C = 8, 100, 1, 13
    counts = np.zeros(E, np.int32)
    counts[3] = T
    kept = np.minimum(counts, C).astype(np.int32)
    h = oracle.routing_health(counts, kept, T, k)
    assert h[0] == 0.0
    assert abs(h[1] - T * T * (E - 1) / E ** 2) < 1e-9
    assert abs(h[2] - C * C * (E - 1) / E ** 2) < 1e-9
    assert abs(h[3] - (1 - C / T)) < 1e-15


def test_health_capacity_example_wrblog_s4_2():
    # §4.2: demand (6, 2) with C = 4 keeps (4, 2): 2 of 8 slots overflow.
    g = golden("wrblog_s4_2_capacity_example.json")
    case = g["cases"][0]
    counts = np.array(case["expert_one_based_demand"], np.int32)
    kept = np.array(case["kept"], np.int32)
    h = oracle.routing_health(counts, kept, g["T"], g["k"])
    assert abs(h[0] - -(0.75 * math.log(0.75) + 0.25 * math.log(0.25))) < 1e-12
    assert abs(h[1] - 4.0) < 1e-12    # mean 4: (2² + 2²)/2
    assert abs(h[2] - 1.0) < 1e-12    # mean 3: (1² + 1²)/2
    assert abs(h[3] - 0.25) < 1e-15


def test_health_against_library_routines():
    rng = np.random.default_rng(5)
    E, T, k = 37, 1000, 3
    ids = rng.integers(0, E, size=T * k)
    counts = np.bincount(ids, minlength=E).astype(np.int32)
    kept = np.minimum(counts, 90).astype(np.int32)
    h = oracle.routing_health(counts, kept, T, k)
    assert abs(h[0] - scipy.stats.entropy(counts / (T * k))) < 1e-12
    assert abs(h[1] - np.var(counts.astype(np.float64))) < 1e-9
    assert abs(h[2] - np.var(kept.astype(np.float64))) < 1e-9
    assert abs(h[3] - (1 - kept.sum() / (T * k))) < 1e-15
