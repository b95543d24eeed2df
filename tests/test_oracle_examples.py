"""Pins for the CPU oracle: the articles' worked examples, closed forms and
special cases that reduce to library routines.  CPU only.

Each expected value below comes from a worked example printed in the
articles (fixtures under tests/golden/, each citing its section), from exact
arithmetic (fractions), or from an independent library computation (numpy /
torch / scipy in float64) — never from the oracle itself.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def two_expert_logits(routing0):
    """Scores giving p = (0.6, 0.4) for tokens routed to expert 0, (0.4, 0.6) else."""
    s = np.empty((len(routing0), 2), np.float32)
    for t, e in enumerate(routing0):
        s[t] = (math.log(0.6), math.log(0.4)) if e == 0 else (math.log(0.4), math.log(0.6))
    return s


# --- MoE 模型原理 §4.2: T=8, E=2, top-1, routing [1,1,1,1,1,1,2,2] ----------------

def test_capacity_example_wrblog_s4_2():
    g = golden("wrblog_s4_2_capacity_example.json")
    routing0 = [r - 1 for r in g["routing_one_based"]]
    ids, w, psum, _ = oracle.select(two_expert_logits(routing0), k=1, renormalize=True)
    assert ids[:, 0].tolist() == routing0
    for case in g["cases"]:
        C = oracle.capacity(g["T"], g["k"], g["E"], case["c"])
        assert C == case["C"]
        fl = oracle.fill(ids, g["E"], C)
        assert fl["kept"].tolist() == case["kept"]
        assert fl["counts"].tolist() == [6, 2]
        dropped = [t for t in range(g["T"]) if fl["slot_row"][t, 0] < 0]
        if case["C"] == 4:
            # the first four expert-1 tokens are kept, the last two overflow
            assert dropped == [4, 5]
            assert fl["row_token"].tolist() == [0, 1, 2, 3, 6, 7]
        else:
            assert dropped == []


def test_aux_example_wrblog_s3_3():
    g = golden("wrblog_s3_3_aux_example.json")
    routing0 = [0, 0, 0, 0, 0, 0, 1, 1]
    ids, w, psum, _ = oracle.select(two_expert_logits(routing0), k=1, renormalize=True)
    fl = oracle.fill(ids, 2, oracle.capacity(8, 1, 2, 1.0))
    for alpha in (1.0, 0.01):
        f, pbar, l_aux = oracle.aux(fl["counts"], psum, 8, alpha)
        np.testing.assert_allclose(f, g["f"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(pbar, g["pbar"], rtol=1e-7)
        assert abs(float(np.dot(f, pbar)) - g["sum_f_pbar"]) < 1e-7
        assert abs(l_aux - g["l_aux_over_alpha"] * alpha) < 1e-7 * max(alpha, 1)
    # exactly, from the printed f and p̄ (counts 6,2 and Σp = T·p̄)
    f, pbar, l_aux = oracle.aux(np.array([6, 2]), np.array([4.4, 3.6]), 8, 1.0)
    assert abs(l_aux - 1.05) < 1e-12


@pytest.mark.parametrize("E,k", [(2, 1), (8, 1), (16, 1), (8, 2), (8, 4)])
def test_uniform_routing_gives_alpha(E, k):
    """§3.2: f_i = p̄_i = 1/E gives L_aux = α for top-1; with f_i = (1/T)Σ1[i∈S_t]
    read literally, top-k uniform routing gives Σ f = k and L_aux = k·α."""
    g = golden("wrblog_s3_3_aux_example.json")
    T = 4 * E
    # round-robin scores: token t prefers experts t, t+1, ... with equal
    # softmax mass per expert over the whole batch
    s = np.zeros((T, E), np.float32)
    for t in range(T):
        for j in range(E):
            s[t, (t + j) % E] = float(E - j)
    ids, w, psum, _ = oracle.select(s, k=k, renormalize=True)
    fl = oracle.fill(ids, E, oracle.capacity(T, k, E, 1.0))
    alpha = 0.01
    f, pbar, l_aux = oracle.aux(fl["counts"], psum, T, alpha)
    np.testing.assert_allclose(f, np.full(E, k / E), rtol=1e-15)
    np.testing.assert_allclose(pbar, np.full(E, 1 / E), rtol=1e-12)
    assert abs(l_aux - k * alpha * g["uniform_l_aux_over_alpha"]) < 1e-12


# --- 111qqz EP article: the A–H routing table -------------------------------------

def test_ep_forward_table_regroups():
    g = golden("111qqz_ep_forward_table.json")
    T, E = 8, 8
    ids = np.array(g["expert"], np.int32)[:, None]
    C = oracle.capacity(T, 1, E, 1.0)
    assert C == 1
    fl = oracle.fill(ids, E, C)
    names = g["tokens"]
    per = g["experts_per_gpu"]
    for gpu, expect in g["after_dispatch"].items():
        gi = int(gpu)
        rows = range(fl["offsets"][gi * per], fl["offsets"][(gi + 1) * per])
        got = [names[fl["row_token"][r]] for r in rows]
        assert sorted(got) == sorted(expect)  # within a group the buffer is in expert order
        for r in rows:
            e = int(np.searchsorted(fl["offsets"], r, side="right") - 1)
            assert g["expert_of_token_after_dispatch"][names[fl["row_token"][r]]] == e
    dest = [fl["offsets"].searchsorted(fl["slot_row"][t, 0], side="right") - 1 for t in range(T)]
    cross = [names[t] for t in range(T) if dest[t] // per != g["source_gpu"][t]]
    assert cross == g["cross_gpu_tokens"]
    n_gpu = T // per
    assert (T // n_gpu) * (n_gpu - 1) * n_gpu == g["allgather_payloads"]
    assert len(cross) == g["all_to_all_payloads"]


def test_capacity_dropping_111qqz():
    g = golden("111qqz_capacity_dropping.json")
    T, E = g["T"], g["E"]
    rng = np.random.default_rng(0)
    ids = np.where(np.arange(T) < g["hot_tokens"], g["hot_expert"], 0)
    others = rng.integers(0, E - 1, size=T)
    others[others >= g["hot_expert"]] += 1
    ids = np.where(np.arange(T) < g["hot_tokens"], g["hot_expert"], others)
    ids = rng.permutation(ids).astype(np.int32)[:, None]
    for case in g["cases"]:
        C = oracle.capacity(T, g["k"], E, case["cf"])
        assert C == case["C"]
        fl = oracle.fill(ids, E, C)
        assert fl["counts"][g["hot_expert"]] == g["hot_tokens"]
        assert fl["counts"][g["hot_expert"]] - fl["kept"][g["hot_expert"]] == case["overflow"]
        assert (fl["kept"] <= C).all()


# --- capacity: exact rational ceiling ----------------------------------------------

@pytest.mark.parametrize("c", [1.0, 1.25, 1.5, 2.0, 0.5, 1.1, 0.3, 1.0 + 2 ** -52, 3.75])
@pytest.mark.parametrize("T,k,E", [(512, 2, 8), (4096, 2, 8), (16384, 1, 8), (8192, 6, 64),
                                   (32768, 8, 256), (7, 3, 5), (1, 1, 1), (3 << 30, 1, 3)])
def test_capacity_is_exact_ceiling(T, k, E, c):
    expect = math.ceil(Fraction(c) * T * k / E)
    assert oracle.capacity(T, k, E, c) == expect


# --- §2.1/§2.2: softmax, top-k, weights against library routines ------------------

@pytest.mark.parametrize("E,k", [(8, 2), (64, 6), (256, 8), (5, 5), (3, 1)])
@pytest.mark.parametrize("renorm", [True, False])
def test_select_matches_library(E, k, renorm):
    rng = np.random.default_rng(E * 10 + k)
    T = 97
    s = rng.standard_normal((T, E)).astype(np.float32)
    s[::7, 1] = s[::7, 0]          # plant exact ties
    s[::11] = 0.25                 # and fully tied rows
    ids, w, psum, probs = oracle.select(s, k, renorm, want_probs=True)
    p = scipy.special.softmax(s.astype(np.float64), axis=1)
    np.testing.assert_allclose(probs, p, rtol=1e-13, atol=1e-300)
    # stable argsort of -s: descending score, equal scores in ascending index
    ref_ids = np.argsort(-s, axis=1, kind="stable")[:, :k]
    np.testing.assert_array_equal(ids, ref_ids)
    sel = np.take_along_axis(p, ref_ids, axis=1)
    ref_w = sel / sel.sum(axis=1, keepdims=True) if renorm else sel
    np.testing.assert_allclose(w, ref_w, rtol=1e-13)
    np.testing.assert_allclose(psum, p.sum(axis=0), rtol=1e-12)


def test_select_tie_lowest_index():
    s = np.zeros((3, 6), np.float32)
    s[1] = [1, 3, 3, 2, 3, 0]
    s[2] = [-1, -1, -1, -1, -1, -1]
    ids, *_ = oracle.select(s, 3, True)
    assert ids.tolist() == [[0, 1, 2], [1, 2, 4], [0, 1, 2]]


def test_top1_renormalised_weight_is_one_raw_weight_is_max_prob():
    """§2.3: top-1 output is E_{i*}(x) (weight 1); without renormalisation the
    weight is the raw max probability."""
    rng = np.random.default_rng(5)
    s = rng.standard_normal((50, 8)).astype(np.float32)
    _, w1, _, _ = oracle.select(s, 1, True)
    assert (w1 == 1.0).all()
    _, w0, _, _ = oracle.select(s, 1, False)
    np.testing.assert_allclose(w0[:, 0], scipy.special.softmax(s.astype(np.float64), 1).max(1),
                               rtol=1e-13)


# --- §2.1: router logits against a library matmul ----------------------------------

@pytest.mark.parametrize("bf16", [False, True])
def test_router_logits_match_matmul(bf16):
    g = torch.Generator().manual_seed(3)
    T, d, E = 33, 96, 12
    x = torch.randn(T, d, generator=g)
    Wr = torch.randn(E, d, generator=g) / math.sqrt(d)
    br = torch.randn(E, generator=g)
    if bf16:
        x, Wr = x.bfloat16(), Wr.bfloat16()
        xn = x.view(torch.int16).numpy().view(np.uint16)
        wn = Wr.view(torch.int16).numpy().view(np.uint16)
    else:
        xn, wn = x.numpy(), Wr.numpy()
    got = oracle.router_logits(xn, wn, br.numpy())
    ref = x.double().numpy() @ Wr.double().numpy().T + br.double().numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


# --- §1: the expert FFN reduces to a dense FFN for E=1, k=1 ------------------------

@pytest.mark.parametrize("act", [oracle.ACT_RELU, oracle.ACT_GELU_TANH])
def test_single_expert_is_dense_ffn(act):
    g = torch.Generator().manual_seed(11)
    T, d, d_ff = 40, 24, 56
    x = torch.randn(T, d, generator=g, dtype=torch.float64).float()
    Wr = torch.randn(1, d, generator=g).float()
    br = torch.zeros(1)
    W1 = torch.randn(1, d_ff, d, generator=g).float() / math.sqrt(d)
    b1 = torch.randn(1, d_ff, generator=g).float()
    W2 = torch.randn(1, d, d_ff, generator=g).float() / math.sqrt(d_ff)
    b2 = torch.randn(1, d, generator=g).float()
    out = oracle.forward(x.numpy(), Wr.numpy(), br.numpy(), W1.numpy(), b1.numpy(), W2.numpy(),
                         b2.numpy(), k=1, capacity_factor=1.0, renormalize=True, act=act)
    assert out["C"] == T and (out["slot_row"][:, 0] == np.arange(T)).all()
    xd = x.double()
    u = xd @ W1[0].double().T + b1[0].double()
    h = torch.relu(u) if act == oracle.ACT_RELU else torch.nn.functional.gelu(u, approximate="tanh")
    ref = h @ W2[0].double().T + b2[0].double()
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-12, atol=1e-12)


def test_activation_matches_torch():
    u = np.linspace(-9, 9, 2001)
    got = oracle.activation(u, oracle.ACT_GELU_TANH)
    ref = torch.nn.functional.gelu(torch.from_numpy(u), approximate="tanh").numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-14, atol=1e-15)
    np.testing.assert_array_equal(oracle.activation(u, oracle.ACT_RELU), np.maximum(u, 0))


# --- §2.2 with k = E and no drops: the dense soft mixture Σ_i p_i E_i(x) -----------

@pytest.mark.parametrize("act", [oracle.ACT_RELU, oracle.ACT_GELU_TANH])
def test_k_equals_E_is_soft_mixture(act):
    g = torch.Generator().manual_seed(17)
    T, d, d_ff, E = 21, 16, 40, 5
    x = torch.randn(T, d, generator=g)
    Wr = torch.randn(E, d, generator=g) / math.sqrt(d)
    br = torch.randn(E, generator=g)
    W1 = torch.randn(E, d_ff, d, generator=g) / math.sqrt(d)
    b1 = torch.randn(E, d_ff, generator=g)
    W2 = torch.randn(E, d, d_ff, generator=g) / math.sqrt(d_ff)
    b2 = torch.randn(E, d, generator=g)
    out = oracle.forward(x.numpy(), Wr.numpy(), br.numpy(), W1.numpy(), b1.numpy(), W2.numpy(),
                         b2.numpy(), k=E, capacity_factor=1.0, renormalize=True, act=act)
    assert out["C"] == T and (out["slot_row"] >= 0).all()
    X, s = x.double(), torch.from_numpy(out["logits"]).double()
    p = torch.softmax(s, dim=1)
    u = torch.einsum("td,efd->tef", X, W1.double()) + b1.double()[None]
    h = torch.relu(u) if act == oracle.ACT_RELU else torch.nn.functional.gelu(u, approximate="tanh")
    ye = torch.einsum("tef,edf->ted", h, W2.double()) + b2.double()[None]
    ref = torch.einsum("te,ted->td", p, ye)
    np.testing.assert_allclose(out["y"], ref.numpy(), rtol=1e-11, atol=1e-12)


# --- small integers: every step exact, so indexing is pinned bit for bit -----------

def test_small_integer_forward_is_exact():
    rng = np.random.default_rng(23)
    T, d, d_ff, E, k = 37, 8, 16, 4, 2
    x = rng.integers(-2, 3, (T, d)).astype(np.float32)
    Wr = rng.integers(-3, 4, (E, d)).astype(np.float32)
    br = np.zeros(E, np.float32)
    W1 = rng.integers(-2, 3, (E, d_ff, d)).astype(np.float32)
    b1 = rng.integers(-4, 5, (E, d_ff)).astype(np.float32)
    W2 = rng.integers(-2, 3, (E, d, d_ff)).astype(np.float32)
    b2 = rng.integers(-4, 5, (E, d)).astype(np.float32)
    out = oracle.forward(x, Wr, br, W1, b1, W2, b2, k=k, capacity_factor=0.75, renormalize=False,
                         act=oracle.ACT_RELU)
    xi = x.astype(np.int64)
    # independent integer evaluation per slot (mask formulation, no buffer)
    ids = out["topk_ids"]
    yd_tok = np.zeros((T, k, d), np.int64)
    for t in range(T):
        for r in range(k):
            e = ids[t, r]
            h = np.maximum(W1[e].astype(np.int64) @ xi[t] + b1[e].astype(np.int64), 0)
            yd_tok[t, r] = W2[e].astype(np.int64) @ h + b2[e].astype(np.int64)
    for row in range(out["offsets"][E]):
        t = out["row_token"][row]
        r = int(np.where(out["slot_row"][t] == row)[0][0])
        assert (out["yd"][row] == yd_tok[t, r]).all()
    kept = out["slot_row"] >= 0
    ref = np.einsum("tk,tkd->td", out["topk_w"] * kept, yd_tok.astype(np.float64))
    np.testing.assert_allclose(out["y"], ref, rtol=1e-15, atol=1e-12)


# --- the toy top-1 router of §7, restated: raw max-prob weight, zero on overflow ---

def test_toy_top1_semantics():
    g = torch.Generator().manual_seed(7)
    T, d, d_ff, E = 64, 4, 8, 2
    for cf in (1.0, 0.75, 1.5):
        x = torch.randn(T, d, generator=g)
        Wr = torch.randn(E, d, generator=g)
        W1 = torch.randn(E, d_ff, d, generator=g)
        b1 = torch.randn(E, d_ff, generator=g)
        W2 = torch.randn(E, d, d_ff, generator=g)
        b2 = torch.randn(E, d, generator=g)
        out = oracle.forward(x.numpy(), Wr.numpy(), np.zeros(E, np.float32), W1.numpy(),
                             b1.numpy(), W2.numpy(), b2.numpy(), k=1, capacity_factor=cf,
                             renormalize=False, act=oracle.ACT_RELU)
        s = torch.from_numpy(out["logits"]).double()
        probs = torch.softmax(s, -1)
        top_prob, top_idx = probs.max(-1)
        cap = math.ceil(Fraction(cf) * T / E)
        assert out["C"] == cap
        y = torch.zeros(T, d, dtype=torch.float64)
        kept = torch.zeros(T, dtype=torch.bool)
        for e in range(E):
            tok = torch.nonzero(top_idx == e).flatten()[:cap]
            h = torch.relu(x[tok].double() @ W1[e].double().T + b1[e].double())
            y[tok] += top_prob[tok, None] * (h @ W2[e].double().T + b2[e].double())
            kept[tok] = True
            assert out["kept"][e] == tok.numel() <= cap
        np.testing.assert_allclose(out["y"], y.numpy(), rtol=1e-12, atol=1e-12)
        assert int((out["slot_row"][:, 0] < 0).sum()) == int((~kept).sum())
        np.testing.assert_allclose(out["pbar"], probs.mean(0).numpy(), rtol=1e-12)


# --- token subsets give the same outputs as the whole batch -------------------------

def test_token_subset_matches_full():
    rng = np.random.default_rng(31)
    T, d, d_ff, E, k = 200, 16, 24, 6, 3
    x = rng.standard_normal((T, d)).astype(np.float32)
    Wr = rng.standard_normal((E, d)).astype(np.float32)
    br = np.linspace(1, -1, E).astype(np.float32)
    W1 = rng.standard_normal((E, d_ff, d)).astype(np.float32)
    W2 = rng.standard_normal((E, d, d_ff)).astype(np.float32)
    b1 = rng.standard_normal((E, d_ff)).astype(np.float32)
    b2 = rng.standard_normal((E, d)).astype(np.float32)
    kw = dict(k=k, capacity_factor=0.8, renormalize=True, act=oracle.ACT_GELU_TANH)
    full = oracle.forward(x, Wr, br, W1, b1, W2, b2, **kw)
    tokens = np.sort(rng.choice(T, 37, replace=False))
    sub = oracle.forward(x, Wr, br, W1, b1, W2, b2, tokens=tokens, **kw)
    np.testing.assert_array_equal(sub["y"], full["y"][tokens])
    assert (full["slot_row"] < 0).any()
