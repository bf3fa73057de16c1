"""Pins of the oracle's dynamic tree construction (no GPU).

Source: "SGLang EAGLE-2 Speculative Decoding" (Tech Radar), section 2: the
entropy H = -sum P log P of the draft distribution; low entropy extends one
branch, high entropy widens the tree up to 8 nodes; per depth, beam search
prunes the low branches; at most 64 nodes.  The pins come from outside the
oracle: closed-form entropies, scipy's entropy and log-softmax, a stable
numpy sort, brute-force enumeration of the candidates, a hand-worked
two-level example (tests/golden/expand_example.txt) and structural invariants
of the grown tree.
"""
import math

import numpy as np
import pytest
from scipy import special, stats

import oracle
from eagle_speculative_decoding_attn_gb300 import workloads as W
from golden_io import read_fixture


# --------------------------------------------------------------------------
# entropy and width
# --------------------------------------------------------------------------
@pytest.mark.parametrize("k", [1, 2, 3, 5, 8, 13])
def test_entropy_of_k_equal_tokens_is_ln_k(k):
    z = np.full(40, -400.0)
    z[np.arange(k) * 3] = 1.5
    assert oracle.draft_entropy(z) == pytest.approx(math.log(k), abs=1e-12)


@pytest.mark.parametrize("p", [0.5, 0.9, 0.99, 0.2])
def test_entropy_of_two_point_distribution(p):
    z = np.array([math.log(p), math.log(1 - p)])
    assert oracle.draft_entropy(z) == pytest.approx(-p * math.log(p) - (1 - p) * math.log(1 - p), abs=1e-13)


def test_entropy_matches_scipy():
    rng = np.random.default_rng(3)
    for _ in range(20):
        z = rng.standard_normal(rng.integers(2, 3000)) * rng.uniform(0.1, 5)
        assert oracle.draft_entropy(z) == pytest.approx(stats.entropy(special.softmax(z)), rel=1e-12, abs=1e-13)


def test_entropy_shift_invariant_and_one_hot():
    rng = np.random.default_rng(4)
    z = rng.standard_normal(500)
    assert oracle.draft_entropy(z + 123.0) == pytest.approx(oracle.draft_entropy(z), abs=1e-11)
    z = np.zeros(100)
    z[7] = 1000.0
    assert oracle.draft_entropy(z) == 0.0


@pytest.mark.parametrize("top_k", range(1, 9))
def test_width_of_k_equal_tokens(top_k):
    # e^H = k exactly: k children up to the cap
    for k in range(1, 12):
        z = np.full(30, -500.0)
        z[:k] = 0.0
        assert oracle.branch_width(oracle.draft_entropy(z), top_k) == min(k, top_k)


def test_width_is_nearest_integer_of_perplexity():
    rng = np.random.default_rng(5)
    for H in rng.uniform(0.0, 3.0, size=2000):
        ppl = math.exp(H)
        if abs(ppl - math.floor(ppl) - 0.5) < 1e-9:
            continue
        expect = min(8, max(1, int(math.floor(ppl + 0.5))))
        assert oracle.branch_width(H, 8) == expect
    # the two ends of the pages' statement
    assert oracle.branch_width(0.0, 8) == 1
    assert oracle.branch_width(math.log(32000), 8) == 8


# --------------------------------------------------------------------------
# top-k expansion
# --------------------------------------------------------------------------
def test_top_tokens_equals_stable_sort():
    rng = np.random.default_rng(6)
    for _ in range(50):
        V = int(rng.integers(1, 60))
        z = np.round(rng.standard_normal(V), 1)  # many equal values
        w = int(rng.integers(1, 9))
        expect = np.argsort(-z, kind="stable")[:w].tolist()
        assert oracle.top_tokens(z, w) == expect


# --------------------------------------------------------------------------
# one level against brute force
# --------------------------------------------------------------------------
def _brute_force_level(rows, parents, tokens, scores, n, ls, top_k, max_new, budget):
    """Every candidate written out with scipy's log-softmax, sorted by Python's
    sorted(); the kept ones re-sorted into (parent, rank) order."""
    cands = []
    for f in range(ls, n):
        lp = special.log_softmax(rows[f].astype(np.float64))
        H = float(stats.entropy(np.exp(lp)))
        w = min(top_k, max(1, int(math.floor(math.exp(H) + 0.5))))
        order = np.argsort(-rows[f].astype(np.float64), kind="stable")[:w]
        for r, t in enumerate(order):
            cands.append((scores[f] + lp[t], f, r, int(t)))
    keep = min(max_new, budget - n, len(cands))
    best = sorted(cands, key=lambda c: (-c[0], c[1], c[2]))[:max(keep, 0)]
    best.sort(key=lambda c: (c[1], c[2]))
    P, T, S = parents.copy(), tokens.copy(), scores.copy()
    for k, (s, f, _r, t) in enumerate(best):
        P[n + k], T[n + k], S[n + k] = f, t, s
    return P, T, S, n + max(keep, 0)


@pytest.mark.parametrize("seed", range(12))
def test_level_equals_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    n_max, V = 64, int(rng.integers(5, 40))
    top_k = int(rng.integers(1, 9))
    max_new = int(rng.integers(1, 20))
    budget = int(rng.integers(8, n_max + 1))
    # a random current tree grown level by level
    n = int(rng.integers(1, 8))
    ls = int(rng.integers(0, n + 1)) if n > 1 else 0
    parents = np.full((1, n_max), -1, dtype=np.int32)
    for i in range(1, n):
        parents[0, i] = rng.integers(0, i)
    tokens = rng.integers(0, V, size=(1, n_max)).astype(np.int32)
    scores = np.zeros((1, n_max))
    scores[0, 1:n] = -rng.uniform(0, 5, size=n - 1)
    rows = (rng.standard_normal((1, n_max, V)) * rng.uniform(0.3, 4)).astype(np.float32)
    rows[0, :, ::3] = np.round(rows[0, :, ::3])  # equal logits for the tie rules
    out = oracle.tree_expand_level(rows, parents, tokens, scores, np.array([n]), np.array([ls]), top_k, max_new,
                                   budget)
    P, T, S, n_new = _brute_force_level(rows[0], parents[0], tokens[0], scores[0], n, ls, top_k, max_new, budget)
    assert out["status"][0] == 0
    assert out["n_nodes"][0] == n_new
    assert out["level_start"][0] == n
    assert out["parents"][0].tolist() == P.tolist()
    assert out["tokens"][0].tolist() == T.tolist()
    np.testing.assert_allclose(out["scores"][0], S, rtol=0, atol=1e-12)


def test_level_hand_worked_example():
    fx = read_fixture("expand_example.txt")
    V, top_k = int(fx["V"][0]), int(fx["top_k"][0])
    rows = np.zeros((1, 8, V))
    for f in range(4):
        rows[0, f] = [float(x) for x in fx[f"row{f}"]]
    ints = lambda key: [int(x) for x in fx[key]]
    floats = lambda key: [float(x) for x in fx[key]]
    st = dict(parents=np.full((1, 8), -1, np.int32), tokens=np.zeros((1, 8), np.int32),
              scores=np.zeros((1, 8)), n_nodes=np.array([1]), level_start=np.array([0]))
    l1 = oracle.tree_expand_level(rows, st["parents"], st["tokens"], st["scores"], st["n_nodes"],
                                  st["level_start"], top_k, 3, 8)
    assert l1["n_nodes"][0] == 4 and l1["level_start"][0] == 1
    assert l1["parents"][0, :4].tolist() == ints("level1_parents")
    assert l1["tokens"][0, :4].tolist() == ints("level1_tokens")
    np.testing.assert_allclose(l1["scores"][0, :4], floats("level1_scores"), atol=1e-12)
    for case, budget, n_new in (("caseA", 8, 8), ("caseB", 6, 6)):
        l2 = oracle.tree_expand_level(rows, l1["parents"], l1["tokens"], l1["scores"], l1["n_nodes"],
                                      l1["level_start"], top_k, 4, budget)
        assert l2["n_nodes"][0] == int(fx[f"{case}_n_nodes"][0]) == n_new
        assert l2["level_start"][0] == 4
        assert l2["parents"][0, :n_new].tolist() == ints(f"{case}_parents")
        assert l2["tokens"][0, :n_new].tolist() == ints(f"{case}_tokens")
        if case == "caseA":
            np.testing.assert_allclose(l2["scores"][0, :n_new], floats("caseA_scores"), atol=1e-9)
        H = np.concatenate([l1["entropy"][0, :1], l2["entropy"][0, 1:4]])
        np.testing.assert_allclose(H, floats("entropy"), atol=1e-9)
        W_ = np.concatenate([l1["width"][0, :1], l2["width"][0, 1:4]])
        assert W_.tolist() == ints("width")


# --------------------------------------------------------------------------
# whole trees
# --------------------------------------------------------------------------
def _depths(p, n):
    d = [0] * n
    for i in range(1, n):
        d[i] = d[p[i]] + 1
    return d


def test_peaked_rows_grow_a_chain():
    rng = np.random.default_rng(7)
    V, n_max, levels = 300, 16, 6
    rows = rng.standard_normal((1, n_max, V)).astype(np.float32)
    spikes = rng.integers(0, V, size=n_max)
    rows[0, np.arange(n_max), spikes] += 40.0
    out = oracle.tree_build_dynamic(rows, [5], levels, 8, 16, n_max)
    n = levels + 1
    assert out["n_nodes"][0] == n
    assert out["parents"][0, :n].tolist() == list(range(-1, n - 1))
    assert out["tokens"][0, 1:n].tolist() == spikes[: n - 1].tolist()
    assert np.all(out["width"][0, :levels] == 1)
    assert abs(out["scores"][0, n - 1]) < 1e-9


def test_fully_kept_levels_give_every_node_its_width():
    rng = np.random.default_rng(8)
    V, n_max = 50, 64
    rows = (rng.standard_normal((1, n_max, V)) * rng.uniform(0.2, 6, size=(1, n_max, 1))).astype(np.float32)
    out = oracle.tree_build_dynamic(rows, [0], 2, 3, 64, 64)   # at most 1 + 3 + 9 nodes: nothing pruned
    n = int(out["n_nodes"][0])
    kids = [0] * n
    for i in range(1, n):
        kids[out["parents"][0, i]] += 1
    for f in range(int(out["level_start"][0])):
        assert kids[f] == out["width"][0, f]


@pytest.mark.parametrize("seed", range(4))
def test_tree_invariants(seed):
    wl = W.make_expand_workload(3, 64, 700, seed=seed, n_levels=6, max_new=16)
    out = oracle.tree_build_dynamic(wl.draft_logits, wl.root_tokens, wl.n_levels, wl.top_k, wl.max_new,
                                    wl.budget)
    for b in range(wl.B):
        n = int(out["n_nodes"][b])
        p = out["parents"][b]
        assert 1 <= n <= wl.budget and p[0] == -1
        assert all(0 <= p[i] < i for i in range(1, n))
        d = _depths(p, n)
        assert max(d) <= wl.n_levels
        # nodes appear level by level, at most max_new per level
        assert d == sorted(d)
        for lv in range(1, max(d) + 1):
            assert d.count(lv) <= wl.max_new
        # siblings are contiguous and ordered by probability; at most w_f of them
        kids = [[] for _ in range(n)]
        for i in range(1, n):
            kids[p[i]].append(i)
        for f in range(n):
            ks = kids[f]
            if not ks:
                continue
            assert ks == list(range(ks[0], ks[0] + len(ks)))
            assert len(ks) <= out["width"][b, f]
            lp = special.log_softmax(wl.draft_logits[b, f].astype(np.float64))
            toks = [int(out["tokens"][b, c]) for c in ks]
            assert toks == np.argsort(-wl.draft_logits[b, f].astype(np.float64), kind="stable")[: len(ks)].tolist()
            # a node's score is the log of the product of the probabilities on its path
            for c in ks:
                assert out["scores"][b, c] == pytest.approx(out["scores"][b, f] + lp[out["tokens"][b, c]], abs=1e-12)
        for i in range(n):
            logp, j = 0.0, i
            while j != 0:
                logp += special.log_softmax(wl.draft_logits[b, p[j]].astype(np.float64))[out["tokens"][b, j]]
                j = p[j]
            assert out["scores"][b, i] == pytest.approx(logp, abs=1e-9)


def test_invalid_state_and_full_budget():
    rows = np.zeros((3, 8, 10), dtype=np.float32)
    parents = np.full((3, 8), -1, np.int32)
    parents[2, 1:8] = [0, 0, 1, 1, 2, 2, 3]
    tokens = np.zeros((3, 8), np.int32)
    scores = np.zeros((3, 8))
    n = np.array([0, 3, 8], np.int32)
    ls = np.array([0, 4, 3], np.int32)
    out = oracle.tree_expand_level(rows, parents, tokens, scores, n, ls, 8, 4, 8)
    assert out["status"].tolist() == [oracle.STATUS_BAD_TREE, oracle.STATUS_BAD_TREE, 0]
    assert out["n_nodes"].tolist() == [0, 3, 8]
    # budget reached: nothing added, the frontier empties
    assert out["level_start"][2] == 8
    assert out["parents"][2].tolist() == parents[2].tolist()


def test_equal_scores_keep_lower_parent_then_lower_rank():
    # two frontier nodes with equal scores and the same uniform row: four
    # candidates of one score; keeping 2 takes both of node 1's (lower f
    # before lower rank)
    rows = np.zeros((1, 8, 6), dtype=np.float32)
    rows[0, 1, 2:] = -300.0     # node 1: tokens 0, 1 equally likely
    rows[0, 2, 2:] = -300.0     # node 2: the same
    parents = np.array([[-1, 0, 0, -1, -1, -1, -1, -1]], np.int32)
    tokens = np.zeros((1, 8), np.int32)
    scores = np.array([[0.0, -1.0, -1.0, 0, 0, 0, 0, 0]])
    out = oracle.tree_expand_level(rows, parents, tokens, scores, np.array([3]), np.array([1]), 8, 2, 8)
    assert out["width"][0, 1:3].tolist() == [2, 2]
    assert out["n_nodes"][0] == 5
    assert out["parents"][0, 3:5].tolist() == [1, 1]
    assert out["tokens"][0, 3:5].tolist() == [0, 1]
    assert out["near_boundary"][0]          # a cut between equal scores is flagged
