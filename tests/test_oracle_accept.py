"""Pins of the oracle's acceptance (no GPU).

Greedy: a hand-worked example (study note case 1: k hits emit k+1 tokens)
and brute force by simulated sequential greedy decoding down the tree.
Sampling: a hand-worked example, exact enumeration of the output
distribution on tiny vocabularies (the lossless property stated by
troisinh.com "Why it works" and the study note, case 3), and a chi-square
test of the walker driven by fresh uniforms.
"""
import itertools
import math
import zlib

import numpy as np
import pytest
from scipy import stats

import oracle
from eagle_speculative_decoding_attn_gb300 import workloads as W
from golden_io import read_fixture


# --------------------------------------------------------------------------
# greedy
# --------------------------------------------------------------------------
def test_greedy_hand_worked_example():
    fx = read_fixture("greedy_example.txt")
    parents = np.array([int(x) for x in fx["parents"]], dtype=np.int32)
    tokens = np.array([int(x) for x in fx["tokens"]], dtype=np.int32)
    tokens[0] = 0
    logits = np.array([[float(x) for x in r] for r in fx["logits"]], dtype=np.float32)
    n = len(parents)
    res = oracle.tree_accept_greedy(logits[None], tokens[None], parents[None], np.array([n]))
    a = int(fx["accept_len"][0])
    assert res["accept_len"][0] == a
    assert res["path_nodes"][0, : a + 1].tolist() == [int(x) for x in fx["path"]]
    assert res["path_nodes"][0, a + 1:].tolist() == [-1] * (n - a - 1)
    assert res["out_tokens"][0, : a + 1].tolist() == [int(x) for x in fx["out_tokens"]]
    assert res["out_tokens"][0, a + 1:].tolist() == [-1] * (n - a)


def _greedy_by_decoding(logits, tokens, parents, n):
    """Brute force: follow greedy decoding from the root; at each node the
    target's next token is argmax of its row; descend into every child that
    drafted that token (depth-first) and keep the longest run (lowest node
    index among equally long runs)."""
    kids = [[] for _ in range(n)]
    for c in range(1, n):
        kids[parents[c]].append(c)
    best = (0, 0)   # (depth, -node) maximised lexicographically -> deepest, lowest index

    def visit(node, depth):
        nonlocal best
        if (depth, -node) > (best[0], -best[1]):
            best = (depth, node)
        nxt = int(np.argmax(logits[node]))
        for c in kids[node]:
            if tokens[c] == nxt:
                visit(c, depth + 1)

    visit(0, 0)
    return best


@pytest.mark.parametrize("n,V", [(1, 3), (2, 2), (8, 3), (20, 2), (64, 3), (64, 4)])
def test_greedy_matches_simulated_decoding(n, V):
    rng = np.random.Generator(np.random.PCG64(100 + n + V))
    for _ in range(30):
        p = W.random_recursive_tree(rng, n)
        toks = rng.integers(0, V, size=n).astype(np.int32)
        logits = rng.integers(0, 3, size=(n, V)).astype(np.float32)   # many ties on purpose
        res = oracle.tree_accept_greedy(logits[None], toks[None], p[None], np.array([n]))
        depth, node = _greedy_by_decoding(logits, toks, p, n)
        a = int(res["accept_len"][0])
        assert a == depth
        path = res["path_nodes"][0, : a + 1].tolist()
        assert path[-1] == node and path[0] == 0
        # the path is node's root-to-node chain
        for k in range(1, a + 1):
            assert p[path[k]] == path[k - 1]
        emitted = res["out_tokens"][0, : a + 1].tolist()
        assert emitted[:a] == [int(toks[c]) for c in path[1:]]
        assert emitted[a] == int(np.argmax(logits[node]))
        assert res["out_tokens"][0, a + 1:].tolist() == [-1] * (n - a)


def test_greedy_rejects_bad_token():
    p = W.chain_tree(3)
    toks = np.array([0, 5, 1], dtype=np.int32)
    res = oracle.tree_accept_greedy(np.zeros((1, 3, 4), np.float32), toks[None], p[None], np.array([3]))
    assert res["status"][0] == oracle.STATUS_BAD_TOKEN


# --------------------------------------------------------------------------
# sampling
# --------------------------------------------------------------------------
def test_sampling_hand_worked_example():
    fx = read_fixture("sampling_example.txt")
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([0.2, 0.6, 0.2])
    tl = np.log(p).astype(np.float32)
    dl = np.log(q).astype(np.float32)
    np.testing.assert_allclose(oracle.softmax_t(tl, 1.0), p, rtol=1e-6)
    cur_list, final = oracle.node_plan(p, q, [int(fx["child_token"][0])])
    x = int(fx["child_token"][0])
    assert cur_list[0][x] / q[x] == pytest.approx(float(fx["accept_prob"][0]))
    np.testing.assert_allclose(final, [float(v) for v in fx["residual_after_reject"]], atol=1e-15)
    # full walk on a root + one leaf child
    parents = np.array([[-1, 0]], dtype=np.int32)
    tokens = np.array([[0, x]], dtype=np.int32)
    T = np.stack([tl, tl])[None]
    D = np.stack([dl, dl])[None]
    for case in fx["case"]:
        ua = np.array([[0.0, float(case["u_accept"])]], dtype=np.float32)
        for us in [0.01, 0.45, 0.6, 0.99]:
            usamp = np.full((1, 2), us, dtype=np.float32)
            r = oracle.tree_accept_sampling(T, D, tokens, parents, np.array([2]), 1.0, ua, usamp)
            assert r["accept_len"][0] == int(case["accepted"])
            if int(case["accepted"]) == 0:
                assert r["out_tokens"][0, 0] == int(case["bonus"])
            else:
                assert r["out_tokens"][0, 0] == x
                # the leaf's bonus comes from its unmodified p = [0.5, 0.3, 0.2]
                expect = 0 if us < 0.5 else (1 if us < 0.8 else 2)
                assert r["out_tokens"][0, 1] == expect


def _exact_first_token_dist(p, q, width):
    """P(first emitted token = v) by enumerating every i.i.d. draw of the
    ``width`` children tokens from q and every accept/reject branch, using the
    oracle's per-node plan for the acceptance probabilities."""
    V = len(p)
    dist = np.zeros(V)
    for toks in itertools.product(range(V), repeat=width):
        w_draw = np.prod([q[t] for t in toks])
        cur_list, final = oracle.node_plan(p, q, list(toks))
        reach = 1.0
        for x, cur in zip(toks, cur_list):
            a = min(1.0, cur[x] / q[x]) if q[x] > 0 else (1.0 if cur[x] > 0 else 0.0)
            dist[x] += w_draw * reach * a
            reach *= 1.0 - a
        dist += w_draw * reach * final
    return dist


@pytest.mark.parametrize("V,width,seed", [(2, 1, 0), (3, 2, 1), (3, 3, 2), (4, 3, 3), (5, 2, 4),
                                          (3, 4, 5)])
def test_sampling_first_token_is_exactly_target(V, width, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    for _ in range(5):
        p = oracle.softmax_t(rng.normal(0, 2, V), 1.0)
        q = oracle.softmax_t(rng.normal(0, 2, V), 1.0)
        dist = _exact_first_token_dist(p, q, width)
        np.testing.assert_allclose(dist, p, rtol=0, atol=1e-12)


def test_sampling_exact_with_zero_probabilities():
    p = np.array([0.0, 0.7, 0.3, 0.0])
    q = np.array([0.5, 0.0, 0.25, 0.25])
    for width in (1, 2, 3):
        np.testing.assert_allclose(_exact_first_token_dist(p, q, width), p, atol=1e-12)
    # identical p and q: the residual is empty and the plan keeps p
    np.testing.assert_allclose(_exact_first_token_dist(q, q, 2), q, atol=1e-12)


def _lm_rows(prefix_tokens, V, seed, kind):
    """Toy language model: logits depend only on the token path (so two nodes
    with the same context get the same distribution)."""
    h = zlib.crc32(repr((seed, kind, tuple(int(t) for t in prefix_tokens))).encode())
    r = np.random.Generator(np.random.PCG64(h))
    return r.normal(0, 1.5, V)


def test_sampling_second_token_given_accepted_child_is_child_target():
    """Depth-2 trees drawn i.i.d. from q at every node: conditional on the
    first emitted token being an accepted draft x, the next emitted token is
    distributed as the target at context (x,), by exact enumeration over all
    drafts and decisions of the oracle's plan."""
    V, width, seed = 3, 2, 77
    p0 = oracle.softmax_t(_lm_rows((), V, seed, "t"), 1.0)
    q0 = oracle.softmax_t(_lm_rows((), V, seed, "d"), 1.0)
    joint = np.zeros((V, V))     # P(first = x via acceptance, second = y)
    acc_mass = np.zeros(V)
    for toks in itertools.product(range(V), repeat=width):
        w0 = np.prod([q0[t] for t in toks])
        cur_list, _ = oracle.node_plan(p0, q0, list(toks))
        reach = 1.0
        for x, cur in zip(toks, cur_list):
            a = min(1.0, cur[x] / q0[x])
            m = w0 * reach * a
            acc_mass[x] += m
            p1 = oracle.softmax_t(_lm_rows((x,), V, seed, "t"), 1.0)
            q1 = oracle.softmax_t(_lm_rows((x,), V, seed, "d"), 1.0)
            joint[x] += m * _exact_first_token_dist(p1, q1, width)
            reach *= 1.0 - a
    for x in range(V):
        p1 = oracle.softmax_t(_lm_rows((x,), V, seed, "t"), 1.0)
        np.testing.assert_allclose(joint[x] / acc_mass[x], p1, atol=1e-12)


def _random_draw_tree(rng, V, T, width, depth, seed):
    """A full tree of the given width/depth whose children tokens are drawn
    i.i.d. from the toy LM's draft at T; returns the batch arrays."""
    parents, tokens, ctx = [-1], [0], [()]
    frontier = [0]
    for _ in range(depth):
        nxt = []
        for n in frontier:
            qd = oracle.softmax_t(_lm_rows(ctx[n], V, seed, "d"), T)
            for _ in range(width):
                x = int(rng.choice(V, p=qd))
                parents.append(n)
                tokens.append(x)
                ctx.append(ctx[n] + (x,))
                nxt.append(len(parents) - 1)
        frontier = nxt
    n = len(parents)
    tl = np.stack([_lm_rows(c, V, seed, "t") for c in ctx]).astype(np.float32)
    dl = np.stack([_lm_rows(c, V, seed, "d") for c in ctx]).astype(np.float32)
    return (np.array(parents, np.int32), np.array(tokens, np.int32), tl, dl, n)


def test_sampling_walker_chi_square():
    """The walker, fed fresh uniforms and freshly drafted trees, emits a first
    token distributed as the (float32-rounded) target at the root."""
    V, T, seed = 4, 0.8, 5
    rng = np.random.Generator(np.random.PCG64(12345))
    counts = np.zeros(V)
    n_draws = 6000
    for _ in range(n_draws):
        parents, tokens, tl, dl, n = _random_draw_tree(rng, V, T, width=2, depth=2, seed=seed)
        ua = rng.random((1, n), dtype=np.float32)
        us = rng.random((1, n), dtype=np.float32)
        r = oracle.tree_accept_sampling(tl[None], dl[None], tokens[None], parents[None],
                                        np.array([n]), T, ua, us)
        counts[r["out_tokens"][0, 0]] += 1
    p_root = oracle.softmax_t(tl[0], T)
    chi2, pval = stats.chisquare(counts, n_draws * p_root)
    assert pval > 1e-4, (counts, n_draws * p_root, pval)


def test_sampling_leaf_root_bonus_from_target():
    """A root without children emits one token drawn from p by inverse CDF."""
    tl = np.log(np.array([[0.1, 0.2, 0.3, 0.4]], dtype=np.float64)).astype(np.float32)
    parents = np.array([[-1]], np.int32)
    tokens = np.zeros((1, 1), np.int32)
    cdf = np.cumsum([0.1, 0.2, 0.3, 0.4])
    for u in [0.05, 0.15, 0.29, 0.31, 0.59, 0.61, 0.95]:
        r = oracle.tree_accept_sampling(tl[None], tl[None], tokens, parents, np.array([1]), 1.0,
                                        np.zeros((1, 1), np.float32),
                                        np.full((1, 1), u, np.float32))
        assert r["accept_len"][0] == 0
        assert r["out_tokens"][0, 0] == int(np.searchsorted(cdf, np.float32(u), side="right"))


def test_inverse_cdf_never_picks_zero_weight():
    w = np.array([0.0, 0.5, 0.0, 0.5, 0.0])
    for u in np.linspace(0, 0.999999, 101):
        j, _ = oracle.inverse_cdf(w, u)
        assert w[j] > 0


def test_near_boundary_flag():
    p = np.array([0.5, 0.3, 0.2])
    q = np.array([0.2, 0.6, 0.2])
    tl = np.log(p).astype(np.float32)
    dl = np.log(q).astype(np.float32)
    parents = np.array([[-1, 0]], np.int32)
    tokens = np.array([[0, 1]], np.int32)
    T = np.stack([tl, tl])[None]
    D = np.stack([dl, dl])[None]
    ratio = oracle.softmax_t(tl, 1.0)[1] / oracle.softmax_t(dl, 1.0)[1]
    r = oracle.tree_accept_sampling(T, D, tokens, parents, np.array([2]), 1.0,
                                    np.array([[0.0, ratio + 2e-7]], np.float32),
                                    np.full((1, 2), 0.3, np.float32))
    assert bool(r["near_boundary"][0])
    r = oracle.tree_accept_sampling(T, D, tokens, parents, np.array([2]), 1.0,
                                    np.array([[0.0, 0.9]], np.float32),
                                    np.full((1, 2), 0.3, np.float32))
    assert not bool(r["near_boundary"][0])


def test_workload_sampling_configs_run():
    w = W.make_workload("tiny")
    r = oracle.tree_accept_sampling(w.target_logits, w.draft_logits, w.tokens, w.parents,
                                    w.n_nodes, w.temperature, w.u_accept, w.u_sample)
    assert r["status"][0] == 0
    a = int(r["accept_len"][0])
    assert 0 <= a <= 3
    g = oracle.tree_accept_greedy(w.target_logits, w.tokens, w.parents, w.n_nodes)
    assert g["status"][0] == 0


# --------------------------------------------------------------------------
# siblings drafted without replacement
# --------------------------------------------------------------------------
def test_wor_hand_worked_example():
    fx = read_fixture("sampling_wor_example.txt")
    p = np.array([float(v) for v in fx["p"]])
    q = np.array([float(v) for v in fx["q"]])
    kids = [int(v) for v in fx["children"]]
    plans, final = oracle.node_plan_wor(p, q, kids)
    acc = [min(1.0, cur[x] / qk[x]) for x, (cur, qk) in zip(kids, plans)]
    np.testing.assert_allclose(acc, [float(v) for v in fx["accept_prob"]], atol=1e-15)
    np.testing.assert_allclose(plans[1][0], [float(v) for v in fx["cur_after_first"]], atol=1e-15)
    np.testing.assert_allclose(plans[1][1], [float(v) for v in fx["q_after_first"]], atol=1e-15)
    np.testing.assert_allclose(final, [float(v) for v in fx["final"]], atol=1e-15)
    parents = np.array([[-1, 0, 0]], dtype=np.int32)
    tokens = np.array([[0] + kids], dtype=np.int32)
    T = np.log(np.stack([p, p, p]))[None].astype(np.float32)
    D = np.log(np.stack([q, q, q]))[None].astype(np.float32)
    for case in fx["case"]:
        ua = np.array([[0.0, float(case["u1"]), float(case["u2"])]], dtype=np.float32)
        us = np.full((1, 3), 0.5, dtype=np.float32)
        r = oracle.tree_accept_sampling(T, D, tokens, parents, np.array([3]), 1.0, ua, us, without_replacement=True)
        acc_node = int(case["accepted"])
        assert r["accept_len"][0] == (1 if acc_node else 0)
        if acc_node:
            assert r["path_nodes"][0, 1] == acc_node
        else:
            assert r["out_tokens"][0, 0] == int(case["bonus"])


def _wor_sequences(q, width):
    """Every ordered draw of `width` distinct tokens without replacement from
    q, with its probability (written out from the definition of the draw)."""
    V = len(q)
    for toks in itertools.permutations(range(V), width):
        prob, left = 1.0, 1.0
        for t in toks:
            prob *= q[t] / left if left > 0 else 0.0
            left -= q[t]
        yield toks, prob


def _exact_first_token_dist_rule(p, q, draws, plan):
    dist = np.zeros(len(p))
    for toks, w_draw in draws:
        if w_draw == 0.0:
            continue
        plans, final = plan(p, q, list(toks))
        reach = 1.0
        for x, (cur, qk) in zip(toks, plans):
            a = min(1.0, cur[x] / qk[x]) if qk[x] > 0 else (1.0 if cur[x] > 0 else 0.0)
            dist[x] += w_draw * reach * a
            reach *= 1.0 - a
        dist += w_draw * reach * final
    return dist


def _plan_fixed_q(p, q, toks):
    cur_list, final = oracle.node_plan(p, q, toks)
    return [(c, np.asarray(q, dtype=np.float64)) for c in cur_list], final


@pytest.mark.parametrize("V,width,seed", [(2, 1, 0), (2, 2, 1), (3, 2, 2), (3, 3, 3), (4, 2, 4), (4, 4, 5),
                                          (5, 3, 6)])
def test_wor_first_token_is_exactly_target(V, width, seed):
    """Siblings drawn without replacement from q and tested with the
    renormalised draft: the first emitted token is distributed exactly as p."""
    rng = np.random.Generator(np.random.PCG64(100 + seed))
    for _ in range(5):
        p = oracle.softmax_t(rng.normal(0, 2, V), 1.0)
        q = oracle.softmax_t(rng.normal(0, 2, V), 1.0)
        dist = _exact_first_token_dist_rule(p, q, list(_wor_sequences(q, width)), oracle.node_plan_wor)
        np.testing.assert_allclose(dist, p, rtol=0, atol=1e-12)


def test_wor_with_zero_probabilities_and_whole_vocabulary():
    p = np.array([0.0, 0.6, 0.4, 0.0])
    q = np.array([0.5, 0.0, 0.3, 0.2])
    for width in (1, 2, 3):  # up to the draft's support: a draw without replacement ends there
        dist = _exact_first_token_dist_rule(p, q, list(_wor_sequences(q, width)), oracle.node_plan_wor)
        np.testing.assert_allclose(dist, p, atol=1e-12)


def test_sibling_rules_are_not_interchangeable():
    """Negative controls: the fixed-draft rule is biased under draws without
    replacement, and the renormalised rule is biased under i.i.d. draws."""
    p = np.array([0.3, 0.5, 0.2])    # the hand-worked case: a two-point residual after a rejection
    q = np.array([0.1, 0.3, 0.6])
    wor = list(_wor_sequences(q, 2))
    iid = [(toks, float(np.prod([q[t] for t in toks]))) for toks in itertools.product(range(3), repeat=2)]
    d_fixed_wor = _exact_first_token_dist_rule(p, q, wor, _plan_fixed_q)
    d_wor_iid = _exact_first_token_dist_rule(p, q, iid, oracle.node_plan_wor)
    assert np.max(np.abs(d_fixed_wor - p)) > 1e-3
    assert np.max(np.abs(d_wor_iid - p)) > 1e-3
    np.testing.assert_allclose(_exact_first_token_dist_rule(p, q, iid, _plan_fixed_q), p, atol=1e-12)


def test_wor_drafts_are_renormalised_without_rejected_tokens():
    rng = np.random.Generator(np.random.PCG64(10))
    p = oracle.softmax_t(rng.normal(0, 2, 6), 1.0)
    q = oracle.softmax_t(rng.normal(0, 2, 6), 1.0)
    kids = [4, 1, 3, 0]
    plans, _ = oracle.node_plan_wor(p, q, kids)
    for k, (_cur, qk) in enumerate(plans):
        assert qk.sum() == pytest.approx(1.0, abs=1e-12)
        assert all(qk[x] == 0.0 for x in kids[:k])
        keep = [t for t in range(6) if t not in kids[:k]]
        np.testing.assert_allclose(qk[keep], q[keep] / q[keep].sum(), atol=1e-15)


def test_wor_second_token_given_accepted_child_is_child_target():
    """Depth-2 trees drawn without replacement at every node: conditional on
    the first emitted token being an accepted draft x, the next emitted token
    is distributed as the target at context (x,)."""
    V, width, seed = 4, 2, 78
    p0 = oracle.softmax_t(_lm_rows((), V, seed, "t"), 1.0)
    q0 = oracle.softmax_t(_lm_rows((), V, seed, "d"), 1.0)
    joint = np.zeros((V, V))
    acc_mass = np.zeros(V)
    for toks, w0 in _wor_sequences(q0, width):
        plans, _ = oracle.node_plan_wor(p0, q0, list(toks))
        reach = 1.0
        for x, (cur, qk) in zip(toks, plans):
            a = min(1.0, cur[x] / qk[x])
            m = w0 * reach * a
            acc_mass[x] += m
            p1 = oracle.softmax_t(_lm_rows((x,), V, seed, "t"), 1.0)
            q1 = oracle.softmax_t(_lm_rows((x,), V, seed, "d"), 1.0)
            joint[x] += m * _exact_first_token_dist_rule(p1, q1, list(_wor_sequences(q1, width)),
                                                         oracle.node_plan_wor)
            reach *= 1.0 - a
    for x in range(V):
        if acc_mass[x] > 0:
            p1 = oracle.softmax_t(_lm_rows((x,), V, seed, "t"), 1.0)
            np.testing.assert_allclose(joint[x] / acc_mass[x], p1, atol=1e-12)


def test_wor_walker_chi_square():
    """The walker on trees whose siblings are Gumbel top-k draws (without
    replacement) emits a first token distributed as the target at the root."""
    V, T, seed, width = 5, 0.8, 6, 3
    rng = np.random.Generator(np.random.PCG64(54321))
    counts = np.zeros(V)
    n_draws = 6000
    for _ in range(n_draws):
        parents, tokens, ctx = [-1], [0], [()]
        frontier = [0]
        for _ in range(2):
            nxt = []
            for n in frontier:
                z = _lm_rows(ctx[n], V, seed, "d") / T + rng.gumbel(size=V)
                for x in np.argsort(-z, kind="stable")[:width]:
                    parents.append(n)
                    tokens.append(int(x))
                    ctx.append(ctx[n] + (int(x),))
                    nxt.append(len(parents) - 1)
            frontier = nxt
        n = len(parents)
        tl = np.stack([_lm_rows(c, V, seed, "t") for c in ctx]).astype(np.float32)
        dl = np.stack([_lm_rows(c, V, seed, "d") for c in ctx]).astype(np.float32)
        ua = rng.random((1, n), dtype=np.float32)
        us = rng.random((1, n), dtype=np.float32)
        r = oracle.tree_accept_sampling(tl[None], dl[None], np.array([tokens], np.int32),
                                        np.array([parents], np.int32), np.array([n]), T, ua, us,
                                        without_replacement=True)
        counts[r["out_tokens"][0, 0]] += 1
    p_root = oracle.softmax_t(_lm_rows((), V, seed, "t").astype(np.float32), T)
    chi2, pval = stats.chisquare(counts, n_draws * p_root)
    assert pval > 1e-4, (counts, n_draws * p_root, pval)


def test_wor_equals_fixed_rule_on_chains():
    """With one child per node the two sibling rules coincide."""
    w = W.make_workload("tiny")
    parents = np.arange(-1, 7, dtype=np.int32)[None]
    rng = np.random.Generator(np.random.PCG64(3))
    tokens = rng.integers(0, w.V, size=(1, 8)).astype(np.int32)
    a = oracle.tree_accept_sampling(w.target_logits, w.draft_logits, tokens, parents, np.array([8]), 1.0,
                                    w.u_accept, w.u_sample)
    b = oracle.tree_accept_sampling(w.target_logits, w.draft_logits, tokens, parents, np.array([8]), 1.0,
                                    w.u_accept, w.u_sample, without_replacement=True)
    for k in ("accept_len", "path_nodes", "out_tokens"):
        assert np.array_equal(a[k], b[k])
