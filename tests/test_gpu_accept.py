"""GPU parity of tv_tree_accept against the oracle.

Greedy results (accepted length, path, emitted tokens) must be bit-exact.
Sampled results must be bit-exact given the same uniforms, except requests
whose walk met a decision within 1e-6 of its threshold (the oracle flags
them); those are counted and reported.  A chi-square test over 10^6 GPU
draws checks the lossless property: the first emitted token is distributed
as the target at the root.
"""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from golden_io import read_fixture
from gpu_helpers import DevWorkload, require_gpu, to_dev

pytestmark = pytest.mark.gpu


def _run(dw, temperature, status=None, wor=False):
    anc, depth, st = dw.mask()
    if status is not None:
        st = status
    if temperature > 0:
        res = tvb.tree_accept(dw.target, dw.draft, dw.tokens, dw.parents, dw.n_nodes, anc, depth, temperature,
                              dw.u_accept, dw.u_sample, st, without_replacement=wor)
    else:
        res = tvb.tree_accept(dw.target, None, dw.tokens, dw.parents, dw.n_nodes, anc, depth, 0.0, None, None, st)
    torch.cuda.synchronize()
    return [r.cpu().numpy() for r in res] + [st.cpu().numpy()]


def _check_greedy(w, dev):
    a, pn, ot, st = _run(DevWorkload(w, dev), 0.0)
    ref = oracle.tree_accept_greedy(w.target_logits, w.tokens, w.parents, w.n_nodes)
    assert np.array_equal(st, ref["status"])
    assert np.array_equal(a, ref["accept_len"])
    assert np.array_equal(pn, ref["path_nodes"])
    assert np.array_equal(ot, ref["out_tokens"])
    return a


def _check_sampling(w, dev, T=None, wor=False):
    T = w.temperature if T is None else T
    a, pn, ot, st = _run(DevWorkload(w, dev), T, wor=wor)
    ref = oracle.tree_accept_sampling(w.target_logits, w.draft_logits, w.tokens, w.parents, w.n_nodes, T,
                                      w.u_accept, w.u_sample, without_replacement=wor)
    assert np.array_equal(st, ref["status"])
    near = ref["near_boundary"]
    same = (a == ref["accept_len"]) & (pn == ref["path_nodes"]).all(1) & (ot == ref["out_tokens"]).all(1)
    bad = np.nonzero(~same & ~near)[0]
    assert bad.size == 0, f"requests {bad.tolist()} differ from the oracle away from any boundary"
    n_near_diff = int((~same & near).sum())
    print(f"sampling parity: {w.B} requests, {int(near.sum())} near-boundary, {n_near_diff} differ there")
    return a


def test_greedy_tiny():
    _check_greedy(W.make_workload("tiny"), require_gpu())


def test_greedy_llama2_7b():
    a = _check_greedy(W.make_workload("llama2_7b"), require_gpu())
    print("7B accept_len", a.tolist())


def test_greedy_serving():
    a = _check_greedy(W.make_workload("serving"), require_gpu())
    print("serving accept_len", a.tolist())


@pytest.mark.parametrize("V,seed", [(2, 0), (3, 1), (7, 2), (1000, 3), (1001, 4)])
def test_greedy_random_trees_with_ties(V, seed):
    """Integer logits make argmax ties frequent; small V makes long accepted
    chains and duplicate sibling tokens common."""
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(seed))
    B = 64
    trees = [W.random_recursive_tree(rng, int(rng.integers(1, 65))) if b % 5 else W.chain_tree(64)
             for b in range(B)]
    w = W.make_custom(B=B, Hq=1, Hkv=1, D=64, prefix_len=[0] * B, parents_list=trees, seed=seed, V=V,
                      n_max=64)
    w.target_logits[:] = rng.integers(0, 3, size=w.target_logits.shape).astype(np.float32)
    w.tokens[:] = rng.integers(0, V, size=w.tokens.shape).astype(np.int32)
    # most drafted tokens follow the target's argmax at the parent (first index among ties),
    # so accepted chains are long and duplicate siblings occur
    for b in range(B):
        for c in range(1, int(w.n_nodes[b])):
            if rng.random() < 0.7:
                w.tokens[b, c] = int(np.argmax(w.target_logits[b, int(w.parents[b, c])]))
    a = _check_greedy(w, dev)
    assert a.max() >= 2


def test_greedy_one_pass_workspace_reuse_and_skips():
    """The one-pass greedy walk on one workspace three times in a row (its arrival
    counters must return to zero), with a request whose status is already set
    (skipped) and one with a malformed tree (BAD_TREE) in the same batch."""
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(42))
    B, V = 6, 5003
    trees = [W.random_recursive_tree(rng, 40) for _ in range(B)]
    w = W.make_custom(B=B, Hq=1, Hkv=1, D=64, prefix_len=[0] * B, parents_list=trees, seed=42, V=V, n_max=64)
    for b in range(B):
        for c in range(1, int(w.n_nodes[b])):
            if rng.random() < 0.8:
                w.tokens[b, c] = int(np.argmax(w.target_logits[b, int(w.parents[b, c])]))
    w.parents[3, 5] = 7                       # parent after the child: malformed
    assert tvb.tree_accept_workspace_bytes(B, 64, V) > 0
    ws = tvb.new_accept_workspace(B, 64, V, dev)
    dw = DevWorkload(w, dev)
    ref = oracle.tree_accept_greedy(w.target_logits, w.tokens, w.parents, w.n_nodes)
    for _ in range(3):
        st = torch.zeros(B, dtype=torch.int32, device=dev)
        st[1] = oracle.STATUS_PAGE_OOB        # set by an earlier stage: this request is skipped
        a, pn, ot = tvb.tree_accept(dw.target, None, dw.tokens, dw.parents, dw.n_nodes, None, None, 0.0, None,
                                    None, st, workspace=ws)
        torch.cuda.synchronize()
        a, pn, ot, st = a.cpu().numpy(), pn.cpu().numpy(), ot.cpu().numpy(), st.cpu().numpy()
        for b in range(B):
            if b == 1:
                assert a[b] == 0 and (pn[b] == -1).all() and (ot[b] == -1).all() and st[b] == oracle.STATUS_PAGE_OOB
                continue
            assert st[b] == ref["status"][b]
            assert a[b] == ref["accept_len"][b]
            assert np.array_equal(pn[b], ref["path_nodes"][b]) and np.array_equal(ot[b], ref["out_tokens"][b])
        assert st[3] == oracle.STATUS_BAD_TREE
        assert a.max() >= 2
    assert int(ws[-4 * B:].view(torch.int32).abs().sum()) == 0   # arrival counters back at zero


def test_sampling_tiny():
    _check_sampling(W.make_workload("tiny"), require_gpu())


def test_sampling_llama3_70b():
    a = _check_sampling(W.make_workload("llama3_70b"), require_gpu())
    print("70B accept_len", a.tolist())


def test_sampling_long():
    _check_sampling(W.make_workload("long"), require_gpu())


@pytest.mark.parametrize("V,T,seed", [(5, 1.0, 0), (50, 0.5, 1), (4096, 1.3, 2), (32003, 0.9, 3)])
def test_sampling_random(V, T, seed):
    """Children drawn i.i.d. from the draft at T, so accepts are frequent."""
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(70 + seed))
    B = 48
    trees = [W.random_recursive_tree(rng, int(rng.integers(1, 65))) for _ in range(B)]
    w = W.make_custom(B=B, Hq=1, Hkv=1, D=64, prefix_len=[0] * B, parents_list=trees, seed=seed, V=V,
                      temperature=T, n_max=64)
    # correlated target/draft so that acceptance happens
    w.target_logits[:] = (w.draft_logits + 0.7 * rng.standard_normal(w.draft_logits.shape)).astype(np.float32)
    for b in range(B):
        n = int(w.n_nodes[b])
        for c in range(1, n):
            par = int(w.parents[b, c])
            g = rng.gumbel(size=V)
            w.tokens[b, c] = int(np.argmax(w.draft_logits[b, par].astype(np.float64) / T + g))
    a = _check_sampling(w, dev)
    print(f"V={V} accept lengths mean {a.mean():.2f} max {a.max()}")


def test_sampling_chi_square_million_draws():
    """Root with 3 children drawn i.i.d. from q (fresh per request); the first
    emitted token over 10^6 GPU draws against p_root (V - 1 dof)."""
    dev = require_gpu()
    V, T = 6, 1.0
    rng = np.random.Generator(np.random.PCG64(2024))
    tl = (1.5 * rng.standard_normal(V)).astype(np.float32)
    dl = (1.5 * rng.standard_normal(V)).astype(np.float32)
    p_root = oracle.softmax_t(tl, T)
    q_root = oracle.softmax_t(dl, T)
    B, n = 125000, 4
    parents = np.tile(np.array([-1, 0, 0, 0], np.int32), (B, 1))
    target = np.broadcast_to(np.tile(tl, (n, 1)), (B, n, V)).astype(np.float32)
    draft = np.broadcast_to(np.tile(dl, (n, 1)), (B, n, V)).astype(np.float32)
    pd, dd = to_dev(parents, dev), to_dev(np.full(B, n, np.int32), dev)
    td, drd = to_dev(target, dev), to_dev(draft, dev)
    anc, depth, st0 = tvb.tree_build_mask(pd, dd)
    counts = np.zeros(V)
    for rep in range(8):
        toks = np.zeros((B, n), np.int32)
        toks[:, 1:] = rng.choice(V, size=(B, n - 1), p=q_root)
        ua = rng.random((B, n), dtype=np.float32)
        us = rng.random((B, n), dtype=np.float32)
        st = st0.clone()
        a, pn, ot = tvb.tree_accept(td, drd, to_dev(toks, dev), pd, dd, anc, depth, T, to_dev(ua, dev),
                                    to_dev(us, dev), st)
        first = ot[:, 0].cpu().numpy()
        assert (st.cpu().numpy() == 0).all()
        counts += np.bincount(first, minlength=V)
    total = counts.sum()
    assert total == 10 ** 6
    chi2, pval = stats.chisquare(counts, total * p_root)
    print(f"chi-square {chi2:.2f}, p = {pval:.4f}; counts {counts.tolist()}")
    assert pval > 1e-3


def test_accept_errors():
    dev = require_gpu()
    w = W.make_workload("tiny")
    dw = DevWorkload(w, dev)
    anc, depth, st = dw.mask()
    bad_tok = dw.tokens.clone()
    bad_tok[0, 3] = w.V + 5
    a, pn, ot = tvb.tree_accept(dw.target, None, bad_tok, dw.parents, dw.n_nodes, anc, depth, 0.0, None, None, st)
    torch.cuda.synchronize()
    assert int(st.cpu()[0]) == tvb.TV_DEV_BAD_TOKEN
    assert int(a.cpu()[0]) == 0 and (pn.cpu().numpy() == -1).all() and (ot.cpu().numpy() == -1).all()
    with pytest.raises(tvb.TreeVerifyError):
        tvb.tree_accept(dw.target, None, dw.tokens, dw.parents, dw.n_nodes, anc, depth, 1.0, None, None, st)
    # sampling keeps each request's rows in registers: at most 16 CTAs of 512
    # threads with 32 entries each
    for B, V in ((1, 16 * 512 * 32 + 4), (12, 16 * 512 * 32 + 64)):
        big = torch.zeros((B, 2, V), dtype=torch.float32, device=dev)
        two = lambda t: t[:, :2].expand(B, 2).contiguous()
        with pytest.raises(tvb.TreeVerifyError):
            tvb.tree_accept(big, big, two(dw.tokens), two(dw.parents), torch.ones(B, dtype=torch.int32, device=dev),
                            None, None, 1.0, two(dw.u_accept), two(dw.u_sample),
                            torch.zeros(B, dtype=torch.int32, device=dev))


# --------------------------------------------------------------------------
# siblings drafted without replacement (renormalised draft after each rejection)
# --------------------------------------------------------------------------
def test_sampling_wor_hand_worked_example():
    dev = require_gpu()
    fx = read_fixture("sampling_wor_example.txt")
    p = np.array([float(v) for v in fx["p"]])
    q = np.array([float(v) for v in fx["q"]])
    kids = [int(v) for v in fx["children"]]
    cases = fx["case"]
    B = len(cases)
    parents = np.tile(np.array([-1, 0, 0], np.int32), (B, 1))
    tokens = np.tile(np.array([0] + kids, np.int32), (B, 1))
    tl = np.broadcast_to(np.log(p).astype(np.float32), (B, 3, 3)).copy()
    dl = np.broadcast_to(np.log(q).astype(np.float32), (B, 3, 3)).copy()
    ua = np.array([[0.0, float(c["u1"]), float(c["u2"])] for c in cases], np.float32)
    us = np.full((B, 3), 0.5, np.float32)
    pd, nd = to_dev(parents, dev), to_dev(np.full(B, 3, np.int32), dev)
    anc, depth, st = tvb.tree_build_mask(pd, nd)
    a, pn, ot = tvb.tree_accept(to_dev(tl, dev), to_dev(dl, dev), to_dev(tokens, dev), pd, nd, anc, depth, 1.0,
                                to_dev(ua, dev), to_dev(us, dev), st, without_replacement=True)
    torch.cuda.synchronize()
    a, pn, ot = a.cpu().numpy(), pn.cpu().numpy(), ot.cpu().numpy()
    for b, c in enumerate(cases):
        acc = int(c["accepted"])
        assert a[b] == (1 if acc else 0)
        if acc:
            assert pn[b, 1] == acc
        else:
            assert ot[b, 0] == int(c["bonus"])


def test_sampling_wor_tiny():
    _check_sampling(W.make_workload("tiny", siblings="wor"), require_gpu(), wor=True)


def test_sampling_wor_llama3_70b():
    a = _check_sampling(W.make_workload("llama3_70b", siblings="wor"), require_gpu(), wor=True)
    print("70B (siblings without replacement) accept_len", a.tolist())


def test_sampling_wor_long():
    _check_sampling(W.make_workload("long", siblings="wor"), require_gpu(), wor=True)


@pytest.mark.parametrize("V,T,seed,dup", [(5, 1.0, 0, False), (50, 0.5, 1, False), (4096, 1.3, 2, False),
                                          (32003, 0.9, 3, False), (7, 1.0, 4, True)])
def test_sampling_wor_random(V, T, seed, dup):
    """Children by Gumbel top-k of the draft at T (distinct siblings), or,
    with dup, i.i.d. draws so that the rule also meets repeated tokens."""
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(170 + seed))
    B = 48
    trees = [W.random_recursive_tree(rng, int(rng.integers(1, 65))) for _ in range(B)]
    w = W.make_custom(B=B, Hq=1, Hkv=1, D=64, prefix_len=[0] * B, parents_list=trees, seed=seed, V=V,
                      temperature=T, n_max=64)
    w.target_logits[:] = (w.draft_logits + 0.7 * rng.standard_normal(w.draft_logits.shape)).astype(np.float32)
    for b in range(B):
        n = int(w.n_nodes[b])
        kids = W.children_lists(w.parents[b], n)
        for node in range(n):
            if not kids[node]:
                continue
            z = w.draft_logits[b, node].astype(np.float64) / T
            if dup:
                toks = [int(np.argmax(z + rng.gumbel(size=V))) for _ in kids[node]]
            else:
                toks = np.argsort(-(z + rng.gumbel(size=V)), kind="stable")[:len(kids[node])].tolist()
            for c, t in zip(kids[node], toks):
                w.tokens[b, c] = t
    a = _check_sampling(w, dev, wor=True)
    print(f"V={V} accept lengths mean {a.mean():.2f} max {a.max()}")


def test_sampling_wor_chi_square_million_draws():
    """Root with 3 children drawn without replacement from q (Gumbel top-3,
    fresh per request); the first emitted token over 10^6 GPU draws against
    p_root (V - 1 dof)."""
    dev = require_gpu()
    V, T = 6, 1.0
    rng = np.random.Generator(np.random.PCG64(2025))
    tl = (1.5 * rng.standard_normal(V)).astype(np.float32)
    dl = (1.5 * rng.standard_normal(V)).astype(np.float32)
    p_root = oracle.softmax_t(tl, T)
    B, n = 125000, 4
    parents = np.tile(np.array([-1, 0, 0, 0], np.int32), (B, 1))
    target = np.broadcast_to(np.tile(tl, (n, 1)), (B, n, V)).astype(np.float32)
    draft = np.broadcast_to(np.tile(dl, (n, 1)), (B, n, V)).astype(np.float32)
    pd, dd = to_dev(parents, dev), to_dev(np.full(B, n, np.int32), dev)
    td, drd = to_dev(target, dev), to_dev(draft, dev)
    anc, depth, st0 = tvb.tree_build_mask(pd, dd)
    counts = np.zeros(V)
    for rep in range(8):
        z = dl.astype(np.float64)[None, :] / T + rng.gumbel(size=(B, V))
        toks = np.zeros((B, n), np.int32)
        toks[:, 1:] = np.argsort(-z, axis=1, kind="stable")[:, : n - 1]
        ua = rng.random((B, n), dtype=np.float32)
        us = rng.random((B, n), dtype=np.float32)
        st = st0.clone()
        a, pn, ot = tvb.tree_accept(td, drd, to_dev(toks, dev), pd, dd, anc, depth, T, to_dev(ua, dev),
                                    to_dev(us, dev), st, without_replacement=True)
        first = ot[:, 0].cpu().numpy()
        assert (st.cpu().numpy() == 0).all()
        counts += np.bincount(first, minlength=V)
    total = counts.sum()
    assert total == 10 ** 6
    chi2, pval = stats.chisquare(counts, total * p_root)
    print(f"chi2 {chi2:.2f} p {pval:.3f}")
    assert pval > 1e-4
