"""Pins of the oracle's tree mask (no GPU).

The mask is defined in "SGLang EAGLE-2 Speculative Decoding" (Tech Radar),
section 2, "Dynamic Tree-Attention Masking": M[i][j] = 1 iff j is an ancestor
of i or i itself.
"""
import numpy as np
import pytest

import oracle
from eagle_speculative_decoding_attn_gb300 import workloads as W
from golden_io import read_fixture


def _mask_matrix(word, n):
    return [(int(word) >> j) & 1 for j in range(n)]


def test_mask_hand_worked_example():
    fx = read_fixture("mask_example.txt")
    parents = np.array([int(x) for x in fx["parents"]], dtype=np.int32)
    n = len(parents)
    anc, depth, status = oracle.tree_build_mask(parents[None, :], np.array([n]))
    assert status[0] == 0
    expect = [[int(x) for x in row] for row in fx["mask"]]
    got = [_mask_matrix(anc[0, i], n) for i in range(n)]
    assert got == expect
    assert depth[0].tolist() == [int(x) for x in fx["depth"]]


def _closure_by_matrix_powers(parents, n):
    """Reflexive-transitive closure of the child->parent relation by repeated
    boolean matrix products (brute force, independent of the parent walk)."""
    A = np.zeros((n, n), dtype=np.int64)
    for i in range(1, n):
        A[i, parents[i]] = 1
    R = np.eye(n, dtype=np.int64)
    P = np.eye(n, dtype=np.int64)
    for _ in range(n):
        P = (P @ A > 0).astype(np.int64)
        R = ((R + P) > 0).astype(np.int64)
    return R


@pytest.mark.parametrize("n", [1, 2, 5, 17, 63, 64])
def test_mask_matches_brute_force_closure(n):
    rng = np.random.Generator(np.random.PCG64(7 + n))
    for _ in range(5):
        p = W.random_recursive_tree(rng, n)
        anc, depth, status = oracle.tree_build_mask(p[None, :], np.array([n]))
        assert status[0] == 0
        R = _closure_by_matrix_powers(p, n)
        for i in range(n):
            assert _mask_matrix(anc[0, i], n) == R[i].tolist()
            # depth = number of strict ancestors
            assert depth[0, i] == R[i].sum() - 1


def test_mask_chain_and_star():
    n = 64
    anc, depth, st = oracle.tree_build_mask(W.chain_tree(n)[None], np.array([n]))
    assert st[0] == 0
    for i in range(n):
        assert int(anc[0, i]) == (1 << (i + 1)) - 1          # all nodes 0..i
        assert depth[0, i] == i
    anc, depth, st = oracle.tree_build_mask(W.star_tree(n)[None], np.array([n]))
    for i in range(1, n):
        assert int(anc[0, i]) == 1 | (1 << i)
        assert depth[0, i] == 1


@pytest.mark.parametrize("bad", [
    ([0, 0, 1], 3),          # root must have parent -1
    ([-1, 1, 0], 3),         # parent must precede the node
    ([-1, 0, 5], 3),         # parent out of range
    ([-1, 0, -1], 3),        # second root
    ([-1], 0),               # empty tree
])
def test_mask_rejects_bad_trees(bad):
    p, n = bad
    arr = np.full((1, max(3, len(p))), -1, dtype=np.int32)
    arr[0, : len(p)] = p
    anc, depth, st = oracle.tree_build_mask(arr, np.array([n]))
    assert st[0] == oracle.STATUS_BAD_TREE
    assert np.all(anc == 0) and np.all(depth == -1)


def test_mask_rejects_65_nodes():
    p = np.concatenate([[-1], np.zeros(64, dtype=np.int32)]).astype(np.int32)
    _, _, st = oracle.tree_build_mask(p[None], np.array([65]))
    assert st[0] == oracle.STATUS_BAD_TREE
