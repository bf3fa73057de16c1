"""Pins of the oracle's KV commit (no GPU).

Tech Radar section 2 (sequence diagram): after verification the target keeps
the KV of the accepted branch and discards the wrong branches.  Checked
against a hand-worked overlapping example and against an independent
formulation (gather the request's logical sequence, rebuild it as
prefix + accepted rows, scatter it back).
"""
import numpy as np
import pytest

import oracle
from eagle_speculative_decoding_attn_gb300 import workloads as W
from golden_io import read_fixture


def test_commit_hand_worked_overlap():
    fx = read_fixture("commit_example.txt")
    L, N = int(fx["prefix_len"][0]), int(fx["n_nodes"][0])
    path = [int(x) for x in fx["path"]]
    labels = fx["before"]
    # one layer, one page, one head, D=1: position t holds the label index t
    k = np.zeros((1, 1, 1, 16, 1), dtype=np.int64)
    k[0, 0, 0, : len(labels), 0] = np.arange(len(labels))
    v = k.copy() + 100
    pt = np.array([[0]], dtype=np.int32)
    pn = np.full((1, N), -1, dtype=np.int32)
    pn[0, : len(path)] = path
    k2, v2, slots, new_len, st = oracle.kv_commit_path(
        k, v, pt, np.array([L]), np.array([N]), np.array([len(path) - 1]), pn)
    assert st[0] == 0
    after = [labels[int(i)] for i in k2[0, 0, 0, : len(labels), 0]]
    assert after == fx["after"]
    assert (v2 - 100 == k2).all()
    assert new_len[0] == int(fx["new_len"][0])
    assert slots[0, : len(path)].tolist() == [int(x) for x in fx["committed_slots"]]
    assert slots[0, len(path):].tolist() == [-1] * (N - len(path))


def _commit_by_sequence_rebuild(k, v, pt, L, path, P):
    """Independent formulation: read the logical sequence, form
    prefix + [rows of the accepted nodes], write it back position by position."""
    k, v = k.copy(), v.copy()
    n_seq = L + max(path) + 1
    def slot(t):
        return int(pt[t // P]), t % P
    seq_k = [k[:, slot(t)[0], :, slot(t)[1], :].copy() for t in range(n_seq)]
    seq_v = [v[:, slot(t)[0], :, slot(t)[1], :].copy() for t in range(n_seq)]
    new_k = seq_k[:L] + [seq_k[L + n] for n in path]
    new_v = seq_v[:L] + [seq_v[L + n] for n in path]
    for t in range(len(new_k)):
        pg, o = slot(t)
        k[:, pg, :, o, :] = new_k[t]
        v[:, pg, :, o, :] = new_v[t]
    return k, v


@pytest.mark.parametrize("seed", range(12))
def test_commit_matches_sequence_rebuild(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    n_layers, Hkv, D, P = 3, 2, 8, 16
    B = 3
    L = rng.integers(0, 50, size=B).astype(np.int32)
    trees = [W.random_recursive_tree(rng, int(rng.integers(1, 65))) for _ in range(B)]
    N = np.array([len(t) for t in trees], dtype=np.int32)
    pages = [(int(L[b]) + int(N[b]) + P - 1) // P for b in range(B)]
    perm = rng.permutation(sum(pages) + 2)
    pt = np.full((B, max(pages)), -1, dtype=np.int32)
    off = 0
    for b in range(B):
        pt[b, : pages[b]] = perm[off: off + pages[b]]
        off += pages[b]
    k = rng.integers(0, 1 << 15, size=(n_layers, len(perm), Hkv, P, D)).astype(np.uint16)
    v = rng.integers(0, 1 << 15, size=(n_layers, len(perm), Hkv, P, D)).astype(np.uint16)
    n_max = 64
    pn = np.full((B, n_max), -1, dtype=np.int32)
    acc = np.zeros(B, dtype=np.int32)
    for b in range(B):
        node = int(rng.integers(0, N[b]))
        path = oracle.ancestors_or_self(trees[b], node)
        pn[b, : len(path)] = path
        acc[b] = len(path) - 1
    k2, v2, slots, new_len, st = oracle.kv_commit_path(k, v, pt, L, N, acc, pn)
    assert (st == 0).all()
    ke, ve = k.copy(), v.copy()
    for b in range(B):
        path = pn[b, : acc[b] + 1].tolist()
        ke, ve = _commit_by_sequence_rebuild(ke, ve, pt[b], int(L[b]), path, P)
        assert new_len[b] == L[b] + acc[b] + 1
        for kk in range(acc[b] + 1):
            t = int(L[b]) + kk
            assert slots[b, kk] == pt[b, t // P] * P + t % P
    assert np.array_equal(k2, ke) and np.array_equal(v2, ve)


def test_commit_rejects_bad_path():
    k = np.zeros((1, 2, 1, 16, 4), np.uint16)
    pt = np.array([[0, 1]], np.int32)
    pn = np.array([[0, 3, 2, -1, -1]], np.int32)     # not increasing
    _, _, _, new_len, st = oracle.kv_commit_path(k, k, pt, np.array([3]), np.array([5]),
                                                 np.array([2]), pn)
    assert st[0] == oracle.STATUS_BAD_TREE and new_len[0] == 3
