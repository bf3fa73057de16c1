"""Pins of the oracle's zero-copy page pruning (no GPU).

Source: Tech Radar, failure mode 2 (rejected branches leave garbage blocks in
the page table; a prefix-tree page manager frees them at once, without a
copy) and section 2's sequence diagram (keep the accepted branch, drop the
wrong ones).  Pinned by a hand-worked fixture (tests/golden/prune_example.txt),
a position-by-position model of which pages still hold a kept row, reference
count conservation, shared pages and the error cases.
"""
import collections

import numpy as np
import pytest

import oracle
from golden_io import read_fixture

P = 16


def test_hand_worked_example():
    fx = read_fixture("prune_example.txt")
    ints = lambda k: np.array([int(x) for x in fx[k]], dtype=np.int32)
    pt = np.stack([ints("row0_before"), ints("row1_before")])
    pt2, rc2, freed, st = oracle.kv_prune_pages(pt, ints("refcount_before"), ints("prefix_len"), ints("n_nodes"),
                                                ints("new_len"))
    assert st.tolist() == [0, 0]
    assert pt2[0].tolist() == ints("row0_after").tolist()
    assert pt2[1].tolist() == ints("row1_after").tolist()
    assert rc2.tolist() == ints("refcount_after").tolist()
    assert freed == ints("freed").tolist()


def _kept_slots(L, N, new_len):
    """Slots that still hold a kept position, and slots that held tree rows,
    from the positions themselves."""
    kept, tree = set(), set()
    for pos in range(L + N):
        if pos < new_len:
            kept.add(pos // P)
        if pos >= L:
            tree.add(pos // P)
    return kept, tree


@pytest.mark.parametrize("seed", range(8))
def test_matches_position_model(seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    B, max_pages = 12, 40
    L = rng.integers(0, 500, size=B)
    N = rng.integers(1, 65, size=B)
    a = np.array([rng.integers(0, n) for n in N])
    new_len = (L + a + 1).astype(np.int32)
    num_pages = int(sum((L + N + P - 1) // P)) + 10
    perm = rng.permutation(num_pages).astype(np.int32)
    pt = np.full((B, max_pages), -1, np.int32)
    off = 0
    for b in range(B):
        k = int((L[b] + N[b] + P - 1) // P)
        pt[b, :k] = perm[off:off + k]
        off += k
    rc = np.zeros(num_pages, np.int32)
    for b in range(B):
        for s in range(max_pages):
            if pt[b, s] >= 0:
                rc[pt[b, s]] += 1
    extra = rng.integers(0, 2, size=num_pages)     # references held by other sequences
    rc = rc + extra.astype(np.int32)
    pt2, rc2, freed, st = oracle.kv_prune_pages(pt, rc, L, N, new_len)
    assert (st == 0).all()
    released = collections.Counter()
    for b in range(B):
        kept, tree = _kept_slots(int(L[b]), int(N[b]), int(new_len[b]))
        for s in range(max_pages):
            if s in tree and s not in kept:
                assert pt2[b, s] == -1
                released[int(pt[b, s])] += 1
            else:
                assert pt2[b, s] == pt[b, s]
    for pid in range(num_pages):
        assert rc2[pid] == rc[pid] - released[pid]
    assert freed == sorted(pid for pid in range(num_pages) if released[pid] and rc2[pid] == 0)
    assert int(rc.sum() - rc2.sum()) == sum(released.values())


def test_shared_page_freed_once():
    # two requests whose last pages are the same physical page (count 2)
    pt = np.array([[0, 3], [1, 3]], np.int32)
    rc = np.array([1, 1, 0, 2], np.int32)
    L = np.array([10, 12], np.int32)
    N = np.array([10, 8], np.int32)
    new_len = np.array([11, 13], np.int32)
    pt2, rc2, freed, st = oracle.kv_prune_pages(pt, rc, L, N, new_len)
    assert (st == 0).all()
    assert pt2.tolist() == [[0, -1], [1, -1]]
    assert rc2.tolist() == [1, 1, 0, 0]
    assert freed == [3]


def test_errors_and_skips():
    pt = np.array([[0, 1, -1], [2, 9, -1], [3, 4, -1], [5, 6, -1], [7, 8, -1]], np.int32)
    rc = np.ones(9, np.int32)
    rc[8] = 0
    L = np.array([10, 10, 10, 10, 10], np.int32)
    N = np.array([10, 10, 10, 40, 10], np.int32)
    new_len = np.array([25, 11, 11, 11, 11], np.int32)
    st_in = np.array([0, 0, 2, 0, 0], np.int32)
    pt2, rc2, freed, st = oracle.kv_prune_pages(pt, rc, L, N, new_len, status_in=st_in)
    # 0: new_len beyond L + N; 1: page id 9 out of range; 2: skipped; 3: L + N does not fit;
    # 4: page 8's count is already zero
    assert st.tolist() == [oracle.STATUS_BAD_TREE, oracle.STATUS_PAGE_OOB, 2, oracle.STATUS_CAPACITY,
                           oracle.STATUS_BAD_REFCOUNT]
    assert pt2[:4].tolist() == pt[:4].tolist()
    assert pt2[4].tolist() == [7, -1, -1]
    assert rc2[8] == 0 and freed == []


def test_nothing_released_when_everything_is_kept():
    pt = np.array([[4, 5, 6]], np.int32)
    rc = np.ones(7, np.int32)
    for L, N in ((0, 48), (5, 43), (31, 1)):
        pt2, rc2, freed, st = oracle.kv_prune_pages(pt, rc, [L], [N], [L + N])
        assert st[0] == 0 and pt2.tolist() == pt.tolist() and rc2.tolist() == rc.tolist() and freed == []


def test_new_length_must_keep_the_root():
    # the root (position L) is always kept: new_len = L is malformed
    pt = np.array([[0, 1]], np.int32)
    pt2, rc2, freed, st = oracle.kv_prune_pages(pt, np.ones(2, np.int32), [16], [10], [16])
    assert st[0] == oracle.STATUS_BAD_TREE and pt2.tolist() == pt.tolist() and freed == []
