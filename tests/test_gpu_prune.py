"""GPU parity of tv_kv_prune_pages against the oracle: page tables and
reference counts bit-exact; the freed pages compared as a set (their order in
the free list depends on which lanes finish first)."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from golden_io import read_fixture
from gpu_helpers import DevWorkload, require_gpu, to_dev

pytestmark = pytest.mark.gpu
P = 16


def _run(pt, rc, L, N, nl, dev, status=None, cap=None):
    B = pt.shape[0]
    ptd, rcd = to_dev(pt, dev), to_dev(rc, dev)
    st = to_dev(np.zeros(B, np.int32) if status is None else status, dev)
    fl = torch.full((B * 8 if cap is None else cap,), -1, dtype=torch.int32, device=dev)
    fc = torch.zeros(1, dtype=torch.int32, device=dev)
    tvb.kv_prune_pages(ptd, rcd, to_dev(np.asarray(L, np.int32), dev), to_dev(np.asarray(N, np.int32), dev),
                       to_dev(np.asarray(nl, np.int32), dev), st, free_list=fl, free_count=fc)
    torch.cuda.synchronize()
    n = int(fc.cpu()[0])
    listed = fl.cpu().numpy()[: min(n, fl.numel())]
    return ptd.cpu().numpy(), rcd.cpu().numpy(), n, listed, st.cpu().numpy()


def _compare(pt, rc, L, N, nl, dev, status=None):
    pt2, rc2, n, listed, st = _run(pt, rc, L, N, nl, dev, status)
    rpt, rrc, rfreed, rst = oracle.kv_prune_pages(pt, rc, L, N, nl, status_in=status)
    assert np.array_equal(st, rst)
    assert np.array_equal(pt2, rpt)
    assert np.array_equal(rc2, rrc)
    assert n == len(rfreed) and sorted(listed.tolist()) == rfreed
    return n


def test_hand_worked_example():
    dev = require_gpu()
    fx = read_fixture("prune_example.txt")
    ints = lambda k: np.array([int(x) for x in fx[k]], dtype=np.int32)
    pt = np.stack([ints("row0_before"), ints("row1_before")])
    pt2, rc2, n, listed, st = _run(pt, ints("refcount_before"), ints("prefix_len"), ints("n_nodes"),
                                   ints("new_len"), dev)
    assert st.tolist() == [0, 0]
    assert pt2[0].tolist() == ints("row0_after").tolist() and pt2[1].tolist() == ints("row1_after").tolist()
    assert rc2.tolist() == ints("refcount_after").tolist()
    assert sorted(listed.tolist()) == ints("freed").tolist()


@pytest.mark.parametrize("seed,B", [(0, 1), (1, 12), (2, 64), (3, 300)])
def test_random_requests_with_shared_pages(seed, B):
    """Tree pages private to each request, some pages referenced by several
    requests (and by sequences outside the batch)."""
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(seed))
    max_pages = 40
    L = rng.integers(0, 500, size=B).astype(np.int32)
    N = rng.integers(1, 65, size=B).astype(np.int32)
    a = np.array([rng.integers(0, n) for n in N])
    nl = (L + a + 1).astype(np.int32)
    num_pages = int(sum((L + N + P - 1) // P)) + 10
    pool = rng.permutation(num_pages).astype(np.int32)
    pt = np.full((B, max_pages), -1, np.int32)
    off = 0
    for b in range(B):
        k = int((L[b] + N[b] + P - 1) // P)
        pt[b, :k] = pool[off:off + k]
        off += k
        # occasionally point a released slot at a page another request also releases
        if b > 0 and rng.random() < 0.3:
            s = int((L[b] + N[b] + P - 1) // P) - 1
            if s * P >= nl[b]:
                pt[b, s] = pt[b - 1, int((L[b - 1] + N[b - 1] + P - 1) // P) - 1]
    rc = np.zeros(num_pages, np.int32)
    for b in range(B):
        for s in range(max_pages):
            if pt[b, s] >= 0:
                rc[pt[b, s]] += 1
    rc += rng.integers(0, 2, size=num_pages).astype(np.int32)
    n = _compare(pt, rc, L, N, nl, dev)
    print(f"B={B}: {n} pages freed")


def test_errors_and_skips():
    dev = require_gpu()
    pt = np.array([[0, 1, -1], [2, 9, -1], [3, 4, -1], [5, 6, -1], [7, 8, -1], [10, 11, -1]], np.int32)
    rc = np.ones(12, np.int32)
    rc[8] = 0
    L = np.array([10, 10, 10, 10, 10, 16], np.int32)
    N = np.array([10, 10, 10, 40, 10, 10], np.int32)
    nl = np.array([25, 11, 11, 11, 11, 16], np.int32)
    st_in = np.array([0, 0, 2, 0, 0, 0], np.int32)
    _compare(pt, rc, L, N, nl, dev, status=st_in)


def test_free_list_overflow_reports_capacity():
    dev = require_gpu()
    B = 6
    pt = np.array([[2 * b, 2 * b + 1] for b in range(B)], np.int32)
    rc = np.ones(2 * B, np.int32)
    L = np.full(B, 10, np.int32)
    N = np.full(B, 10, np.int32)
    nl = np.full(B, 11, np.int32)
    pt2, rc2, n, listed, st = _run(pt, rc, L, N, nl, dev, cap=2)
    assert n == B                                   # every second page was freed
    assert (pt2[:, 1] == -1).all() and (rc2[1::2] == 0).all()
    assert len(listed) == 2 and set(listed.tolist()) <= set(range(1, 2 * B, 2))
    assert int((st == oracle.STATUS_CAPACITY).sum()) == B - 2 and int((st == 0).sum()) == 2


def test_after_commit_on_serving_batch():
    """The step's tail on the serving workload: greedy accept, commit of the
    accepted paths, then release of the pages beyond each new length."""
    dev = require_gpu()
    w = W.make_workload("serving")
    dw = DevWorkload(w, dev)
    anc, depth, st = dw.mask()
    acc = tvb.tree_accept(dw.target, None, dw.tokens, dw.parents, dw.n_nodes, anc, depth, 0.0, None, None, st)
    slots, new_len = tvb.kv_commit_path(dw.k, dw.v, dw.page_table, dw.prefix_len, dw.n_nodes, acc[0], acc[1], st)
    torch.cuda.synchronize()
    rc = np.ones(w.num_pages, np.int32)
    nl = new_len.cpu().numpy()
    ref = oracle.tree_accept_greedy(w.target_logits, w.tokens, w.parents, w.n_nodes)
    assert np.array_equal(nl, w.prefix_len + ref["accept_len"] + 1)
    n = _compare(w.page_table, rc, w.prefix_len, w.n_nodes, nl, dev)
    print(f"serving: {n} pages freed of {w.num_pages}")
