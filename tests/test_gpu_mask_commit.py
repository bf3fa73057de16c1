"""GPU parity of tv_tree_build_mask and tv_kv_commit_path against the oracle
(bit-exact integer / byte results)."""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from gpu_helpers import require_gpu, to_dev
from golden_io import read_fixture

pytestmark = pytest.mark.gpu


def _run_mask(parents, n_nodes, dev):
    anc, depth, st = tvb.tree_build_mask(to_dev(parents, dev), to_dev(n_nodes, dev))
    torch.cuda.synchronize()
    return anc.cpu().numpy().view(np.uint64), depth.cpu().numpy(), st.cpu().numpy()


def test_mask_golden():
    dev = require_gpu()
    fx = read_fixture("mask_example.txt")
    p = np.array([[int(x) for x in fx["parents"]]], dtype=np.int32)
    n = p.shape[1]
    anc, depth, st = _run_mask(p, np.array([n], np.int32), dev)
    assert st[0] == 0
    for i, row in enumerate(fx["mask"]):
        assert [(int(anc[0, i]) >> j) & 1 for j in range(n)] == [int(x) for x in row]
    assert depth[0].tolist() == [int(x) for x in fx["depth"]]


def test_mask_random_trees_bit_exact():
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(31))
    B, n_max = 200, 64
    parents = np.full((B, n_max), -1, np.int32)
    n_nodes = np.zeros(B, np.int32)
    for b in range(B):
        n = int(rng.integers(1, n_max + 1)) if b % 4 else n_max
        kind = b % 3
        p = W.chain_tree(n) if kind == 0 else (W.star_tree(n) if kind == 1 else W.random_recursive_tree(rng, n))
        parents[b, :n] = p
        n_nodes[b] = n
    # invalid trees mixed in
    parents[5, 3] = 7          # parent after the node
    parents[9, 0] = 0          # root with a parent
    n_nodes[13] = 0            # empty
    n_nodes[17] = 65           # too many
    anc, depth, st = _run_mask(parents, n_nodes, dev)
    ra, rd, rs = oracle.tree_build_mask(parents, n_nodes)
    assert np.array_equal(st, rs)
    assert np.array_equal(anc, ra)
    assert np.array_equal(depth, rd)
    assert set(np.nonzero(st)[0].tolist()) == {5, 9, 13, 17}


def test_mask_n_max_smaller_than_64():
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(2))
    parents = np.stack([W.random_recursive_tree(rng, 8) for _ in range(7)]).astype(np.int32)
    n_nodes = np.array([8, 1, 2, 3, 5, 8, 7], np.int32)
    anc, depth, st = _run_mask(parents, n_nodes, dev)
    ra, rd, rs = oracle.tree_build_mask(parents, n_nodes)
    assert np.array_equal(anc, ra) and np.array_equal(depth, rd) and np.array_equal(st, rs)


# ------------------------------------------------------------------ commit
def _commit_case(seed, B, n_layers, Hkv, D, max_n=64, overlap_path=None):
    rng = np.random.Generator(np.random.PCG64(seed))
    P = 16
    L = rng.integers(0, 90, size=B).astype(np.int32)
    trees = [W.random_recursive_tree(rng, int(rng.integers(1, max_n + 1))) for _ in range(B)]
    N = np.array([len(t) for t in trees], np.int32)
    n_max = 64
    pages = [(int(L[b]) + int(N[b]) + P - 1) // P for b in range(B)]
    num_pages = sum(pages) + 3
    perm = rng.permutation(num_pages).astype(np.int32)
    pt = np.full((B, max(pages)), -1, np.int32)
    off = 0
    for b in range(B):
        pt[b, : pages[b]] = perm[off: off + pages[b]]
        off += pages[b]
    k = rng.integers(0, 1 << 16, size=(n_layers, num_pages, Hkv, P, D), dtype=np.uint16)
    v = rng.integers(0, 1 << 16, size=(n_layers, num_pages, Hkv, P, D), dtype=np.uint16)
    pn = np.full((B, n_max), -1, np.int32)
    acc = np.zeros(B, np.int32)
    for b in range(B):
        node = int(rng.integers(0, N[b]))
        path = oracle.ancestors_or_self(trees[b], node)
        pn[b, : len(path)] = path
        acc[b] = len(path) - 1
    if overlap_path is not None:
        N[0] = max(N[0], max(overlap_path) + 1)
        trees[0] = W.chain_tree(int(N[0]))
        L[0] = min(L[0], pt.shape[1] * P - int(N[0]))
        pn[0] = -1
        pn[0, : len(overlap_path)] = overlap_path
        acc[0] = len(overlap_path) - 1
    return k, v, pt, L, N, acc, pn


@pytest.mark.parametrize("seed,B,n_layers,Hkv,D", [(0, 4, 1, 8, 128), (1, 6, 3, 2, 64), (2, 3, 2, 32, 128),
                                                    (3, 8, 5, 8, 128)])
def test_commit_bit_exact(seed, B, n_layers, Hkv, D):
    dev = require_gpu()
    k, v, pt, L, N, acc, pn = _commit_case(seed, B, n_layers, Hkv, D)
    kd = to_dev(k.view(np.int16), dev).view(torch.bfloat16)
    vd = to_dev(v.view(np.int16), dev).view(torch.bfloat16)
    st = torch.zeros(B, dtype=torch.int32, device=dev)
    slots, new_len = tvb.kv_commit_path(kd, vd, to_dev(pt, dev), to_dev(L, dev), to_dev(N, dev), to_dev(acc, dev),
                                        to_dev(pn, dev), st)
    torch.cuda.synchronize()
    ke, ve, rs, rl, rst = oracle.kv_commit_path(k, v, pt, L, N, acc, pn)
    assert np.array_equal(st.cpu().numpy(), rst)
    assert np.array_equal(slots.cpu().numpy(), rs)
    assert np.array_equal(new_len.cpu().numpy(), rl)
    assert np.array_equal(kd.view(torch.int16).cpu().numpy().view(np.uint16), ke)
    assert np.array_equal(vd.view(torch.int16).cpu().numpy().view(np.uint16), ve)


def test_commit_overlapping_moves():
    """Path 0,2,5 style overlaps: a destination is an earlier move's source."""
    dev = require_gpu()
    for path in ([0, 2, 5], [0, 1, 3, 4, 9, 10], [0, 5, 6, 7, 8, 30], list(range(0, 64, 2))[:20]):
        k, v, pt, L, N, acc, pn = _commit_case(7, 2, 2, 4, 128, overlap_path=path)
        kd = to_dev(k.view(np.int16), dev).view(torch.bfloat16)
        vd = to_dev(v.view(np.int16), dev).view(torch.bfloat16)
        st = torch.zeros(2, dtype=torch.int32, device=dev)
        slots, new_len = tvb.kv_commit_path(kd, vd, to_dev(pt, dev), to_dev(L, dev), to_dev(N, dev),
                                            to_dev(acc, dev), to_dev(pn, dev), st)
        torch.cuda.synchronize()
        ke, ve, rs, rl, rst = oracle.kv_commit_path(k, v, pt, L, N, acc, pn)
        assert (rst == 0).all() and np.array_equal(st.cpu().numpy(), rst)
        assert np.array_equal(kd.view(torch.int16).cpu().numpy().view(np.uint16), ke)
        assert np.array_equal(vd.view(torch.int16).cpu().numpy().view(np.uint16), ve)
        assert np.array_equal(slots.cpu().numpy(), rs)


def test_commit_error_status():
    dev = require_gpu()
    k, v, pt, L, N, acc, pn = _commit_case(11, 4, 1, 2, 64)
    pn[1, 1], pn[1, 2] = 5, 3 if acc[1] >= 2 else pn[1, 2]
    acc[1] = max(acc[1], 2)
    N[1] = max(N[1], 6)
    pt2 = pt.copy()
    pt2[2, (int(L[2]) // 16)] = 10 ** 6          # page of the root out of range
    kd = to_dev(k.view(np.int16), dev).view(torch.bfloat16)
    vd = to_dev(v.view(np.int16), dev).view(torch.bfloat16)
    st = torch.zeros(4, dtype=torch.int32, device=dev)
    st[3] = tvb.TV_DEV_BAD_TREE                   # skipped on entry
    slots, new_len = tvb.kv_commit_path(kd, vd, to_dev(pt2, dev), to_dev(L, dev), to_dev(N, dev), to_dev(acc, dev),
                                        to_dev(pn, dev), st)
    torch.cuda.synchronize()
    s = st.cpu().numpy()
    assert s[1] & tvb.TV_DEV_BAD_TREE and s[2] & tvb.TV_DEV_PAGE_OOB and s[0] == 0
    nl = new_len.cpu().numpy()
    assert nl[1] == L[1] and nl[2] == L[2] and nl[3] == L[3]
    assert (slots.cpu().numpy()[1:] == -1).all()
