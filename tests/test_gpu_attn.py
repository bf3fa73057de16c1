"""GPU parity of tv_tree_verify_attn against the fp64 oracle.

Tolerance (bf16 inputs, fp32 accumulation, bf16 P and output): max |err| <=
1e-2 and mean |err| <= 1e-3 per compared set of rows; the log-sum-exp within
2e-3.  The hand-shaped edge cases (rows over a handful of keys, outputs as
large as single V entries) add the bf16 output's own rounding, 2^-8 |ref|,
to the per-element bound; the Llama-shaped workloads use the plain bound.  Invariances (page placement, non-ancestor K/V, garbage past the data)
are checked bit for bit on the GPU output.
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from gpu_helpers import DevWorkload, compare_attn, require_gpu, sample_rows, to_dev, bf16_dev

pytestmark = pytest.mark.gpu


def _oracle(w, rows=None):
    return oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table, w.prefix_len, w.n_nodes,
                                   w.parents, w.scale, rows=rows)


CASES = [
    # (B, Hq, Hkv, D, prefixes, tree kinds)
    (1, 4, 4, 64, [0], ["chain8"]),
    (1, 4, 4, 64, [1], ["star5"]),
    (2, 8, 2, 64, [15, 16], ["rand12", "chain17"]),
    (3, 8, 8, 128, [17, 127, 128], ["rand64", "chain64", "star64"]),
    (2, 32, 4, 128, [129, 300], ["rand33", "one"]),      # G = 8
    (2, 32, 2, 128, [250, 5], ["rand64", "chain40"]),    # G = 16: four M-tile pairs
    (4, 8, 4, 128, [1000, 2047, 513, 64], ["rand63", "rand64", "chain2", "one"]),  # G = 2
    (1, 64, 8, 128, [4000], ["rand64"]),                 # 70B-shaped, one request
    (2, 16, 16, 64, [700, 33], ["rand64", "rand31"]),    # MHA, D = 64
    (2, 64, 1, 128, [300, 1], ["rand64", "rand9"]),      # G = 64 (one KV head): two nodes per M tile
    (2, 32, 1, 64, [64, 65], ["chain64", "rand20"]),     # G = 32, D = 64
]


def _tree(kind, rng):
    if kind == "one":
        return W.chain_tree(1)
    if kind.startswith("chain"):
        return W.chain_tree(int(kind[5:]))
    if kind.startswith("star"):
        return W.star_tree(int(kind[4:]))
    return W.random_recursive_tree(rng, int(kind[4:]))


@pytest.mark.parametrize("case", range(len(CASES)))
def test_attn_edge_cases(case):
    dev = require_gpu()
    B, Hq, Hkv, D, prefixes, kinds = CASES[case]
    rng = np.random.Generator(np.random.PCG64(500 + case))
    w = W.make_custom(B=B, Hq=Hq, Hkv=Hkv, D=D, prefix_len=prefixes, parents_list=[_tree(k, rng) for k in kinds],
                      seed=900 + case, n_max=64 if case % 2 else None)
    dw = DevWorkload(w, dev, logits=False)
    out, lse, st = dw.attn()
    ref_out, ref_lse, ref_st = _oracle(w)
    assert np.array_equal(st, ref_st) and (st == 0).all()
    compare_attn(out, lse, ref_out, ref_lse, w, output_rounding=True)


def test_attn_tiny_config_full():
    dev = require_gpu()
    w = W.make_workload("tiny")
    out, lse, st = DevWorkload(w, dev, logits=False).attn()
    ref_out, ref_lse, _ = _oracle(w)
    assert (st == 0).all()
    compare_attn(out, lse, ref_out, ref_lse, w)


def test_attn_llama2_7b_config_full():
    dev = require_gpu()
    w = W.make_workload("llama2_7b", with_logits=False)
    out, lse, st = DevWorkload(w, dev, logits=False).attn()
    ref_out, ref_lse, _ = _oracle(w)
    assert (st == 0).all()
    compare_attn(out, lse, ref_out, ref_lse, w)


@pytest.mark.parametrize("name", ["llama3_70b", "serving", "long"])
def test_attn_large_configs_sampled(name):
    dev = require_gpu()
    w = W.make_workload(name, with_logits=False)
    out, lse, st = DevWorkload(w, dev, logits=False).attn()
    assert (st == 0).all()
    rows = sample_rows(w, np.random.Generator(np.random.PCG64(1)))
    ref_out, ref_lse, _ = _oracle(w, rows=rows)
    compare_attn(out, lse, ref_out, ref_lse, w, rows=rows)
    # every valid row is finite
    for b in range(w.B):
        assert np.isfinite(out[b, : int(w.n_nodes[b])]).all()


@pytest.mark.parametrize("name,which", [("llama3_70b", "longest"), ("llama3_70b", "shortest"), ("long", "first")])
def test_attn_full_request_every_row(name, which):
    """Every (node, query head) row of one whole request of a G = 8 workload at
    the plain bound: all eight KV heads, both M-tile pairs of each, and every
    split of the request's key range with its merge (the sampled comparison
    above covers a few rows of every request; this covers one request whole)."""
    dev = require_gpu()
    w = W.make_workload(name, with_logits=False)
    out, lse, st = DevWorkload(w, dev, logits=False).attn()
    assert (st == 0).all()
    b = {"longest": int(np.argmax(w.prefix_len)), "shortest": int(np.argmin(w.prefix_len)), "first": 0}[which]
    rows = [(b, i, h) for i in range(int(w.n_nodes[b])) for h in range(w.Hq)]
    ref_out, ref_lse, _ = _oracle(w, rows=rows)
    mx, mean = compare_attn(out, lse, ref_out, ref_lse, w, rows=rows)
    print(f"{name} request {b} (prefix {int(w.prefix_len[b])}): {len(rows)} rows, max err {mx:.2e}, mean {mean:.2e}")


def test_attn_page_shuffle_bit_exact():
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(44))
    w = W.make_custom(B=2, Hq=16, Hkv=4, D=128, prefix_len=[333, 70],
                      parents_list=[W.random_recursive_tree(rng, 40), W.chain_tree(9)], seed=3, extra_pages=5)
    dw = DevWorkload(w, dev, logits=False)
    out1, lse1, _ = dw.attn()
    perm = rng.permutation(w.num_pages)
    inv = np.argsort(perm)
    pt = w.page_table.copy()
    pt[pt >= 0] = inv[pt[pt >= 0]]
    out2, lse2, _ = dw.attn(k=bf16_dev(w.k_bits[perm], dev), v=bf16_dev(w.v_bits[perm], dev),
                            page_table=to_dev(pt, dev))
    for b in range(w.B):
        n = int(w.n_nodes[b])
        assert np.array_equal(out1[b, :n], out2[b, :n])
        assert np.array_equal(lse1[b, :n], lse2[b, :n])


def test_attn_non_ancestor_and_garbage_do_not_matter():
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(45))
    parents = W.random_recursive_tree(rng, 30)
    L = 100
    w = W.make_custom(B=1, Hq=8, Hkv=2, D=128, prefix_len=[L], parents_list=[parents], seed=8, extra_pages=2)
    dw = DevWorkload(w, dev, logits=False)
    base, lse0, _ = dw.attn()
    anc, _, _ = oracle.tree_build_mask(w.parents, w.n_nodes)
    k2, v2 = w.k_bits.copy(), w.v_bits.copy()
    j = 17
    pos = L + j
    # a moderate perturbation keeps |out| < 2, where a bf16 ulp is <= 2^-7
    k2[w.page_table[0, pos // 16], :, pos % 16] = W.to_bf16_bits(np.full((2, 128), 1.5, np.float32))
    v2[w.page_table[0, pos // 16], :, pos % 16] = W.to_bf16_bits(np.full((2, 128), -1.5, np.float32))
    # poison every slot past L + N in the last page, and the unused pages, with NaN / Inf
    end = L + 30
    last = w.page_table[0, (end - 1) // 16]
    for s in range(end % 16 or 16, 16):
        k2[last, :, s] = 0x7FC0
        v2[last, :, s] = 0x7F80
    used = set(w.page_table[0][w.page_table[0] >= 0].tolist())
    for pg in range(w.num_pages):
        if pg not in used:
            k2[pg], v2[pg] = 0x7FC0, 0xFF80
    out, lse, st = dw.attn(k=bf16_dev(k2, dev), v=bf16_dev(v2, dev))
    assert (st == 0).all()
    for i in range(30):
        sees = (int(anc[0, i]) >> j) & 1
        if not sees:
            assert np.array_equal(out[0, i], base[0, i]), i
            assert np.array_equal(lse[0, i], lse0[0, i])
        else:
            assert not np.array_equal(out[0, i], base[0, i])
    assert np.isfinite(out[0, :30]).all()
    ref_out, ref_lse, _ = oracle.tree_verify_attn(w.q_bits, k2, v2, w.page_table, w.prefix_len, w.n_nodes,
                                                  w.parents, w.scale)
    compare_attn(out, lse, ref_out, ref_lse, w)


def test_attn_status_errors_zero_outputs():
    dev = require_gpu()
    w = W.make_custom(B=4, Hq=8, Hkv=4, D=64, prefix_len=[40, 50, 60, 10],
                      parents_list=[W.chain_tree(5)] * 4, seed=12)
    dw = DevWorkload(w, dev, logits=False)
    anc, _, status = dw.mask()
    pt = w.page_table.copy()
    pt[1, 2] = w.num_pages + 100          # page of request 1 out of range
    L = w.prefix_len.copy()
    L[2] = 16 * w.max_pages                # request 2 no longer fits
    status[3] = tvb.TV_DEV_BAD_TREE        # request 3 flagged on entry
    out = torch.full_like(dw.q, 5.0)
    o, lse = tvb.tree_verify_attn(dw.q, dw.k, dw.v, to_dev(pt, dev), to_dev(L, dev), dw.n_nodes, anc, w.scale,
                                  status, out=out)
    torch.cuda.synchronize()
    st = status.cpu().numpy()
    assert st[0] == 0 and st[1] == tvb.TV_DEV_PAGE_OOB and st[2] == tvb.TV_DEV_CAPACITY
    assert st[3] == tvb.TV_DEV_BAD_TREE
    of = o.float().cpu().numpy()
    assert (of[1:] == 0).all()
    ref_out, ref_lse, _ = _oracle(w, rows=[(0, i, h) for i in range(5) for h in range(8)])
    compare_attn(of, lse.cpu().numpy(), ref_out, ref_lse, w, rows=[(0, i, h) for i in range(5) for h in range(8)])


def test_attn_host_argument_errors():
    dev = require_gpu()
    w = W.make_custom(B=1, Hq=4, Hkv=4, D=64, prefix_len=[10], parents_list=[W.chain_tree(3)], seed=1)
    dw = DevWorkload(w, dev, logits=False)
    anc, _, status = dw.mask()
    lib = tvb.load_library()
    ws = tvb.new_attn_workspace(1, w.n_max, 4, 4, 64, dev)
    o = torch.empty_like(dw.q)
    import ctypes
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [P(dw.q), P(dw.k), P(dw.v), w.num_pages, P(dw.page_table), w.max_pages, P(dw.prefix_len),
            P(dw.n_nodes), P(anc), 1, w.n_max, 4, 4, 64, 16, 0.125, P(o), None, P(ws), ws.numel(), P(status), s]
    a = list(args); a[13] = 96                        # head dim
    assert lib.tv_tree_verify_attn(*a) == tvb.TV_ERR_UNSUPPORTED
    a = list(args); a[14] = 32                        # page size
    assert lib.tv_tree_verify_attn(*a) == tvb.TV_ERR_UNSUPPORTED
    a = list(args); a[11] = 6; a[12] = 4              # Hq not a multiple of Hkv
    assert lib.tv_tree_verify_attn(*a) == tvb.TV_ERR_UNSUPPORTED
    a = list(args); a[19] = 1024                      # workspace too small
    assert lib.tv_tree_verify_attn(*a) == tvb.TV_ERR_WORKSPACE
    a = list(args); a[0] = None                       # NULL q
    assert lib.tv_tree_verify_attn(*a) == tvb.TV_ERR_INVALID_ARG
    assert b"NULL" in lib.tv_last_error()
    assert lib.tv_tree_verify_attn(*args) == tvb.TV_OK
    torch.cuda.synchronize()


def test_attn_many_small_requests():
    """300 requests of 1..12 nodes over short, ragged prefixes: the plan over many
    requests, items that start mid-request and requests with a single KV tile."""
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(77))
    B = 300
    trees = [W.random_recursive_tree(rng, int(rng.integers(1, 13))) for _ in range(B)]
    prefixes = rng.integers(0, 400, size=B).tolist()
    w = W.make_custom(B=B, Hq=8, Hkv=2, D=64, prefix_len=prefixes, parents_list=trees, seed=78, n_max=12)
    dw = DevWorkload(w, dev, logits=False)
    out, lse, st = dw.attn()
    ref_out, ref_lse, ref_st = _oracle(w)
    assert np.array_equal(st, ref_st) and (st == 0).all()
    compare_attn(out, lse, ref_out, ref_lse, w, output_rounding=True)


def test_attn_split_partials_past_fp16_range():
    """Split partials are stored in fp16; a row with a value past the fp16 range
    is stored again as O / max |O|.  One KV head over a 6000-key prefix splits
    across ~30 CTAs; the V row of tree node 5 carries an offset of 1e9, so the
    rows of node 5 and its descendants have partials and outputs past the fp16
    range while the other rows of the same warps do not.  An output dominated by
    one V value carries that key's probability rounded to bf16 (up to 2^-8
    relative), the bf16 output's rounding (up to 2^-8) and the fp16 partial's
    (2^-11 of its largest value): the bound is 1e-2 + (2^-7 + 2^-10) |ref|."""
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(91))
    parents = W.random_recursive_tree(rng, 40)
    L, j = 6000, 5
    w = W.make_custom(B=1, Hq=8, Hkv=1, D=128, prefix_len=[L], parents_list=[parents], seed=92)
    v = oracle.bf16_to_f64(w.v_bits)
    pos = L + j
    v[w.page_table[0, pos // 16], 0, pos % 16] += 1.0e9
    w.v_bits = W.to_bf16_bits(v.astype(np.float32))
    out, lse, st = DevWorkload(w, dev, logits=False).attn()
    assert (st == 0).all()
    ref_out, ref_lse, _ = _oracle(w)
    n = int(w.n_nodes[0])
    big = np.abs(ref_out[0, :n]).max(axis=-1) > 65504.0
    assert big.any() and (~big).any()                      # both paths are taken
    got, ref = out[0, :n], ref_out[0, :n]
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    rel = err[big] / np.abs(ref[big])
    assert np.all(err <= 1e-2 + (2.0 ** -7 + 2.0 ** -10) * np.abs(ref)), \
        f"large rows: max relative error {rel.max():.3e}; other rows: max error {err[~big].max():.3e}"
    assert np.abs(lse[0, :n] - ref_lse[0, :n]).max() <= 2e-3


def test_attn_stray_mask_bits_ignored():
    """Bits j >= n_nodes of a node's ancestor word name no node of the tree.
    The attention ignores them: with every such bit set (and the cache slots
    they would name filled with large keys) the outputs equal those of the
    clean words bit for bit."""
    dev = require_gpu()
    rng = np.random.Generator(np.random.PCG64(46))
    trees = [W.random_recursive_tree(rng, 20), W.chain_tree(5), W.random_recursive_tree(rng, 63)]
    w = W.make_custom(B=3, Hq=16, Hkv=4, D=128, prefix_len=[100, 37, 500], parents_list=trees, seed=47,
                      n_max=64)
    k2 = w.k_bits.copy()
    for b in range(w.B):
        L, N = int(w.prefix_len[b]), int(w.n_nodes[b])
        cap = 16 * int((w.page_table[b] >= 0).sum())
        for pos in range(L + N, cap):          # slots past the tree in the request's own pages
            k2[w.page_table[b, pos // 16], :, pos % 16] = W.to_bf16_bits(np.full((w.Hkv, w.D), 8.0, np.float32))
    dw = DevWorkload(w, dev, logits=False)
    kd = bf16_dev(k2, dev)
    out0, lse0, st0 = dw.attn(k=kd)
    anc, _, status = dw.mask()
    words = anc.cpu().numpy().view(np.uint64).copy()
    for b in range(w.B):
        N = int(w.n_nodes[b])
        stray = np.uint64(0) if N >= 64 else ~np.uint64((1 << N) - 1)
        words[b, :N] |= stray
    anc2 = to_dev(words.view(np.int64), dev)
    out1, lse1, st1 = dw.attn(status=status, anc=anc2, k=kd)
    assert (st0 == 0).all() and (st1 == 0).all()
    for b in range(w.B):
        n = int(w.n_nodes[b])
        assert np.array_equal(out0[b, :n], out1[b, :n]), b
        assert np.array_equal(lse0[b, :n], lse1[b, :n]), b
