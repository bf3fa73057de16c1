"""GPU parity of tv_tree_verify_attn_q4 (tree attention over a 4-bit paged
KV cache) against the fp64 oracle, which decodes the cache with
``dequantize_q4`` and runs its plain attention on the decoded values.

Tolerances are those of the bf16 attention (max |err| <= 1e-2, mean <= 1e-3,
log-sum-exp within 2e-3; hand-shaped edge cases add the bf16 output's own
rounding, 2^-8 |ref|).  The decode itself is checked exactly: a node that
sees a single key returns that key's decoded V row bit for bit.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from gpu_helpers import compare_attn, require_gpu, sample_rows, to_dev, bf16_dev

pytestmark = pytest.mark.gpu


def _q4_cache(w, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    kc, kp = W.make_q4_cache(rng, w.num_pages, w.Hkv, w.D)
    vc, vp = W.make_q4_cache(rng, w.num_pages, w.Hkv, w.D)
    return kc, kp, vc, vp


def _run(w, cache, dev, page_table=None, prefix_len=None, status=None, out=None):
    kc, kp, vc, vp = (to_dev(a, dev) for a in cache)
    parents, n_nodes = to_dev(w.parents, dev), to_dev(w.n_nodes, dev)
    anc, _, st = tvb.tree_build_mask(parents, n_nodes)
    if status is not None:
        st = status(st)
    o, lse = tvb.tree_verify_attn_q4(bf16_dev(w.q_bits, dev), kc, kp, vc, vp,
                                     to_dev(w.page_table if page_table is None else page_table, dev),
                                     to_dev(w.prefix_len if prefix_len is None else prefix_len, dev), n_nodes,
                                     anc, w.scale, st, out=out)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy(), st.cpu().numpy()


def _oracle(w, cache, rows=None):
    kc, kp, vc, vp = cache
    return oracle.tree_verify_attn_q4(w.q_bits, kc, kp, vc, vp, w.page_table, w.prefix_len, w.n_nodes, w.parents,
                                      w.scale, rows=rows)


def _oracle_sampled(w, cache, rows):
    """The oracle on the requests of `rows` only, over their own pages (the
    decode of a whole large cache in fp64 is not needed for a sample)."""
    bs = sorted({b for b, _, _ in rows})
    pos = {b: k for k, b in enumerate(bs)}
    pt = w.page_table[bs]
    used = np.unique(pt[pt >= 0])
    remap = np.zeros(w.num_pages, dtype=np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    pt2 = np.where(pt >= 0, remap[np.maximum(pt, 0)], -1).astype(np.int32)
    kc, kp, vc, vp = (a[used] for a in cache)
    sub_rows = [(pos[b], i, h) for b, i, h in rows]
    ref_out, ref_lse, _ = oracle.tree_verify_attn_q4(w.q_bits[bs], kc, kp, vc, vp, pt2, w.prefix_len[bs],
                                                     w.n_nodes[bs], w.parents[bs], w.scale, rows=sub_rows)
    return bs, sub_rows, ref_out, ref_lse


def _tree(kind, rng):
    if kind == "one":
        return W.chain_tree(1)
    if kind.startswith("chain"):
        return W.chain_tree(int(kind[5:]))
    if kind.startswith("star"):
        return W.star_tree(int(kind[4:]))
    return W.random_recursive_tree(rng, int(kind[4:]))


CASES = [
    # (B, Hq, Hkv, D, prefixes, tree kinds)
    (1, 4, 4, 64, [0], ["chain8"]),
    (2, 8, 2, 64, [15, 16], ["rand12", "chain17"]),
    (3, 8, 8, 128, [17, 127, 128], ["rand64", "chain64", "star64"]),
    (2, 32, 4, 128, [129, 300], ["rand33", "one"]),      # G = 8
    (2, 32, 2, 128, [250, 5], ["rand64", "chain40"]),    # G = 16: four M-tile pairs
    (4, 8, 4, 128, [1000, 2047, 513, 64], ["rand63", "rand64", "chain2", "one"]),  # G = 2
    (1, 64, 8, 128, [4000], ["rand64"]),                 # 70B-shaped, one request
    (2, 16, 16, 64, [700, 33], ["rand64", "rand31"]),    # MHA, D = 64
    (2, 64, 1, 128, [300, 1], ["rand64", "rand9"]),      # G = 64 (one KV head)
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_q4_attn_edge_cases(case):
    dev = require_gpu()
    B, Hq, Hkv, D, prefixes, kinds = CASES[case]
    rng = np.random.Generator(np.random.PCG64(700 + case))
    w = W.make_custom(B=B, Hq=Hq, Hkv=Hkv, D=D, prefix_len=prefixes, parents_list=[_tree(k, rng) for k in kinds],
                      seed=1100 + case, n_max=64 if case % 2 else None, extra_pages=case % 3)
    cache = _q4_cache(w, 1300 + case)
    out, lse, st = _run(w, cache, dev)
    ref_out, ref_lse, ref_st = _oracle(w, cache)
    assert np.array_equal(st, ref_st) and (st == 0).all()
    compare_attn(out, lse, ref_out, ref_lse, w, output_rounding=True)


def test_q4_attn_tiny_and_7b_full():
    dev = require_gpu()
    for name, seed in (("tiny", 21), ("llama2_7b", 22)):
        w = W.make_workload(name, with_logits=False)
        cache = _q4_cache(w, seed)
        out, lse, st = _run(w, cache, dev)
        ref_out, ref_lse, _ = _oracle(w, cache)
        assert (st == 0).all()
        compare_attn(out, lse, ref_out, ref_lse, w)


@pytest.mark.parametrize("name", ["llama3_70b", "serving", "long"])
def test_q4_attn_large_configs_sampled(name):
    dev = require_gpu()
    w = W.make_workload(name, with_logits=False)
    cache = _q4_cache(w, 31)
    out, lse, st = _run(w, cache, dev)
    assert (st == 0).all()
    rows = sample_rows(w, np.random.Generator(np.random.PCG64(2)), per_request=8)
    rng = np.random.Generator(np.random.PCG64(3))
    rows = [rows[i] for i in sorted(rng.choice(len(rows), size=min(len(rows), 96), replace=False))]
    bs, sub_rows, ref_out, ref_lse = _oracle_sampled(w, cache, rows)
    compare_attn(out[bs], lse[bs], ref_out, ref_lse, w, rows=sub_rows)
    for b in range(w.B):
        assert np.isfinite(out[b, : int(w.n_nodes[b])]).all()


def test_q4_decode_exact_through_single_key_rows():
    """Requests with no prefix and a lone root: the root sees one key, so its
    output is that key's decoded V row, bit for bit, for every head of the
    group; the log-sum-exp is scale * <q, k> of the decoded K row."""
    dev = require_gpu()
    B, Hq, Hkv, D = 200, 8, 4, 128
    w = W.make_custom(B=B, Hq=Hq, Hkv=Hkv, D=D, prefix_len=[0] * B, parents_list=[W.chain_tree(1)] * B, seed=41,
                      extra_pages=7)
    cache = _q4_cache(w, 42)
    out, lse, st = _run(w, cache, dev)
    assert (st == 0).all()
    kc, kp, vc, vp = cache
    G = Hq // Hkv
    for b in range(B):
        pg = int(w.page_table[b, 0])
        vdec = oracle.bf16_to_f64(oracle.dequantize_q4(vc[pg, :, 0], vp[pg, :, 0]))   # [Hkv, D]
        kdec = oracle.bf16_to_f64(oracle.dequantize_q4(kc[pg, :, 0], kp[pg, :, 0]))
        for h in range(Hq):
            assert np.array_equal(out[b, 0, h], vdec[h // G]), (b, h)
            s = w.scale * float(oracle.bf16_to_f64(w.q_bits[b, 0, h]) @ kdec[h // G])
            assert abs(float(lse[b, 0, h]) - s) <= 1e-4 * max(1.0, abs(s)), (b, h)


def test_q4_matches_bf16_kernel_on_the_decoded_cache():
    """The 4-bit kernel against the bf16 kernel run on the oracle-decoded cache:
    the same products and probabilities, but the 4-bit plan charges each KV tile
    for its decode, so the two kernels cut a group's tiles into splits at other
    places.  A split's partial is stored in fp16 (O / max |O|), off by at most
    2^-11 of its largest value, and that value is at most max |V|; each output
    then takes one bf16 rounding (2^-7 relative at most).  So outputs agree to
    2^-7 |o| + 2 * 2^-11 max |V|, and the log-sum-exps (fp32 merges) to 1e-5."""
    dev = require_gpu()
    w = W.make_workload("llama2_7b", with_logits=False)
    cache = _q4_cache(w, 51)
    out, lse, _ = _run(w, cache, dev)
    kc, kp, vc, vp = cache
    kd, vd = oracle.dequantize_q4(kc, kp), oracle.dequantize_q4(vc, vp)
    parents, n_nodes = to_dev(w.parents, dev), to_dev(w.n_nodes, dev)
    anc, _, st = tvb.tree_build_mask(parents, n_nodes)
    o2, l2 = tvb.tree_verify_attn(bf16_dev(w.q_bits, dev), bf16_dev(kd, dev), bf16_dev(vd, dev),
                                  to_dev(w.page_table, dev), to_dev(w.prefix_len, dev), n_nodes, anc, w.scale, st)
    torch.cuda.synchronize()
    o2 = o2.float().cpu().numpy()
    n = int(w.n_nodes[0])
    d = np.abs(out[0, :n] - o2[0, :n])
    vmax = float(np.abs(oracle.bf16_to_f64(vd)).max())
    bound = 2.0 ** -7 * np.abs(o2[0, :n]) + 2.0 ** -10 * vmax
    print(f"max |d| {d.max():.3g}, max d / bound {(d / bound).max():.3f}, differing {(d > 0).mean():.4f}")
    assert np.all(d <= bound)
    assert np.abs(lse[0, :n] - l2.cpu().numpy()[0, :n]).max() <= 1e-5


def test_q4_status_errors_zero_outputs():
    dev = require_gpu()
    w = W.make_custom(B=4, Hq=8, Hkv=4, D=64, prefix_len=[40, 50, 60, 10], parents_list=[W.chain_tree(5)] * 4,
                      seed=61)
    cache = _q4_cache(w, 62)
    pt = w.page_table.copy()
    pt[1, 2] = w.num_pages + 100          # page of request 1 out of range
    L = w.prefix_len.copy()
    L[2] = 16 * w.max_pages                # request 2 no longer fits

    def flag3(st):
        st[3] = tvb.TV_DEV_BAD_TREE        # request 3 flagged on entry
        return st

    out0 = torch.full((4, w.n_max, 8, 64), 5.0, dtype=torch.bfloat16, device=dev)
    out, lse, st = _run(w, cache, dev, page_table=pt, prefix_len=L, status=flag3, out=out0)
    assert st[0] == 0 and st[1] == tvb.TV_DEV_PAGE_OOB and st[2] == tvb.TV_DEV_CAPACITY
    assert st[3] == tvb.TV_DEV_BAD_TREE
    assert (out[1:] == 0).all()
    rows = [(0, i, h) for i in range(5) for h in range(8)]
    ref_out, ref_lse, _ = _oracle(w, cache, rows=rows)
    compare_attn(out, lse, ref_out, ref_lse, w, rows=rows)


def test_q4_host_argument_errors():
    dev = require_gpu()
    w = W.make_custom(B=1, Hq=4, Hkv=4, D=64, prefix_len=[10], parents_list=[W.chain_tree(3)], seed=71)
    kc, kp, vc, vp = (to_dev(a, dev) for a in _q4_cache(w, 72))
    anc, _, status = tvb.tree_build_mask(to_dev(w.parents, dev), to_dev(w.n_nodes, dev))
    q = bf16_dev(w.q_bits, dev)
    pt, L, N = to_dev(w.page_table, dev), to_dev(w.prefix_len, dev), to_dev(w.n_nodes, dev)
    lib = tvb.load_library()
    ws = tvb.new_attn_workspace(1, w.n_max, 4, 4, 64, dev)
    o = torch.empty_like(q)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [P(q), P(kc), P(kp), P(vc), P(vp), w.num_pages, P(pt), w.max_pages, P(L), P(N), P(anc), 1, w.n_max, 4,
            4, 64, 16, 0.125, P(o), None, P(ws), ws.numel(), P(status), s]
    a = list(args); a[15] = 96                        # head dim
    assert lib.tv_tree_verify_attn_q4(*a) == tvb.TV_ERR_UNSUPPORTED
    a = list(args); a[11] = 257                       # more requests than the 4-bit plan holds
    assert lib.tv_tree_verify_attn_q4(*a) == tvb.TV_ERR_UNSUPPORTED
    a = list(args); a[2] = None                       # NULL K params
    assert lib.tv_tree_verify_attn_q4(*a) == tvb.TV_ERR_INVALID_ARG
    a = list(args); a[4] = ctypes.c_void_p(vp.data_ptr() + 4)   # misaligned V params
    assert lib.tv_tree_verify_attn_q4(*a) == tvb.TV_ERR_INVALID_ARG
    a = list(args); a[21] = 1024                      # workspace too small
    assert lib.tv_tree_verify_attn_q4(*a) == tvb.TV_ERR_WORKSPACE
    assert lib.tv_tree_verify_attn_q4(*args) == tvb.TV_OK
    torch.cuda.synchronize()
