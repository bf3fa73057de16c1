"""GPU parity of the 3-bit KV path against the oracle.

tv_kv_quantize_q3: codes and parameters bit-exact against ``quantize_q3``
(both take the integer decisions in float32 IEEE steps with fp16
parameters).  tv_tree_verify_attn_q3: against ``tree_verify_attn_q3`` (the
cache decoded by ``dequantize_q3``, then the plain attention), with the
tolerances of the bf16 attention (max |err| <= 1e-2, mean <= 1e-3, log-sum-exp
within 2e-3; hand-shaped edge cases add the bf16 output's own rounding), and
the decode exactly: a node that sees a single key returns that key's decoded V
row bit for bit.  (troisinh.com "EAGLE - Draft head ...", further reading:
INT4/INT3 KV-cache quantisation.)
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from gpu_helpers import bf16_dev, compare_attn, require_gpu, sample_rows, to_dev

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- encoder
def _check_enc(bits, dev):
    codes, params = tvb.kv_quantize_q3(bf16_dev(bits, dev))
    torch.cuda.synchronize()
    rc, rp = oracle.quantize_q3(bits)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(params.cpu().numpy().view(np.uint16), rp.view(np.uint16))


@pytest.mark.parametrize("D,rows,seed", [(32, 1, 0), (64, 333, 1), (128, 5000, 2), (256, 77, 3)])
def test_encoder_random_rows(D, rows, seed):
    dev = require_gpu()
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, D)) * rng.uniform(1e-3, 50, size=(rows, 1))).astype(np.float32)
    _check_enc(W.to_bf16_bits(x), dev)


def test_encoder_constant_groups_ties_and_extremes():
    dev = require_gpu()
    rng = np.random.default_rng(4)
    rows = [np.full(128, 3.0),                                   # constant: scale 0
            np.repeat([0.0, 1.0, -2.5, 7.0], 32),                # constant per group
            np.tile(np.arange(32) * 0.25 % 3.75, 4),             # half steps of the scale: ties
            np.tile(np.linspace(-1, 1, 32), 4) * 60000.0,        # near the fp16 range
            np.tile(np.linspace(0, 1, 32), 4) * 1e-6,            # tiny: fp16 subnormal scales
            rng.integers(-4, 4, size=128).astype(np.float64)]    # small integers
    _check_enc(W.to_bf16_bits(np.stack(rows).astype(np.float32)), dev)


def test_encoder_paged_cache_llama2_7b_shape():
    dev = require_gpu()
    w = W.make_workload("llama2_7b", with_logits=False)
    _check_enc(w.k_bits, dev)


# ---------------------------------------------------------------- attention
def _cache(w, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    kc, kp = W.make_q3_cache(rng, w.num_pages, w.Hkv, w.D)
    vc, vp = W.make_q3_cache(rng, w.num_pages, w.Hkv, w.D)
    return kc, kp, vc, vp


def _run(w, cache, dev, page_table=None, prefix_len=None, status=None, out=None):
    kc, kp, vc, vp = (to_dev(a, dev) for a in cache)
    parents, n_nodes = to_dev(w.parents, dev), to_dev(w.n_nodes, dev)
    anc, _, st = tvb.tree_build_mask(parents, n_nodes)
    if status is not None:
        st = status(st)
    o, lse = tvb.tree_verify_attn_q3(bf16_dev(w.q_bits, dev), kc, kp, vc, vp,
                                     to_dev(w.page_table if page_table is None else page_table, dev),
                                     to_dev(w.prefix_len if prefix_len is None else prefix_len, dev), n_nodes,
                                     anc, w.scale, st, out=out)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy(), st.cpu().numpy()


def _oracle(w, cache, rows=None):
    kc, kp, vc, vp = cache
    return oracle.tree_verify_attn_q3(w.q_bits, kc, kp, vc, vp, w.page_table, w.prefix_len, w.n_nodes, w.parents,
                                      w.scale, rows=rows)


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
    (4, 8, 4, 128, [1000, 2047, 513, 64], ["rand63", "rand64", "chain2", "one"]),  # G = 2
    (1, 64, 8, 128, [4000], ["rand64"]),                 # 70B-shaped, one request
    (2, 16, 16, 64, [700, 33], ["rand64", "rand31"]),    # MHA, D = 64
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_q3_attn_edge_cases(case):
    dev = require_gpu()
    B, Hq, Hkv, D, prefixes, kinds = CASES[case]
    rng = np.random.Generator(np.random.PCG64(800 + case))
    w = W.make_custom(B=B, Hq=Hq, Hkv=Hkv, D=D, prefix_len=prefixes, parents_list=[_tree(k, rng) for k in kinds],
                      seed=1500 + case, n_max=64 if case % 2 else None, extra_pages=case % 3)
    cache = _cache(w, 1600 + case)
    out, lse, st = _run(w, cache, dev)
    ref_out, ref_lse, ref_st = _oracle(w, cache)
    assert np.array_equal(st, ref_st) and (st == 0).all()
    compare_attn(out, lse, ref_out, ref_lse, w, output_rounding=True)


def test_q3_attn_tiny_and_7b_full():
    dev = require_gpu()
    for name, seed in (("tiny", 23), ("llama2_7b", 24)):
        w = W.make_workload(name, with_logits=False)
        cache = _cache(w, seed)
        out, lse, st = _run(w, cache, dev)
        ref_out, ref_lse, _ = _oracle(w, cache)
        assert (st == 0).all()
        compare_attn(out, lse, ref_out, ref_lse, w)


def test_q3_attn_70b_sampled():
    dev = require_gpu()
    w = W.make_workload("llama3_70b", with_logits=False)
    cache = _cache(w, 33)
    out, lse, st = _run(w, cache, dev)
    assert (st == 0).all()
    rows = sample_rows(w, np.random.Generator(np.random.PCG64(4)), per_request=8)
    rng = np.random.Generator(np.random.PCG64(5))
    rows = [rows[i] for i in sorted(rng.choice(len(rows), size=min(len(rows), 64), replace=False))]
    bs = sorted({b for b, _, _ in rows})
    pos = {b: k for k, b in enumerate(bs)}
    pt = w.page_table[bs]
    used = np.unique(pt[pt >= 0])
    remap = np.zeros(w.num_pages, dtype=np.int32)
    remap[used] = np.arange(len(used), dtype=np.int32)
    pt2 = np.where(pt >= 0, remap[np.maximum(pt, 0)], -1).astype(np.int32)
    kc, kp, vc, vp = (a[used] for a in cache)
    sub_rows = [(pos[b], i, h) for b, i, h in rows]
    ref_out, ref_lse, _ = oracle.tree_verify_attn_q3(w.q_bits[bs], kc, kp, vc, vp, pt2, w.prefix_len[bs],
                                                     w.n_nodes[bs], w.parents[bs], w.scale, rows=sub_rows)
    compare_attn(out[bs], lse[bs], ref_out, ref_lse, w, rows=sub_rows)


def test_q3_decode_exact_through_single_key_rows():
    """Requests with no prefix and a lone root: the root sees one key, so its
    output is that key's decoded V row, bit for bit, for every head of the
    group; the log-sum-exp is scale * <q, k> of the decoded K row."""
    dev = require_gpu()
    B, Hq, Hkv, D = 200, 8, 4, 128
    w = W.make_custom(B=B, Hq=Hq, Hkv=Hkv, D=D, prefix_len=[0] * B, parents_list=[W.chain_tree(1)] * B, seed=43,
                      extra_pages=7)
    cache = _cache(w, 44)
    out, lse, st = _run(w, cache, dev)
    assert (st == 0).all()
    kc, kp, vc, vp = cache
    G = Hq // Hkv
    for b in range(B):
        pg = int(w.page_table[b, 0])
        vdec = oracle.bf16_to_f64(oracle.dequantize_q3(vc[pg, :, 0], vp[pg, :, 0]))   # [Hkv, D]
        kdec = oracle.bf16_to_f64(oracle.dequantize_q3(kc[pg, :, 0], kp[pg, :, 0]))
        for h in range(Hq):
            assert np.array_equal(out[b, 0, h], vdec[h // G]), (b, h)
            s = w.scale * float(oracle.bf16_to_f64(w.q_bits[b, 0, h]) @ kdec[h // G])
            assert abs(float(lse[b, 0, h]) - s) <= 1e-4 * max(1.0, abs(s)), (b, h)


def test_q3_encoded_cache_end_to_end():
    """bf16 cache -> tv_kv_quantize_q3 -> tv_tree_verify_attn_q3 against the
    oracle's encoder and quantised attention on the same bf16 cache."""
    dev = require_gpu()
    w = W.make_workload("tiny", with_logits=False)
    kc, kp = tvb.kv_quantize_q3(bf16_dev(w.k_bits, dev))
    vc, vp = tvb.kv_quantize_q3(bf16_dev(w.v_bits, dev))
    cache = tuple(t.cpu().numpy() for t in (kc, kp, vc, vp))
    rk, rkp = oracle.quantize_q3(w.k_bits)
    assert np.array_equal(cache[0], rk) and np.array_equal(cache[1].view(np.uint16), rkp.view(np.uint16))
    out, lse, st = _run(w, cache, dev)
    ref_out, ref_lse, _ = _oracle(w, cache)
    assert (st == 0).all()
    compare_attn(out, lse, ref_out, ref_lse, w)


def test_q3_status_errors_zero_outputs():
    dev = require_gpu()
    w = W.make_custom(B=4, Hq=8, Hkv=4, D=64, prefix_len=[40, 50, 60, 10], parents_list=[W.chain_tree(5)] * 4,
                      seed=63)
    cache = _cache(w, 64)
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
