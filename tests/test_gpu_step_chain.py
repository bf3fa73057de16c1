"""Two steps in one stream: this step's mask, attention, acceptance and commit,
then the next step's mask and attention over the cache the commit compacted,
with the commit's new_len output passed as the next step's prefix_len.

The attention reads the lengths, q, the page table and the cache before it waits
for the previous kernel in the stream; no call that writes those lets its
successor start early, so the next step must see the committed rows.  Expected
values are the oracle's alone: its greedy acceptance on the same logits (the
GPU's must equal it), its commit on a host copy of the cache with that path, and
its attention over the result.  (Tech Radar, SGLang EAGLE-2, section 2 sequence
diagram: the accepted branch's KV is kept, and the next step attends to it.)
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from gpu_helpers import bf16_dev, compare_attn, require_gpu, to_dev

pytestmark = pytest.mark.gpu


def test_commit_then_next_step_attention():
    dev = require_gpu()
    trees = [[-1, 0, 0, 1, 2, 4, 4, 2], [-1, 0, 1, 2, 3], [-1, 0, 0, 0, 3, 3, 5]]
    # position L + a + 1 (the next step's node) lies in the request's pages: a is at
    # most the tree's depth (3, 4 and 3), so L + a + 1 < L + N, or < 112 for request 1
    prefixes = [40, 101, 7]
    w = W.make_custom(B=3, Hq=8, Hkv=2, D=128, prefix_len=prefixes, parents_list=trees, seed=71, V=16)
    # one branch of each tree carries the target's argmax, so the commit moves rows
    tokens = w.tokens.copy()
    for b, path in enumerate([[0, 2, 4, 5], [0, 1, 2], [0, 3, 5]]):
        for par, node in zip(path[:-1], path[1:]):
            tokens[b, node] = int(np.argmax(w.target_logits[b, par]))

    # the oracle's two steps
    ref_acc = oracle.tree_accept_greedy(w.target_logits, tokens, w.parents, w.n_nodes)
    a_ref, p_ref = ref_acc["accept_len"], ref_acc["path_nodes"]
    assert (a_ref >= 2).all(), "each request's planted branch should be accepted"
    k2, v2, _, new_len_ref, _ = oracle.kv_commit_path(w.k_bits[None], w.v_bits[None], w.page_table, w.prefix_len,
                                                      w.n_nodes, a_ref, p_ref)
    B, Hq, D = w.B, w.Hq, w.D
    parents2 = np.full((B, 1), -1, dtype=np.int32)
    n2 = np.ones(B, dtype=np.int32)
    rng = np.random.Generator(np.random.PCG64(72))
    q2 = oracle.f64_to_bf16_bits_via_f32(rng.normal(size=(B, 1, Hq, D)))
    out_ref, lse_ref, _ = oracle.tree_verify_attn(q2, k2[0], v2[0], w.page_table, new_len_ref, n2, parents2, w.scale)

    # the same two steps on the GPU, one stream, no synchronisation in between
    parents_d, n_d = to_dev(w.parents, dev), to_dev(w.n_nodes, dev)
    pt_d = to_dev(w.page_table, dev)
    k_d, v_d = bf16_dev(w.k_bits, dev), bf16_dev(w.v_bits, dev)
    L_d = to_dev(w.prefix_len, dev)
    anc, depth, st = tvb.tree_build_mask(parents_d, n_d)
    out1, lse1 = tvb.tree_verify_attn(bf16_dev(w.q_bits, dev), k_d, v_d, pt_d, L_d, n_d, anc, w.scale, st)
    acc_len, path, _ = tvb.tree_accept(to_dev(w.target_logits, dev), None, to_dev(tokens, dev), parents_d, n_d, anc,
                                       depth, 0.0, None, None, st)
    _, new_len = tvb.kv_commit_path(k_d, v_d, pt_d, L_d, n_d, acc_len, path, st)
    n2_d = to_dev(n2, dev)
    anc2, _, st2 = tvb.tree_build_mask(to_dev(parents2, dev), n2_d)
    out, lse = tvb.tree_verify_attn(bf16_dev(q2, dev), k_d, v_d, pt_d, new_len, n2_d, anc2, w.scale, st2)
    torch.cuda.synchronize()

    out1_ref, lse1_ref, _ = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table, w.prefix_len,
                                                    w.n_nodes, w.parents, w.scale)
    compare_attn(out1.float().cpu().numpy(), lse1.cpu().numpy(), out1_ref, lse1_ref, w, output_rounding=True)
    np.testing.assert_array_equal(acc_len.cpu().numpy(), a_ref)
    np.testing.assert_array_equal(new_len.cpu().numpy(), new_len_ref)
    assert (st.cpu().numpy() == 0).all() and (st2.cpu().numpy() == 0).all()
    w2 = W.make_custom(B=B, Hq=Hq, Hkv=w.Hkv, D=D, prefix_len=list(new_len_ref), parents_list=[[-1]] * B, seed=73)
    compare_attn(out.float().cpu().numpy(), lse.cpu().numpy(), out_ref, lse_ref, w2, output_rounding=True)


@pytest.mark.parametrize("bits", [4, 3])
def test_quantize_then_lowbit_attention_same_stream(bits):
    """The encoder writes the low-bit cache and the attention reads it right after,
    in the same stream with no synchronisation: the attention's producers copy
    codes before their kernel waits for the previous one, and the encoder starts
    its successor only once it has finished.  Against the oracle's encoder and its
    attention over the decoded cache."""
    dev = require_gpu()
    w = W.make_workload("tiny", with_logits=False)
    quant = tvb.kv_quantize_q4 if bits == 4 else tvb.kv_quantize_q3
    attn = tvb.tree_verify_attn_q4 if bits == 4 else tvb.tree_verify_attn_q3
    oq = oracle.quantize_q4 if bits == 4 else oracle.quantize_q3
    oattn = oracle.tree_verify_attn_q4 if bits == 4 else oracle.tree_verify_attn_q3
    parents_d, n_d = to_dev(w.parents, dev), to_dev(w.n_nodes, dev)
    anc, _, st = tvb.tree_build_mask(parents_d, n_d)
    kc, kp = quant(bf16_dev(w.k_bits, dev))
    vc, vp = quant(bf16_dev(w.v_bits, dev))
    out, lse = attn(bf16_dev(w.q_bits, dev), kc, kp, vc, vp, to_dev(w.page_table, dev), to_dev(w.prefix_len, dev), n_d,
                    anc, w.scale, st)
    torch.cuda.synchronize()
    rk, rkp = oq(w.k_bits)
    rv, rvp = oq(w.v_bits)
    ref_out, ref_lse, _ = oattn(w.q_bits, rk, rkp, rv, rvp, w.page_table, w.prefix_len, w.n_nodes, w.parents, w.scale)
    assert (st.cpu().numpy() == 0).all()
    compare_attn(out.float().cpu().numpy(), lse.cpu().numpy(), ref_out, ref_lse, w)
