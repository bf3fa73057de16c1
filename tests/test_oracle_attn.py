"""Pins of the oracle's tree-verify attention (no GPU).

Each check compares the oracle with something that does not come from it:
torch's fp64 scaled_dot_product_attention (a chain tree is ordinary causal
attention over the appended tokens; a one-node tree is plain decode
attention), a closed form (all keys equal => mean of the visible values),
and invariances the definition implies (non-ancestors and page placement do
not matter).  Mask definition: Tech Radar section 2, "Dynamic Tree-Attention
Masking".
"""
import math

import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import workloads as W


def _logical_kv(w, b):
    """K/V of request b at logical positions 0..L+N-1 as float64 [T, Hkv, D]."""
    L, N = int(w.prefix_len[b]), int(w.n_nodes[b])
    pos = np.arange(L + N)
    page = w.page_table[b][pos // w.page_size]
    slot = pos % w.page_size
    K = W.bf16_bits_to_f32(w.k_bits[page, :, slot, :]).astype(np.float64)
    V = W.bf16_bits_to_f32(w.v_bits[page, :, slot, :]).astype(np.float64)
    return K, V


def _sdpa(q, K, V, mask, scale):
    """torch fp64 attention: q [Hq, M, D], K/V [Hq, T, D], mask [M, T] bool."""
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(K), torch.from_numpy(V),
        attn_mask=torch.from_numpy(mask), scale=scale).numpy()


@pytest.mark.parametrize("L,N,Hq,Hkv,D", [(37, 9, 4, 2, 64), (0, 5, 2, 2, 64), (128, 64, 8, 1, 128),
                                          (16, 16, 4, 4, 64)])
def test_chain_tree_is_causal_attention(L, N, Hq, Hkv, D):
    w = W.make_custom(B=1, Hq=Hq, Hkv=Hkv, D=D, prefix_len=[L], parents_list=[W.chain_tree(N)],
                      seed=11 + L + N)
    out, lse, st = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table,
                                           w.prefix_len, w.n_nodes, w.parents, w.scale)
    assert st[0] == 0
    K, V = _logical_kv(w, 0)
    G = Hq // Hkv
    q = W.bf16_bits_to_f32(w.q_bits[0, :N]).astype(np.float64)       # [N, Hq, D]
    qh = np.transpose(q, (1, 0, 2)).copy()                            # [Hq, N, D]
    Kh = np.repeat(np.transpose(K, (1, 0, 2)), G, axis=0).copy()       # [Hq, T, D]
    Vh = np.repeat(np.transpose(V, (1, 0, 2)), G, axis=0).copy()
    # query i sits at position L+i and sees every position up to its own
    mask = np.arange(L + N)[None, :] <= (L + np.arange(N))[:, None]
    ref = _sdpa(qh, Kh, Vh, mask, w.scale)                             # [Hq, N, D]
    np.testing.assert_allclose(out[0, :N], np.transpose(ref, (1, 0, 2)), rtol=0, atol=1e-12)
    # log-sum-exp of the same scores, via torch.logsumexp
    s = torch.from_numpy(qh) @ torch.from_numpy(Kh).transpose(1, 2) * w.scale
    s = s.masked_fill(~torch.from_numpy(mask), -math.inf)
    np.testing.assert_allclose(lse[0, :N], torch.logsumexp(s, dim=-1).numpy().T, rtol=0, atol=1e-12)


def test_single_node_is_decode_attention():
    L, Hq, Hkv, D = 200, 8, 2, 128
    w = W.make_custom(B=1, Hq=Hq, Hkv=Hkv, D=D, prefix_len=[L], parents_list=[[-1]], seed=5)
    out, lse, st = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table,
                                           w.prefix_len, w.n_nodes, w.parents, w.scale)
    K, V = _logical_kv(w, 0)
    G = Hq // Hkv
    q = W.bf16_bits_to_f32(w.q_bits[0, 0]).astype(np.float64)        # [Hq, D]
    Kh = np.repeat(np.transpose(K, (1, 0, 2)), G, axis=0).copy()
    Vh = np.repeat(np.transpose(V, (1, 0, 2)), G, axis=0).copy()
    ref = _sdpa(q[:, None, :].copy(), Kh, Vh, np.ones((1, L + 1), dtype=bool), w.scale)
    np.testing.assert_allclose(out[0, 0], ref[:, 0], rtol=0, atol=1e-12)


def test_constant_keys_give_mean_of_visible_values():
    L, Hq, Hkv, D = 21, 4, 2, 64
    rng = np.random.Generator(np.random.PCG64(3))
    parents = W.random_recursive_tree(rng, 12)
    w = W.make_custom(B=1, Hq=Hq, Hkv=Hkv, D=D, prefix_len=[L], parents_list=[parents], seed=9)
    w.k_bits[:] = W.to_bf16_bits(np.full(D, 0.25, dtype=np.float32))
    out, lse, _ = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table,
                                          w.prefix_len, w.n_nodes, w.parents, w.scale)
    K, V = _logical_kv(w, 0)
    G = Hq // Hkv
    for i in range(12):
        # visible set written out by hand: the prefix and i's ancestors-or-self
        vis, j = list(range(L)), i
        chain = [i]
        while j != 0:
            j = int(parents[j])
            chain.append(j)
        vis += [L + c for c in chain]
        for h in range(Hq):
            np.testing.assert_allclose(out[0, i, h], V[vis, h // G].mean(axis=0), rtol=0, atol=1e-12)
            qk = 0.25 * W.bf16_bits_to_f32(w.q_bits[0, i, h]).astype(np.float64).sum() * w.scale
            np.testing.assert_allclose(lse[0, i, h], qk + math.log(len(vis)), rtol=0, atol=1e-12)


def test_non_ancestor_kv_does_not_matter():
    L, Hq, Hkv, D = 33, 4, 4, 64
    rng = np.random.Generator(np.random.PCG64(21))
    parents = W.random_recursive_tree(rng, 20)
    w = W.make_custom(B=1, Hq=Hq, Hkv=Hkv, D=D, prefix_len=[L], parents_list=[parents], seed=4)
    base, _, _ = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table,
                                         w.prefix_len, w.n_nodes, w.parents, w.scale)
    anc, _, _ = oracle.tree_build_mask(w.parents, w.n_nodes)
    for j in [3, 11, 19]:
        k2, v2 = w.k_bits.copy(), w.v_bits.copy()
        pos = L + j
        pg, sl = w.page_table[0, pos // 16], pos % 16
        k2[pg, :, sl, :] = W.to_bf16_bits(np.full((Hkv, D), 7.0, dtype=np.float32))
        v2[pg, :, sl, :] = W.to_bf16_bits(np.full((Hkv, D), -5.0, dtype=np.float32))
        out, _, _ = oracle.tree_verify_attn(w.q_bits, k2, v2, w.page_table, w.prefix_len,
                                            w.n_nodes, w.parents, w.scale)
        for i in range(20):
            sees_j = (int(anc[0, i]) >> j) & 1
            same = np.array_equal(out[0, i], base[0, i])
            assert same == (not sees_j), (i, j)


def test_page_placement_does_not_matter():
    L, Hq, Hkv, D = 70, 4, 2, 64
    rng = np.random.Generator(np.random.PCG64(8))
    parents = W.random_recursive_tree(rng, 10)
    w = W.make_custom(B=1, Hq=Hq, Hkv=Hkv, D=D, prefix_len=[L], parents_list=[parents], seed=6,
                      extra_pages=3)
    out, lse, _ = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table,
                                          w.prefix_len, w.n_nodes, w.parents, w.scale)
    perm = rng.permutation(w.num_pages)
    inv = np.argsort(perm)
    k2, v2 = w.k_bits[perm], w.v_bits[perm]     # new page x holds old page perm[x]
    pt = w.page_table.copy()
    used = pt >= 0
    pt[used] = inv[pt[used]]
    out2, lse2, _ = oracle.tree_verify_attn(w.q_bits, k2, v2, pt, w.prefix_len, w.n_nodes,
                                            w.parents, w.scale)
    assert np.array_equal(out, out2, equal_nan=True) and np.array_equal(lse, lse2, equal_nan=True)


def test_row_sampling_matches_full():
    w = W.make_custom(B=2, Hq=4, Hkv=2, D=64, prefix_len=[17, 40],
                      parents_list=[W.chain_tree(6), W.star_tree(5)], seed=2)
    full, lse, _ = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table,
                                           w.prefix_len, w.n_nodes, w.parents, w.scale)
    rows = [(0, 5, 3), (1, 4, 0), (1, 0, 2)]
    part, lse2, _ = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table,
                                            w.prefix_len, w.n_nodes, w.parents, w.scale, rows=rows)
    for (b, i, h) in rows:
        assert np.array_equal(part[b, i, h], full[b, i, h])
        assert lse2[b, i, h] == lse[b, i, h]


def test_capacity_and_page_errors():
    w = W.make_custom(B=2, Hq=2, Hkv=2, D=64, prefix_len=[30, 30],
                      parents_list=[W.chain_tree(4), W.chain_tree(4)], seed=1)
    pt = w.page_table.copy()
    pt[1, 1] = w.num_pages + 5          # second page of request 1 out of range
    _, _, st = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, pt, w.prefix_len,
                                       w.n_nodes, w.parents, w.scale)
    assert st.tolist() == [0, oracle.STATUS_PAGE_OOB]
    L = np.array([30, 50], dtype=np.int32)      # 50 + 4 positions need 4 pages of 16
    _, _, st = oracle.tree_verify_attn(w.q_bits, w.k_bits, w.v_bits, w.page_table[:, :3], L,
                                       w.n_nodes, w.parents, w.scale)
    assert st.tolist() == [0, oracle.STATUS_CAPACITY]
