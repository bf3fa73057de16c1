"""tv_kv_commit_path at full workload size, byte for byte against the oracle.

The step's tail as the bench runs it: the GPU acceptance picks each request's
path, then the commit moves the accepted rows of every layer (32 layers on the
7B shape, 80 on the G = 8 shapes) in one call.  Every K/V byte is checked:

* the pages holding any request's tree positions (at most five per request)
  are gathered, before the commit, into a compact cache with its own page
  table (prefix pages point at a zero page); the oracle's kv_commit_path runs
  on that compact cache with the GPU's accepted paths, and the same pages read
  back after the commit must equal its result exactly, as must the committed
  slots (mapped back to the real page ids) and the new lengths;
* every other page of every layer must still hold its original bytes.

Layer l of the cache holds the workload's bf16 bits plus 7 l (16-bit wrap), so
the layers differ and any layer-stride mistake shows.  (Source: Tech Radar,
SGLang EAGLE-2, section 2 sequence diagram: keep the accepted branch's KV and
drop the wrong branches.)
"""
import numpy as np
import pytest
import torch

import oracle
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from gpu_helpers import DevWorkload, require_gpu, to_dev

pytestmark = pytest.mark.gpu


def _layer_bits(base16, layer):
    """Layer `layer` of the test cache: the base bits plus 7 * layer (int16 wrap)."""
    return base16 + 7 * layer


@pytest.mark.parametrize("name", ["llama2_7b", "serving", "llama3_70b"])
def test_commit_full_size_byte_exact(name):
    dev = require_gpu()
    cfg = W.CONFIG_BY_NAME[name]
    layers = cfg.n_layers_commit
    w = W.make_workload(name)
    dw = DevWorkload(w, dev)
    B, P = w.B, 16
    kb = dw.k.view(torch.int16)
    vb = dw.v.view(torch.int16)
    num_pages = kb.shape[0]
    kL = torch.empty((layers,) + tuple(kb.shape), dtype=torch.int16, device=dev)
    vL = torch.empty_like(kL)
    for l in range(layers):
        kL[l] = _layer_bits(kb, l)
        vL[l] = _layer_bits(vb, l)

    anc, depth, st = dw.mask()
    sampling = w.temperature > 0
    acc_len, path, _ = tvb.tree_accept(dw.target, dw.draft if sampling else None, dw.tokens, dw.parents,
                                       dw.n_nodes, anc, depth, w.temperature, dw.u_accept if sampling else None,
                                       dw.u_sample if sampling else None, st)
    torch.cuda.synchronize()
    a_host, p_host = acc_len.cpu().numpy(), path.cpu().numpy()
    assert (st.cpu().numpy() == 0).all()
    assert a_host.max() >= 1, "no request accepted anything: nothing would move"

    # the pages holding tree positions, gathered before the commit
    span = []
    for b in range(B):
        L, N = int(w.prefix_len[b]), int(w.n_nodes[b])
        span += [int(w.page_table[b, j]) for j in range(L // P, (L + N - 1) // P + 1)]
    span = sorted(set(span))
    cidx = {pg: i for i, pg in enumerate(span)}
    zero_page = len(span)
    cpt = np.full_like(w.page_table, -1)
    for b in range(B):
        L, N = int(w.prefix_len[b]), int(w.n_nodes[b])
        for j in range((L + N + P - 1) // P):
            pg = int(w.page_table[b, j])
            cpt[b, j] = cidx.get(pg, zero_page) if j >= L // P else zero_page
    span_t = torch.tensor(span, dtype=torch.int64, device=dev)

    def gather(t):
        g = t.index_select(1, span_t).cpu().numpy()
        z = np.zeros((g.shape[0], 1) + g.shape[2:], dtype=g.dtype)
        return np.concatenate([g, z], axis=1).view(np.uint16)

    kc0, vc0 = gather(kL), gather(vL)

    slots, new_len = tvb.kv_commit_path(kL.view(torch.bfloat16), vL.view(torch.bfloat16), dw.page_table,
                                        dw.prefix_len, dw.n_nodes, acc_len, path, st)
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()

    ke, ve, cslots, rl, rst = oracle.kv_commit_path(kc0, vc0, cpt, w.prefix_len, w.n_nodes, a_host, p_host)
    assert (rst == 0).all()
    assert np.array_equal(new_len.cpu().numpy(), rl)
    real = np.where(cslots >= 0, np.asarray(span + [-1], np.int64)[np.maximum(cslots, 0) // P] * P + cslots % P, -1)
    assert np.array_equal(slots.cpu().numpy(), real)
    kc1, vc1 = gather(kL), gather(vL)
    assert np.array_equal(kc1[:, :-1], ke[:, :-1]), "tree pages of K differ from the oracle"
    assert np.array_equal(vc1[:, :-1], ve[:, :-1]), "tree pages of V differ from the oracle"

    # every other page of every layer is untouched
    others = torch.ones(num_pages, dtype=torch.bool, device=dev)
    others[span_t] = False
    for l in range(layers):
        assert torch.equal(kL[l][others], _layer_bits(kb, l)[others]), f"K layer {l} changed outside the tree pages"
        assert torch.equal(vL[l][others], _layer_bits(vb, l)[others]), f"V layer {l} changed outside the tree pages"
    moved = sum(int(np.sum(p_host[b, 1:a_host[b] + 1] != np.arange(1, a_host[b] + 1))) for b in range(B))
    print(f"{name}: {layers} layers, {moved} moved rows per layer and head, {len(span)} tree pages compared")
