"""GPU test of tv_tree_verify_attn_noalloc, the attention entry point for
callers that cannot allocate device memory themselves (its scratch is an
array built into the library).  It is called through the C ABI and must
reproduce tv_tree_verify_attn (which runs on a caller workspace) within the
attention tolerance of the other tests, on two calls in a row: the second
call finds the first call's leftovers in the shared array.

This file is collected last so that a run stopping at the first failure has
already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W
from gpu_helpers import ATOL_MAX, ATOL_MEAN, LSE_ATOL, DevWorkload, require_gpu

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _call_noalloc(lib, dw, w, anc, status, out, lse):
    num_pages, Hkv, P, D = dw.k.shape
    B, n_max, Hq, _ = dw.q.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.tv_tree_verify_attn_noalloc(
        _p(dw.q), _p(dw.k), _p(dw.v), num_pages, _p(dw.page_table), dw.page_table.shape[1], _p(dw.prefix_len),
        _p(dw.n_nodes), _p(anc), B, n_max, Hq, Hkv, D, P, float(w.scale), _p(out), _p(lse), _p(status), stream)


def _valid_rows(w, a):
    return np.concatenate([a[b, : int(w.n_nodes[b])].reshape(-1) for b in range(w.B)])


@pytest.mark.parametrize("name", ["llama2_7b", "tiny"])
def test_noalloc_matches_workspace_entry_twice(name):
    dev = require_gpu()
    lib = tvb.load_library()
    w = W.make_workload(name, with_logits=False)
    dw = DevWorkload(w, dev, logits=False)
    anc, _, status0 = dw.mask()
    ref_out, ref_lse = tvb.tree_verify_attn(dw.q, dw.k, dw.v, dw.page_table, dw.prefix_len, dw.n_nodes, anc,
                                            w.scale, status0.clone())
    torch.cuda.synchronize()
    ref_o = ref_out.float().cpu().numpy()
    ref_l = ref_lse.cpu().numpy()
    for _ in range(2):
        out = torch.full_like(dw.q, float("nan"))
        lse = torch.full(ref_lse.shape, float("nan"), dtype=torch.float32, device=dev)
        status = status0.clone()
        rc = _call_noalloc(lib, dw, w, anc, status, out, lse)
        assert rc == tvb.TV_OK, lib.tv_last_error()
        torch.cuda.synchronize()
        assert (status.cpu().numpy() == 0).all()
        o = _valid_rows(w, out.float().cpu().numpy())
        r = _valid_rows(w, ref_o)
        err = np.abs(o - r)
        assert np.isfinite(o).all()
        assert err.max() <= ATOL_MAX and err.mean() <= ATOL_MEAN
        le = np.abs(_valid_rows(w, lse.cpu().numpy()) - _valid_rows(w, ref_l))
        assert le.max() <= LSE_ATOL
