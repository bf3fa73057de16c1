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


def test_noalloc_alternating_sizes():
    """Calls of different sizes in turn (7B-shaped, tiny, 7B-shaped, tiny): each
    call finds the other size's split partials, tickets and error bits in the
    shared array and must still reproduce the workspace entry point."""
    dev = require_gpu()
    lib = tvb.load_library()
    runs = {}
    for name in ("llama2_7b", "tiny"):
        w = W.make_workload(name, with_logits=False)
        dw = DevWorkload(w, dev, logits=False)
        anc, _, status0 = dw.mask()
        ref_out, ref_lse = tvb.tree_verify_attn(dw.q, dw.k, dw.v, dw.page_table, dw.prefix_len, dw.n_nodes, anc,
                                                w.scale, status0.clone())
        torch.cuda.synchronize()
        runs[name] = (w, dw, anc, status0, _valid_rows(w, ref_out.float().cpu().numpy()),
                      _valid_rows(w, ref_lse.cpu().numpy()))
    for name in ("llama2_7b", "tiny", "llama2_7b", "tiny"):
        w, dw, anc, status0, r, rl = runs[name]
        out = torch.full_like(dw.q, float("nan"))
        lse = torch.full((w.B, w.n_max, w.Hq), float("nan"), dtype=torch.float32, device=dev)
        status = status0.clone()
        assert _call_noalloc(lib, dw, w, anc, status, out, lse) == tvb.TV_OK, lib.tv_last_error()
        torch.cuda.synchronize()
        assert (status.cpu().numpy() == 0).all()
        o = _valid_rows(w, out.float().cpu().numpy())
        err = np.abs(o - r)
        assert np.isfinite(o).all()
        assert err.max() <= ATOL_MAX and err.mean() <= ATOL_MEAN, name
        assert np.abs(_valid_rows(w, lse.cpu().numpy()) - rl).max() <= LSE_ATOL


_RESET_SCRIPT = r'''
import ctypes, sys
import numpy as np
sys.path.insert(0, sys.argv[1])
from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
from eagle_speculative_decoding_attn_gb300 import workloads as W

lib = tvb.load_library()
rt = ctypes.CDLL("libcudart.so.13")
w = W.make_workload("tiny", with_logits=False)
P = ctypes.c_void_p


def dev_buf(nbytes):
    p = P()
    assert rt.cudaMalloc(ctypes.byref(p), ctypes.c_size_t(max(nbytes, 16))) == 0
    assert rt.cudaMemset(p, 0, ctypes.c_size_t(max(nbytes, 16))) == 0
    return p


def upload(a):
    a = np.ascontiguousarray(a)
    p = dev_buf(a.nbytes)
    assert rt.cudaMemcpy(p, a.ctypes.data_as(P), ctypes.c_size_t(a.nbytes), 1) == 0
    return p


def download(p, shape, dtype):
    a = np.empty(shape, dtype=dtype)
    assert rt.cudaMemcpy(a.ctypes.data_as(P), p, ctypes.c_size_t(a.nbytes), 2) == 0
    return a


def run():
    B, n_max, Hq, D = w.q_bits.shape
    num_pages, Hkv = w.k_bits.shape[0], w.k_bits.shape[1]
    q, k, v = upload(w.q_bits), upload(w.k_bits), upload(w.v_bits)
    pt, L, n, par = upload(w.page_table), upload(w.prefix_len), upload(w.n_nodes), upload(w.parents)
    anc, depth = dev_buf(B * n_max * 8), dev_buf(B * n_max * 4)
    st_mask, st_ws, st_na = dev_buf(B * 4), dev_buf(B * 4), dev_buf(B * 4)
    assert lib.tv_tree_build_mask(par, n, B, n_max, anc, depth, st_mask, None) == 0, lib.tv_last_error()
    ws_bytes = lib.tv_tree_verify_attn_workspace(B, n_max, Hq, Hkv, D, 0)
    ws = dev_buf(ws_bytes)
    o_ws, l_ws = dev_buf(B * n_max * Hq * D * 2), dev_buf(B * n_max * Hq * 4)
    o_na, l_na = dev_buf(B * n_max * Hq * D * 2), dev_buf(B * n_max * Hq * 4)
    common = (num_pages, pt, w.page_table.shape[1], L, n, anc, B, n_max, Hq, Hkv, D, 16, float(w.scale))
    assert lib.tv_tree_verify_attn(q, k, v, *common, o_ws, l_ws, ws, ws_bytes, st_ws, None) == 0, \
        lib.tv_last_error()
    assert lib.tv_tree_verify_attn_noalloc(q, k, v, *common, o_na, l_na, st_na, None) == 0, lib.tv_last_error()
    assert rt.cudaDeviceSynchronize() == 0
    a = download(o_ws, (B, n_max, Hq, D), np.uint16).astype(np.uint32) << 16
    b = download(o_na, (B, n_max, Hq, D), np.uint16).astype(np.uint32) << 16
    a, b = a.view(np.float32), b.view(np.float32)
    N = int(w.n_nodes[0])
    err = np.abs(a[:, :N] - b[:, :N])
    assert np.isfinite(b[:, :N]).all()
    assert (download(st_na, (B,), np.int32) == 0).all()
    for p in (q, k, v, pt, L, n, par, anc, depth, st_mask, st_ws, st_na, ws, o_ws, l_ws, o_na, l_na):
        rt.cudaFree(p)
    return float(err.max()), float(err.mean())


e1 = run()
assert rt.cudaDeviceReset() == 0
e2 = run()
print("RESET_OK", e1[0], e2[0])
'''


def test_noalloc_after_device_reset():
    """A device reset ends the context the built-in scratch's address was found
    in; the next call must look it up again in the new context.  Run in a child
    process on plain CUDA runtime buffers (no torch allocations to invalidate):
    a call, cudaDeviceReset, and a call again, each compared with the workspace
    entry point."""
    require_gpu()
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _RESET_SCRIPT, root], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "RESET_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-2000:]
    e1, e2 = (float(x) for x in r.stdout.split("RESET_OK")[1].split()[:2])
    assert e1 <= ATOL_MAX and e2 <= ATOL_MAX
