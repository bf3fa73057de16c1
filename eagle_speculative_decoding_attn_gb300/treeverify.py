"""Python binding of libtreeverify.so (ctypes; argument marshalling only).

Every step of the tree-verification path runs in the library's CUDA kernels;
this module only passes torch tensors' device pointers, sizes and the current
CUDA stream through the C ABI declared in ``include/treeverify.h``, and
allocates output tensors with torch when the caller does not supply them.
There is no CPU fallback: when the library is missing or a call fails, an
exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtreeverify.so")

TV_OK = 0
TV_ERR_INVALID_ARG = -1
TV_ERR_UNSUPPORTED = -2
TV_ERR_WORKSPACE = -3
TV_ERR_CUDA = -4

TV_ACCEPT_SIBLINGS_WITHOUT_REPLACEMENT = 1

TV_DEV_BAD_TREE = 1
TV_DEV_PAGE_OOB = 2
TV_DEV_CAPACITY = 4
TV_DEV_TIMEOUT = 8
TV_DEV_BAD_TOKEN = 16
TV_DEV_BAD_REFCOUNT = 32

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_F = ctypes.c_float

_SIGNATURES = {
    "tv_tree_build_mask": (_I, [_P, _P, _I, _I, _P, _P, _P, _P]),
    "tv_tree_verify_attn_workspace": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "tv_tree_verify_attn": (_I, [_P, _P, _P, _I64, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P, _P,
                                 _SZ, _P, _P]),
    "tv_tree_verify_attn_noalloc": (_I, [_P, _P, _P, _I64, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                                         _P, _P]),
    "tv_tree_accept_workspace": (_SZ, [_I, _I, _I]),
    "tv_tree_accept": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _F, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tv_kv_commit_path": (_I, [_P, _P, _I, _I64, _I64, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "tv_tree_expand_workspace": (_SZ, [_I, _I, _I]),
    "tv_tree_expand": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _SZ, _P, _P]),
    "tv_kv_prune_pages": (_I, [_P, _I, _P, _I64, _P, _P, _P, _I, _I, _P, _I64, _P, _P, _P]),
    "tv_kv_quantize_q4": (_I, [_P, _I64, _I, _P, _P, _P]),
    "tv_tree_verify_attn_q4": (_I, [_P, _P, _P, _P, _P, _I64, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P,
                                    _P, _P, _SZ, _P, _P]),
    "tv_kv_quantize_q3": (_I, [_P, _I64, _I, _P, _P, _P]),
    "tv_tree_verify_attn_q3": (_I, [_P, _P, _P, _P, _P, _I64, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P,
                                    _P, _P, _SZ, _P, _P]),
    "tv_selftest_wait_timeout": (_I, [_P, _P]),
    "tv_last_error": (ctypes.c_char_p, []),
    "tv_version": (ctypes.c_char_p, []),
}

_lib = None


class TreeVerifyError(RuntimeError):
    pass


def load_library(path: Optional[str] = None):
    """Load libtreeverify.so (once) and declare every entry point's signature."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise TreeVerifyError(
            f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(p)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def _check(rc: int, what: str):
    if rc != TV_OK:
        msg = load_library().tv_last_error().decode(errors="replace")
        raise TreeVerifyError(f"{what} failed with code {rc}: {msg}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise TreeVerifyError("tensors passed to the library must live on a CUDA device")
    if not t.is_contiguous():
        raise TreeVerifyError("tensors passed to the library must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _expect(t: torch.Tensor, dtype, shape, name):
    if t.dtype != dtype:
        raise TreeVerifyError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise TreeVerifyError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


# --------------------------------------------------------------------------
def tree_build_mask(parents: torch.Tensor, n_nodes: torch.Tensor, *, anc_mask=None, depth=None, status=None):
    """Ancestor bit-mask (int64 view of the uint64 words) and depth per node.

    parents int32 [B, n_max], n_nodes int32 [B] -> (anc_mask int64 [B, n_max],
    depth int32 [B, n_max], status int32 [B]).
    """
    B, n_max = parents.shape
    dev = parents.device
    anc_mask = torch.empty((B, n_max), dtype=torch.int64, device=dev) if anc_mask is None else anc_mask
    depth = torch.empty((B, n_max), dtype=torch.int32, device=dev) if depth is None else depth
    status = torch.empty((B,), dtype=torch.int32, device=dev) if status is None else status
    _expect(parents, torch.int32, (B, n_max), "parents")
    _expect(n_nodes, torch.int32, (B,), "n_nodes")
    rc = load_library().tv_tree_build_mask(_ptr(parents), _ptr(n_nodes), B, n_max, _ptr(anc_mask), _ptr(depth),
                                           _ptr(status), _stream(dev))
    _check(rc, "tv_tree_build_mask")
    return anc_mask, depth, status


def tree_verify_attn_workspace_bytes(B, n_max, Hq, Hkv, D, max_kv_len=0) -> int:
    return int(load_library().tv_tree_verify_attn_workspace(B, n_max, Hq, Hkv, D, max_kv_len))


def new_attn_workspace(B, n_max, Hq, Hkv, D, device) -> torch.Tensor:
    """A zero-filled workspace for tv_tree_verify_attn, reusable for later
    calls of the same sizes on the same stream."""
    nbytes = tree_verify_attn_workspace_bytes(B, n_max, Hq, Hkv, D)
    return torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)


def tree_verify_attn(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, page_table: torch.Tensor,
                     prefix_len: torch.Tensor, n_nodes: torch.Tensor, anc_mask: torch.Tensor, scale: float,
                     status: torch.Tensor, *, out=None, lse=None, want_lse=True, workspace=None):
    """Tree-masked paged attention.  q bf16 [B, n_max, Hq, D]; caches bf16
    [num_pages, Hkv, 16, D]; page_table int32 [B, max_pages]; anc_mask int64
    [B, n_max].  Returns (out bf16 [B, n_max, Hq, D], lse f32 [B, n_max, Hq] or None)."""
    B, n_max, Hq, D = q.shape
    num_pages, Hkv, P, Dk = k_cache.shape
    dev = q.device
    if Dk != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise TreeVerifyError("k_cache / v_cache shapes do not match q")
    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        if t.dtype != torch.bfloat16:
            raise TreeVerifyError(f"{nm} must be bfloat16")
    _expect(page_table, torch.int32, page_table.shape, "page_table")
    _expect(anc_mask, torch.int64, (B, n_max), "anc_mask")
    out = torch.empty_like(q) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, n_max, Hq), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_attn_workspace(B, n_max, Hq, Hkv, D, dev)
    rc = load_library().tv_tree_verify_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), num_pages, _ptr(page_table), page_table.shape[1],
        _ptr(prefix_len), _ptr(n_nodes), _ptr(anc_mask), B, n_max, Hq, Hkv, D, P, float(scale), _ptr(out),
        _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev))
    _check(rc, "tv_tree_verify_attn")
    return out, lse


def tree_accept_workspace_bytes(B, n_max, V) -> int:
    return int(load_library().tv_tree_accept_workspace(B, n_max, V))


def new_accept_workspace(B, n_max, V, device) -> Optional[torch.Tensor]:
    """A zero-filled workspace for tv_tree_accept (None when the sizes need
    none), reusable for later calls of the same sizes on the same stream."""
    nbytes = tree_accept_workspace_bytes(B, n_max, V)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device) if nbytes > 0 else None


def tree_accept(target_logits: torch.Tensor, draft_logits: Optional[torch.Tensor], tokens: torch.Tensor,
                parents: torch.Tensor, n_nodes: torch.Tensor, anc_mask: Optional[torch.Tensor],
                depth: Optional[torch.Tensor], temperature: float, u_accept: Optional[torch.Tensor],
                u_sample: Optional[torch.Tensor], status: torch.Tensor, *, outputs=None, workspace=None,
                without_replacement: bool = False):
    """Greedy (temperature 0) or rejection-sampling acceptance; with
    ``without_replacement`` the sampling walk renormalises the draft without
    each rejected sibling's token.  Returns (accept_len int32 [B], path_nodes
    int32 [B, n_max], out_tokens int32 [B, n_max+1])."""
    B, n_max, V = target_logits.shape
    dev = target_logits.device
    if workspace is None:
        workspace = new_accept_workspace(B, n_max, V, dev)
    if outputs is None:
        accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
        path_nodes = torch.empty((B, n_max), dtype=torch.int32, device=dev)
        out_tokens = torch.empty((B, n_max + 1), dtype=torch.int32, device=dev)
    else:
        accept_len, path_nodes, out_tokens = outputs
    rc = load_library().tv_tree_accept(
        _ptr(target_logits), _ptr(draft_logits), _ptr(tokens), _ptr(parents), _ptr(n_nodes), _ptr(anc_mask),
        _ptr(depth), B, n_max, V, float(temperature), TV_ACCEPT_SIBLINGS_WITHOUT_REPLACEMENT if without_replacement else 0,
        _ptr(u_accept), _ptr(u_sample), _ptr(accept_len),
        _ptr(path_nodes), _ptr(out_tokens), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _ptr(status), _stream(dev))
    _check(rc, "tv_tree_accept")
    return accept_len, path_nodes, out_tokens


def kv_commit_path(k_cache: torch.Tensor, v_cache: torch.Tensor, page_table: torch.Tensor,
                   prefix_len: torch.Tensor, n_nodes: torch.Tensor, accept_len: torch.Tensor,
                   path_nodes: torch.Tensor, status: torch.Tensor, *, outputs=None):
    """Compact the accepted path's K/V in place.  Caches bf16 [num_pages, Hkv,
    16, D] (one layer) or [n_layers, num_pages, Hkv, 16, D].  Returns
    (committed_slots int64 [B, n_max], new_len int32 [B])."""
    if k_cache.dim() == 4:
        n_layers, (num_pages, Hkv, P, D) = 1, k_cache.shape
        stride = num_pages * Hkv * P * D
    else:
        n_layers, num_pages, Hkv, P, D = k_cache.shape
        stride = num_pages * Hkv * P * D
    B, n_max = path_nodes.shape
    dev = k_cache.device
    if outputs is None:
        slots = torch.empty((B, n_max), dtype=torch.int64, device=dev)
        new_len = torch.empty((B,), dtype=torch.int32, device=dev)
    else:
        slots, new_len = outputs
    rc = load_library().tv_kv_commit_path(
        _ptr(k_cache), _ptr(v_cache), n_layers, stride, num_pages, _ptr(page_table), page_table.shape[1],
        _ptr(prefix_len), _ptr(n_nodes), _ptr(accept_len), _ptr(path_nodes), B, n_max, Hkv, D, P, _ptr(slots),
        _ptr(new_len), _ptr(status), _stream(dev))
    _check(rc, "tv_kv_commit_path")
    return slots, new_len


def tree_expand_workspace_bytes(B, max_frontier, V) -> int:
    return int(load_library().tv_tree_expand_workspace(B, max_frontier, V))


def new_expand_workspace(B, max_frontier, V, device) -> torch.Tensor:
    """A zero-filled workspace for tv_tree_expand, reusable for later calls of
    the same sizes on the same stream."""
    return torch.zeros(tree_expand_workspace_bytes(B, max_frontier, V), dtype=torch.uint8, device=device)


def tree_expand(draft_logits: torch.Tensor, parents: torch.Tensor, tokens: torch.Tensor, scores: torch.Tensor,
                n_nodes: torch.Tensor, level_start: torch.Tensor, status: torch.Tensor, *, top_k: int,
                max_new: int, budget: int, max_frontier: Optional[int] = None, entropy=None, width=None,
                workspace=None):
    """One level of dynamic tree construction; updates parents, tokens,
    scores, n_nodes and level_start in place.  Returns (entropy, width) of the
    frontier rows (tensors the caller passed, else None)."""
    B, n_max, V = draft_logits.shape
    _expect(draft_logits, torch.float32, (B, n_max, V), "draft_logits")
    _expect(parents, torch.int32, (B, n_max), "parents")
    _expect(tokens, torch.int32, (B, n_max), "tokens")
    _expect(scores, torch.float32, (B, n_max), "scores")
    _expect(n_nodes, torch.int32, (B,), "n_nodes")
    _expect(level_start, torch.int32, (B,), "level_start")
    if max_frontier is None:
        max_frontier = max(1, min(max_new, n_max))
    if workspace is None:
        workspace = new_expand_workspace(B, max_frontier, V, draft_logits.device)
    rc = load_library().tv_tree_expand(
        _ptr(draft_logits), _ptr(parents), _ptr(tokens), _ptr(scores), _ptr(n_nodes), _ptr(level_start),
        _ptr(entropy), _ptr(width), B, n_max, V, int(top_k), int(max_new), int(budget), int(max_frontier),
        _ptr(workspace), workspace.numel(), _ptr(status), _stream(draft_logits.device))
    _check(rc, "tv_tree_expand")
    return entropy, width


def kv_prune_pages(page_table: torch.Tensor, refcount: torch.Tensor, prefix_len: torch.Tensor,
                   n_nodes: torch.Tensor, new_len: torch.Tensor, status: torch.Tensor, *, free_list=None,
                   free_count=None):
    """Release the pages that hold only rejected tree rows (page-table slots
    cleared, reference counts decremented in place).  Returns (free_list int32
    [capacity], free_count int32 [1]): the pages whose count reached zero are
    free_list[old count : new count]."""
    B, max_pages = page_table.shape
    dev = page_table.device
    _expect(refcount, torch.int32, refcount.shape, "refcount")
    if free_list is None:
        free_list = torch.full((B * 8,), -1, dtype=torch.int32, device=dev)
    if free_count is None:
        free_count = torch.zeros(1, dtype=torch.int32, device=dev)
    rc = load_library().tv_kv_prune_pages(
        _ptr(page_table), max_pages, _ptr(refcount), refcount.numel(), _ptr(prefix_len), _ptr(n_nodes),
        _ptr(new_len), B, 16, _ptr(free_list), free_list.numel(), _ptr(free_count), _ptr(status),
        _stream(dev))
    _check(rc, "tv_kv_prune_pages")
    return free_list, free_count


def _code_row(bits: int, D: int) -> int:
    """Bytes of one row's codes in the 4-bit (D/2) or 3-bit (3D/8) format."""
    return D // 2 if bits == 4 else 3 * D // 8


def _kv_quantize(bits: int, x: torch.Tensor, codes, params):
    name = f"tv_kv_quantize_q{bits}"
    if x.dtype != torch.bfloat16:
        raise TreeVerifyError(f"x: expected torch.bfloat16, got {x.dtype}")
    D = x.shape[-1]
    rows = x.numel() // D
    if codes is None:
        codes = torch.empty(x.shape[:-1] + (_code_row(bits, D),), dtype=torch.uint8, device=x.device)
    if params is None:
        params = torch.empty(x.shape[:-1] + (2 * D // 32,), dtype=torch.float16, device=x.device)
    rc = getattr(load_library(), name)(_ptr(x), rows, D, _ptr(codes), _ptr(params), _stream(x.device))
    _check(rc, name)
    return codes, params


def kv_quantize_q4(x: torch.Tensor, *, codes=None, params=None):
    """Encode bf16 rows [..., D] in the 4-bit cache format.  Returns (codes
    uint8 [..., D/2], params float16 [..., 2*D/32])."""
    return _kv_quantize(4, x, codes, params)


def kv_quantize_q3(x: torch.Tensor, *, codes=None, params=None):
    """Encode bf16 rows [..., D] in the 3-bit cache format.  Returns (codes
    uint8 [..., 3*D/8], params float16 [..., 2*D/32])."""
    return _kv_quantize(3, x, codes, params)


def _verify_attn_lowbit(bits, q, k_codes, k_params, v_codes, v_params, page_table, prefix_len, n_nodes, anc_mask,
                        scale, status, out, lse, want_lse, workspace):
    name = f"tv_tree_verify_attn_q{bits}"
    B, n_max, Hq, D = q.shape
    num_pages, Hkv, P, Dc = k_codes.shape
    dev = q.device
    if q.dtype != torch.bfloat16:
        raise TreeVerifyError("q must be bfloat16")
    if Dc != _code_row(bits, D) or tuple(v_codes.shape) != tuple(k_codes.shape):
        raise TreeVerifyError("k_codes / v_codes shapes do not match q")
    for t, nm in ((k_codes, "k_codes"), (v_codes, "v_codes")):
        _expect(t, torch.uint8, (num_pages, Hkv, P, Dc), nm)
    for t, nm in ((k_params, "k_params"), (v_params, "v_params")):
        _expect(t, torch.float16, (num_pages, Hkv, P, 2 * D // 32), nm)
    _expect(page_table, torch.int32, page_table.shape, "page_table")
    _expect(anc_mask, torch.int64, (B, n_max), "anc_mask")
    out = torch.empty_like(q) if out is None else out
    if lse is None and want_lse:
        lse = torch.empty((B, n_max, Hq), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = new_attn_workspace(B, n_max, Hq, Hkv, D, dev)
    rc = getattr(load_library(), name)(
        _ptr(q), _ptr(k_codes), _ptr(k_params), _ptr(v_codes), _ptr(v_params), num_pages, _ptr(page_table),
        page_table.shape[1], _ptr(prefix_len), _ptr(n_nodes), _ptr(anc_mask), B, n_max, Hq, Hkv, D, P,
        float(scale), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(status), _stream(dev))
    _check(rc, name)
    return out, lse


def tree_verify_attn_q4(q: torch.Tensor, k_codes: torch.Tensor, k_params: torch.Tensor, v_codes: torch.Tensor,
                        v_params: torch.Tensor, page_table: torch.Tensor, prefix_len: torch.Tensor,
                        n_nodes: torch.Tensor, anc_mask: torch.Tensor, scale: float, status: torch.Tensor, *,
                        out=None, lse=None, want_lse=True, workspace=None):
    """Tree-masked paged attention over a 4-bit cache: codes uint8
    [num_pages, Hkv, 16, D/2] and params float16 [num_pages, Hkv, 16, 2*D/32]
    for K and for V (the format of ``kv_quantize_q4``); everything else as
    ``tree_verify_attn``, whose workspace it shares."""
    return _verify_attn_lowbit(4, q, k_codes, k_params, v_codes, v_params, page_table, prefix_len, n_nodes,
                               anc_mask, scale, status, out, lse, want_lse, workspace)


def tree_verify_attn_q3(q: torch.Tensor, k_codes: torch.Tensor, k_params: torch.Tensor, v_codes: torch.Tensor,
                        v_params: torch.Tensor, page_table: torch.Tensor, prefix_len: torch.Tensor,
                        n_nodes: torch.Tensor, anc_mask: torch.Tensor, scale: float, status: torch.Tensor, *,
                        out=None, lse=None, want_lse=True, workspace=None):
    """Tree-masked paged attention over a 3-bit cache: codes uint8
    [num_pages, Hkv, 16, 3*D/8] and params float16 [num_pages, Hkv, 16, 2*D/32]
    for K and for V (the format of ``kv_quantize_q3``); everything else as
    ``tree_verify_attn``, whose workspace it shares."""
    return _verify_attn_lowbit(3, q, k_codes, k_params, v_codes, v_params, page_table, prefix_len, n_nodes,
                               anc_mask, scale, status, out, lse, want_lse, workspace)


def version() -> str:
    return load_library().tv_version().decode()


# kernel launches each call enqueues (mask, attention, accept, commit)
LAUNCHES = {"tree_build_mask": 1, "tree_verify_attn": 1, "tree_accept": 1, "kv_commit_path": 1}


def launches_per_step() -> int:
    """Kernel launches of one verification step (the four calls once each)."""
    return sum(LAUNCHES.values())


def selftest_wait_timeout(status: torch.Tensor):
    """Run the bounded-wait self-test: sets TV_DEV_TIMEOUT (8) in status[0]."""
    _expect(status, torch.int32, status.shape, "status")
    rc = load_library().tv_selftest_wait_timeout(_ptr(status), _stream(status.device))
    _check(rc, "tv_selftest_wait_timeout")
    return status
