"""The C ABI library builds, loads without a GPU and exports every entry point
that include/treeverify.h declares (no compute calls here)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treeverify.h")


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(tv_[a-z0-9_]+)\s*\(", txt)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available to build the library")
    from eagle_speculative_decoding_attn_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_four_calls():
    names = _declared()
    for n in ["tv_tree_build_mask", "tv_tree_verify_attn", "tv_tree_accept", "tv_kv_commit_path",
              "tv_tree_verify_attn_workspace", "tv_tree_accept_workspace", "tv_last_error", "tv_version"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in treeverify.h but not exported"


def test_host_only_calls(lib):
    lib.tv_version.restype = ctypes.c_char_p
    assert b"sm_103a" in lib.tv_version()
    lib.tv_last_error.restype = ctypes.c_char_p
    assert lib.tv_last_error() is not None
    lib.tv_tree_accept_workspace.restype = ctypes.c_size_t
    assert lib.tv_tree_accept_workspace(8, 64, 128256) == 0


def test_binding_declares_every_symbol():
    from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
    assert set(_declared()) == set(tvb._SIGNATURES)


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "eagle_speculative_decoding_attn_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f


def _declarations():
    """{name: (return type, [parameter types])} of every call in the header."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    out = {}
    for m in re.finditer(r"([A-Za-z_][A-Za-z0-9_ ]*?\**)\s*\b(tv_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", txt):
        ret, name, params = m.group(1).strip(), m.group(2), m.group(3).strip()
        types = []
        if params and params != "void":
            for prm in params.split(","):
                prm = " ".join(prm.split())
                # drop the parameter's name: the last identifier
                t = re.sub(r"\b[A-Za-z_][A-Za-z0-9_]*\s*$", "", prm).strip()
                types.append(t)
        out[name] = (ret, types)
    return out


def _ctype_of(c_type):
    if "*" in c_type:
        return ctypes.c_char_p if c_type.replace(" ", "") == "constchar*" else ctypes.c_void_p
    base = c_type.replace("const", "").strip()
    return {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "size_t": ctypes.c_size_t,
            "float": ctypes.c_float}[base]


def test_binding_argument_types_match_the_header():
    from eagle_speculative_decoding_attn_gb300 import treeverify as tvb
    decl = _declarations()
    assert set(decl) == set(tvb._SIGNATURES)
    for name, (ret, params) in decl.items():
        restype, argtypes = tvb._SIGNATURES[name]
        assert len(argtypes) == len(params), f"{name}: {len(argtypes)} binding arguments, header has {len(params)}"
        for i, (c_type, a) in enumerate(zip(params, argtypes)):
            assert a is _ctype_of(c_type), f"{name} argument {i}: header {c_type!r}, binding {a}"
        assert restype is _ctype_of(ret), f"{name} return: header {ret!r}, binding {restype}"
