"""Host-side checks of the C ABI that need no GPU: the libraries load, export every symbol
the headers declare, and refuse bad arguments with the documented codes before any CUDA
call is made."""
import ctypes
import os
import re

import pytest

import invariant_bi_gemm_gb300 as bg
from invariant_bi_gemm_gb300 import build as bgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared(header):
    d = os.path.join(ROOT, "include")
    if not os.path.exists(os.path.join(d, header)):
        d = os.path.join(ROOT, "tests", "include")   # the test-only controls header
    src = open(os.path.join(d, header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w[\w\s\*]*?\b(bi_\w+)\s*\(", src, flags=re.M)))


def test_header_symbols_exported():
    declared = _declared("bi_gemm.h")
    assert set(declared) == set(bg.EXPORTED_SYMBOLS)
    L = ctypes.CDLL(bgbuild.lib_path("libbi_gemm.so"))
    for name in declared:
        assert hasattr(L, name), name


def test_rmsnorm_header_symbols_exported():
    declared = _declared("bi_rmsnorm.h")
    assert set(declared) == set(bg.RMSNORM_EXPORTED_SYMBOLS)
    L = ctypes.CDLL(bgbuild.lib_path("libbi_gemm.so"))
    for name in declared:
        assert hasattr(L, name), name


@pytest.mark.parametrize("d,eps,want", [
    (4096, -1.0, bg.BI_GEMM_ERR_INVALID_ARG),
    (4096, float("nan"), bg.BI_GEMM_ERR_INVALID_ARG),
    (4096, float("inf"), bg.BI_GEMM_ERR_INVALID_ARG),
    (0, 1e-6, bg.BI_GEMM_ERR_UNSUPPORTED),
    (4, 1e-6, bg.BI_GEMM_ERR_UNSUPPORTED),
    (4100, 1e-6, bg.BI_GEMM_ERR_UNSUPPORTED),          # row not a whole number of 16-byte vectors
    (32776, 1e-6, bg.BI_GEMM_ERR_UNSUPPORTED),         # past 1024 threads x 4 vectors x 8
    (-8, 1e-6, bg.BI_GEMM_ERR_UNSUPPORTED),
])
def test_rmsnorm_create_refuses_before_touching_cuda(d, eps, want):
    h = ctypes.c_void_p()
    assert bg.library().bi_rmsnorm_create(ctypes.byref(h), d, eps) == want
    assert h.value is None


def test_rmsnorm_null_arguments():
    L = bg.library()
    assert L.bi_rmsnorm_create(None, 4096, 1e-6) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_rmsnorm_run(None, None, 4, None, None, None) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_rmsnorm_get_config(None, None) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_rmsnorm_destroy(None) == bg.BI_GEMM_OK


def test_attention_header_symbols_exported():
    declared = _declared("bi_attention.h")
    assert set(declared) == set(bg.ATTENTION_EXPORTED_SYMBOLS)
    L = ctypes.CDLL(bgbuild.lib_path("libbi_gemm.so"))
    for name in declared:
        assert hasattr(L, name), name


@pytest.mark.parametrize("Hq,Hkv,D,page,scale,split,want", [
    (32, 8, 128, 16, 0.0, 0, bg.BI_GEMM_ERR_INVALID_ARG),
    (32, 8, 128, 16, float("nan"), 0, bg.BI_GEMM_ERR_INVALID_ARG),
    (32, 8, 128, 0, 0.1, 0, bg.BI_GEMM_ERR_INVALID_ARG),
    (32, 8, 128, 16, 0.1, -1, bg.BI_GEMM_ERR_INVALID_ARG),
    (30, 8, 128, 16, 0.1, 0, bg.BI_GEMM_ERR_UNSUPPORTED),       # heads not a multiple
    (32, 2, 128, 16, 0.1, 0, bg.BI_GEMM_ERR_UNSUPPORTED),       # group of 16
    (32, 8, 96, 16, 0.1, 0, bg.BI_GEMM_ERR_UNSUPPORTED),        # head dim
    (32, 8, 128, 16, 0.1, 200, bg.BI_GEMM_ERR_UNSUPPORTED),     # split not a multiple of 128
    (32, 8, 128, 16, 0.1, 2048, bg.BI_GEMM_ERR_UNSUPPORTED),
])
def test_attention_create_refuses_before_touching_cuda(Hq, Hkv, D, page, scale, split, want):
    h = ctypes.c_void_p()
    assert bg.library().bi_attention_create(ctypes.byref(h), Hq, Hkv, D, page, scale, split) == want
    assert h.value is None


def test_attention_null_arguments():
    L = bg.library()
    assert L.bi_attention_create(None, 32, 8, 128, 16, 0.1, 0) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_attention_run(None, None, 1, None, None, None, None, 1, None, 1, 1, 0, None, None) == \
        bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_attention_get_device_error(None, None) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_attention_get_config(None, None) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_attention_destroy(None) == bg.BI_GEMM_OK


def test_prenorm_header_symbols_exported():
    declared = _declared("bi_prenorm.h")
    assert set(declared) == set(bg.PRENORM_EXPORTED_SYMBOLS)
    L = ctypes.CDLL(bgbuild.lib_path("libbi_gemm.so"))
    for name in declared:
        assert hasattr(L, name), name


@pytest.mark.parametrize("K,N,eps,chunk,want", [
    (16384, 24, -1.0, 0, bg.BI_GEMM_ERR_INVALID_ARG),
    (16384, 24, float("nan"), 0, bg.BI_GEMM_ERR_INVALID_ARG),
    (16384, 24, 1e-6, -64, bg.BI_GEMM_ERR_INVALID_ARG),
    (16380, 24, 1e-6, 0, bg.BI_GEMM_ERR_UNSUPPORTED),     # K not a whole number of 16-byte pieces
    (16384, 20, 1e-6, 0, bg.BI_GEMM_ERR_UNSUPPORTED),     # N % 8
    (16384, 40, 1e-6, 0, bg.BI_GEMM_ERR_UNSUPPORTED),     # N > 32
    (16384, 24, 1e-6, 96, bg.BI_GEMM_ERR_UNSUPPORTED),    # chunk % 64
    (16384, 24, 1e-6, 2048, bg.BI_GEMM_ERR_UNSUPPORTED),
])
def test_prenorm_create_refuses_before_touching_cuda(K, N, eps, chunk, want):
    h = ctypes.c_void_p()
    assert bg.library().bi_prenorm_create(ctypes.byref(h), K, N, eps, chunk) == want
    assert h.value is None


def test_prenorm_null_arguments():
    L = bg.library()
    assert L.bi_prenorm_create(None, 16384, 24, 1e-6, 0) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_prenorm_run(None, None, 4, None, None, None) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_prenorm_get_config(None, None) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_prenorm_destroy(None) == bg.BI_GEMM_OK


def test_controls_symbols_exported():
    declared = _declared("bi_gemm_controls.h")
    assert declared, "controls header declares nothing"
    L = ctypes.CDLL(bgbuild.lib_path("libbi_gemm_controls.so"))
    for name in declared:
        assert hasattr(L, name), name
    # the control library hides its private copy of the product ABI
    assert not hasattr(L, "bi_gemm_run")


def test_version_and_strerror():
    assert bg.bi_gemm_version() >> 16 == 1
    for code in range(0, -7, -1):
        assert bg.bi_gemm_strerror(code) and "unknown" not in bg.bi_gemm_strerror(code)
    assert "unknown" in bg.bi_gemm_strerror(-99)


@pytest.mark.parametrize("K,N,dtype,layout,want", [
    (256, 128, 7, 0, bg.BI_GEMM_ERR_INVALID_ARG),        # bad dtype
    (256, 128, 0, 5, bg.BI_GEMM_ERR_INVALID_ARG),        # bad scale layout
    (-1, 128, 0, 0, bg.BI_GEMM_ERR_INVALID_ARG),
    (0, 128, 0, 0, bg.BI_GEMM_ERR_UNSUPPORTED),
    (250, 128, 0, 0, bg.BI_GEMM_ERR_UNSUPPORTED),        # bf16 row pitch not 16 B
    (256, 100, 1, 0, bg.BI_GEMM_ERR_UNSUPPORTED),
    (256, 128, 0, 1, bg.BI_GEMM_ERR_UNSUPPORTED),        # bf16 with scales
    (192, 128, 2, 1, bg.BI_GEMM_ERR_UNSUPPORTED),        # MXFP8 K % 128
    (256, 120, 2, 1, bg.BI_GEMM_ERR_UNSUPPORTED),        # MXFP8 N % 16
    (256, 128, 2, 0, bg.BI_GEMM_ERR_UNSUPPORTED),        # MXFP8 without scales
])
def test_create_refuses_before_touching_cuda(K, N, dtype, layout, want):
    h = ctypes.c_void_p()
    rc = bg.library().bi_gemm_create(ctypes.byref(h), K, N, dtype, layout)
    assert rc == want
    assert h.value is None


def test_null_arguments():
    L = bg.library()
    assert L.bi_gemm_create(None, 256, 128, 0, 0) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_gemm_run(None, None, 4, None, None, None, None) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_gemm_get_device_error(None, None) == bg.BI_GEMM_ERR_INVALID_ARG
    assert L.bi_gemm_destroy(None) == bg.BI_GEMM_OK
    assert L.bi_gemm_get_config(None, None) == bg.BI_GEMM_ERR_INVALID_ARG
    b = ctypes.c_uint64()
    assert L.bi_gemm_workspace_size(None, 4, ctypes.byref(b)) == bg.BI_GEMM_ERR_INVALID_ARG
    opts = bg.bi_gemm_options(-1, 0, 0)
    h = ctypes.c_void_p()
    assert L.bi_gemm_create_ex(ctypes.byref(h), 256, 128, 0, 0, ctypes.byref(opts)) == bg.BI_GEMM_ERR_INVALID_ARG
    opts = bg.bi_gemm_options(5, 0, 0)   # 5 > ceil(256 / 64) k-blocks
    assert L.bi_gemm_create_ex(ctypes.byref(h), 256, 128, 0, 0, ctypes.byref(opts)) == bg.BI_GEMM_ERR_INVALID_ARG
    opts = bg.bi_gemm_options(0, -3, 0)   # negative grid bound
    assert L.bi_gemm_create_ex(ctypes.byref(h), 256, 128, 0, 0, ctypes.byref(opts)) == bg.BI_GEMM_ERR_INVALID_ARG


def test_product_binding_has_no_fallback(monkeypatch, tmp_path):
    """Without the built library the binding raises instead of computing anything."""
    monkeypatch.setattr(bgbuild, "lib_path", lambda name="libbi_gemm.so": str(tmp_path / name))
    monkeypatch.setattr(bg, "_lib", None)
    with pytest.raises(ImportError):
        bg.library()


def test_product_path_does_not_import_oracle():
    pkg = os.path.join(ROOT, "invariant_bi_gemm_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "bi_oracle" not in src and "from oracle" not in src and "import oracle" not in src


def _structs(header):
    """{typedef name: [(C type, field), ...]} of the plain structs a header declares."""
    src = open(os.path.join(ROOT, "include", header)).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for body, name in re.findall(r"typedef struct\s*\{(.*?)\}\s*(\w+)\s*;", src, flags=re.S):
        fields = []
        for decl in body.split(";"):
            decl = decl.strip()
            if not decl:
                continue
            m = re.match(r"((?:const\s+)?\w+\s*\**)\s*(.+)", decl)
            ctype, names = m.group(1).replace(" ", ""), m.group(2)
            fields += [(ctype, n.strip()) for n in names.split(",")]
        out[name] = fields
    return out


@pytest.mark.parametrize("header,name,cls", [
    ("bi_gemm.h", "bi_gemm_config", "bi_gemm_config"),
    ("bi_gemm.h", "bi_gemm_options", "bi_gemm_options"),
    ("bi_gemm.h", "bi_gemm_block", "bi_gemm_block"),
    ("bi_gemm.h", "bi_gemm_scales", "bi_gemm_scales"),
    ("bi_rmsnorm.h", "bi_rmsnorm_config", "bi_rmsnorm_config"),
    ("bi_attention.h", "bi_attention_config", "bi_attention_config"),
    ("bi_prenorm.h", "bi_prenorm_config", "bi_prenorm_config"),
])
def test_binding_structs_match_the_headers(header, name, cls):
    """The ctypes structures of the binding list the header's fields in the header's order with
    the header's widths, so a field added on one side only is caught without a GPU."""
    width = {"int32_t": ctypes.c_int32, "uint32_t": ctypes.c_uint32, "uint64_t": ctypes.c_uint64,
             "int64_t": ctypes.c_int64}
    fields = _structs(header)[name]
    py = getattr(bg, cls)._fields_
    assert [n for _, n in fields] == [n for n, _ in py]
    assert [ctypes.c_void_p if t.endswith("*") else width[t] for t, _ in fields] == [t for _, t in py]
