"""CPU-side checks of the C ABI: the library builds, loads and exports every
symbol include/twell.h declares, and host-detectable argument errors return
their codes before anything touches a GPU."""
import ctypes
import os
import re

import pytest

import activation_sparse_transformer_gate_gb300 as tw
from activation_sparse_transformer_gate_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return tw.load()


def header_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ \t\*]*?\b(twell_[a-z0-9_]+)\s*\(",
                            src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = header_functions()
    for n in tw.EXPORTS:
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    for n in header_functions():
        assert hasattr(lib, n), f"libtwell.so does not export {n}"
    assert "sm_103a" in tw.twell_version()


def test_test_hooks_stay_out_of_the_product_library(lib):
    """The measurement hooks (GEMM engine test entry, gather probe) are built
    into the test-hooks variant only."""
    for n in ("twell_test_tc_gemm", "twell_test_gather_probe"):
        assert not hasattr(lib, n), f"libtwell.so exports the test hook {n}"
    _build.build(variants=("hooks",))
    hooks = tw.load(_build.lib_path("hooks"))
    for n in ("twell_test_tc_gemm", "twell_test_gather_probe"):
        assert hasattr(hooks, n), n
    for n in header_functions():
        assert hasattr(hooks, n), n


def test_workspace_size(lib):
    a = tw.twell_workspace_size(4096, 2048, 8192, 128, 8, tw.TWELL_BF16, 0)
    b = tw.twell_workspace_size(4096, 2048, 8192, 128, 8, tw.TWELL_BF16, 1)
    assert a > 4096 * 8192 * 2 and b > a
    assert tw.twell_workspace_size(4096, 2048, 8192, 100, 8, tw.TWELL_BF16, 0) == 0   # C
    assert tw.twell_workspace_size(4096, 2048, 8192, 128, 3, tw.TWELL_BF16, 0) == 0   # K
    assert tw.twell_workspace_size(4096, 2048, 8192, 64, 128, tw.TWELL_BF16, 0) == 0  # K > C
    assert tw.twell_workspace_size(0, 2048, 8192, 128, 8, tw.TWELL_BF16, 0) == 0      # T
    assert tw.twell_workspace_size(64, 2048, 8192, 128, 8, 7, 0) == 0                 # dtype
    assert tw.twell_workspace_size(64, 2050, 8192, 128, 8, tw.TWELL_BF16, 0) == 0     # pitch


def _fake_tw(**kw):
    # Fake, 16-byte aligned "device" addresses: validation must fail before any
    # pointer is dereferenced or any CUDA call is made.
    base = 1 << 40
    t = tw.twell_t(T=64, F=512, C=64, K=4, dtype=tw.TWELL_F32, idx=base, val=base + 4096,
                   nnz=base + 8192, ovf_rows=base + 12288, n_ovf=base + 16384, ovf_cap=64,
                   g_fb=base + 20480, u_val=None, u_fb=None, status=base + 24576, dense_switch=0.0)
    for k, v in kw.items():
        setattr(t, k, v)
    return t


def _code(fn, *args):
    return fn(*args)


@pytest.mark.parametrize("field,value,code", [
    ("C", 48, -1), ("K", 3, -1), ("K", 128, -1), ("T", 0, -1), ("dtype", 9, -3),
    ("idx", None, -1), ("status", None, -1), ("ovf_cap", -1, -1), ("val", (1 << 40) + 4100, -2),
])
def test_pack_dense_rejects_bad_twell(lib, field, value, code):
    t = _fake_tw(**{field: value})
    assert lib.twell_pack_dense(ctypes.c_void_p(1 << 41), ctypes.byref(t), None) == code


def test_forward_rejects_bad_args(lib):
    t = _fake_tw()
    P = ctypes.c_void_p
    good = P(1 << 41)
    ws = P(1 << 42)
    need = tw.twell_workspace_size(64, 128, 512, 64, 4, tw.TWELL_F32, 0)
    f = lib.twell_ffn_forward
    # NULL x
    assert f(None, good, good, None, None, good, 128, 0, ctypes.byref(t), good, ws, need, None) == -1
    # misaligned W_down
    assert f(good, good, good, None, None, P((1 << 41) + 8), 128, 0, ctypes.byref(t), good, ws,
             need, None) == -2
    # workspace too small, NULL, misaligned
    assert f(good, good, good, None, None, good, 128, 0, ctypes.byref(t), good, ws, need - 1,
             None) == -8
    assert f(good, good, good, None, None, good, 128, 0, ctypes.byref(t), good, None, need,
             None) == -8
    assert f(good, good, good, None, None, good, 128, 0, ctypes.byref(t), good, P((1 << 42) + 16),
             need, None) == -8
    # d_model whose row pitch is not 16 bytes / too large
    assert f(good, good, good, None, None, good, 130, 0, ctypes.byref(t), good, ws, need, None) == -2
    assert f(good, good, good, None, None, good, 8192, 0, ctypes.byref(t), good, ws, 1 << 40,
             None) == -1
    # training without the u buffers (gated)
    assert f(good, good, good, None, good, good, 128, 1, ctypes.byref(t), good, ws, need,
             None) == -1


def test_backward_rejects_bad_args(lib):
    t = _fake_tw()
    P = ctypes.c_void_p
    good = P(1 << 41)
    need = tw.twell_workspace_size(64, 128, 512, 64, 4, tw.TWELL_F32, 1)
    f = lib.twell_ffn_backward
    assert f(good, good, None, good, ctypes.byref(t), good, ctypes.c_float(0.0), 128, good, good,
             None, good, good, P(1 << 42), need, None) == -1          # NULL dbg
    assert f(good, good, None, good, ctypes.byref(t), good, ctypes.c_float(0.0), 128, good, good,
             good, good, good, P(1 << 42), need - 1, None) == -8      # workspace


def header_struct_fields(name):
    """Field names, in order, of `typedef struct { ... } name;` in include/twell.h."""
    src = open(os.path.join(ROOT, "include", "twell.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    m = re.search(r"typedef\s+struct\s*\{([^{}]*)\}\s*" + name + r"\s*;", src)
    assert m, name
    fields = []
    for decl in m.group(1).split(";"):
        decl = decl.strip()
        if not decl:
            continue
        # "type a, *b, c" -> a, b, c
        parts = decl.split(",")
        first = re.findall(r"\*?\s*([A-Za-z_][A-Za-z0-9_]*)\s*$", parts[0])
        fields += first + [re.sub(r"[\s\*]", "", p) for p in parts[1:]]
    return fields


@pytest.mark.parametrize("name", ["twell_t", "twell_rowell_t"])
def test_binding_structs_match_the_header(name):
    """The ctypes mirrors of the ABI structs list the header's fields in the
    header's order (a field added on one side only would shift the others)."""
    py = [f[0] for f in getattr(tw, name)._fields_]
    assert py == header_struct_fields(name)


def test_workspace_size_with_a_dense_row_cap(lib):
    """A cap on the dense-path rows sizes those row buffers for the cap:
    at the training-step shape, 256 rows instead of 4096."""
    full = tw.twell_workspace_size(4096, 2048, 8192, 128, 8, tw.TWELL_BF16, 1)
    assert tw.twell_workspace_size_rows(4096, 2048, 8192, 128, 8, tw.TWELL_BF16, 1, 0) == full
    assert tw.twell_workspace_size_rows(4096, 2048, 8192, 128, 8, tw.TWELL_BF16, 1, 4096) == full
    assert tw.twell_workspace_size_rows(4096, 2048, 8192, 128, 8, tw.TWELL_BF16, 1, 9999) == full
    capped = tw.twell_workspace_size_rows(4096, 2048, 8192, 128, 8, tw.TWELL_BF16, 1, 256)
    # per dense row: h (2F), u rows (2F), dz/du/h rows (3 x 4F) bytes, x and dy
    # rows, and the dbg column sums (4F per 32 rows)
    per_row = 2 * 8192 + 2 * 8192 + 3 * 4 * 8192 + 2 * 2 * 2048 + 4 * 8192 // 32
    assert full - capped == (4096 - 256) * per_row
    assert capped < full / 3
    # rounded up to whole 128-row tiles
    assert (tw.twell_workspace_size_rows(4096, 2048, 8192, 128, 8, tw.TWELL_BF16, 1, 200) ==
            capped)


def test_workspace_without_dense_path_rows(lib):
    """A cap below one 128-row tile admits no dense-path row: the workspace
    then holds no dense-path GEMM buffers or fp16 weight copies, only the
    gather path's overflow-row arrays (128 rows)."""
    T, D, F = 4096, 2048, 8192
    small = tw.twell_workspace_size_rows(T, D, F, 128, 8, tw.TWELL_BF16, 1, 64)
    tile = tw.twell_workspace_size_rows(T, D, F, 128, 8, tw.TWELL_BF16, 1, 128)
    dense_row_bytes = 128 * (2 * F + 2 * F + 2 * D + 2 * D)  # h, u rows, x and dy rows
    f16_copies = 3 * 2 * F * D
    dbg_groups = 4 * (128 // 32) * F                          # dbg column sums per 32 rows
    assert tile - small == dense_row_bytes + f16_copies + dbg_groups
    # T below one tile: every row may run densely, the buffers are kept
    assert (tw.twell_workspace_size_rows(100, D, F, 128, 8, tw.TWELL_BF16, 1, 100) ==
            tw.twell_workspace_size(100, D, F, 128, 8, tw.TWELL_BF16, 1))
