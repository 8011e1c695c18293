"""Python binding of libtwell.so (the C ABI in include/twell.h).

Argument marshalling only: every computation runs in the CUDA kernels of the
library.  Torch tensors (CUDA) or raw integer device pointers are accepted
wherever the ABI takes a pointer; PyTorch provides device memory and streams.
The library must have been built (``_build.build()``); importing this module
without it raises instead of falling back to anything else.

Names follow the ABI: ``twell_workspace_size``, ``twell_pack_dense``,
``twell_pack``, ``twell_ffn_forward``, ``twell_ffn_backward``,
``twell_get_status``, and the row-ELL comparison baseline
``twell_rowell_pack_dense`` / ``twell_rowell_forward``.  ``TwellBuffers`` and
``RowEllBuffers`` allocate the device buffers of a ``twell_t`` /
``twell_rowell_t`` with torch.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

LIB_PATH = _build.LIB

TWELL_OK = 0
TWELL_ERR = {
    -1: "TWELL_ERR_ARG", -2: "TWELL_ERR_ALIGN", -3: "TWELL_ERR_DTYPE",
    -4: "TWELL_ERR_CAPACITY", -5: "TWELL_ERR_INDEX", -6: "TWELL_ERR_TIMEOUT",
    -7: "TWELL_ERR_CUDA", -8: "TWELL_ERR_WORKSPACE", -9: "TWELL_ERR_UNSUPPORTED",
    -10: "TWELL_ERR_STATIC_LIMIT", -11: "TWELL_ERR_RANGE",
}
TWELL_F32, TWELL_BF16 = 0, 1

EXPORTS = ("twell_workspace_size", "twell_workspace_size_rows", "twell_pack_dense", "twell_pack",
           "twell_ffn_forward", "twell_ffn_backward", "twell_get_status", "twell_version",
           "twell_rowell_pack_dense", "twell_rowell_forward")


class TwellError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {TWELL_ERR.get(code, code)}")
        self.code = code


class twell_t(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("F", ctypes.c_int32), ("C", ctypes.c_int32), ("K", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("idx", ctypes.c_void_p), ("val", ctypes.c_void_p), ("nnz", ctypes.c_void_p),
        ("ovf_rows", ctypes.c_void_p), ("n_ovf", ctypes.c_void_p), ("ovf_cap", ctypes.c_int32),
        ("g_fb", ctypes.c_void_p), ("u_val", ctypes.c_void_p), ("u_fb", ctypes.c_void_p),
        ("status", ctypes.c_void_p), ("dense_switch", ctypes.c_float),
        ("dense_density", ctypes.c_float), ("dh_density", ctypes.c_float),
        ("dense_rows_cap", ctypes.c_int32),
        ("gather_passes", ctypes.c_int32),
    ]


class twell_rowell_t(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("F", ctypes.c_int32), ("E", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("idx", ctypes.c_void_p), ("val", ctypes.c_void_p), ("nnz", ctypes.c_void_p),
        ("status", ctypes.c_void_p),
    ]


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load libtwell.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libtwell.so is not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    P, I, F32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    S = ctypes.c_size_t
    TP = ctypes.POINTER(twell_t)
    lib.twell_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.twell_workspace_size.restype = S
    lib.twell_workspace_size_rows.argtypes = [I, I, I, I, I, I, I, I]
    lib.twell_workspace_size_rows.restype = S
    lib.twell_pack_dense.argtypes = [P, TP, P]
    lib.twell_pack.argtypes = [P, P, P, P, I, TP, P, S, P]
    lib.twell_ffn_forward.argtypes = [P, P, P, P, P, P, I, I, TP, P, P, S, P]
    lib.twell_ffn_backward.argtypes = [P, P, P, P, TP, P, F32, I, P, P, P, P, P, P, S, P]
    lib.twell_get_status.argtypes = [TP, P, ctypes.POINTER(ctypes.c_int32)]
    lib.twell_version.restype = ctypes.c_char_p
    RP = ctypes.POINTER(twell_rowell_t)
    lib.twell_rowell_pack_dense.argtypes = [P, RP, P]
    lib.twell_rowell_forward.argtypes = [P, P, P, I, RP, P, P]
    for name in ("twell_pack_dense", "twell_pack", "twell_ffn_forward", "twell_ffn_backward",
                 "twell_get_status", "twell_rowell_pack_dense", "twell_rowell_forward"):
        getattr(lib, name).restype = I
    if path is None:
        _lib = lib
    return lib


def _ptr(a) -> Optional[int]:
    if a is None:
        return None
    if isinstance(a, int):
        return a
    return a.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str) -> None:
    if code != TWELL_OK:
        raise TwellError(code, where)


def twell_version() -> str:
    return load().twell_version().decode()


def twell_workspace_size(T: int, D: int, F: int, C: int, K: int, dtype: int, train: int) -> int:
    return int(load().twell_workspace_size(T, D, F, C, K, dtype, int(train)))


def twell_workspace_size_rows(T: int, D: int, F: int, C: int, K: int, dtype: int, train: int,
                              dense_rows_cap: int) -> int:
    return int(load().twell_workspace_size_rows(T, D, F, C, K, dtype, int(train),
                                                int(dense_rows_cap)))


def twell_pack_dense(H, tw: twell_t, stream=None) -> None:
    _check(load().twell_pack_dense(_ptr(H), ctypes.byref(tw), _stream(stream)), "twell_pack_dense")


def twell_pack(x, Wg, bg, row_bias, D: int, tw: twell_t, workspace, workspace_bytes: int,
               stream=None) -> None:
    _check(load().twell_pack(_ptr(x), _ptr(Wg), _ptr(bg), _ptr(row_bias), D, ctypes.byref(tw),
                             _ptr(workspace), int(workspace_bytes), _stream(stream)), "twell_pack")


def twell_ffn_forward(x, Wg, bg, row_bias, Wu, Wd, D: int, train: int, tw: twell_t, y, workspace,
                      workspace_bytes: int, stream=None) -> None:
    _check(load().twell_ffn_forward(_ptr(x), _ptr(Wg), _ptr(bg), _ptr(row_bias), _ptr(Wu),
                                    _ptr(Wd), D, int(train), ctypes.byref(tw), _ptr(y),
                                    _ptr(workspace), int(workspace_bytes), _stream(stream)),
           "twell_ffn_forward")


def twell_ffn_backward(x, Wg, Wu, Wd, tw: twell_t, dy, lam: float, D: int, dx, dWg, dbg, dWu,
                       dWd, workspace, workspace_bytes: int, stream=None) -> None:
    _check(load().twell_ffn_backward(_ptr(x), _ptr(Wg), _ptr(Wu), _ptr(Wd), ctypes.byref(tw),
                                     _ptr(dy), float(lam), D, _ptr(dx), _ptr(dWg), _ptr(dbg),
                                     _ptr(dWu), _ptr(dWd), _ptr(workspace), int(workspace_bytes),
                                     _stream(stream)), "twell_ffn_backward")


def twell_rowell_pack_dense(H, re: twell_rowell_t, stream=None) -> None:
    _check(load().twell_rowell_pack_dense(_ptr(H), ctypes.byref(re), _stream(stream)),
           "twell_rowell_pack_dense")


def twell_rowell_forward(x, Wu, Wd, D: int, re: twell_rowell_t, y, stream=None) -> None:
    _check(load().twell_rowell_forward(_ptr(x), _ptr(Wu), _ptr(Wd), D, ctypes.byref(re), _ptr(y),
                                       _stream(stream)), "twell_rowell_forward")


def twell_get_status(tw: twell_t, stream=None):
    """Returns (status_code, n_ovf); synchronises the stream."""
    n = ctypes.c_int32(0)
    code = load().twell_get_status(ctypes.byref(tw), _stream(stream), ctypes.byref(n))
    return int(code), int(n.value)


class TwellBuffers:
    """Device buffers of one twell_t, allocated with torch (plumbing only)."""

    def __init__(self, T: int, F: int, C: int, K: int, dtype: int, ovf_cap: Optional[int] = None,
                 train: bool = False, device="cuda", dense_switch: float = 0.0,
                 dense_density: float = 0.0, dh_density: float = 0.0, dense_rows_cap: int = 0,
                 gather_passes: int = 0):
        import torch
        tdt = torch.bfloat16 if dtype == TWELL_BF16 else torch.float32
        nt = F // C
        cap = T if ovf_cap is None else int(ovf_cap)
        self.T, self.F, self.C, self.K, self.dtype, self.cap = T, F, C, K, dtype, cap
        self.idx = torch.empty((nt, T, K), dtype=torch.uint8, device=device)
        self.val = torch.empty((nt, T, K), dtype=tdt, device=device)
        self.nnz = torch.empty((nt, T), dtype=torch.uint8, device=device)
        self.ovf_rows = torch.empty((max(cap, 1),), dtype=torch.int32, device=device)
        self.n_ovf = torch.zeros((1,), dtype=torch.int32, device=device)
        self.g_fb = torch.empty((max(cap, 1), F), dtype=tdt, device=device)
        self.u_val = torch.empty((nt, T, K), dtype=tdt, device=device) if train else None
        self.u_fb = torch.empty((max(cap, 1), F), dtype=tdt, device=device) if train else None
        self.status = torch.zeros((4,), dtype=torch.int32, device=device)
        self.t = twell_t(T=T, F=F, C=C, K=K, dtype=dtype, idx=_ptr(self.idx), val=_ptr(self.val),
                         nnz=_ptr(self.nnz), ovf_rows=_ptr(self.ovf_rows), n_ovf=_ptr(self.n_ovf),
                         ovf_cap=cap, g_fb=_ptr(self.g_fb), u_val=_ptr(self.u_val),
                         u_fb=_ptr(self.u_fb), status=_ptr(self.status),
                         dense_switch=float(dense_switch), dense_density=float(dense_density),
                         dh_density=float(dh_density), dense_rows_cap=int(dense_rows_cap),
                         gather_passes=int(gather_passes))


class RowEllBuffers:
    """Device buffers of one twell_rowell_t (row-ELL baseline), allocated with torch."""

    def __init__(self, T: int, F: int, E: int, dtype: int, device="cuda"):
        import torch
        tdt = torch.bfloat16 if dtype == TWELL_BF16 else torch.float32
        self.T, self.F, self.E, self.dtype = T, F, E, dtype
        self.idx = torch.empty((T, E), dtype=torch.int16, device=device)
        self.val = torch.empty((T, E), dtype=tdt, device=device)
        self.nnz = torch.empty((T,), dtype=torch.int32, device=device)
        self.status = torch.zeros((4,), dtype=torch.int32, device=device)
        self.t = twell_rowell_t(T=T, F=F, E=E, dtype=dtype, idx=_ptr(self.idx),
                                val=_ptr(self.val), nnz=_ptr(self.nnz), status=_ptr(self.status))


def workspace(T: int, D: int, F: int, C: int, K: int, dtype: int, train: bool, device="cuda",
              dense_rows_cap: int = 0):
    """Allocate a workspace tensor of twell_workspace_size_rows bytes (256-byte
    aligned by torch); dense_rows_cap must match the twell_t's."""
    import torch
    n = twell_workspace_size_rows(T, D, F, C, K, dtype, int(train), int(dense_rows_cap))
    if n == 0:
        raise TwellError(-1, "twell_workspace_size")
    return torch.empty((n,), dtype=torch.uint8, device=device), n
