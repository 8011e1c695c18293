"""CPU oracle for the activation-sparse FFN (TEST INFRASTRUCTURE ONLY).

Plain C loops in double precision (``twell_oracle.c``) behind ctypes.  Only
the tests, the smoke check and the benchmark's CPU-baseline / reference leg
use this package; the CUDA library and its Python binding never import it,
and it imports nothing from them.

What each function follows (pages: "Sparser, Faster, Lighter Transformer
Language Models", technical summary):

* ``gate``           -- the dense gate matmul whose epilogue produces TwELL (2.A).
* ``twell_pack``     -- TwELL slots + hybrid split into overflow rows (2.A).
* ``twell_unpack``   -- inverse of the pack.
* ``ffn_dense``      -- the FFN by its definition over all neurons.
* ``ffn_twell``      -- the FFN consuming TwELL + dense backup (2.B inference).
* ``ffn_backward``   -- gradients with the L1 term (2.B training).
* ``ffn_loss``       -- the scalar loss, for finite differences.

Parity status: every function here is pinned by the tests in
``tests/test_oracle.py`` (hand-worked cases, numpy closed forms, invariants,
finite differences and the sparse == dense identity).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "twell_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

Q_F32, Q_BF16, Q_NONE = 0, 1, 2
DT = {"f32": 0, "bf16": 1}
QMODE = {"f32": Q_F32, "bf16": Q_BF16, "none": Q_NONE}


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (no fast-math, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-shared",
               "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_set_threads.argtypes = [I]
            lib.oracle_get_threads.restype = I
            lib.oracle_bf16_round.argtypes = [P, P, ctypes.c_int64]
            lib.oracle_gate.argtypes = [I, I, I, I, P, P, P, P, P]
            lib.oracle_twell_pack.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P]
            lib.oracle_twell_pack.restype = I
            lib.oracle_twell_unpack.argtypes = [I, I, I, I, P, P, P, P, P, I, P, P]
            lib.oracle_ffn_dense.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P]
            lib.oracle_ffn_twell.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, P, P, I, P, P]
            lib.oracle_ffn_backward.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P,
                                                ctypes.c_double, P, I, P, I, P, P, P, P, P]
            lib.oracle_ffn_loss.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, ctypes.c_double]
            lib.oracle_ffn_loss.restype = ctypes.c_double
            lib.oracle_rowell_pack.argtypes = [I, I, I, P, P, P, P]
            lib.oracle_ffn_rowell.argtypes = [I, I, I, I, P, P, P, P, P, P, P]
            _lib = lib
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype) if dtype is not None else np.ascontiguousarray(a)


def _storage(a, dt: str):
    if a is None:
        return None
    return _c(a, np.uint16 if dt == "bf16" else np.float32)


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def get_threads() -> int:
    return int(_load().oracle_get_threads())


def bf16_round(a: np.ndarray) -> np.ndarray:
    a = _c(a, np.float32)
    out = np.empty(a.shape, dtype=np.uint16)
    _load().oracle_bf16_round(_p(a), _p(out), a.size)
    return out


def gate(x, Wg, bg, rb, dt: str) -> np.ndarray:
    """z [T][F] in float64."""
    x, Wg = _storage(x, dt), _storage(Wg, dt)
    T, D = x.shape
    F = Wg.shape[0]
    z = np.empty((T, F), dtype=np.float64)
    _load().oracle_gate(T, D, F, DT[dt], _p(x), _p(Wg), _p(_c(bg, np.float32)),
                        _p(_c(rb, np.float32)), _p(z))
    return z


def twell_pack(z: np.ndarray, C: int, K: int, q: str) -> dict:
    """TwELL + hybrid split of a pre-activation matrix z [T][F]."""
    z = _c(z, np.float64)
    T, F = z.shape
    nt = F // C
    idx = np.empty((nt, T, K), dtype=np.uint8)
    val = np.empty((nt, T, K), dtype=np.float64)
    nnz = np.empty((nt, T), dtype=np.uint8)
    row_ovf = np.empty((T,), dtype=np.uint8)
    ovf_rows = np.empty((T,), dtype=np.int32)
    g_fb = np.empty((T, F), dtype=np.float64)
    n = _load().oracle_twell_pack(T, F, C, K, QMODE[q], _p(z), _p(idx), _p(val), _p(nnz),
                                  _p(row_ovf), _p(ovf_rows), _p(g_fb))
    return dict(idx=idx, val=val, nnz=nnz, row_ovf=row_ovf, ovf_rows=ovf_rows[:n].copy(),
                n_ovf=n, g_fb=g_fb[:n].copy(), C=C, K=K, T=T, F=F)


def twell_unpack(tw: dict) -> np.ndarray:
    T, F, C, K = tw["T"], tw["F"], tw["C"], tw["K"]
    g = np.empty((T, F), dtype=np.float64)
    ovf = _c(tw["ovf_rows"], np.int32)
    gfb = _c(tw["g_fb"], np.float64)
    if gfb.size == 0:
        gfb = np.zeros((1, F), dtype=np.float64)
    _load().oracle_twell_unpack(T, F, C, K, _p(_c(tw["idx"], np.uint8)), _p(_c(tw["val"], np.float64)),
                                _p(_c(tw["nnz"], np.uint8)), _p(_c(tw["row_ovf"], np.uint8)),
                                _p(ovf), int(tw["n_ovf"]), _p(gfb), _p(g))
    return g


def ffn_dense(x, Wg, bg, rb, Wu, Wd, dt: str, q: str, want_h: bool = False):
    x, Wg, Wu, Wd = (_storage(a, dt) for a in (x, Wg, Wu, Wd))
    T, D = x.shape
    F = Wg.shape[0]
    y = np.empty((T, D), dtype=np.float64)
    h = np.empty((T, F), dtype=np.float64) if want_h else None
    _load().oracle_ffn_dense(T, D, F, DT[dt], QMODE[q], _p(x), _p(Wg), _p(_c(bg, np.float32)),
                             _p(_c(rb, np.float32)), _p(Wu), _p(Wd), _p(y), _p(h))
    return (y, h) if want_h else y


def ffn_twell(x, Wu, Wd, tw: dict, dt: str) -> np.ndarray:
    x, Wu, Wd = (_storage(a, dt) for a in (x, Wu, Wd))
    T, D = x.shape
    F, C, K = tw["F"], tw["C"], tw["K"]
    y = np.empty((T, D), dtype=np.float64)
    gfb = _c(tw["g_fb"], np.float64)
    if gfb.size == 0:
        gfb = np.zeros((1, F), dtype=np.float64)
    _load().oracle_ffn_twell(T, D, F, C, K, DT[dt], _p(x), _p(Wu), _p(Wd),
                             _p(_c(tw["idx"], np.uint8)), _p(_c(tw["val"], np.float64)),
                             _p(_c(tw["nnz"], np.uint8)), _p(_c(tw["row_ovf"], np.uint8)),
                             _p(_c(tw["ovf_rows"], np.int32)), int(tw["n_ovf"]), _p(gfb), _p(y))
    return y


def ffn_backward(x, Wg, bg, rb, Wu, Wd, dy, lam: float, dt: str, q: str,
                 tok_sel=None, neu_sel=None) -> dict:
    x, Wg, Wu, Wd, dy = (_storage(a, dt) for a in (x, Wg, Wu, Wd, dy))
    T, D = x.shape
    F = Wg.shape[0]
    ts = None if tok_sel is None else _c(tok_sel, np.int32)
    ns = None if neu_sel is None else _c(neu_sel, np.int32)
    nt = T if ts is None else ts.size
    nn = F if ns is None else ns.size
    dx = np.empty((nt, D), dtype=np.float64)
    dWg = np.empty((nn, D), dtype=np.float64)
    dbg = np.empty((nn,), dtype=np.float64)
    dWu = np.empty((nn, D), dtype=np.float64) if Wu is not None else None
    dWd = np.empty((nn, D), dtype=np.float64)
    _load().oracle_ffn_backward(T, D, F, DT[dt], QMODE[q], _p(x), _p(Wg), _p(_c(bg, np.float32)),
                                _p(_c(rb, np.float32)), _p(Wu), _p(Wd), _p(dy), float(lam),
                                _p(ts), nt if ts is not None else 0, _p(ns),
                                nn if ns is not None else 0,
                                _p(dx), _p(dWg), _p(dbg), _p(dWu), _p(dWd))
    return dict(dx=dx, dWg=dWg, dbg=dbg, dWu=dWu, dWd=dWd)


def ffn_loss(x, Wg, bg, rb, Wu, Wd, dy, lam: float, dt: str, q: str) -> float:
    x, Wg, Wu, Wd, dy = (_storage(a, dt) for a in (x, Wg, Wu, Wd, dy))
    T, D = x.shape
    F = Wg.shape[0]
    return float(_load().oracle_ffn_loss(T, D, F, DT[dt], QMODE[q], _p(x), _p(Wg),
                                         _p(_c(bg, np.float32)), _p(_c(rb, np.float32)),
                                         _p(Wu), _p(Wd), _p(dy), float(lam)))


def rowell_pack(h: np.ndarray, E: int) -> dict:
    """Classic row-ELL of a dense activation matrix h [T][F] (entries >= 0)."""
    h = _c(h, np.float64)
    T, F = h.shape
    idx = np.empty((T, E), dtype=np.uint16)
    val = np.empty((T, E), dtype=np.float64)
    nnz = np.empty((T,), dtype=np.int32)
    _load().oracle_rowell_pack(T, F, E, _p(h), _p(idx), _p(val), _p(nnz))
    return dict(idx=idx, val=val, nnz=nnz, T=T, F=F, E=E)


def ffn_rowell(x, Wu, Wd, re: dict, dt: str) -> np.ndarray:
    """y = up + down projection from row-ELL gate values."""
    x, Wu, Wd = (_storage(a, dt) for a in (x, Wu, Wd))
    T, D = x.shape
    y = np.empty((T, D), dtype=np.float64)
    _load().oracle_ffn_rowell(T, D, re["E"], DT[dt], _p(x), _p(Wu), _p(Wd),
                              _p(_c(re["idx"], np.uint16)), _p(_c(re["val"], np.float64)),
                              _p(_c(re["nnz"], np.int32)), _p(y))
    return y
