"""Seeded synthetic inputs for the activation-sparse FFN.

This module is shared by the tests, the benchmark and the smoke check.  It
holds no arithmetic of the method itself: it only draws random numbers with
numpy's PCG64 generator, scales them to the stated variance and stores them in
the storage type of the workload (fp32, or bf16 bit patterns obtained by
round-to-nearest-even).  Both the CUDA path and the oracle receive the
identical arrays.

Workloads follow the shapes and distributions of the pages' setting
("Sparser, Faster, Lighter Transformer Language Models", technical summary
section 2: a transformer FFN with ReLU activations that is >99% sparse after L1
regularisation; section 4: denser early/informative tokens).  The trained
FineWeb activations of the pages are not available, so these draws stand in for
them:

* x ~ N(0, 1) per element, weights ~ N(0, 1/fan_in) (variance), so that the
  gate pre-activation is approximately N(b, 1) and the active fraction is
  1 - Phi(-b): b = -2.33 gives ~0.99% active (~99% sparse).
* the dense-leading-token workload adds a per-token bias of +1.49 to the first
  16 tokens of each 1024-token sequence (effective bias -0.84, ~20% active).

Draw order: x, W_gate (W1), W_up (gated only), W_down (W2), dy (training).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even) and
    return the 16-bit patterns as uint16.  Inputs here are finite normals."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 view of a stored array (bf16 bits or float32)."""
    if dtype == BF16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float32).astype(np.float64)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int                 # tokens (rows)
    D: int                 # d_model
    F: int                 # d_ff (hidden neurons)
    C: int                 # TwELL tile width (columns of the hidden axis)
    K: int                 # slots per (row, tile)
    dtype: str             # storage type of x, weights, y: "f32" or "bf16"
    gated: bool            # gated (gate*up) or plain ReLU FFN
    bias: float            # uniform per-neuron gate bias
    seed: int
    hot_tokens: int = 0    # leading tokens per sequence that get hot_bias
    seq_len: int = 0       # sequence length for the hot-token pattern
    hot_bias: float = 0.0  # per-token bias added to the hot tokens
    lam: float = 0.0       # L1 coefficient (training)
    train: bool = False    # draw dy as well

    @property
    def n_tiles(self) -> int:
        return self.F // self.C

    def describe(self) -> str:
        return (f"{self.name}: T={self.T} D={self.D} F={self.F} C={self.C} K={self.K} "
                f"{self.dtype} {'gated' if self.gated else 'non-gated'} b={self.bias}")


def config1() -> Workload:
    """Non-gated fp32 ReLU FFN, T=64, D=128, F=512, tile 64, K=4."""
    return Workload("c1_f32_nongated", 64, 128, 512, 64, 4, F32, False, -2.33, 1001)


def config2() -> Workload:
    """Gated bf16 FFN, T=4096, D=2048, F=8192, tile 128, K=8, ~99% sparse."""
    return Workload("c2_bf16_gated_T4096", 4096, 2048, 8192, 128, 8, BF16, True, -2.33, 1002)


def config3() -> Workload:
    """As config 2 with T=16384 = 16 x 1024 and dense leading tokens."""
    return Workload("c3_bf16_gated_T16384_hot16", 16384, 2048, 8192, 128, 8, BF16, True,
                    -2.33, 1003, hot_tokens=16, seq_len=1024, hot_bias=1.49)


SWEEP_BIASES = (-1.28, -1.64, -2.33, -2.58)
SWEEP_KS = (4, 8, 16)


def config4(bias: float, K: int) -> Workload:
    """Larger gated bf16 FFN, T=8192, D=4096, F=14336, tile 128, swept bias and K."""
    i = SWEEP_BIASES.index(bias) * len(SWEEP_KS) + SWEEP_KS.index(K)
    return Workload(f"c4_bf16_gated_T8192_b{bias}_K{K}", 8192, 4096, 14336, 128, K, BF16,
                    True, bias, 1040 + i)


def config5() -> Workload:
    """Training step of config 2: forward + backward, L1 lambda = 1e-4, dy ~ N(0,1)."""
    return dataclasses.replace(config2(), name="c5_bf16_gated_T4096_train", seed=1005,
                               lam=1e-4, train=True)


def scaled(w: Workload, **kw) -> Workload:
    """Same distributions at other sizes (small parity cases)."""
    return dataclasses.replace(w, **kw)


def generate(w: Workload, rows: Optional[int] = None) -> dict:
    """Draw the arrays of a workload.

    Returns a dict with numpy arrays: x [T][D], Wg [F][D], Wu [F][D] (gated)
    or None, Wd [F][D] (neuron-major down weight), bg [F] fp32, rb [T] fp32
    or None, dy [T][D] (train) or None.  Storage arrays are float32 or
    uint16 bf16 bit patterns.  ``rows`` (optional) keeps only the first rows
    of x / rb / dy after drawing everything (same values as the full draw).
    """
    rng = np.random.default_rng(w.seed)
    T, D, F = w.T, w.D, w.F

    def draw(shape, var):
        a = rng.standard_normal(shape, dtype=np.float32)
        if var != 1.0:
            a *= np.float32(np.sqrt(var))
        return f32_to_bf16_bits(a) if w.dtype == BF16 else a

    x = draw((T, D), 1.0)
    Wg = draw((F, D), 1.0 / D)
    Wu = draw((F, D), 1.0 / D) if w.gated else None
    Wd = draw((F, D), 1.0 / F)
    dy = draw((T, D), 1.0) if w.train else None
    bg = np.full((F,), w.bias, dtype=np.float32)
    rb = None
    if w.hot_tokens:
        rb = np.zeros((T,), dtype=np.float32)
        pos = np.arange(T) % w.seq_len
        rb[pos < w.hot_tokens] = np.float32(w.hot_bias)
    if rows is not None:
        x = np.ascontiguousarray(x[:rows])
        rb = None if rb is None else np.ascontiguousarray(rb[:rows])
        dy = None if dy is None else np.ascontiguousarray(dy[:rows])
    return dict(x=x, Wg=Wg, Wu=Wu, Wd=Wd, bg=bg, rb=rb, dy=dy)


def generate_grid(T: int, D: int, F: int, dtype: str, gated: bool, seed: int,
                  bias_units: int, row_bias_units: Optional[np.ndarray] = None,
                  train: bool = False) -> dict:
    """Integer-grid inputs for bit-exact comparisons.

    x and dy are integers in [-3, 3]; weights are integers in [-3, 3] times
    2^-4; biases are integers times 2^-4.  Every product and every partial sum
    of the gate contraction is a multiple of 2^-4 below 2^20 in magnitude for
    D <= 16384, so any fp32 summation order gives the same exact value, and
    exact zeros (ReLU ties) occur.  All values are exact in bf16.
    """
    rng = np.random.default_rng(seed)
    unit = np.float32(1.0 / 16.0)

    def ints(shape, scale):
        a = rng.integers(-3, 4, size=shape).astype(np.float32) * np.float32(scale)
        return f32_to_bf16_bits(a) if dtype == BF16 else a

    x = ints((T, D), 1.0)
    Wg = ints((F, D), unit)
    Wu = ints((F, D), unit) if gated else None
    Wd = ints((F, D), unit)
    dy = ints((T, D), 1.0) if train else None
    bg = np.full((F,), np.float32(bias_units) * unit, dtype=np.float32)
    rb = None
    if row_bias_units is not None:
        rb = np.asarray(row_bias_units, dtype=np.float32) * unit
    return dict(x=x, Wg=Wg, Wu=Wu, Wd=Wd, bg=bg, rb=rb, dy=dy)
