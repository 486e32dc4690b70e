"""Seeded synthetic inputs for the block-quantized product.

This module only draws random fp32 arrays; it holds none of the method's
arithmetic (no scales, codes or dot products), so both the CUDA path and the
CPU oracle may take their inputs from it.

Generator: numpy ``Generator(PCG64(seed))``, values drawn as fp32 in the order
each function lists.  The workloads mirror the shapes the pages discuss for
llama.cpp decode and prefill (7B / 8B / 70B transformer weight matrices);
no trained weights exist here, so every matrix is random with the stated
distribution.
"""
from __future__ import annotations

import numpy as np


def rng(seed: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    x = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def gemv_q4_0(seed: int = 0, rows: int = 512, cols: int = 1024):
    """Small Q4_0 x Q8_0 GEMV workload: W ~ N(0, 0.02^2) [rows, cols], then
    x ~ N(0, 1) [cols]."""
    g = rng(seed)
    W = normal(g, (rows, cols), 0.02)
    x = normal(g, (cols,))
    return W, x


def outlier_weights(g: np.random.Generator, rows: int, cols: int,
                    frac: float = 0.001, sigma: float = 0.02) -> np.ndarray:
    """Weights with per-row std sigma * exp(U(ln 0.5, ln 2)) (log-uniform in
    [0.5, 2] x sigma) and a fraction `frac` of all entries, chosen uniformly
    without replacement, replaced by +-10 row-sigma with a random sign.
    Draw order: row scales, the normal matrix, outlier positions, signs."""
    s = sigma * np.exp(g.uniform(np.log(0.5), np.log(2.0), size=rows)).astype(np.float32)
    W = normal(g, (rows, cols))
    W *= s[:, None]
    n_out = int(frac * rows * cols)
    if n_out:
        idx = g.choice(rows * cols, size=n_out, replace=False)
        sign = np.where(g.integers(0, 2, size=n_out) == 0, -1.0, 1.0).astype(np.float32)
        r = idx // cols
        W.reshape(-1)[idx] = sign * np.float32(10.0) * s[r]
    return W


def gemv_q4_k(seed: int = 0, rows: int = 4096, cols: int = 4096):
    """Q4_K x Q8_K GEMV workload with row-scale spread and 0.1% outliers,
    then x ~ N(0, 1) [cols]."""
    g = rng(seed)
    W = outlier_weights(g, rows, cols)
    x = normal(g, (cols,))
    return W, x


# 7B-shape decode: per layer four 4096x4096 attention projections, the
# 11008x4096 gate/up projections and the 4096x11008 down projection (Q4_K),
# then a 32000x4096 output head (Q8_0).
DECODE_LAYER = (("wq", 4096, 4096), ("wk", 4096, 4096), ("wv", 4096, 4096),
                ("wo", 4096, 4096), ("w1", 11008, 4096), ("w3", 11008, 4096),
                ("w2", 4096, 11008))
DECODE_HEAD = ("head", 32000, 4096)
DECODE_LAYERS = 32


def decode_weights(seed: int = 0, scale: int = 1):
    """One layer's weights plus the head, all ~N(0, 0.02^2), drawn in the
    order of DECODE_LAYER then DECODE_HEAD.  `scale` divides every row count
    (for small test versions of the same structure)."""
    g = rng(seed)
    out = {}
    for name, r, c in DECODE_LAYER + (DECODE_HEAD,):
        out[name] = normal(g, (max(1, r // scale), c), 0.02)
    x = normal(g, (4096,))
    return out, x


def batch_columns(g: np.random.Generator, batch: int, cols: int) -> np.ndarray:
    """`batch` activation vectors of N(0, 1), stored as [batch, cols]."""
    return normal(g, (batch, cols))


def gemm_q4_k(seed: int = 0, rows: int = 14336, cols: int = 4096, batch: int = 64):
    """W ~ N(0, 0.02^2) [rows, cols], then X ~ N(0, 1) [batch, cols]."""
    g = rng(seed)
    W = normal(g, (rows, cols), 0.02)
    X = batch_columns(g, batch, cols)
    return W, X
