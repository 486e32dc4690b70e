"""CPU oracle for the block-quantized product -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or executes anything here, and this
package never imports the product: the two share nothing but the seeded input
generators, which hold none of the method's arithmetic.

The arithmetic lives in ``gq_oracle.c`` (plain C, compiled with
``-O2 -ffp-contract=off``); this module compiles it with gcc on first use and
wraps it with numpy arrays.  Formats and citations are documented in the C
file's header.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_0, Q8_0, Q4_K, Q8_K, Q6_K, Q5_K = 0, 1, 2, 3, 4, 5
TYPE_NAMES = {Q4_0: "Q4_0", Q8_0: "Q8_0", Q4_K: "Q4_K", Q8_K: "Q8_K", Q6_K: "Q6_K", Q5_K: "Q5_K"}
ACT_TYPE = {Q4_0: Q8_0, Q8_0: Q8_0, Q4_K: Q8_K, Q6_K: Q8_K, Q5_K: Q8_K}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gq_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-std=c11",
           "-Wall", "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc) if missing or stale."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            L.or_f16_rn.argtypes = [ctypes.c_float]
            L.or_f16_rn.restype = ctypes.c_uint16
            L.or_f16_ru.argtypes = [ctypes.c_float]
            L.or_f16_ru.restype = ctypes.c_uint16
            L.or_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.or_f16_to_f32.restype = ctypes.c_float
            L.or_f16_rn_array.argtypes = [vp, vp, i64]
            L.or_f16_ru_array.argtypes = [vp, vp, i64]
            L.or_block_elems.argtypes = [i32]
            L.or_block_elems.restype = i64
            L.or_block_bytes.argtypes = [i32]
            L.or_block_bytes.restype = i64
            L.or_quantize.argtypes = [i32, vp, vp, i64]
            L.or_quantize.restype = i32
            L.or_quantize_errmin.argtypes = [i32, vp, vp, i64]
            L.or_quantize_errmin.restype = i32
            L.or_dequantize.argtypes = [i32, vp, vp, i64]
            L.or_dequantize.restype = i32
            L.or_dequantize_f64.argtypes = [i32, vp, vp, i64]
            L.or_dequantize_f64.restype = i32
            L.or_block_sums.argtypes = [i32, vp, vp, i64, i64, i64, vp]
            L.or_block_sums.restype = i32
            L.or_matmul_ref.argtypes = [i32, vp, vp, i64, i64, i64, vp, vp, i32]
            L.or_matmul_ref.restype = i32
            L.or_quantize_rows_mt.argtypes = [i32, vp, vp, i64, i64, i32]
            L.or_quantize_rows_mt.restype = i32
            L.or_max_threads.restype = i32
            _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def block_elems(t: int) -> int:
    return int(lib().or_block_elems(t))


def block_bytes(t: int) -> int:
    return int(lib().or_block_bytes(t))


def f16_rn(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().or_f16_rn_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_ru(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().or_f16_ru_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_to_f32(h: int) -> float:
    return float(lib().or_f16_to_f32(h))


def quantize(t: int, x: np.ndarray, errmin: bool = False) -> np.ndarray:
    """Quantize a flat (or row-major 2-D) fp32 array to packed blocks.

    errmin (Q4_K and Q5_K only): the error-minimizing refinement of the
    sub-block scales and mins instead of the plain min/max fit.

    Returns a uint8 array of shape [n / block_elems, block_bytes] for flat
    input, or [rows, cols / block_elems * block_bytes] for 2-D input."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    be, bb = block_elems(t), block_bytes(t)
    n = x.size
    if n % be:
        raise ValueError("element count must be a multiple of the block size")
    out = np.empty(n // be * bb, dtype=np.uint8)
    fn = lib().or_quantize_errmin if errmin else lib().or_quantize
    rc = fn(t, _ptr(x), _ptr(out), n)
    if rc != 0:
        raise ValueError(f"oracle quantize failed ({rc})")
    if x.ndim == 2:
        return out.reshape(x.shape[0], x.shape[1] // be * bb)
    return out.reshape(n // be, bb)


def quantize_rows_mt(t: int, x: np.ndarray, nthreads: int) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, cols = x.shape
    be, bb = block_elems(t), block_bytes(t)
    out = np.empty((rows, cols // be * bb), dtype=np.uint8)
    rc = lib().or_quantize_rows_mt(t, _ptr(x), _ptr(out), rows, cols, nthreads)
    if rc != 0:
        raise ValueError("oracle quantize failed")
    return out


def dequantize(t: int, q: np.ndarray, n: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.empty(n, dtype=np.float32)
    rc = lib().or_dequantize(t, _ptr(q), _ptr(out), n)
    if rc != 0:
        raise ValueError("oracle dequantize failed")
    return out


def dequantize_f64(t: int, q: np.ndarray, n: int) -> np.ndarray:
    """Exact per-element reconstruction in double (no fp32 rounding)."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.empty(n, dtype=np.float64)
    rc = lib().or_dequantize_f64(t, _ptr(q), _ptr(out), n)
    if rc != 0:
        raise ValueError("oracle dequantize failed")
    return out


def block_sums(wtype: int, W: np.ndarray, xq: np.ndarray, rows: int, cols: int,
               batch: int) -> np.ndarray:
    """Integer per-block sums, shape [batch, rows, cols/B] (Q4_0, Q8_0, Q6_K)
    or [batch, rows, cols/256, 2] (Q4_K, Q5_K: S1, S2)."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    nb = cols // block_elems(wtype)
    shape = (batch, rows, nb, 2) if wtype in (Q4_K, Q5_K) else (batch, rows, nb)
    out = np.empty(shape, dtype=np.int32)
    rc = lib().or_block_sums(wtype, _ptr(W), _ptr(xq), rows, cols, batch, _ptr(out))
    if rc != 0:
        raise ValueError("oracle block_sums failed")
    return out


def matmul_ref(wtype: int, W: np.ndarray, xq: np.ndarray, rows: int, cols: int,
               batch: int, nthreads: int = 1):
    """Reference product in double: returns (y, T), each [batch, rows]."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    y = np.empty((batch, rows), dtype=np.float64)
    T = np.empty((batch, rows), dtype=np.float64)
    rc = lib().or_matmul_ref(wtype, _ptr(W), _ptr(xq), rows, cols, batch, _ptr(y), _ptr(T),
                             nthreads)
    if rc != 0:
        raise ValueError("oracle matmul failed")
    return y, T


def max_threads() -> int:
    return int(lib().or_max_threads())


# ------------------------------------------------------------ KV cache
# "llama.cpp 推理引擎" §3.7.3 (KV Cache 量化): the attention keys and values
# are cached as Q8_0 or Q4_0 blocks.  A cache is a uint8 array
# [n_heads, capacity, head_dim / 32 * block_bytes]: row (h, p) holds head h's
# key (or value) at position p.

def kv_append(t: int, x: np.ndarray, cache: np.ndarray, pos: int) -> np.ndarray:
    """Writes x [n_heads, head_dim], each head's row quantized with the block
    encoding of type t (§5.1), into row (h, pos) of every head; returns cache."""
    if t not in (Q8_0, Q4_0):
        raise ValueError("KV cache blocks are Q8_0 or Q4_0")
    for h in range(cache.shape[0]):
        cache[h, pos] = quantize(t, x[h]).reshape(-1)
    return cache


def kv_scores_ref(t: int, cache: np.ndarray, q: np.ndarray, n_pos: int):
    """Scores of the queries q [n_heads, head_dim] against the first n_pos keys
    of each head: the query quantized to Q8_0, then per head the block-dot
    product of §6.4 with the key rows as the weight rows (matmul_ref).
    Returns (scores, T), each [n_heads, n_pos] in double, T the sum of
    |block terms| per output for the tolerance."""
    n_heads = cache.shape[0]
    head_dim = q.shape[1]
    S = np.empty((n_heads, n_pos))
    T = np.empty((n_heads, n_pos))
    for h in range(n_heads):
        qq = quantize(Q8_0, q[h:h + 1])
        y, tt = matmul_ref(t, cache[h, :n_pos], qq, n_pos, head_dim, 1)
        S[h], T[h] = y[0], tt[0]
    return S, T
