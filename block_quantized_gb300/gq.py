"""Thin Python binding of the C ABI in include/gq.h (libgq.so).

Argument marshalling only: every function forwards device pointers and sizes
to the library, where all of the work runs in CUDA kernels.  Functions named
``gq_*`` mirror the C entry points one to one and accept either torch CUDA
tensors or raw integer device pointers; a stream argument of ``None`` means
the current torch stream.  The convenience helpers below them only allocate
outputs with torch and call the same entry points.

There is no fallback: if the library cannot be loaded, or a call returns an
error status, a GQError is raised.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

Q4_0, Q8_0, Q4_K, Q8_K, Q6_K, Q5_K = 0, 1, 2, 3, 4, 5
PATH_AUTO, PATH_GEMV, PATH_MMA, PATH_SKINNY = 0, 1, 2, 3
FLAG_W_STATIC = 1
QUANT_ERRMIN = 1
ACT_TYPE = {Q4_0: Q8_0, Q8_0: Q8_0, Q4_K: Q8_K, Q6_K: Q8_K, Q5_K: Q8_K}
BLOCK_ELEMS = {Q4_0: 32, Q8_0: 32, Q4_K: 256, Q8_K: 256, Q6_K: 256, Q5_K: 256}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q4_K: 144, Q8_K: 276, Q6_K: 194, Q5_K: 176}

STATUS = {0: "GQ_OK", 1: "GQ_ERR_NULL", 2: "GQ_ERR_TYPE", 3: "GQ_ERR_SHAPE",
          4: "GQ_ERR_ALIGN", 5: "GQ_ERR_CUDA", 6: "GQ_ERR_TIMEOUT", 7: "GQ_ERR_ARCH"}

# Every symbol the header declares, with its ctypes signature.
_i64, _i32, _vp, _u32p = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)
SIGNATURES = {
    "gq_block_elems": ([_i32], _i64),
    "gq_block_bytes": ([_i32], _i64),
    "gq_status_string": ([_i32], ctypes.c_char_p),
    "gq_last_cuda_error": ([], _i32),
    "gq_quantize_rows": ([_i32, _vp, _vp, _i64], _i32),
    "gq_quantize_rows_async": ([_i32, _vp, _vp, _i64, _vp], _i32),
    "gq_quantize_rows_ex": ([_i32, _vp, _vp, _i64, ctypes.c_uint, _vp], _i32),
    "gq_dequantize_rows": ([_i32, _vp, _vp, _i64], _i32),
    "gq_dequantize_rows_async": ([_i32, _vp, _vp, _i64, _vp], _i32),
    "gq_matmul": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, _vp], _i32),
    "gq_matmul_path": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp], _i32),
    "gq_matmul_ex": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, _i32, ctypes.c_uint, _vp], _i32),
    "gq_matmul_f32": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, ctypes.c_uint, _vp], _i32),
    "gq_block_sums": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp], _i32),
    "gq_block_sums_f32": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, _vp], _i32),
    "gq_matmul_workspace_bytes": ([_i32, _i64, _i64, _i64], ctypes.c_size_t),
    "gq_matmul_ws": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, _i32, ctypes.c_uint, _vp,
                      ctypes.c_size_t, _vp], _i32),
    "gq_block_sums_ws": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, ctypes.c_size_t,
                          _vp], _i32),
    "gq_matmul_noalloc": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, _vp], _i32),
    "gq_kv_append": ([_i32, _vp, _vp, _i64, _i64, _i64, _i64, _vp], _i32),
    "gq_kv_scores": ([_i32, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _vp], _i32),
    "gq_debug_kv_timeout": ([_i32], _i32),
    "gq_tc_min_batch": ([], _i64),
    "gq_auto_path": ([_i32, _i64, _i64, _i64, _i32, ctypes.POINTER(ctypes.c_int32)], _i32),
    "gq_device_status": ([_u32p, _i32], _i32),
}


class GQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        detail = ""
        if status == 5 and _lib is not None:
            detail = f" (cudaError {_lib.gq_last_cuda_error()})"
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}{detail}")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libgq.so (optionally compiling it first)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and _build.needs_build():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libgq.so not built ({path}); run __graft_entry__.build() first")
            L = ctypes.CDLL(path)
            for name, (args, res) in SIGNATURES.items():
                f = getattr(L, name)
                f.argtypes = args
                f.restype = res
            _lib = L
    return _lib


def _p(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int) -> None:
    if st != 0:
        raise GQError(fn, st)


# ----------------------------------------------------------- 1:1 entry points

def gq_block_elems(t: int) -> int:
    return int(load().gq_block_elems(t))


def gq_block_bytes(t: int) -> int:
    return int(load().gq_block_bytes(t))


def gq_quantize_rows_async(t: int, src, dst, n: int, stream=None) -> None:
    _check("gq_quantize_rows_async",
           load().gq_quantize_rows_async(t, _p(src), _p(dst), n, _s(stream)))


def gq_quantize_rows_ex(t: int, src, dst, n: int, flags: int = 0, stream=None) -> None:
    _check("gq_quantize_rows_ex",
           load().gq_quantize_rows_ex(t, _p(src), _p(dst), n, flags, _s(stream)))


def gq_quantize_rows(t: int, src, dst, n: int) -> None:
    _check("gq_quantize_rows", load().gq_quantize_rows(t, _p(src), _p(dst), n))


def gq_dequantize_rows_async(t: int, src, dst, n: int, stream=None) -> None:
    _check("gq_dequantize_rows_async",
           load().gq_dequantize_rows_async(t, _p(src), _p(dst), n, _s(stream)))


def gq_dequantize_rows(t: int, src, dst, n: int) -> None:
    _check("gq_dequantize_rows", load().gq_dequantize_rows(t, _p(src), _p(dst), n))


def gq_matmul(wtype: int, W, xq, y, rows: int, cols: int, batch: int, stream=None) -> None:
    _check("gq_matmul", load().gq_matmul(wtype, _p(W), _p(xq), _p(y), rows, cols, batch,
                                         _s(stream)))


def gq_matmul_path(wtype: int, W, xq, y, rows: int, cols: int, batch: int, path: int,
                   stream=None) -> None:
    _check("gq_matmul_path", load().gq_matmul_path(wtype, _p(W), _p(xq), _p(y), rows, cols,
                                                   batch, path, _s(stream)))


def gq_matmul_ex(wtype: int, W, xq, y, rows: int, cols: int, batch: int, path: int = PATH_AUTO,
                 flags: int = 0, stream=None) -> None:
    _check("gq_matmul_ex", load().gq_matmul_ex(wtype, _p(W), _p(xq), _p(y), rows, cols, batch,
                                               path, flags, _s(stream)))


def gq_matmul_f32(wtype: int, W, x, y, rows: int, cols: int, batch: int, flags: int = 0,
                  stream=None) -> None:
    _check("gq_matmul_f32", load().gq_matmul_f32(wtype, _p(W), _p(x), _p(y), rows, cols, batch,
                                                 flags, _s(stream)))


def gq_block_sums_f32(wtype: int, W, x, sums, rows: int, cols: int, batch: int,
                      stream=None) -> None:
    _check("gq_block_sums_f32", load().gq_block_sums_f32(wtype, _p(W), _p(x), _p(sums), rows, cols,
                                                         batch, _s(stream)))


def gq_block_sums(wtype: int, W, xq, sums, rows: int, cols: int, batch: int, path: int,
                  stream=None) -> None:
    _check("gq_block_sums", load().gq_block_sums(wtype, _p(W), _p(xq), _p(sums), rows, cols,
                                                 batch, path, _s(stream)))


def gq_matmul_workspace_bytes(wtype: int, rows: int, cols: int, batch: int) -> int:
    return int(load().gq_matmul_workspace_bytes(wtype, rows, cols, batch))


def gq_matmul_ws(wtype: int, W, xq, y, rows: int, cols: int, batch: int, path: int, flags: int,
                 workspace, workspace_bytes: int, stream=None) -> None:
    _check("gq_matmul_ws", load().gq_matmul_ws(wtype, _p(W), _p(xq), _p(y), rows, cols, batch, path,
                                               flags, _p(workspace), workspace_bytes, _s(stream)))


def gq_block_sums_ws(wtype: int, W, xq, sums, rows: int, cols: int, batch: int, path: int,
                     workspace, workspace_bytes: int, stream=None) -> None:
    _check("gq_block_sums_ws", load().gq_block_sums_ws(wtype, _p(W), _p(xq), _p(sums), rows, cols,
                                                       batch, path, _p(workspace), workspace_bytes,
                                                       _s(stream)))


def gq_matmul_noalloc(wtype: int, W, xq, y, rows: int, cols: int, batch: int,
                      stream=None) -> None:
    """Tensor-core product using the library's static scratch (no allocation
    anywhere); see gq.h for the size limit and the sharing rules."""
    _check("gq_matmul_noalloc", load().gq_matmul_noalloc(wtype, _p(W), _p(xq), _p(y), rows, cols,
                                                         batch, _s(stream)))


def gq_kv_append(t: int, x, cache, n_heads: int, head_dim: int, capacity: int, pos: int,
                 stream=None) -> None:
    _check("gq_kv_append", load().gq_kv_append(t, _p(x), _p(cache), n_heads, head_dim, capacity, pos,
                                               _s(stream)))


def gq_kv_scores(t: int, cache, q, scores, n_heads: int, head_dim: int, capacity: int, n_pos: int,
                 stream=None) -> None:
    _check("gq_kv_scores", load().gq_kv_scores(t, _p(cache), _p(q), _p(scores), n_heads, head_dim, capacity,
                                               n_pos, _s(stream)))


def gq_debug_kv_timeout(on: bool) -> None:
    """Test switch: make gq_kv_scores' bounded waits run out (see gq.h)."""
    _check("gq_debug_kv_timeout", load().gq_debug_kv_timeout(1 if on else 0))


def gq_tc_min_batch() -> int:
    return int(load().gq_tc_min_batch())


def gq_auto_path(wtype: int, rows: int, cols: int, batch: int, with_workspace: bool = False) -> int:
    """The family (PATH_GEMV, PATH_MMA or PATH_SKINNY) GQ_PATH_AUTO takes;
    host only."""
    out = ctypes.c_int32(-1)
    _check("gq_auto_path", load().gq_auto_path(wtype, rows, cols, batch, 1 if with_workspace else 0,
                                                ctypes.byref(out)))
    return int(out.value)


def gq_device_status(reset: bool = True) -> int:
    """Returns the device status word (0 = no bounded wait ran out)."""
    w = ctypes.c_uint32(0)
    st = load().gq_device_status(ctypes.byref(w), 1 if reset else 0)
    if st not in (0, 6):
        raise GQError("gq_device_status", st)
    return int(w.value)


# ------------------------------------------------------ convenience (torch)

def packed_bytes(t: int, n: int) -> int:
    return n // BLOCK_ELEMS[t] * BLOCK_BYTES[t]


def quantize(t: int, x, stream=None, flags: int = 0):
    """Quantize a CUDA fp32 tensor [..., cols] into a uint8 tensor
    [..., cols / block_elems * block_bytes] (flags: QUANT_ERRMIN for the
    error-minimizing Q4_K / Q5_K encoder)."""
    import torch
    assert x.is_cuda and x.dtype == torch.float32 and x.is_contiguous()
    cols = x.shape[-1]
    out = torch.empty(*x.shape[:-1], cols // BLOCK_ELEMS[t] * BLOCK_BYTES[t],
                      dtype=torch.uint8, device=x.device)
    gq_quantize_rows_ex(t, x, out, x.numel(), flags, stream)
    return out


def dequantize(t: int, q, n: int, stream=None):
    import torch
    out = torch.empty(n, dtype=torch.float32, device=q.device)
    gq_dequantize_rows_async(t, q, out, n, stream)
    return out


def matmul(wtype: int, W, xq, rows: int, cols: int, batch: int, path: int = PATH_AUTO,
           out=None, stream=None):
    import torch
    y = out if out is not None else torch.empty(batch, rows, dtype=torch.float32, device=W.device)
    gq_matmul_path(wtype, W, xq, y, rows, cols, batch, path, stream)
    return y


def matmul_f32(wtype: int, W, x, rows: int, cols: int, batch: int, flags: int = 0, out=None,
               stream=None):
    """Fused activation quantize + product from fp32 activations [batch, cols]."""
    import torch
    y = out if out is not None else torch.empty(batch, rows, dtype=torch.float32, device=W.device)
    gq_matmul_f32(wtype, W, x, y, rows, cols, batch, flags, stream)
    return y


def _sums_buffer(wtype, W, rows, cols, batch):
    import torch
    nb = cols // BLOCK_ELEMS[wtype]
    shape = (batch, rows, nb, 2) if wtype in (Q4_K, Q5_K) else (batch, rows, nb)
    return torch.empty(shape, dtype=torch.int32, device=W.device)


def workspace(wtype: int, rows: int, cols: int, batch: int, device=None):
    """A torch uint8 device buffer sized for the tensor-core path (or None)."""
    import torch
    n = gq_matmul_workspace_bytes(wtype, rows, cols, batch)
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda") if n else None


def matmul_ws(wtype: int, W, xq, rows: int, cols: int, batch: int, path: int = PATH_AUTO,
              flags: int = 0, ws=None, out=None, stream=None):
    import torch
    y = out if out is not None else torch.empty(batch, rows, dtype=torch.float32, device=W.device)
    if ws is None:
        ws = workspace(wtype, rows, cols, batch, W.device)
    gq_matmul_ws(wtype, W, xq, y, rows, cols, batch, path, flags, ws,
                 0 if ws is None else ws.numel(), stream)
    return y


def block_sums(wtype: int, W, xq, rows: int, cols: int, batch: int, path: int = PATH_GEMV,
               stream=None):
    s = _sums_buffer(wtype, W, rows, cols, batch)
    if path == PATH_MMA:
        ws = workspace(wtype, rows, cols, batch, W.device)
        gq_block_sums_ws(wtype, W, xq, s, rows, cols, batch, path, ws,
                         0 if ws is None else ws.numel(), stream)
    else:
        gq_block_sums(wtype, W, xq, s, rows, cols, batch, path, stream)
    return s


def block_sums_f32(wtype: int, W, x, rows: int, cols: int, batch: int, stream=None):
    s = _sums_buffer(wtype, W, rows, cols, batch)
    gq_block_sums_f32(wtype, W, x, s, rows, cols, batch, stream)
    return s


def kv_cache(t: int, n_heads: int, capacity: int, head_dim: int, device=None):
    """A zeroed uint8 device tensor [n_heads, capacity, head_dim / 32 * block_bytes]
    laid out as gq_kv_append / gq_kv_scores expect."""
    import torch
    return torch.zeros(n_heads, capacity, head_dim // BLOCK_ELEMS[t] * BLOCK_BYTES[t], dtype=torch.uint8,
                       device=device or "cuda")


def kv_scores(t: int, cache, q, n_pos: int, stream=None):
    """Scores [n_heads, n_pos] of fp32 queries q [n_heads, head_dim] against the
    first n_pos cached keys of each head."""
    import torch
    n_heads, capacity = cache.shape[0], cache.shape[1]
    head_dim = q.shape[-1]
    out = torch.empty(n_heads, n_pos, dtype=torch.float32, device=q.device)
    gq_kv_scores(t, cache, q, out, n_heads, head_dim, capacity, n_pos, stream)
    return out
