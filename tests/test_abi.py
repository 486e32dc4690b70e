"""Host-side tests of the C ABI (no GPU needed): the library builds and loads,
exports every entry point include/gq.h declares, and rejects invalid
arguments on the host with the documented status codes before touching CUDA.
"""
import ctypes
import os
import re

import pytest

from block_quantized_gb300 import build as gqbuild
from block_quantized_gb300 import gq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, NULL, TYPE, SHAPE, ALIGN, CUDA = 0, 1, 2, 3, 4, 5


@pytest.fixture(scope="module")
def lib():
    gqbuild.build()
    return gq.load()


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "gq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gq_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(gq.SIGNATURES), "binding and header disagree"


def test_block_geometry(lib):
    assert [gq.gq_block_elems(t) for t in range(6)] == [32, 32, 256, 256, 256, 256]
    assert [gq.gq_block_bytes(t) for t in range(6)] == [18, 34, 144, 276, 194, 176]
    assert gq.gq_block_elems(9) == -1 and gq.gq_block_bytes(-1) == -1


def test_status_strings(lib):
    for s in range(8):
        assert lib.gq_status_string(s)
    assert lib.gq_status_string(123) == b"unknown status"


# Fake, never-dereferenced device addresses: validation happens on the host
# and returns before any CUDA call.
A16 = 0x10000
MIS = 0x10002


def test_matmul_validation(lib):
    f = lib.gq_matmul
    assert f(3, A16, A16, A16, 8, 256, 1, None) == TYPE          # Q8_K is not a weight type
    assert f(7, A16, A16, A16, 8, 256, 1, None) == TYPE
    assert f(2, A16, A16, A16, 8, 100, 1, None) == SHAPE         # not a block multiple
    assert f(0, A16, A16, A16, 8, 48, 1, None) == SHAPE
    assert f(2, A16, A16, A16, -1, 256, 1, None) == SHAPE
    assert f(2, A16, A16, A16, 8, 256, -3, None) == SHAPE
    assert f(2, A16, A16, A16, 1 << 40, 256, 1, None) == SHAPE   # size overflow
    assert f(2, A16, A16, A16, 8, 1 << 30, 1, None) == SHAPE     # cols above the maximum
    assert f(2, 0, A16, A16, 8, 256, 1, None) == NULL
    assert f(2, A16, 0, A16, 8, 256, 1, None) == NULL
    assert f(2, A16, A16, 0, 8, 256, 1, None) == NULL
    assert f(2, MIS, A16, A16, 8, 256, 1, None) == ALIGN
    assert f(2, A16, MIS, A16, 8, 256, 1, None) == ALIGN
    assert f(2, A16, A16, A16 + 1, 8, 256, 1, None) == ALIGN
    # zero sizes are a no-op, even with NULL pointers
    assert f(2, 0, 0, 0, 0, 256, 1, None) == OK
    assert f(2, 0, 0, 0, 8, 256, 0, None) == OK
    # path and pairing rules
    g = lib.gq_matmul_path
    assert g(2, A16, A16, A16, 8, 256, 1, 9, None) == TYPE
    # tensor-core Q4_0 / Q8_0: cols a multiple of 256, no workspace (accepted,
    # then no device here)
    assert g(0, A16, A16, A16, 8, 288, 64, 2, None) == SHAPE
    assert g(1, A16, A16, A16, 8, 96, 64, 2, None) == SHAPE
    assert g(0, A16, A16, A16, 8, 256, 64, 2, None) == CUDA
    assert g(1, A16, A16, A16, 8, 512, 64, 2, None) == CUDA
    assert g(4, A16, A16, A16, 8, 256, 64, 2, None) == TYPE
    assert f(4, A16, A16, A16, 8, 32, 1, None) == SHAPE          # Q6_K needs 256-multiples
    assert f(4, 0, 0, 0, 8, 256, 0, None) == OK
    assert g(5, A16, A16, A16, 8, 256, 64, 2, None) == TYPE      # no tensor-core Q5_K kernel
    # the warp-level tensor-core path: Q4_K, Q5_K, Q4_0 and Q8_0, cols a
    # multiple of 256 (larger batches run as 64- or 32-column chunks)
    assert g(4, A16, A16, A16, 8, 256, 8, 3, None) == TYPE
    assert g(5, A16, A16, A16, 8, 256, 40, 3, None) == CUDA
    assert g(0, A16, A16, A16, 8, 288, 8, 3, None) == SHAPE
    assert g(1, A16, A16, A16, 8, 256, 8, 3, None) == CUDA
    assert g(2, A16, A16, A16, 8, 256, 65, 3, None) == CUDA
    assert g(2, A16, A16, A16, 8, 256, 64, 3, None) == CUDA
    assert f(5, A16, A16, A16, 8, 32, 1, None) == SHAPE          # Q5_K needs 256-multiples
    assert f(6, A16, A16, A16, 8, 256, 1, None) == TYPE
    assert lib.gq_block_sums(2, A16, A16, 0, 8, 256, 1, 1, None) == NULL


def test_codec_validation(lib):
    q = lib.gq_quantize_rows
    assert q(6, A16, A16, 32) == TYPE
    assert q(5, A16, A16, 32) == SHAPE                          # Q5_K needs 256-multiples
    assert q(5, A16, A16 + 2, 256) == ALIGN                     # Q5_K dst 4-aligned
    assert q(0, A16, A16, 33) == SHAPE
    assert q(2, A16, A16, 32) == SHAPE                          # Q4_K needs 256-multiples
    assert q(1, A16, A16, -32) == SHAPE
    assert q(1, 0, A16, 32) == NULL
    assert q(1, A16, 0, 32) == NULL
    assert q(1, A16 + 2, A16, 32) == ALIGN                      # src must be 4-aligned
    assert q(3, A16, A16 + 2, 256) == ALIGN                     # Q8_K dst 4-aligned
    assert q(1, A16, A16 + 1, 32) == ALIGN                      # Q8_0 dst 2-aligned
    assert q(4, A16, A16 + 1, 256) == ALIGN                     # Q6_K dst 2-aligned
    assert q(4, A16, A16, 32) == SHAPE
    assert q(1, 0, 0, 0) == OK
    e = lib.gq_quantize_rows_ex
    assert e(2, A16, A16, 256, 2, None) == TYPE                  # unknown flag bit
    assert e(1, A16, A16, 32, 1, None) == TYPE                   # error-minimizing: K-quants only
    assert e(4, A16, A16, 256, 1, None) == TYPE
    assert e(2, A16, A16, 32, 1, None) == SHAPE
    assert e(5, A16, A16 + 2, 256, 1, None) == ALIGN
    assert e(2, 0, 0, 0, 1, None) == OK
    assert e(0, A16, A16, 33, 0, None) == SHAPE                  # flags 0: the default encoder's rules
    d = lib.gq_dequantize_rows
    assert d(0, A16, A16, 31) == SHAPE
    assert d(2, A16 + 2, A16, 256) == ALIGN
    assert d(0, 0, 0, 0) == OK


def test_valid_call_without_gpu_fails_loudly(lib):
    """With arguments that pass validation, the library needs a CUDA device;
    without one it reports GQ_ERR_CUDA (never a silent CPU result)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert lib.gq_matmul(2, A16, A16, A16, 8, 256, 1, None) == CUDA
    assert lib.gq_debug_kv_timeout(1) == CUDA
    assert lib.gq_last_cuda_error() != 0
    with pytest.raises(gq.GQError):
        gq.gq_matmul(2, A16, A16, A16, 8, 256, 1, stream=0)


def test_fused_and_flag_validation(lib):
    f = lib.gq_matmul_f32
    assert f(2, A16, A16 + 4, A16, 8, 256, 1, 0, None) == ALIGN     # x must be 16-aligned
    assert f(0, A16, A16, A16, 8, 96, 1, 0, None) == SHAPE          # fused needs cols % 256 == 0
    assert f(2, A16, A16, A16, 8, 256, 1, 2, None) == TYPE          # unknown flag bit
    assert f(3, A16, A16, A16, 8, 256, 1, 0, None) == TYPE
    # Q5_K / Q6_K fuse only into the streaming kernel: the vector must fit its
    # shared memory (Q6_K also wants whole 16-byte rows, cols % 2048 == 0)
    assert f(5, A16, A16, A16, 8, 19200, 1, 0, None) == SHAPE
    assert f(4, A16, A16, A16, 8, 18432, 1, 0, None) == SHAPE
    assert f(4, A16, A16, A16, 8, 2304, 1, 0, None) == SHAPE
    assert lib.gq_block_sums_f32(4, A16, A16, A16, 8, 768, 1, None) == SHAPE
    assert f(2, 0, 0, 0, 0, 256, 1, 0, None) == OK
    e = lib.gq_matmul_ex
    assert e(2, A16, A16, A16, 8, 256, 1, 1, 4, None) == TYPE
    assert e(2, A16, A16, MIS + 1, 8, 256, 1, 1, 1, None) == ALIGN
    assert lib.gq_block_sums_f32(2, A16, A16, 0, 8, 256, 1, None) == NULL


def test_workspace_rules_on_host(lib):
    wb = lib.gq_matmul_workspace_bytes
    # tiles of 32 columns up to batch 32, 64 up to 64, then 128; one unit per
    # (column tile, super-block) of 4 * tn * 128 + tn * 40 bytes
    assert wb(2, 14336, 4096, 8) == 1 * 16 * 17664
    assert wb(2, 14336, 4096, 32) == 1 * 16 * 17664
    assert wb(2, 14336, 4096, 33) == 1 * 16 * 35328
    assert wb(2, 14336, 4096, 64) == 1 * 16 * 35328
    assert wb(2, 14336, 4096, 65) == 1 * 16 * 70656
    assert wb(2, 14336, 4096, 129) == 2 * 16 * 70656
    assert wb(2, 28672, 8192, 512) == 4 * 32 * 70656
    assert wb(0, 128, 256, 64) == 0 and wb(2, 128, 100, 64) == 0 and wb(2, 0, 256, 64) == 0
    m = lib.gq_matmul_ws
    need = wb(2, 128, 256, 64)
    # no workspace: the tensor-core kernel packs the activations itself (so
    # on a machine without a GPU the call gets as far as the device query)
    assert m(2, A16, A16, A16, 128, 256, 64, 2, 0, 0, need, None) == CUDA
    assert m(2, A16, A16, A16, 128, 256, 64, 2, 0, A16, need - 1, None) == SHAPE
    assert m(2, A16, A16, A16, 128, 256, 64, 2, 0, A16 + 8, need, None) == ALIGN
    assert m(4, A16, A16, A16, 128, 256, 64, 2, 0, A16, need, None) == TYPE  # no tensor-core Q6_K kernel
    assert m(0, A16, A16, A16, 128, 256, 64, 2, 0, 0, 0, None) == CUDA      # Q4_0 needs no workspace
    assert lib.gq_matmul_path(2, A16, A16, A16, 128, 256, 64, 2, None) == CUDA


def test_kv_validation(lib):
    ap, sc = lib.gq_kv_append, lib.gq_kv_scores
    A16 = 1 << 20
    # append(type, x, cache, n_heads, head_dim, capacity, pos, stream)
    assert ap(2, A16, A16, 4, 128, 64, 0, None) == TYPE          # Q4_K cache
    assert ap(3, A16, A16, 4, 128, 64, 0, None) == TYPE
    assert ap(1, A16, A16, 4, 48, 64, 0, None) == SHAPE          # head_dim not a multiple of 32
    assert ap(1, A16, A16, 4, 288, 64, 0, None) == SHAPE         # head_dim > 256
    assert ap(1, A16, A16, 4, 128, 48, 0, None) == SHAPE         # capacity not a multiple of 32
    assert ap(1, A16, A16, 4, 128, 64, 64, None) == SHAPE        # pos past the capacity
    assert ap(1, A16, A16, 4, 128, 64, -1, None) == SHAPE
    assert ap(1, A16, A16, -1, 128, 64, 0, None) == SHAPE
    assert ap(1, A16, 0, 4, 128, 64, 0, None) == NULL
    assert ap(1, 0, A16, 4, 128, 64, 0, None) == NULL
    assert ap(1, A16, A16 + 8, 4, 128, 64, 0, None) == ALIGN     # cache 16-byte aligned
    assert ap(1, A16 + 2, A16, 4, 128, 64, 0, None) == ALIGN     # x 4-byte aligned
    assert ap(1, A16, A16, 0, 128, 64, 0, None) == OK            # no heads: nothing to do
    # scores(type, cache, q, scores, n_heads, head_dim, capacity, n_pos, stream)
    assert sc(2, A16, A16, A16, 4, 128, 64, 10, None) == TYPE
    assert sc(0, A16, A16, A16, 4, 128, 64, 65, None) == SHAPE   # n_pos past the capacity
    assert sc(0, A16, A16, A16, 4, 128, 50, 10, None) == SHAPE
    assert sc(0, A16, 0, A16, 4, 128, 64, 10, None) == NULL
    assert sc(0, A16, A16, 0, 4, 128, 64, 10, None) == NULL
    assert sc(0, A16 + 4, A16, A16, 4, 128, 64, 10, None) == ALIGN
    assert sc(0, A16, A16, A16 + 2, 4, 128, 64, 10, None) == ALIGN
    assert sc(0, A16, A16, A16, 4, 128, 64, 0, None) == OK       # no positions


# The dispatch table of GQ_PATH_AUTO, pinned on the host (gq_auto_path does
# no device call): weight type, rows, batch, workspace given -> family.  The
# thresholds are the crossovers measured on 14336 x 4096 and 4096 x 4096;
# the GPU tests check that gq_matmul's results equal the named family's.
GEMV, MMA, SKINNY = 1, 2, 3
AUTO_TABLE = [
    # Q4_K: warp-level kernel 4..32 (>= 8192 rows) or 16..32 (>= 2048 rows),
    # tcgen05 beyond (with or without a workspace), with a workspace also
    # from 9 (>= 14336 rows) or 16 on smaller matrices, GEMV otherwise
    (2, 14336, 3, False, GEMV), (2, 14336, 4, False, SKINNY), (2, 14336, 32, True, SKINNY),
    (2, 14336, 33, False, MMA), (2, 14336, 33, True, MMA), (2, 14336, 512, False, MMA),
    (2, 14336, 9, True, SKINNY), (2, 4096, 15, False, GEMV), (2, 4096, 16, False, SKINNY),
    (2, 4096, 33, False, MMA), (2, 4096, 9, True, GEMV), (2, 1024, 16, True, MMA), (2, 1024, 16, False, GEMV),
    (2, 1024, 64, False, GEMV),
    # Q4_0 / Q8_0: warp-level kernel 2..64 (>= 8192 rows) or 8..64 (>= 2048),
    # tcgen05 from 16 otherwise; the workspace changes nothing
    (0, 8192, 1, False, GEMV), (0, 8192, 2, False, SKINNY), (1, 14336, 64, True, SKINNY),
    (1, 14336, 65, False, MMA), (0, 4096, 7, False, GEMV), (0, 4096, 8, False, SKINNY),
    (1, 1024, 15, False, GEMV), (1, 1024, 16, False, MMA),
    # Q5_K: warp-level kernel from 4 (>= 8192 rows) or 16 (>= 2048), GEMV
    # otherwise; Q6_K: always the GEMV
    (5, 14336, 3, False, GEMV), (5, 14336, 4, False, SKINNY), (5, 8192, 200, True, SKINNY),
    (5, 4096, 15, False, GEMV), (5, 4096, 16, False, SKINNY), (5, 1024, 64, False, GEMV),
    (4, 14336, 64, True, GEMV),
]


@pytest.mark.skipif(bool(os.environ.get("GQ_TC_MIN_BATCH")), reason="threshold overridden")
@pytest.mark.parametrize("wtype,rows,batch,ws,want", AUTO_TABLE)
def test_auto_path_rules(lib, wtype, rows, batch, ws, want):
    assert gq.gq_auto_path(wtype, rows, 4096, batch, ws) == want


def test_auto_path_validation(lib):
    out = ctypes.c_int32(-1)
    f = lib.gq_auto_path
    assert f(3, 8, 256, 1, 0, ctypes.byref(out)) == TYPE       # Q8_K is not a weight type
    assert f(2, 8, 100, 1, 0, ctypes.byref(out)) == SHAPE      # not a block multiple
    assert f(2, -1, 256, 1, 0, ctypes.byref(out)) == SHAPE
    assert f(2, 8, 256, 1, 0, None) == NULL
    assert f(2, 0, 256, 1, 0, ctypes.byref(out)) == OK and out.value == GEMV
    # cols % 256 != 0 keeps Q4_0 on the GEMV at any batch
    assert f(0, 14336, 288, 32, 0, ctypes.byref(out)) == OK and out.value == GEMV


def test_build_lists_every_source():
    """Every kernel source and header under csrc is compiled or tracked by the
    build (a header missing from the list would leave a stale library after
    an edit)."""
    files = set(os.listdir(gqbuild.CSRC))
    assert {f for f in files if f.endswith(".cu")} == set(gqbuild.SOURCES)
    assert {f for f in files if f.endswith((".cuh", ".h"))} == set(gqbuild.HEADERS)
