"""GPU parity of the tcgen05 tensor-core path (Q4_K x Q8_K, batched) against
the CPU oracle: integer super-block sums S1 / S2 bit-identical, y within
1e-4 * sum|terms|, and the same y as the GEMV path within that tolerance."""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as orc  # noqa: E402
from block_quantized_gb300 import gq, inputs  # noqa: E402

pytestmark = pytest.mark.gpu

Q4_K, Q8_K = 2, 3
TOL = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    gq.load(build_if_missing=True)
    yield
    torch.cuda.synchronize()
    assert gq.gq_device_status(reset=True) == 0


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    torch.cuda.synchronize()
    return t.cpu().numpy()


def assert_close(y, y_ref, T):
    err = np.abs(y.astype(np.float64) - y_ref)
    bad = err > TOL * T
    assert not bad.any(), (
        f"{bad.sum()} outputs out of tolerance; worst ratio {np.max(err / np.maximum(T, 1e-300)):.3g}")


# tile widths 32 (batch <= 32), 64 (<= 64) and 128; ragged row tiles and
# column tiles; K loops longer than the activation and weight rings
SHAPES = [(128, 256, 128), (128, 512, 16), (200, 768, 40), (256, 1024, 130), (77, 256, 1),
          (384, 4096, 64), (130, 2048, 32), (300, 1280, 33), (64, 512, 65), (513, 4096, 7),
          (257, 3072, 50)]


@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_mma_sums_and_y(rows, cols, batch):
    g = inputs.rng(rows + cols + batch)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q4_K, W), orc.quantize(Q8_K, X)
    Wd, Xd = dev(Wq), dev(Xq)
    s = host(gq.block_sums(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    np.testing.assert_array_equal(s, orc.block_sums(Q4_K, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul_ws(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)
    # and the GEMV path agrees within the same bound
    y_g = host(gq.matmul(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_GEMV))
    assert_close(y_g, y_ref, T)


def test_mma_auto_dispatch_and_workspace_rules():
    rows, cols, batch = 256, 512, 48
    g = inputs.rng(5)
    Wq = orc.quantize(Q4_K, inputs.normal(g, (rows, cols), 0.02))
    Xq = orc.quantize(Q8_K, inputs.normal(g, (batch, cols)))
    need = gq.gq_matmul_workspace_bytes(Q4_K, rows, cols, batch)
    assert need == 1 * 2 * 35328  # one 64-column tile
    assert gq.gq_matmul_workspace_bytes(0, rows, cols, batch) == 0
    y = torch.empty(batch, rows, device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(gq.GQError):  # workspace too small
        gq.gq_matmul_ws(Q4_K, dev(Wq), dev(Xq), y, rows, cols, batch, gq.PATH_MMA, 0, ws, need - 16)
    gq.gq_matmul_ws(Q4_K, dev(Wq), dev(Xq), y, rows, cols, batch, gq.PATH_AUTO, 0, ws, need)
    y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch)
    assert_close(host(y), y_ref, T)


def test_mma_degenerate_blocks():
    """Zero weights / activations, constant and all-negative rows."""
    rows, cols, batch = 130, 512, 20
    W = np.zeros((rows, cols), np.float32)
    W[1] = 1.0
    W[2] = -3.0
    W[3, ::2] = 7.0
    W[4] = np.linspace(-1, 1, cols, dtype=np.float32)
    W[5:] = inputs.normal(inputs.rng(3), (rows - 5, cols), 0.02)
    X = inputs.normal(inputs.rng(4), (batch, cols))
    X[0] = 0.0
    X[1] = 1000.0  # large activation scale: the min-term split keeps fp32 range
    Wq, Xq = orc.quantize(Q4_K, W), orc.quantize(Q8_K, X)
    s = host(gq.block_sums(Q4_K, dev(Wq), dev(Xq), rows, cols, batch, gq.PATH_MMA))
    np.testing.assert_array_equal(s, orc.block_sums(Q4_K, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul_ws(Q4_K, dev(Wq), dev(Xq), rows, cols, batch, gq.PATH_MMA))
    y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch)
    assert np.all(y[0] == 0)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("batch", [5, 40, 100])  # tile widths 32, 64 and 128
def test_mma_sums_beyond_fp32_integers(batch):
    """Super-block sums S1 = sum_j sc_j * s_j reach 63 * 15 * 127 * 256 =
    30,723,840, beyond 2^24, where fp32 holds only even integers: constant
    rows (every sc = 63, every code 15) with one or several codes lowered to
    14, against constant activations (every code +-127), give odd S1 near
    3.07e7.  The tensor-core sums must still equal the oracle's bit for bit
    ("llama.cpp 推理引擎" §5.5: the two-level dequantization whose integer
    sums are exact)."""
    rows, cols = 131, 512
    W = inputs.outlier_weights(inputs.rng(7), rows, cols, frac=0.001)
    W[0] = 1.0
    W[0, 5] = 0.93                                  # one code 14 among 15s
    W[1] = 1.0                                      # every code 15
    W[2] = 1.0
    W[2, 1::2] = 0.93                               # alternating 15 / 14
    W[3] = 1.0
    W[3, 300] = 0.0                                 # one zero, second super-block
    W[4] = np.where(np.arange(cols) % 3 == 0, 1.0, 0.55)
    W[130] = 1.0                                    # last row of a ragged tile
    W[130, 255] = 0.93
    X = inputs.normal(inputs.rng(8), (batch, cols))
    X[0] = 1.0                                      # every code +127
    X[1] = -1.0                                     # every code -127
    X[2] = 1.0
    X[2, 7] = 0.99
    X[3] = 1.0
    X[3, ::5] = -1.0
    X[batch - 1] = 1.0                              # last column of the tile
    Wq, Xq = orc.quantize(Q4_K, W), orc.quantize(Q8_K, X)
    s_ref = orc.block_sums(Q4_K, Wq, Xq, rows, cols, batch)
    S1 = s_ref[..., 0]
    assert np.sum((np.abs(S1) > 2**24) & (S1 % 2 != 0)) >= 10  # the case is exercised
    Wd, Xd = dev(Wq), dev(Xq)
    s = host(gq.block_sums(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    np.testing.assert_array_equal(s, s_ref)
    y = host(gq.matmul_ws(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)
    s_g = host(gq.block_sums(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_GEMV))
    np.testing.assert_array_equal(s_g, s_ref)


def sampled_rows(rows, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return np.unique(np.concatenate([[0, rows - 1], g.choice(rows, size=min(k, rows), replace=False)]))


@pytest.mark.parametrize("rows,cols,batch", [(14336, 4096, 16), (14336, 4096, 64),
                                             (28672, 8192, 512)])
def test_mma_full_size(rows, cols, batch):
    """The batch-sweep and prefill shapes at full size; the oracle recomputes
    sampled rows from the same fp32 inputs."""
    W, X = inputs.gemm_q4_k(0, rows, cols, batch)
    Wd = gq.quantize(Q4_K, dev(W))
    Xd = gq.quantize(Q8_K, dev(X))
    y = host(gq.matmul_ws(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    idx = sampled_rows(rows, 32, rows + batch)
    Wq_s = orc.quantize(Q4_K, W[idx])
    assert host(Wd)[idx].tobytes() == Wq_s.tobytes()
    Xq = orc.quantize(Q8_K, X)
    y_ref, T = orc.matmul_ref(Q4_K, Wq_s, Xq, len(idx), cols, batch, nthreads=orc.max_threads())
    assert_close(y[:, idx], y_ref, T)


@pytest.mark.skipif(bool(os.environ.get("GQ_TC_MIN_BATCH")), reason="threshold overridden")
@pytest.mark.parametrize("rows,batch,ws,want", [
    (14336, 3, True, "gemv"), (14336, 4, True, "skinny"), (14336, 9, True, "skinny"), (14336, 32, True, "skinny"),
    (14336, 33, True, "mma"), (14336, 33, False, "mma"), (14336, 65, False, "mma"), (14336, 65, True, "mma"),
    (4096, 9, True, "gemv"), (4096, 15, False, "gemv"), (4096, 16, True, "skinny"), (4096, 16, False, "skinny"),
    (4096, 33, True, "mma"), (4096, 40, False, "mma"), (1024, 16, True, "mma"), (1024, 16, False, "gemv"),
    (8192, 32, False, "skinny"), (8192, 33, False, "mma")])
def test_auto_dispatch_rule(rows, batch, ws, want):
    """GQ_PATH_AUTO for Q4_K: the warp-level tensor-core kernel from batch 4
    on matrices of 8192 rows or more and from 16 on 2048 or more, up to 32;
    beyond, the tcgen05 kernel (with a workspace, or the variant that packs
    its activations in the CTA without one); with a workspace the tcgen05
    kernel also below that band, from batch 9 on 14336 rows and 16
    otherwise; the GEMV below.  Every family is deterministic, so the AUTO result equals the
    chosen family's bit for bit."""
    cols = 1024
    g = inputs.rng(rows + batch)
    Wd = gq.quantize(Q4_K, torch.from_numpy(inputs.normal(g, (rows, cols), 0.02)).cuda())
    Xd = gq.quantize(Q8_K, torch.from_numpy(inputs.normal(g, (batch, cols))).cuda())
    if ws:
        y_auto = host(gq.matmul_ws(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_AUTO))
    else:
        y_auto = host(gq.matmul(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_AUTO))
    path = {"mma": gq.PATH_MMA, "gemv": gq.PATH_GEMV, "skinny": gq.PATH_SKINNY}[want]
    assert gq.gq_auto_path(Q4_K, rows, cols, batch, ws) == path  # the host-side query agrees
    y_want = host(gq.matmul_ws(Q4_K, Wd, Xd, rows, cols, batch, path))
    assert y_auto.tobytes() == y_want.tobytes()


# ----------------------------------- the tcgen05 kernel without a workspace

NOWS_SHAPES = [(128, 256, 1), (200, 768, 40), (77, 512, 32), (300, 1280, 33), (130, 2048, 64),
               (257, 1024, 65), (384, 4096, 130), (96, 3072, 200)]


@pytest.mark.parametrize("rows,cols,batch", NOWS_SHAPES)
def test_mma_without_workspace(rows, cols, batch):
    """GQ_PATH_MMA with no workspace: tiles of 32 / 64 columns whose idle
    epilogue warps pack the activations in the CTA.  Sums equal the oracle's;
    y equals the workspace variant's bit for bit (same per-output arithmetic
    in the same super-block order, whatever the tile width) and the oracle's
    within the bar."""
    g = inputs.rng(rows * 3 + cols + batch)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q4_K, W), orc.quantize(Q8_K, X)
    Wd, Xd = dev(Wq), dev(Xq)
    s = torch.empty(batch, rows, cols // 256, 2, dtype=torch.int32, device="cuda")
    gq.gq_block_sums(Q4_K, Wd, Xd, s, rows, cols, batch, gq.PATH_MMA)
    np.testing.assert_array_equal(host(s), orc.block_sums(Q4_K, Wq, Xq, rows, cols, batch))
    y = torch.empty(batch, rows, device="cuda")
    gq.gq_matmul_path(Q4_K, Wd, Xd, y, rows, cols, batch, gq.PATH_MMA)
    y_ws = host(gq.matmul_ws(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    assert host(y).tobytes() == y_ws.tobytes()
    y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch)
    assert_close(host(y), y_ref, T)


@pytest.mark.parametrize("batch", [5, 40, 100])
def test_mma_without_workspace_beyond_fp32_integers(batch):
    """The odd S1 above 2^24 case of the workspace variant, packed in the
    CTA (raw -128 activation codes included)."""
    rows, cols = 131, 512
    W = inputs.outlier_weights(inputs.rng(7), rows, cols, frac=0.001)
    W[0] = 1.0
    W[0, 5] = 0.93
    W[2] = 1.0
    W[2, 1::2] = 0.93
    X = inputs.normal(inputs.rng(8), (batch, cols))
    X[0] = 1.0
    X[batch - 1] = 1.0
    Wq, Xq = orc.quantize(Q4_K, W), orc.quantize(Q8_K, X)
    blk = Xq.reshape(batch, cols // 256, 276)
    blk[1, :, 4:260] = 0x80
    blk[1, :, 260:276] = np.frombuffer(np.full(8, -128 * 32, np.int16).tobytes(), np.uint8)
    s_ref = orc.block_sums(Q4_K, Wq, Xq, rows, cols, batch)
    assert np.sum((np.abs(s_ref[..., 0]) > 2**24) & (s_ref[..., 0] % 2 != 0)) >= 2
    s = torch.empty(batch, rows, cols // 256, 2, dtype=torch.int32, device="cuda")
    gq.gq_block_sums(Q4_K, dev(Wq), dev(Xq), s, rows, cols, batch, gq.PATH_MMA)
    np.testing.assert_array_equal(host(s), s_ref)


def test_mma_without_workspace_full_size():
    """The prefill shape through gq_matmul_path(GQ_PATH_MMA) with no
    workspace; the oracle recomputes sampled rows."""
    rows, cols, batch = 28672, 8192, 512
    W, X = inputs.gemm_q4_k(0, rows, cols, batch)
    Wd = gq.quantize(Q4_K, dev(W))
    Xd = gq.quantize(Q8_K, dev(X))
    y = torch.empty(batch, rows, device="cuda")
    gq.gq_matmul_path(Q4_K, Wd, Xd, y, rows, cols, batch, gq.PATH_MMA)
    yh = host(y)
    idx = sampled_rows(rows, 24, 99)
    Wq_s = orc.quantize(Q4_K, W[idx])
    Xq = orc.quantize(Q8_K, X)
    y_ref, T = orc.matmul_ref(Q4_K, Wq_s, Xq, len(idx), cols, batch, nthreads=orc.max_threads())
    assert_close(yh[:, idx], y_ref, T)

