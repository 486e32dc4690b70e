"""GPU parity of the tcgen05 tensor-core path for Q4_0 / Q8_0 weights x Q8_0
activations against the CPU oracle: per-block integer sums bit-identical, y
within 1e-4 * sum|terms|, and the same y as the GEMV path within that bound
("llama.cpp 推理引擎" §5.3-5.4 and §6.4: per-block integer products scaled by
the two block factors and summed)."""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as orc  # noqa: E402
from block_quantized_gb300 import gq, inputs  # noqa: E402

pytestmark = pytest.mark.gpu

Q4_0, Q8_0 = 0, 1
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


# tile widths 32 (batch <= 32), 64 (<= 64) and 128; ragged row and column
# tiles; K loops of one to sixteen raw stages (longer than the stage, operand
# and accumulator rings)
SHAPES = [(128, 256, 128), (130, 512, 16), (200, 768, 40), (257, 2048, 130), (77, 256, 1),
          (384, 4096, 64), (300, 1280, 33), (513, 1024, 7), (64, 512, 65), (129, 256, 200)]


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_mma_q0_sums_and_y(wtype, rows, cols, batch):
    g = inputs.rng(rows * 7 + cols + batch + wtype)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(wtype, W), orc.quantize(Q8_0, X)
    Wd, Xd = dev(Wq), dev(Xq)
    s = host(gq.block_sums(wtype, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    np.testing.assert_array_equal(s, orc.block_sums(wtype, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)
    y_g = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_GEMV))
    assert_close(y_g, y_ref, T)


def raw_blocks(g, wtype, n, extreme):
    """n blocks of raw bytes: fp16 scale 0.5 .. 2, codes drawn over the whole
    byte range (Q8_0: -128..127, Q4_0: nibbles 0..15) or, with `extreme`, only
    the range ends."""
    bb = 34 if wtype == Q8_0 else 18
    out = np.zeros((n, bb), np.uint8)
    d = g.uniform(0.5, 2.0, n).astype(np.float16)
    out[:, 0:2] = d.view(np.uint8).reshape(n, 2)
    if wtype == Q8_0:
        c = g.choice(np.array([-128, 127], np.int8), size=(n, 32)) if extreme else \
            g.integers(-128, 128, size=(n, 32)).astype(np.int8)
        out[:, 2:] = c.view(np.uint8)
    else:
        nib = g.choice(np.array([0, 15], np.uint8), size=(n, 32)) if extreme else \
            g.integers(0, 16, size=(n, 32)).astype(np.uint8)
        out[:, 2:] = nib[:, 0::2] | (nib[:, 1::2] << 4)
    return out


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("extreme", [False, True])
def test_mma_q0_full_code_range(wtype, extreme):
    """Codes the quantizer never writes (Q8_0 -128) and the range ends only:
    |S| reaches 32 * 128 * 128 = 2^19 and every block sum is still exact."""
    rows, cols, batch = 160, 768, 72
    g = inputs.rng(11 + wtype + 2 * extreme)
    nb = cols // 32
    Wq = raw_blocks(g, wtype, rows * nb, extreme).reshape(rows, -1)
    Xq = raw_blocks(g, Q8_0, batch * nb, extreme).reshape(batch, -1)
    if extreme:
        # one row and one column of nothing but the most negative codes:
        # S = 32 * (-128) * (-128) = 524288 (Q8_0) or 32 * (-8) * (-128) (Q4_0)
        for k in range(nb):
            Wq[3, k * Wq.shape[1] // nb + 2:(k + 1) * Wq.shape[1] // nb] = 0x80 if wtype == Q8_0 else 0
            Xq[5, k * 34 + 2:(k + 1) * 34] = 0x80
    Wd, Xd = dev(Wq), dev(Xq)
    s_ref = orc.block_sums(wtype, Wq, Xq, rows, cols, batch)
    if extreme:
        assert s_ref[5, 3, 0] == (524288 if wtype == Q8_0 else 32768)
    s = host(gq.block_sums(wtype, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    np.testing.assert_array_equal(s, s_ref)
    y = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
def test_mma_q0_degenerate_blocks(wtype):
    """Zero, constant and all-negative weight rows; zero and large activation
    columns."""
    rows, cols, batch = 130, 512, 20
    W = np.zeros((rows, cols), np.float32)
    W[1] = 1.0
    W[2] = -3.0
    W[3, ::2] = 7.0
    W[4] = np.linspace(-1, 1, cols, dtype=np.float32)
    W[5:] = inputs.normal(inputs.rng(3), (rows - 5, cols), 0.02)
    X = inputs.normal(inputs.rng(4), (batch, cols))
    X[0] = 0.0
    X[1] = 1000.0
    Wq, Xq = orc.quantize(wtype, W), orc.quantize(Q8_0, X)
    s = host(gq.block_sums(wtype, dev(Wq), dev(Xq), rows, cols, batch, gq.PATH_MMA))
    np.testing.assert_array_equal(s, orc.block_sums(wtype, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul(wtype, dev(Wq), dev(Xq), rows, cols, batch, gq.PATH_MMA))
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert np.all(y[0] == 0) and np.all(y[:, 0] == 0)
    assert_close(y, y_ref, T)


def test_mma_q0_shape_rules():
    """The tensor-core kernel wants cols a multiple of 256 (8 blocks per
    16-byte-aligned TMA row): GQ_PATH_MMA refuses other widths, AUTO takes
    the GEMV for them, and no workspace is ever needed."""
    rows, cols, batch = 128, 288, 32
    g = inputs.rng(21)
    Wq = orc.quantize(Q4_0, inputs.normal(g, (rows, cols), 0.02))
    Xq = orc.quantize(Q8_0, inputs.normal(g, (batch, cols)))
    Wd, Xd = dev(Wq), dev(Xq)
    y = torch.empty(batch, rows, device="cuda")
    with pytest.raises(gq.GQError):
        gq.gq_matmul_path(Q4_0, Wd, Xd, y, rows, cols, batch, gq.PATH_MMA)
    gq.gq_matmul(Q4_0, Wd, Xd, y, rows, cols, batch)
    y_ref, T = orc.matmul_ref(Q4_0, Wq, Xq, rows, cols, batch)
    assert_close(host(y), y_ref, T)
    assert gq.gq_matmul_workspace_bytes(Q4_0, rows, 256, batch) == 0
    assert gq.gq_matmul_workspace_bytes(Q8_0, rows, 256, batch) == 0


@pytest.mark.skipif(bool(os.environ.get("GQ_TC_MIN_BATCH")), reason="threshold overridden")
@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("batch,want", [(15, "gemv"), (16, "mma"), (100, "mma")])
def test_mma_q0_auto_dispatch(wtype, batch, want):
    """gq_matmul itself (no workspace) takes the tensor-core kernel from batch
    16 on; both families are deterministic, so its result equals the chosen
    family's bit for bit."""
    rows, cols = 1024, 1024
    g = inputs.rng(rows + batch + wtype)
    Wd = gq.quantize(wtype, dev(inputs.normal(g, (rows, cols), 0.02)))
    Xd = gq.quantize(Q8_0, dev(inputs.normal(g, (batch, cols))))
    y = torch.empty(batch, rows, device="cuda")
    gq.gq_matmul(wtype, Wd, Xd, y, rows, cols, batch)
    y_want = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_MMA if want == "mma" else gq.PATH_GEMV))
    assert host(y).tobytes() == y_want.tobytes()


def sampled_rows(rows, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return np.unique(np.concatenate([[0, rows - 1], g.choice(rows, size=min(k, rows), replace=False)]))


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("rows,cols,batch", [(14336, 4096, 64), (28672, 8192, 512)])
def test_mma_q0_full_size(wtype, rows, cols, batch):
    """The batch-sweep and prefill shapes at full size with Q4_0 / Q8_0
    weights; the oracle recomputes sampled rows from the same fp32 inputs."""
    W, X = inputs.gemm_q4_k(0, rows, cols, batch)
    Wd = gq.quantize(wtype, dev(W))
    Xd = gq.quantize(Q8_0, dev(X))
    y = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_MMA))
    idx = sampled_rows(rows, 32, rows + batch + wtype)
    Wq_s = orc.quantize(wtype, W[idx])
    assert host(Wd)[idx].tobytes() == Wq_s.tobytes()
    Xq = orc.quantize(Q8_0, X)
    assert host(Xd).tobytes() == Xq.tobytes()
    y_ref, T = orc.matmul_ref(wtype, Wq_s, Xq, len(idx), cols, batch, nthreads=orc.max_threads())
    assert_close(y[:, idx], y_ref, T)
