"""GPU parity of the warp-level tensor-core kernel for Q4_0 / Q8_0 weights x
Q8_0 activations at small batches (GQ_PATH_SKINNY) against the CPU oracle:
per-block integer sums bit-identical, y within 1e-4 * sum|terms|
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


# N tiles of 8, 16, 32 and 64 columns with ragged batches; row tiles of 96
# with ragged tails; stage counts from one to sixteen (activation chunks of
# two to eight stages, some ragged)
SHAPES = [(96, 256, 1), (100, 512, 2), (200, 768, 8), (300, 1280, 9), (77, 256, 16), (513, 2048, 17),
          (192, 1024, 32), (130, 2304, 33), (257, 4096, 64), (1000, 512, 40), (96, 3072, 5)]


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_skinny_q0_sums_and_y(wtype, rows, cols, batch):
    g = inputs.rng(rows * 5 + cols + batch + wtype)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(wtype, W), orc.quantize(Q8_0, X)
    Wd, Xd = dev(Wq), dev(Xq)
    s = host(gq.block_sums(wtype, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    np.testing.assert_array_equal(s, orc.block_sums(wtype, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)


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
@pytest.mark.parametrize("batch", [7, 64])
def test_skinny_q0_full_code_range(wtype, extreme, batch):
    """Codes the quantizer never writes (Q8_0 -128) and the range ends only:
    a block dot reaches 32 * 128 * 128 = 2^19 and every block sum is still
    exact."""
    rows, cols = 160, 768
    g = inputs.rng(13 + wtype + 2 * extreme + batch)
    nb = cols // 32
    Wq = raw_blocks(g, wtype, rows * nb, extreme).reshape(rows, -1)
    Xq = raw_blocks(g, Q8_0, batch * nb, extreme).reshape(batch, -1)
    if extreme:
        for k in range(nb):
            Wq[3, k * Wq.shape[1] // nb + 2:(k + 1) * Wq.shape[1] // nb] = 0x80 if wtype == Q8_0 else 0
            Xq[5, k * 34 + 2:(k + 1) * 34] = 0x80
    s_ref = orc.block_sums(wtype, Wq, Xq, rows, cols, batch)
    if extreme:
        assert s_ref[5, 3, 0] == (524288 if wtype == Q8_0 else 32768)
    Wd, Xd = dev(Wq), dev(Xq)
    np.testing.assert_array_equal(host(gq.block_sums(wtype, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY)), s_ref)
    y = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
def test_skinny_q0_degenerate_blocks(wtype):
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
    s = host(gq.block_sums(wtype, dev(Wq), dev(Xq), rows, cols, batch, gq.PATH_SKINNY))
    np.testing.assert_array_equal(s, orc.block_sums(wtype, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul(wtype, dev(Wq), dev(Xq), rows, cols, batch, gq.PATH_SKINNY))
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert np.all(y[0] == 0) and np.all(y[:, 0] == 0)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("batch", [65, 130])
def test_skinny_q0_batches_beyond_one_tile(wtype, batch):
    """Batches beyond 64 run as 64-column chunks (one launch each)."""
    rows, cols = 200, 768
    g = inputs.rng(37 + batch + wtype)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(wtype, W), orc.quantize(Q8_0, X)
    Wd, Xd = dev(Wq), dev(Xq)
    np.testing.assert_array_equal(host(gq.block_sums(wtype, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY)),
                                  orc.block_sums(wtype, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
def test_skinny_q0_static_weights_flag_same_result(wtype):
    rows, cols, batch, n = 500, 1024, 12, 4
    g = inputs.rng(61 + wtype)
    Ws = [gq.quantize(wtype, dev(inputs.normal(g, (rows, cols), 0.02))) for _ in range(n)]
    X = gq.quantize(Q8_0, dev(inputs.normal(g, (batch, cols))))
    ya = torch.empty(n, batch, rows, device="cuda")
    yb = torch.empty(n, batch, rows, device="cuda")
    for i in range(n):
        gq.gq_matmul_ex(wtype, Ws[i], X, ya[i], rows, cols, batch, gq.PATH_SKINNY, gq.FLAG_W_STATIC)
    for i in range(n):
        gq.gq_matmul_path(wtype, Ws[i], X, yb[i], rows, cols, batch, gq.PATH_SKINNY)
    assert host(ya).tobytes() == host(yb).tobytes()


@pytest.mark.skipif(bool(os.environ.get("GQ_TC_MIN_BATCH")), reason="threshold overridden")
@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("rows,batch,want", [(8192, 1, "gemv"), (8192, 2, "skinny"), (14336, 33, "skinny"),
                                             (14336, 64, "skinny"), (14336, 65, "mma"), (4096, 7, "gemv"),
                                             (4096, 8, "skinny"), (4096, 65, "mma"), (1024, 16, "mma"),
                                             (1024, 8, "gemv")])
def test_skinny_q0_auto_dispatch(wtype, rows, batch, want):
    """gq_matmul (no workspace) picks the family by rows and batch; every
    family is deterministic, so its result equals the chosen one's bit for
    bit."""
    cols = 512
    g = inputs.rng(rows + batch + wtype)
    Wd = gq.quantize(wtype, dev(inputs.normal(g, (rows, cols), 0.02)))
    Xd = gq.quantize(Q8_0, dev(inputs.normal(g, (batch, cols))))
    y = torch.empty(batch, rows, device="cuda")
    gq.gq_matmul(wtype, Wd, Xd, y, rows, cols, batch)
    path = {"gemv": gq.PATH_GEMV, "skinny": gq.PATH_SKINNY, "mma": gq.PATH_MMA}[want]
    assert gq.gq_auto_path(wtype, rows, cols, batch) == path  # the host-side query agrees
    assert host(y).tobytes() == host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, path)).tobytes()


def sampled_rows(rows, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return np.unique(np.concatenate([[0, rows - 1], g.choice(rows, size=min(k, rows), replace=False)]))


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("batch", [4, 16, 32, 64])
def test_skinny_q0_full_size(wtype, batch):
    """The 14336 x 4096 batch-sweep shape; the oracle recomputes sampled rows
    from the same fp32 inputs."""
    rows, cols = 14336, 4096
    W, X = inputs.gemm_q4_k(0, rows, cols, batch)
    Wd = gq.quantize(wtype, dev(W))
    Xd = gq.quantize(Q8_0, dev(X))
    y = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    idx = sampled_rows(rows, 32, rows + batch + wtype)
    Wq_s = orc.quantize(wtype, W[idx])
    assert host(Wd)[idx].tobytes() == Wq_s.tobytes()
    Xq = orc.quantize(Q8_0, X)
    assert host(Xd).tobytes() == Xq.tobytes()
    y_ref, T = orc.matmul_ref(wtype, Wq_s, Xq, len(idx), cols, batch, nthreads=orc.max_threads())
    assert_close(y[:, idx], y_ref, T)
