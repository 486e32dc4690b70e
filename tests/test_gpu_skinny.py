"""GPU parity of the warp-level tensor-core kernel for Q4_K x Q8_K at small
batches (GQ_PATH_SKINNY) against the CPU oracle: integer super-block sums S1
and S2 bit-identical, y within 1e-4 * sum|terms| ("llama.cpp 推理引擎" §5.5,
the two-level scales whose integer sums are exact)."""
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


# N tiles of 8, 16, 32 and 64 columns with ragged batches; row tiles of 96
# with ragged tails; odd and even super-block counts (the activation chunks
# hold two)
SHAPES = [(96, 256, 1), (100, 512, 2), (200, 768, 8), (300, 1280, 9), (77, 256, 16), (513, 2048, 17),
          (192, 1024, 32), (130, 2304, 33), (257, 4096, 64), (1000, 512, 40), (96, 3072, 5)]


@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_skinny_sums_and_y(rows, cols, batch):
    g = inputs.rng(rows * 3 + cols + batch)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q4_K, W), orc.quantize(Q8_K, X)
    Wd, Xd = dev(Wq), dev(Xq)
    s = host(gq.block_sums(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    np.testing.assert_array_equal(s, orc.block_sums(Q4_K, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("batch", [3, 16, 40, 64])
def test_skinny_sums_beyond_fp32_integers(batch):
    """Constant rows (sc = 63, codes 15) with single codes lowered, against
    constant activations (codes +-127): S1 near 3.07e7 > 2^24 and odd, and
    raw activation codes of -128, must still match the oracle bit for bit."""
    rows, cols = 131, 512
    W = inputs.outlier_weights(inputs.rng(7), rows, cols, frac=0.001)
    W[0] = 1.0
    W[0, 5] = 0.93
    W[1] = 1.0
    W[2] = 1.0
    W[2, 1::2] = 0.93
    W[130] = 1.0
    W[130, 255] = 0.93
    X = inputs.normal(inputs.rng(8), (batch, cols))
    X[0] = 1.0
    X[1] = -1.0
    X[batch - 1] = 1.0
    Wq, Xq = orc.quantize(Q4_K, W), orc.quantize(Q8_K, X)
    # a column of raw -128 codes (never written by the quantizer; the bsums
    # are set to match so the block stays self-consistent)
    blk = Xq.reshape(batch, cols // 256, 276)
    blk[1, :, 4:260] = 0x80
    blk[1, :, 260:276] = np.frombuffer(np.full(8, -128 * 32, np.int16).tobytes(), np.uint8)
    s_ref = orc.block_sums(Q4_K, Wq, Xq, rows, cols, batch)
    assert np.sum((np.abs(s_ref[..., 0]) > 2**24) & (s_ref[..., 0] % 2 != 0)) >= 2
    Wd, Xd = dev(Wq), dev(Xq)
    np.testing.assert_array_equal(host(gq.block_sums(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY)), s_ref)
    y = host(gq.matmul(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("batch", [65, 130, 200])
def test_skinny_batches_beyond_one_tile(batch):
    """Batches beyond 64 run as 64-column chunks (one launch each): sums and
    y still match the oracle, the last chunk ragged."""
    rows, cols = 200, 768
    g = inputs.rng(31 + batch)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q4_K, W), orc.quantize(Q8_K, X)
    Wd, Xd = dev(Wq), dev(Xq)
    np.testing.assert_array_equal(host(gq.block_sums(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY)),
                                  orc.block_sums(Q4_K, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("batch", [1, 16, 40])
def test_skinny_static_weights_flag_same_result(batch):
    """GQ_FLAG_W_STATIC only moves the first weight tiles before the
    dependency wait: a chain of products over distinct matrices gives the
    same bytes with and without it."""
    rows, cols, n = 500, 1024, 5
    g = inputs.rng(51 + batch)
    Ws = [gq.quantize(Q4_K, dev(inputs.normal(g, (rows, cols), 0.02))) for _ in range(n)]
    X = gq.quantize(Q8_K, dev(inputs.normal(g, (batch, cols))))
    ya = torch.empty(n, batch, rows, device="cuda")
    yb = torch.empty(n, batch, rows, device="cuda")
    for i in range(n):
        gq.gq_matmul_ex(Q4_K, Ws[i], X, ya[i], rows, cols, batch, gq.PATH_SKINNY, gq.FLAG_W_STATIC)
    for i in range(n):
        gq.gq_matmul_path(Q4_K, Ws[i], X, yb[i], rows, cols, batch, gq.PATH_SKINNY)
    assert host(ya).tobytes() == host(yb).tobytes()
    y_ref, T = orc.matmul_ref(Q4_K, host(Ws[-1]), host(X), rows, cols, batch)
    assert_close(host(ya[-1]), y_ref, T)


def test_skinny_shape_rules():
    """Q4_K, Q5_K, Q4_0 and Q8_0 weights with cols a multiple of 256 only:
    Q6_K is refused, and so is a Q4_0 row of 288 columns."""
    rows, cols = 128, 2048
    g = inputs.rng(31)
    y = torch.empty(65, rows, device="cuda")
    W6 = gq.quantize(4, dev(inputs.normal(g, (rows, cols), 0.02)))
    X8k = gq.quantize(Q8_K, dev(inputs.normal(g, (8, cols))))
    with pytest.raises(gq.GQError):
        gq.gq_matmul_path(4, W6, X8k, y, rows, cols, 8, gq.PATH_SKINNY)
    W0 = gq.quantize(0, dev(inputs.normal(g, (rows, 288), 0.02)))
    X0 = gq.quantize(1, dev(inputs.normal(g, (8, 288))))
    with pytest.raises(gq.GQError):
        gq.gq_matmul_path(0, W0, X0, y, rows, 288, 8, gq.PATH_SKINNY)


def sampled_rows(rows, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    return np.unique(np.concatenate([[0, rows - 1], g.choice(rows, size=min(k, rows), replace=False)]))


@pytest.mark.parametrize("rows,cols,batch", [(14336, 4096, 2), (14336, 4096, 8), (14336, 4096, 16),
                                             (14336, 4096, 32), (14336, 4096, 64), (28672, 8192, 512)])
def test_skinny_full_size(rows, cols, batch):
    """The batch-sweep shape and the prefill shape (eight 64-column chunks);
    the oracle recomputes sampled rows."""
    W, X = inputs.gemm_q4_k(0, rows, cols, batch)
    Wd = gq.quantize(Q4_K, dev(W))
    Xd = gq.quantize(Q8_K, dev(X))
    y = host(gq.matmul(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    idx = sampled_rows(rows, 32, rows + batch)
    Wq_s = orc.quantize(Q4_K, W[idx])
    assert host(Wd)[idx].tobytes() == Wq_s.tobytes()
    Xq = orc.quantize(Q8_K, X)
    y_ref, T = orc.matmul_ref(Q4_K, Wq_s, Xq, len(idx), cols, batch, nthreads=orc.max_threads())
    assert_close(y[:, idx], y_ref, T)
