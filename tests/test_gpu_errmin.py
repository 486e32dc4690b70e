"""GPU parity of the error-minimizing Q4_K / Q5_K encoder (gq_quantize_rows_ex
with GQ_QUANT_ERRMIN) against the CPU oracle: the bytes are bit-identical
(the search's error measure is fp32 in a fixed order on both sides, so both
make the same choice), and the products of the refined weights match the
oracle's within 1e-4 * sum|block terms|."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as orc  # noqa: E402
from block_quantized_gb300 import gq, inputs  # noqa: E402

pytestmark = pytest.mark.gpu

Q4_K, Q8_K, Q5_K = 2, 3, 5
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


def encoder_inputs():
    g = inputs.rng(21)
    parts = [
        inputs.outlier_weights(g, 16, 2048, frac=0.01).reshape(-1),
        inputs.normal(g, (64 * 256,), 0.02),
        inputs.normal(g, (8 * 256,)),
        np.abs(inputs.normal(g, (4 * 256,))),
        -np.abs(inputs.normal(g, (4 * 256,))),
        np.full(2 * 256, 0.37, np.float32),
        np.zeros(2 * 256, np.float32),
        inputs.normal(g, (2 * 256,), 1e-6),
        inputs.normal(g, (2 * 256,), 300.0),
    ]
    x = np.concatenate(parts).astype(np.float32)
    # the hand-derived case: a sub-block the min/max fit scales too coarsely
    c = np.array([0, 15, 3, 8, 1, 12, 7, 4] * 4, np.float32)
    x[0:32] = c * 5 / 256
    x[1] = np.float32(75.01 / 256)
    x[32:64] = np.arange(32, dtype=np.float32) * 945 / 256 / 31
    return x


@pytest.mark.parametrize("t", [Q4_K, Q5_K])
def test_errmin_bytes_bit_exact(t):
    x = encoder_inputs()
    got = host(gq.quantize(t, dev(x), flags=gq.QUANT_ERRMIN))
    ref = orc.quantize(t, x, errmin=True)
    assert got.tobytes() == ref.tobytes()
    # and it differs from the default encoder where the search found better pairs
    assert got.tobytes() != orc.quantize(t, x).tobytes()


@pytest.mark.parametrize("t", [Q4_K, Q5_K])
def test_errmin_weights_in_the_product(t):
    rows, cols, batch = 96, 2048, 3
    g = inputs.rng(22)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wd = gq.quantize(t, dev(W), flags=gq.QUANT_ERRMIN)
    Wq = orc.quantize(t, W, errmin=True)
    assert host(Wd).tobytes() == Wq.tobytes()
    Xq = orc.quantize(Q8_K, X)
    y = host(gq.matmul(t, Wd, dev(Xq), rows, cols, batch))
    y_ref, T = orc.matmul_ref(t, Wq, Xq, rows, cols, batch)
    assert np.all(np.abs(y.astype(np.float64) - y_ref) <= TOL * T)
