"""GPU test of gq_matmul_noalloc, the tensor-core product for callers that
cannot allocate device memory (its scratch is a static array inside the
library).  Called through the C ABI twice in a row on different inputs; each
result must match the oracle's y, and the same product through gq_matmul_ws
(the entry point with a caller-allocated workspace), within the suite's
tolerance, so the second call is not disturbed by what the first left in the
shared scratch.  A product at the scratch's size limit is accepted and
correct, and larger ones are refused.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own in a
fresh process."""
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


def case(seed, rows, cols, batch):
    g = inputs.rng(seed)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q4_K, W), orc.quantize(Q8_K, X)
    return Wq, Xq, torch.from_numpy(Wq).cuda(), torch.from_numpy(Xq).cuda()


def test_noalloc_matches_workspace_entry_twice():
    rows, cols = 300, 2048
    results = []
    for seed, batch in ((1, 200), (2, 77)):
        Wq, Xq, Wd, Xd = case(seed, rows, cols, batch)
        y_na = torch.full((batch, rows), float("nan"), device="cuda")
        gq.gq_matmul_noalloc(Q4_K, Wd, Xd, y_na, rows, cols, batch)
        y_ws = gq.matmul_ws(Q4_K, Wd, Xd, rows, cols, batch, gq.PATH_MMA)
        torch.cuda.synchronize()
        y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch)
        y_na_h = y_na.cpu().numpy().astype(np.float64)
        # against the oracle itself, and against the workspace entry point
        assert np.all(np.abs(y_na_h - y_ref) <= TOL * T)
        assert np.all(np.abs(y_na_h - y_ws.cpu().numpy()) <= TOL * T)
        results.append(y_na.cpu().numpy())
    assert results[0].shape != results[1].shape or not np.array_equal(results[0], results[1])


def test_noalloc_at_the_scratch_limit():
    """The largest product the scratch holds at 8192 columns (batch 896:
    7 column tiles x 32 super-blocks x 70656 bytes) is accepted and correct;
    one more column tile is not."""
    rows, cols, batch = 128, 8192, 896
    need = gq.gq_matmul_workspace_bytes(Q4_K, rows, cols, batch)
    assert need <= 16 << 20 < gq.gq_matmul_workspace_bytes(Q4_K, rows, cols, batch + 1)
    Wq, Xq, Wd, Xd = case(3, rows, cols, batch)
    y = torch.full((batch, rows), float("nan"), device="cuda")
    gq.gq_matmul_noalloc(Q4_K, Wd, Xd, y, rows, cols, batch)
    torch.cuda.synchronize()
    y_ref, T = orc.matmul_ref(Q4_K, Wq, Xq, rows, cols, batch, nthreads=orc.max_threads())
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - y_ref) <= TOL * T)


def test_noalloc_rejects_products_beyond_the_scratch():
    rows, cols, batch = 128, 8192, 1024  # needs 8 * 32 * 70656 bytes > 16 MiB
    assert gq.gq_matmul_workspace_bytes(Q4_K, rows, cols, batch) > 16 << 20
    W = torch.zeros(rows, cols // 256 * 144, dtype=torch.uint8, device="cuda")
    X = torch.zeros(batch, cols // 256 * 276, dtype=torch.uint8, device="cuda")
    y = torch.zeros(batch, rows, device="cuda")
    with pytest.raises(gq.GQError) as e:
        gq.gq_matmul_noalloc(Q4_K, W, X, y, rows, cols, batch)
    assert e.value.status == 3  # GQ_ERR_SHAPE
    with pytest.raises(gq.GQError) as e:
        gq.gq_matmul_noalloc(0, W, X, y, rows, cols, 8)
    assert e.value.status == 2  # GQ_ERR_TYPE
