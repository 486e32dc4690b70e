"""GPU parity for Q5_K weights (the Q4_K super-block with 5-bit codes and a
fifth-bit plane, paired with Q8_K activations): the codecs and the GEMV
through the C ABI against the CPU oracle.

Bar: quantized bytes and int32 block sums (S1, S2) bit-identical; y within
1e-4 * sum|block terms| per output.  The shapes cover both GEMV kernels: the
streaming kernel (whole rows through a per-warp shared-memory ring, 16 or 8
warps, several rows per warp on the tall shapes) and the plain kernel (rows
too long for a two-stage ring).
"""
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as orc  # noqa: E402
from block_quantized_gb300 import gq, inputs  # noqa: E402

pytestmark = pytest.mark.gpu

Q8_K, Q5_K = 3, 5
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


def codec_inputs():
    g = inputs.rng(6)
    be = 256
    parts = [
        inputs.normal(g, (37 * be,), 0.02),
        inputs.outlier_weights(g, 8, 4 * be, frac=0.01).reshape(-1),
        inputs.normal(g, (16 * be,)),
        np.abs(inputs.normal(g, (3 * be,))),
        -np.abs(inputs.normal(g, (3 * be,))),
        np.full(2 * be, 0.37, np.float32),
        np.zeros(2 * be, np.float32),
        inputs.normal(g, (3 * be,), 1e-6),     # subnormal fp16 scales, clipped codes
        inputs.normal(g, (2 * be,), 1e-9),     # scale 0
        inputs.normal(g, (2 * be,), 300.0),
    ]
    x = np.concatenate(parts).astype(np.float32)
    # exact ties in the first super-block: sub-block 1 of range 1953/512
    # (dmin = 2^-6, d = 2^-9) and sub-block 0 with min 0 and step 3/512, its
    # elements at 0.5, 2.5 and 30.5 steps (codes 1, 3, 31)
    r = np.arange(32)
    x[0:32] = 0.0
    x[1:4] = np.array([0.5, 2.5, 30.5], np.float32) * 3 / 512
    x[32:64] = (63 * r - 504) / 512.0
    return x


def test_quantize_bit_exact():
    x = codec_inputs()
    assert host(gq.quantize(Q5_K, dev(x))).tobytes() == orc.quantize(Q5_K, x).tobytes()


@pytest.mark.parametrize("nblocks", [1, 3, 9, 1000])
def test_quantize_sizes(nblocks):
    x = inputs.normal(inputs.rng(nblocks), (nblocks * 256,), 0.5)
    assert host(gq.quantize(Q5_K, dev(x))).tobytes() == orc.quantize(Q5_K, x).tobytes()


def test_dequantize_bit_exact():
    x = codec_inputs()
    q = orc.quantize(Q5_K, x)
    ref = orc.dequantize(Q5_K, q, x.size)
    got = host(gq.dequantize(Q5_K, dev(q.reshape(-1)), x.size))
    assert got.view(np.uint32).tobytes() == ref.view(np.uint32).tobytes()


SHAPES = [
    # streaming kernel (every multiple of 256 whose rows fit a two-stage ring)
    (1, 256, 1), (7, 2048, 1), (130, 4096, 1), (40, 4096, 2), (9, 16384, 3), (33, 768, 5),
    (19, 2816, 3), (64, 11008, 1), (5, 18432, 2),
    # plain kernel: rows too long for a two-stage ring of eight warps
    (2, 131072, 1), (3, 65536, 2),
]


@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_gemv_block_sums_and_y(rows, cols, batch):
    g = inputs.rng(rows * 7 + cols + batch)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q5_K, W), orc.quantize(Q8_K, X)
    Wd, Xd = gq.quantize(Q5_K, dev(W)), gq.quantize(Q8_K, dev(X))
    assert host(Wd).tobytes() == Wq.tobytes()
    assert host(Xd).tobytes() == Xq.tobytes()
    s = host(gq.block_sums(Q5_K, Wd, Xd, rows, cols, batch, gq.PATH_GEMV))
    np.testing.assert_array_equal(s, orc.block_sums(Q5_K, Wq, Xq, rows, cols, batch))
    y_ref, T = orc.matmul_ref(Q5_K, Wq, Xq, rows, cols, batch)
    assert_close(host(gq.matmul(Q5_K, Wd, Xd, rows, cols, batch)), y_ref, T)


# Several vectors per CTA (W streamed once per group of up to eight): group
# sizes 2, 4 and 8, ragged last groups, and more groups than one launch row.
@pytest.mark.parametrize("rows,cols,batch", [(130, 4096, 2), (300, 2048, 3), (77, 4096, 8), (64, 1024, 9),
                                             (200, 8192, 17), (33, 18432, 6)])
def test_gemv_vector_groups(rows, cols, batch):
    g = inputs.rng(rows * 11 + cols + batch)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q5_K, W), orc.quantize(Q8_K, X)
    Wd, Xd = dev(Wq), dev(Xq)
    s = host(gq.block_sums(Q5_K, Wd, Xd, rows, cols, batch, gq.PATH_GEMV))
    np.testing.assert_array_equal(s, orc.block_sums(Q5_K, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul(Q5_K, Wd, Xd, rows, cols, batch))
    y_ref, T = orc.matmul_ref(Q5_K, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)
    # each vector's y equals its own single-vector product within the bar
    for b in (0, batch - 1):
        y1 = host(gq.matmul(Q5_K, Wd, Xd[b:b + 1], rows, cols, 1))
        assert_close(y[b:b + 1], y_ref[b:b + 1], T[b:b + 1])
        assert_close(y1, y_ref[b:b + 1], T[b:b + 1])


# More rows than the grid has warps: each warp streams several rows through
# its ring (stage reuse, barrier phase flips), with a ragged last pass.
TALL_SHAPES = [(4867, 4096, 1), (2435, 8192, 2), (1300, 16384, 1), (3000, 11008, 1)]


@pytest.mark.parametrize("rows,cols,batch", TALL_SHAPES)
def test_gemv_tall(rows, cols, batch):
    g = inputs.rng(rows + cols)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q5_K, W), orc.quantize(Q8_K, X)
    y_ref, T = orc.matmul_ref(Q5_K, Wq, Xq, rows, cols, batch, nthreads=orc.max_threads())
    assert_close(host(gq.matmul(Q5_K, dev(Wq), dev(Xq), rows, cols, batch)), y_ref, T)
    s = host(gq.block_sums(Q5_K, dev(Wq), dev(Xq), rows, cols, batch, gq.PATH_GEMV))
    idx = np.array([0, 1, rows // 2, rows - 2, rows - 1])
    np.testing.assert_array_equal(s[:, idx], orc.block_sums(Q5_K, Wq[idx], Xq, len(idx), cols, batch))


def test_degenerate_blocks():
    """Zero, constant, all-negative and tiny weight blocks, a block at the
    extremes (every sc = 63 and code 31, which drives S1 to 63 * 31 * 127 *
    256 = 63,499,968 with constant activations) and a zero activation vector."""
    rows, cols = 8, 2048
    W = inputs.normal(inputs.rng(3), (rows, cols), 0.02)
    W[0] = 0.0
    W[1] = 0.37
    W[2, :256] = 1e-9
    W[3, 256:512] = -2.5
    W[4] = 1.0
    W[4, 5] = 0.97
    W[5] = -np.abs(W[5])
    X = inputs.normal(inputs.rng(4), (2, cols))
    X[1] = 0.0
    X[0, :256] = 1.0
    Wq, Xq = orc.quantize(Q5_K, W), orc.quantize(Q8_K, X)
    assert host(gq.quantize(Q5_K, dev(W))).tobytes() == Wq.tobytes()
    s = host(gq.block_sums(Q5_K, dev(Wq), dev(Xq), rows, cols, 2, gq.PATH_GEMV))
    np.testing.assert_array_equal(s, orc.block_sums(Q5_K, Wq, Xq, rows, cols, 2))
    y = host(gq.matmul(Q5_K, dev(Wq), dev(Xq), rows, cols, 2))
    y_ref, T = orc.matmul_ref(Q5_K, Wq, Xq, rows, cols, 2)
    assert_close(y, y_ref, T)
    assert np.all(y[1] == 0.0) and np.all(y[0, 0] == 0.0)


def test_gemv_4096_outlier_weights():
    """The 4096 x 4096 batch-1 GEMV on the row-spread + 0.1% outlier weights,
    every row against the oracle."""
    W, x = inputs.gemv_q4_k(0)
    Wq, xq = orc.quantize(Q5_K, W), orc.quantize(Q8_K, x)
    Wd = gq.quantize(Q5_K, dev(W))
    assert host(Wd).tobytes() == Wq.tobytes()
    y_ref, T = orc.matmul_ref(Q5_K, Wq, xq, 4096, 4096, 1, nthreads=orc.max_threads())
    assert_close(host(gq.matmul(Q5_K, Wd, dev(xq), 4096, 4096, 1)), y_ref, T)


def test_static_weights_flag_same_result():
    """GQ_FLAG_W_STATIC only moves the first weight copies before the
    dependency wait: a chain of products gives the same bytes with and
    without it."""
    rows, cols, n = 1000, 2048, 6
    g = inputs.rng(77)
    Ws = [gq.quantize(Q5_K, torch.from_numpy(inputs.normal(g, (rows, cols), 0.02)).cuda()) for _ in range(n)]
    X = gq.quantize(Q8_K, torch.from_numpy(inputs.normal(g, (n, cols))).cuda())
    ya = torch.empty(n, rows, device="cuda")
    yb = torch.empty(n, rows, device="cuda")
    for i in range(n):
        gq.gq_matmul_ex(Q5_K, Ws[i], X[i], ya[i], rows, cols, 1, gq.PATH_AUTO, gq.FLAG_W_STATIC)
    for i in range(n):
        gq.gq_matmul(Q5_K, Ws[i], X[i], yb[i], rows, cols, 1)
    torch.cuda.synchronize()
    assert ya.cpu().numpy().tobytes() == yb.cpu().numpy().tobytes()


# ------------------------------------------- fused activation quantize path

FUSED_SHAPES = [(1, 256, 1), (7, 2048, 1), (130, 4096, 2), (33, 768, 5), (19, 2816, 3),
                (64, 11008, 1), (4867, 4096, 1), (5, 18944, 2), (40, 4096, 8), (21, 2048, 11)]


@pytest.mark.parametrize("rows,cols,batch", FUSED_SHAPES)
def test_fused_f32_matches_unfused_and_oracle(rows, cols, batch):
    """gq_matmul_f32 quantizes the fp32 vector to Q8_K inside the streaming
    kernel: its integer sums equal the oracle's, and y equals quantize +
    gq_matmul bit for bit."""
    g = inputs.rng(5 * rows + cols + batch)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q5_K, W), orc.quantize(Q8_K, X)
    Wd, Xf = dev(Wq), dev(X)
    s = host(gq.block_sums_f32(Q5_K, Wd, Xf, rows, cols, batch))
    idx = np.unique(np.array([0, rows // 2, rows - 1]))
    np.testing.assert_array_equal(s[:, idx], orc.block_sums(Q5_K, Wq[idx], Xq, len(idx), cols, batch))
    y_f = host(gq.matmul_f32(Q5_K, Wd, Xf, rows, cols, batch))
    y_u = host(gq.matmul(Q5_K, Wd, gq.quantize(Q8_K, Xf), rows, cols, batch))
    assert y_f.view(np.uint32).tobytes() == y_u.view(np.uint32).tobytes()
    y_ref, T = orc.matmul_ref(Q5_K, Wq[idx], Xq, len(idx), cols, batch)
    assert_close(y_f[:, idx], y_ref, T)


def test_fused_quantize_ties_match_oracle():
    """Identity weights expose every activation code through the block sums
    (S1 = sc * code); activations on and next to rounding ties."""
    cols = 1024
    g = np.random.default_rng(41)
    X = np.empty((2, cols), np.float32)
    for r in range(2):
        for b0 in range(0, cols, 256):
            d = np.float32(2.0 ** int(g.integers(-12, 3))) if (b0 // 256 + r) % 2 == 0 else \
                np.float32(g.uniform(0.01, 3.0) / 127.0)
            v = ((g.integers(-126, 126, 256) + 0.5) * d).astype(np.float32)
            nudge = g.integers(-1, 2, 256)
            v = np.where(nudge > 0, np.nextafter(v, np.float32(np.inf)), v)
            v = np.where(nudge < 0, np.nextafter(v, np.float32(-np.inf)), v)
            v[0] = np.float32(127.0) * d
            X[r, b0:b0 + 256] = v
    Wq = orc.quantize(Q5_K, np.eye(cols, dtype=np.float32))
    Xq = orc.quantize(Q8_K, X)
    s = host(gq.block_sums_f32(Q5_K, dev(Wq), dev(X), cols, cols, 2))
    np.testing.assert_array_equal(s, orc.block_sums(Q5_K, Wq, Xq, cols, cols, 2))


def test_fused_f32_degenerate_vectors():
    """A zero vector (scale 0: every code 0), a constant one and tiny values."""
    rows, cols = 40, 2048
    W = inputs.normal(inputs.rng(8), (rows, cols), 0.02)
    X = inputs.normal(inputs.rng(9), (4, cols))
    X[0] = 0.0
    X[1] = 0.37
    X[2, :512] = 1e-30
    X[3, ::3] = -5.0
    Wq, Xq = orc.quantize(Q5_K, W), orc.quantize(Q8_K, X)
    s = host(gq.block_sums_f32(Q5_K, dev(Wq), dev(X), rows, cols, 4))
    np.testing.assert_array_equal(s, orc.block_sums(Q5_K, Wq, Xq, rows, cols, 4))
    y = host(gq.matmul_f32(Q5_K, dev(Wq), dev(X), rows, cols, 4))
    y_ref, T = orc.matmul_ref(Q5_K, Wq, Xq, rows, cols, 4)
    assert_close(y, y_ref, T)
    assert np.all(y[0] == 0.0)


def test_fused_f32_width_limit():
    """Wider vectors than the streaming kernel holds are refused (no fallback)."""
    Wd = torch.zeros(1, 19200 // 256 * 176, dtype=torch.uint8, device="cuda")
    x = torch.zeros(1, 19200, device="cuda")
    y = torch.empty(1, 1, device="cuda")
    with pytest.raises(gq.GQError):
        gq.gq_matmul_f32(Q5_K, Wd, x, y, 1, 19200, 1)


# ------------------------------------------- warp-level tensor-core path

SKINNY_SHAPES = [(96, 256, 1), (100, 512, 2), (200, 768, 8), (300, 1280, 9), (77, 256, 16), (513, 2048, 17),
                 (192, 1024, 32), (130, 2304, 33), (257, 4096, 64), (96, 3072, 5)]


@pytest.mark.parametrize("rows,cols,batch", SKINNY_SHAPES)
def test_skinny_sums_and_y(rows, cols, batch):
    """GQ_PATH_SKINNY for Q5_K (mma.sync on A = sc q - 1024, the even and
    odd sub-blocks in separate exact accumulators, 32 columns per launch):
    S1, S2 bit-identical to the oracle, y within the bar."""
    g = inputs.rng(rows * 13 + cols + batch)
    W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    X = inputs.normal(g, (batch, cols))
    Wq, Xq = orc.quantize(Q5_K, W), orc.quantize(Q8_K, X)
    Wd, Xd = dev(Wq), dev(Xq)
    s = host(gq.block_sums(Q5_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    np.testing.assert_array_equal(s, orc.block_sums(Q5_K, Wq, Xq, rows, cols, batch))
    y = host(gq.matmul(Q5_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    y_ref, T = orc.matmul_ref(Q5_K, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("batch", [3, 16, 40])
def test_skinny_sums_beyond_fp32_integers(batch):
    """Constant rows (sc = 63, codes 31) with single codes lowered, against
    constant activations (codes +-127) and a column of raw -128 codes: S1
    near 6.3e7, far above 2^24 and odd, still matches the oracle bit for
    bit (each half's partial sums stay within 2^24)."""
    rows, cols = 131, 512
    W = inputs.outlier_weights(inputs.rng(9), rows, cols, frac=0.001)
    W[0] = 1.0
    W[0, 5] = 0.97
    W[1] = 1.0
    W[2] = 1.0
    W[2, 1::2] = 0.97
    W[130] = 1.0
    W[130, 255] = 0.97
    X = inputs.normal(inputs.rng(10), (batch, cols))
    X[0] = 1.0
    X[1] = -1.0
    X[batch - 1] = 1.0
    Wq, Xq = orc.quantize(Q5_K, W), orc.quantize(Q8_K, X)
    blk = Xq.reshape(batch, cols // 256, 276)
    blk[2, :, 4:260] = 0x80
    blk[2, :, 260:276] = np.frombuffer(np.full(8, -128 * 32, np.int16).tobytes(), np.uint8)
    s_ref = orc.block_sums(Q5_K, Wq, Xq, rows, cols, batch)
    assert np.sum((np.abs(s_ref[..., 0]) > 2**25) & (s_ref[..., 0] % 2 != 0)) >= 2
    Wd, Xd = dev(Wq), dev(Xq)
    np.testing.assert_array_equal(host(gq.block_sums(Q5_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY)), s_ref)
    y = host(gq.matmul(Q5_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    y_ref, T = orc.matmul_ref(Q5_K, Wq, Xq, rows, cols, batch)
    assert_close(y, y_ref, T)


@pytest.mark.parametrize("batch", [8, 32, 64])
def test_skinny_full_size(batch):
    """14336 x 4096 (the batch-sweep shape); the oracle recomputes sampled
    rows from the same fp32 inputs."""
    rows, cols = 14336, 4096
    W, X = inputs.gemm_q4_k(0, rows, cols, batch)
    Wd = gq.quantize(Q5_K, dev(W))
    Xd = gq.quantize(Q8_K, dev(X))
    y = host(gq.matmul(Q5_K, Wd, Xd, rows, cols, batch, gq.PATH_SKINNY))
    g = np.random.Generator(np.random.PCG64(rows + batch))
    idx = np.unique(np.concatenate([[0, rows - 1], g.choice(rows, size=32, replace=False)]))
    Wq_s = orc.quantize(Q5_K, W[idx])
    assert host(Wd)[idx].tobytes() == Wq_s.tobytes()
    Xq = orc.quantize(Q8_K, X)
    y_ref, T = orc.matmul_ref(Q5_K, Wq_s, Xq, len(idx), cols, batch, nthreads=orc.max_threads())
    assert_close(y[:, idx], y_ref, T)


@pytest.mark.skipif(bool(os.environ.get("GQ_TC_MIN_BATCH")), reason="threshold overridden")
@pytest.mark.parametrize("rows,batch,want", [(14336, 3, "gemv"), (14336, 4, "skinny"), (8192, 70, "skinny"),
                                             (4096, 15, "gemv"), (4096, 16, "skinny"), (1024, 64, "gemv")])
def test_auto_dispatch(rows, batch, want):
    """gq_matmul for Q5_K: the warp-level kernel from batch 4 on matrices of
    8192 rows or more and from 16 on 2048 or more (32-column chunks beyond),
    the multi-vector GEMV otherwise; both are deterministic, so the AUTO
    result equals the chosen family's bit for bit."""
    cols = 512
    g = inputs.rng(rows + batch)
    Wd = gq.quantize(Q5_K, dev(inputs.normal(g, (rows, cols), 0.02)))
    Xd = gq.quantize(Q8_K, dev(inputs.normal(g, (batch, cols))))
    y = host(gq.matmul(Q5_K, Wd, Xd, rows, cols, batch))
    path = gq.PATH_SKINNY if want == "skinny" else gq.PATH_GEMV
    assert gq.gq_auto_path(Q5_K, rows, cols, batch) == path  # the host-side query agrees
    assert y.tobytes() == host(gq.matmul(Q5_K, Wd, Xd, rows, cols, batch, path)).tobytes()
