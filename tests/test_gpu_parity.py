"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: quantized bytes and int32 block sums bit-identical; y within
1e-4 * sum|block terms| per output.  Inputs are seeded and synthetic; the
oracle always quantizes from the same fp32 arrays itself, so no oracle input
comes from the GPU.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle as orc  # noqa: E402
from block_quantized_gb300 import gq, inputs  # noqa: E402

pytestmark = pytest.mark.gpu

Q4_0, Q8_0, Q4_K, Q8_K = 0, 1, 2, 3
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


# ------------------------------------------------------------------ codecs

def codec_inputs(be):
    g = inputs.rng(5)
    parts = [
        inputs.normal(g, (37 * be,), 0.02),
        inputs.outlier_weights(g, 8, 4 * be, frac=0.01).reshape(-1),
        inputs.normal(g, (16 * be,)),
        np.abs(inputs.normal(g, (3 * be,))),
        -np.abs(inputs.normal(g, (3 * be,))),
        np.full(2 * be, 0.37, np.float32),
        np.zeros(2 * be, np.float32),
        inputs.normal(g, (3 * be,), 1e-6),
        inputs.normal(g, (2 * be,), 1e-9),
        inputs.normal(g, (2 * be,), 300.0),
    ]
    x = np.concatenate(parts).astype(np.float32)
    x[7] = 63.5  # exact ties in the first block
    x[8], x[9] = 1.25, -0.25
    return x


@pytest.mark.parametrize("t", [Q4_0, Q8_0, Q4_K, Q8_K])
def test_quantize_bit_exact(t):
    be = orc.block_elems(t)
    x = codec_inputs(be)
    ref = orc.quantize(t, x).reshape(-1)
    got = host(gq.quantize(t, dev(x)))
    assert got.tobytes() == ref.tobytes()


@pytest.mark.parametrize("t", [Q4_0, Q8_0, Q4_K, Q8_K])
@pytest.mark.parametrize("nblocks", [1, 3, 9, 1000])
def test_quantize_sizes(t, nblocks):
    be = orc.block_elems(t)
    x = inputs.normal(inputs.rng(nblocks), (nblocks * be,), 0.5)
    assert host(gq.quantize(t, dev(x))).tobytes() == orc.quantize(t, x).tobytes()


@pytest.mark.parametrize("t", [Q4_0, Q8_0, Q4_K, Q8_K])
def test_dequantize_bit_exact(t):
    be = orc.block_elems(t)
    x = codec_inputs(be)
    q = orc.quantize(t, x)
    ref = orc.dequantize(t, q, x.size)
    got = host(gq.dequantize(t, dev(q.reshape(-1)), x.size))
    assert got.view(np.uint32).tobytes() == ref.view(np.uint32).tobytes()


def test_quantize_empty_is_noop():
    x = torch.empty(0, device="cuda")
    out = torch.empty(0, dtype=torch.uint8, device="cuda")
    gq.gq_quantize_rows_async(Q8_0, x, out, 0)


# ----------------------------------------------------------------- product

def make_case(wtype, rows, cols, batch, seed=0, outliers=True):
    g = inputs.rng(seed)
    if outliers:
        W = inputs.outlier_weights(g, rows, cols, frac=0.001)
    else:
        W = inputs.normal(g, (rows, cols), 0.02)
    X = inputs.normal(g, (batch, cols))
    atype = orc.ACT_TYPE[wtype]
    Wq = orc.quantize(wtype, W)
    Xq = orc.quantize(atype, X)
    return W, X, Wq, Xq


SHAPES = [
    # rows, cols, batch -- several CTAs, a ragged row tail, chunk tails
    (1, 256, 1), (7, 256, 1), (8, 512, 1), (37, 1024, 1), (130, 4096, 1),
    (64, 11008, 1), (19, 2816, 3), (40, 4096, 2), (33, 768, 5), (24, 1280, 8),
    (17, 512, 13), (9, 4352, 16), (21, 1024, 65),
]


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0, Q4_K])
@pytest.mark.parametrize("rows,cols,batch", SHAPES)
def test_gemv_block_sums_and_y(wtype, rows, cols, batch):
    W, X, Wq, Xq = make_case(wtype, rows, cols, batch, seed=rows * 7 + cols + batch)
    # the GPU quantizes too: its bytes must equal the oracle's
    Wd = gq.quantize(wtype, dev(W))
    Xd = gq.quantize(orc.ACT_TYPE[wtype], dev(X))
    assert host(Wd).tobytes() == Wq.tobytes()
    assert host(Xd).tobytes() == Xq.tobytes()
    s_ref = orc.block_sums(wtype, Wq, Xq, rows, cols, batch)
    s = host(gq.block_sums(wtype, Wd, Xd, rows, cols, batch, gq.PATH_GEMV))
    np.testing.assert_array_equal(s, s_ref)
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    y = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_GEMV))
    assert_close(y, y_ref, T)


# Tall enough that the GEMV ring carries two or four whole rows per bulk copy
# (rows >= 2 x warps on the GPU), rows spanning several 16-super-block chunks,
# ragged last row groups, and batches through the multi-vector item path.
TALL_SHAPES = [(4867, 4096, 1), (4867, 4096, 5), (2435, 8192, 1), (2435, 8192, 3), (2435, 8192, 8)]


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0, Q4_K])
@pytest.mark.parametrize("rows,cols,batch", TALL_SHAPES)
def test_gemv_tall_whole_row_items(wtype, rows, cols, batch):
    W, X, Wq, Xq = make_case(wtype, rows, cols, batch, seed=rows + cols + 31 * batch, outliers=False)
    Wd, Xd = dev(Wq), dev(Xq)
    s = host(gq.block_sums(wtype, Wd, Xd, rows, cols, batch, gq.PATH_GEMV))
    np.testing.assert_array_equal(s, orc.block_sums(wtype, Wq, Xq, rows, cols, batch))
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert_close(host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_GEMV)), y_ref, T)


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("rows,cols,batch", [(5, 32, 1), (11, 96, 2), (9, 4128, 3)])
def test_gemv_unaligned_rows(wtype, rows, cols, batch):
    """cols % 256 != 0: rows are not 16-byte multiples (plain kernel)."""
    W, X, Wq, Xq = make_case(wtype, rows, cols, batch, seed=cols)
    s_ref = orc.block_sums(wtype, Wq, Xq, rows, cols, batch)
    s = host(gq.block_sums(wtype, dev(Wq), dev(Xq), rows, cols, batch, gq.PATH_GEMV))
    np.testing.assert_array_equal(s, s_ref)
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert_close(host(gq.matmul(wtype, dev(Wq), dev(Xq), rows, cols, batch)), y_ref, T)


def test_degenerate_blocks():
    """All-zero weights and activations, constant rows, extreme codes."""
    rows, cols = 16, 512
    W = np.zeros((rows, cols), np.float32)
    W[1] = 1.0
    W[2] = -3.0
    W[3, ::2] = 7.0
    W[4] = np.linspace(-1, 1, cols, dtype=np.float32)
    X = np.zeros((2, cols), np.float32)
    X[1] = np.linspace(-5, 5, cols, dtype=np.float32)
    for wtype in (Q4_0, Q8_0, Q4_K):
        Wq = orc.quantize(wtype, W)
        Xq = orc.quantize(orc.ACT_TYPE[wtype], X)
        assert host(gq.quantize(wtype, dev(W))).tobytes() == Wq.tobytes()
        s_ref = orc.block_sums(wtype, Wq, Xq, rows, cols, 2)
        np.testing.assert_array_equal(
            host(gq.block_sums(wtype, dev(Wq), dev(Xq), rows, cols, 2, gq.PATH_GEMV)), s_ref)
        y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, 2)
        y = host(gq.matmul(wtype, dev(Wq), dev(Xq), rows, cols, 2, gq.PATH_GEMV))
        assert np.all(y[0] == 0)
        assert_close(y, y_ref, T)


def test_zero_size_matmul_is_noop():
    y = torch.full((1, 4), 7.0, device="cuda")
    gq.gq_matmul(Q4_K, 0, 0, y, 4, 256, 0)
    assert host(y).tolist() == [[7.0] * 4]


# ------------------------------------------------ full-size configurations

def sampled_rows(rows, k, seed):
    g = np.random.Generator(np.random.PCG64(seed))
    r = np.sort(g.choice(rows, size=min(k, rows), replace=False))
    return np.unique(np.concatenate([[0, rows - 1], r]))


def check_full(wtype, W, X, rows, cols, batch, path, nsample=48):
    """GPU quantize + product at full size; the oracle recomputes sampled rows
    from the same fp32 inputs."""
    atype = orc.ACT_TYPE[wtype]
    Wd = gq.quantize(wtype, dev(W))
    Xd = gq.quantize(atype, dev(X))
    y = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, path))
    Xq = orc.quantize(atype, X)
    assert host(Xd).tobytes() == Xq.tobytes()
    idx = sampled_rows(rows, nsample, rows + batch)
    Wq_s = orc.quantize(wtype, W[idx])
    Wd_h = host(Wd)
    assert Wd_h[idx].tobytes() == Wq_s.tobytes()
    y_ref, T = orc.matmul_ref(wtype, Wq_s, Xq, len(idx), cols, batch)
    assert_close(y[:, idx], y_ref, T)


def test_config_q4_0_gemv_512x1024():
    W, x = inputs.gemv_q4_0(0)
    Wq = orc.quantize(Q4_0, W)
    xq = orc.quantize(Q8_0, x)
    assert host(gq.quantize(Q4_0, dev(W))).tobytes() == Wq.tobytes()
    s = host(gq.block_sums(Q4_0, dev(Wq), dev(xq), 512, 1024, 1, gq.PATH_GEMV))
    np.testing.assert_array_equal(s, orc.block_sums(Q4_0, Wq, xq, 512, 1024, 1))
    y_ref, T = orc.matmul_ref(Q4_0, Wq, xq, 512, 1024, 1)
    assert_close(host(gq.matmul(Q4_0, dev(Wq), dev(xq), 512, 1024, 1)), y_ref, T)


def test_config_q4_k_gemv_4096():
    W, x = inputs.gemv_q4_k(0)
    Wq = orc.quantize(Q4_K, W)
    xq = orc.quantize(Q8_K, x)
    Wd = gq.quantize(Q4_K, dev(W))
    assert host(Wd).tobytes() == Wq.tobytes()
    s = host(gq.block_sums(Q4_K, Wd, dev(xq), 4096, 4096, 1, gq.PATH_GEMV))
    np.testing.assert_array_equal(s, orc.block_sums(Q4_K, Wq, xq, 4096, 4096, 1))
    y_ref, T = orc.matmul_ref(Q4_K, Wq, xq, 4096, 4096, 1)
    assert_close(host(gq.matmul(Q4_K, Wd, dev(xq), 4096, 4096, 1)), y_ref, T)


@pytest.mark.parametrize("name", ["wq", "w1", "w2", "head"])
def test_config_decode_shapes(name):
    ws, x = inputs.decode_weights(0)
    W = ws[name]
    rows, cols = W.shape
    wtype = Q8_0 if name == "head" else Q4_K
    X = inputs.normal(inputs.rng(3), (1, cols))
    check_full(wtype, W, X, rows, cols, 1, gq.PATH_AUTO)


@pytest.mark.parametrize("batch", [1, 2, 4, 8, 16, 32, 64])
def test_config_batch_sweep_gemv(batch):
    W, X = inputs.gemm_q4_k(0, 14336, 4096, batch)
    check_full(Q4_K, W, X, 14336, 4096, batch, gq.PATH_GEMV, nsample=24)


# ------------------------------------------- fused activation quantize path

FUSED_SHAPES = [(1, 256, 1), (37, 1024, 1), (130, 4096, 1), (64, 11008, 1), (19, 2816, 3),
                (33, 768, 5), (24, 1280, 8), (9, 4352, 16)]


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0, Q4_K])
@pytest.mark.parametrize("rows,cols,batch", FUSED_SHAPES)
def test_fused_f32_matches_unfused_and_oracle(wtype, rows, cols, batch):
    W, X, Wq, Xq = make_case(wtype, rows, cols, batch, seed=3 * rows + cols + batch)
    Wd, Xf = dev(Wq), dev(X)
    Xd = gq.quantize(orc.ACT_TYPE[wtype], Xf)
    # integer sums of the fused path equal the oracle's
    s = host(gq.block_sums_f32(wtype, Wd, Xf, rows, cols, batch))
    np.testing.assert_array_equal(s, orc.block_sums(wtype, Wq, Xq, rows, cols, batch))
    # the fused result is the unfused result, bit for bit
    y_f = host(gq.matmul_f32(wtype, Wd, Xf, rows, cols, batch))
    y_u = host(gq.matmul(wtype, Wd, Xd, rows, cols, batch, gq.PATH_GEMV))
    assert y_f.view(np.uint32).tobytes() == y_u.view(np.uint32).tobytes()
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert_close(y_f, y_ref, T)


# 32-element formats: the fused quantizer takes eight blocks per warp pass,
# six passes per batch, two at a time; these pass counts (1, 9, 49, 51) leave
# a batch, or the second pass of a pair, empty
RAGGED_FUSED_SHAPES = [(2, 256, 3), (5, 2304, 2), (3, 12544, 1), (4, 13056, 9)]


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0])
@pytest.mark.parametrize("rows,cols,batch", RAGGED_FUSED_SHAPES)
def test_fused_f32_ragged_blocks(wtype, rows, cols, batch):
    test_fused_f32_matches_unfused_and_oracle(wtype, rows, cols, batch)


def tie_heavy_activations(cols, blk, seed):
    """fp32 rows whose codes sit on or next to rounding ties: per block the
    scale is either a power of two (ties exact) or arbitrary (quotients a few
    ulps from a half-integer), and most entries are (k + 1/2) * scale or one
    ulp to either side."""
    g = np.random.default_rng(seed)
    x = np.empty(cols, dtype=np.float32)
    for b0 in range(0, cols, blk):
        if (b0 // blk) % 2 == 0:
            d = np.float32(2.0 ** int(g.integers(-12, 3)))
        else:
            d = np.float32(g.uniform(0.01, 3.0) / 127.0)
        v = ((g.integers(-126, 126, blk) + 0.5) * d).astype(np.float32)
        nudge = g.integers(-1, 2, blk)
        v = np.where(nudge > 0, np.nextafter(v, np.float32(np.inf)), v)
        v = np.where(nudge < 0, np.nextafter(v, np.float32(-np.inf)), v)
        v[0] = np.float32(127.0) * d  # the block maximum fixes the scale
        x[b0:b0 + blk] = v
    return x


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0, Q4_K])
def test_fused_quantize_ties_match_oracle(wtype):
    """Identity weights make each block sum expose single activation codes,
    so the in-kernel quantizer is checked code by code on tie cases."""
    for cols in ((1024,) if wtype == Q4_K else (1024, 2304)):
        check_fused_ties(wtype, cols)


def check_fused_ties(wtype, cols):
    blk = 256 if wtype == Q4_K else 32
    X = np.stack([tie_heavy_activations(cols, blk, 40 + i) for i in range(2)])
    Wq = orc.quantize(wtype, np.eye(cols, dtype=np.float32))
    Xq = orc.quantize(orc.ACT_TYPE[wtype], X)
    s = host(gq.block_sums_f32(wtype, dev(Wq), dev(X), cols, cols, 2))
    np.testing.assert_array_equal(s, orc.block_sums(wtype, Wq, Xq, cols, cols, 2))
    # and the standalone quantizer gives the same bytes
    assert host(gq.quantize(orc.ACT_TYPE[wtype], dev(X))).tobytes() == Xq.tobytes()


@pytest.mark.parametrize("wtype", [Q4_0, Q8_0, Q4_K])
def test_w_static_flag_same_result(wtype):
    rows, cols, batch = 300, 4096, 2
    W, X, Wq, Xq = make_case(wtype, rows, cols, batch, seed=11)
    Wd, Xd = dev(Wq), dev(Xq)
    torch.cuda.synchronize()
    y0 = torch.empty(batch, rows, device="cuda")
    y1 = torch.empty(batch, rows, device="cuda")
    gq.gq_matmul_ex(wtype, Wd, Xd, y0, rows, cols, batch, gq.PATH_GEMV, 0)
    gq.gq_matmul_ex(wtype, Wd, Xd, y1, rows, cols, batch, gq.PATH_GEMV, gq.FLAG_W_STATIC)
    assert host(y0).view(np.uint32).tobytes() == host(y1).view(np.uint32).tobytes()
    y_ref, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert_close(host(y1), y_ref, T)


def test_weights_written_by_previous_kernel_are_read_after_it():
    """Without GQ_FLAG_W_STATIC, a product issued right after the kernel that
    writes W (its quantize) must see the new weights, repeatedly."""
    rows, cols = 2048, 4096
    g = inputs.rng(21)
    Wa = inputs.normal(g, (rows, cols), 0.02)
    Wb = inputs.normal(g, (rows, cols), 0.02)
    x = inputs.normal(g, (1, cols))
    Wd = torch.empty(rows, cols // 256 * 144, dtype=torch.uint8, device="cuda")
    Xd = gq.quantize(Q8_K, dev(x))
    Wa_d, Wb_d = dev(Wa), dev(Wb)
    y = torch.empty(1, rows, device="cuda")
    ref = {}
    for name, Wf in (("a", Wa), ("b", Wb)):
        Wq = orc.quantize(Q4_K, Wf)
        ref[name] = orc.matmul_ref(Q4_K, Wq, orc.quantize(Q8_K, x), rows, cols, 1)
    for it in range(6):
        name, src = ("a", Wa_d) if it % 2 == 0 else ("b", Wb_d)
        gq.gq_quantize_rows_async(Q4_K, src, Wd, rows * cols)
        gq.gq_matmul(Q4_K, Wd, Xd, y, rows, cols, 1)
        y_ref, T = ref[name]
        assert_close(host(y), y_ref, T)
