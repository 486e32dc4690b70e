"""Pins for the CPU oracle: values the pages print, closed forms, invariants,
special cases that reduce to a library routine, and brute force on tiny inputs.

None of the expected values here comes from the oracle itself or from the CUDA
path: they are the pages' numbers (tests/golden, each with its citation),
numpy's own fp16 conversion and float64/int64 matmul, or properties that hold
by the definition of the formats.
"""
import numpy as np
import pytest

import oracle as orc
from block_quantized_gb300 import inputs
from conftest import read_golden

Q4_0, Q8_0, Q4_K, Q8_K, Q6_K, Q5_K = orc.Q4_0, orc.Q8_0, orc.Q4_K, orc.Q8_K, orc.Q6_K, orc.Q5_K


def hexbytes(tokens):
    return np.array([int(t, 16) for t in tokens], dtype=np.uint8)


# --------------------------------------------------------------------------
# Block sizes ("llama.cpp 推理引擎" §5.3: 144 bits per 32 weights = 4.5 bpw;
# the format definition: 18 / 34 / 144 bytes; Q8_K 276 bytes by construction)
# --------------------------------------------------------------------------

def test_block_sizes():
    assert [orc.block_elems(t) for t in (Q4_0, Q8_0, Q4_K, Q8_K)] == [32, 32, 256, 256]
    assert [orc.block_bytes(t) for t in (Q4_0, Q8_0, Q4_K, Q8_K)] == [18, 34, 144, 276]
    assert orc.block_bytes(Q4_0) * 8 / 32 == 4.5
    assert orc.block_bytes(Q4_0) * 8 == 144
    assert orc.block_bytes(Q4_K) * 8 / 256 == 4.5
    # Q6_K: 256 six-bit codes (192 bytes) and one fp16 scale
    assert (orc.block_elems(Q6_K), orc.block_bytes(Q6_K)) == (256, 194)
    assert orc.block_bytes(Q6_K) == 256 * 6 // 8 + 2
    # Q5_K: the 144 Q4_K bytes plus one bit per element (5.5 bits per weight)
    assert (orc.block_elems(Q5_K), orc.block_bytes(Q5_K)) == (256, 176)
    assert orc.block_bytes(Q5_K) == orc.block_bytes(Q4_K) + 256 // 8
    for t in (Q4_0, Q8_0, Q4_K, Q8_K, Q6_K, Q5_K):
        x = np.zeros(orc.block_elems(t) * 3, np.float32)
        assert orc.quantize(t, x).shape == (3, orc.block_bytes(t))


# --------------------------------------------------------------------------
# Printed examples
# --------------------------------------------------------------------------

def test_q4_0_worked_example():
    g = read_golden("q4_0_worked_example.txt")
    x = np.zeros(32, np.float32)
    x[:5] = np.array(g["x"], dtype=np.float32)
    blk = orc.quantize(Q4_0, x)[0]
    assert blk.tobytes() == hexbytes(g["bytes"]).tobytes()
    # the scale printed is 0.5
    assert blk[:2].view(np.float16)[0] == np.float16(0.5)
    # codes: stored nibble minus 8, element 2j in the low nibble of byte j
    nib = np.empty(32, np.int32)
    nib[0::2] = blk[2:] & 0x0F
    nib[1::2] = blk[2:] >> 4
    assert list(nib[:5] - 8) == [int(v) for v in g["codes"]]
    xh = orc.dequantize(Q4_0, blk, 32)
    np.testing.assert_array_equal(xh[:5], np.array(g["dequant"], np.float32))
    np.testing.assert_allclose(np.abs(x[:5] - xh[:5]), np.array(g["abs_err"], np.float32),
                               atol=1e-6)
    assert np.all(xh[5:] == 0)


def test_rounding_illustration():
    g = read_golden("rounding_illustration.txt")
    x = np.zeros(256, np.float32)
    x[:4] = np.array(g["x"], dtype=np.float32)
    x[4] = np.float32(g["amax_pad"][0])
    blk = orc.quantize(Q8_K, x)[0]
    d = blk[:4].view(np.float32)[0]
    assert abs(d - 0.08) < 1e-7
    codes = blk[4:260].view(np.int8)
    assert list(codes[:4]) == [int(v) for v in g["codes"]]
    assert codes[4] == 127
    xh = orc.dequantize(Q8_K, blk, 256)
    np.testing.assert_allclose(xh[:4], np.array(g["dequant"], np.float32), atol=2e-7)


def test_q8_0_ties_round_half_away():
    g = read_golden("q8_0_ties.txt")
    x = np.zeros(32, np.float32)
    x[:5] = np.array(g["x"], dtype=np.float32)
    blk = orc.quantize(Q8_0, x)[0]
    assert blk.tobytes() == hexbytes(g["bytes"]).tobytes()
    assert list(blk[2:7].view(np.int8)) == [int(v) for v in g["codes"]]
    # the same ties through the fp32-scale block
    x8 = np.zeros(256, np.float32)
    x8[:5] = x[:5]
    b8 = orc.quantize(Q8_K, x8)[0]
    assert b8[:4].view(np.float32)[0] == np.float32(0.5)
    assert list(b8[4:9].view(np.int8)) == [127, 3, -3, 1, -1]


def test_q4_k_handmade_block():
    g = read_golden("q4_k_handmade.txt")
    k0 = np.array(g["sub0_k"], np.int64)
    k1 = np.array(g["sub1_k"], np.int64)
    k2 = np.array(g["sub2_k"], np.int64)
    x = np.zeros(256, np.float32)
    x[0:32] = (63 * k0 - 252) / 256.0
    x[32:64] = 5 * k1 / 256.0
    x[64:96] = -0.5 + k2 / 128.0
    blk = orc.quantize(Q4_K, x)[0]
    expect = np.concatenate([hexbytes(g["header"]), hexbytes(g["scales"]), hexbytes(g["qs0"]),
                             hexbytes(g["qs1"]), hexbytes(g["qs2"]), np.zeros(80, np.uint8)])
    assert blk.tobytes() == expect.tobytes()
    # every element lies on its grid, so the reconstruction is exact
    np.testing.assert_array_equal(orc.dequantize(Q4_K, blk, 256), x)


def test_q5_k_handmade_block():
    g = read_golden("q5_k_handmade.txt")
    r = np.arange(32)
    x = np.zeros(256, np.float32)
    x[0:32] = (63 * r - 504) / 512.0
    x[32:64] = 3 * (31 - r) / 512.0
    x[64:96] = -0.5 + ((7 * r) % 32) / 256.0
    blk = orc.quantize(Q5_K, x)[0]
    expect = np.concatenate([hexbytes(g["header"]), hexbytes(g["scales"]), hexbytes(g["qs0"]),
                             hexbytes(g["qs1"]), hexbytes(g["qs2"]), np.zeros(80, np.uint8),
                             hexbytes(g["qh0"]), hexbytes(g["qh1"]), hexbytes(g["qh2"]), np.zeros(20, np.uint8)])
    assert blk.tobytes() == expect.tobytes()
    # every element lies on its grid, so the reconstruction is exact
    np.testing.assert_array_equal(orc.dequantize(Q5_K, blk, 256), x)


def test_q5_k_ties_round_half_away():
    """Codes round half away from zero: in a sub-block with min 0 (m = 0) and
    step 3/512 (sc = 3, d = 2^-9 set by a second sub-block of range 1953/512),
    x = 0.5, 2.5 and 30.5 steps give codes 1, 3 and 31 (ties-to-even would
    give 0, 2 and 30).  Codes are read back through the exact reconstruction
    (x_hat = step * q when m = 0)."""
    r = np.arange(32)
    x = np.zeros(256, np.float32)
    x[1:4] = np.array([0.5, 2.5, 30.5], np.float32) * 3 / 512
    x[32:64] = (63 * r - 504) / 512.0
    blk = orc.quantize(Q5_K, x)[0]
    assert blk[:4].tobytes() == bytes([0x00, 0x18, 0x00, 0x24])
    q = orc.dequantize_f64(Q5_K, blk, 256)[:32] / (3 / 512)
    np.testing.assert_array_equal(q[:4], [0, 1, 3, 31])
    assert np.all(q[4:] == 0)


def test_q6_k_handmade_block():
    g = read_golden("q6_k_handmade.txt")
    q1 = np.array(g["q_first"], np.int64)
    q2 = np.array(g["q_second"], np.int64)
    x = np.concatenate([np.tile(q1, 32), np.tile(q2, 32)]).astype(np.float32) / 16.0
    blk = orc.quantize(Q6_K, x)[0]
    expect = np.concatenate([hexbytes(g["d"]),
                             np.tile(hexbytes(g["ql_first"]), 32), np.tile(hexbytes(g["ql_second"]), 32),
                             np.tile(hexbytes(g["qh_first"]), 32), np.tile(hexbytes(g["qh_second"]), 32)])
    assert blk.tobytes() == expect.tobytes()
    # every element is a multiple of the scale, so the reconstruction is exact
    np.testing.assert_array_equal(orc.dequantize(Q6_K, blk, 256), x)


def test_q6_k_ties_round_half_away():
    """Codes round half away from zero: with d = 1/16 (max|x| = 31/16), x = +-2.5 d
    gives +-3, x = +-0.5 d gives +-1 and 1.5 d gives 2 (ties-to-even would give
    +-2, 0 and 2).  Codes are read back through the exact reconstruction."""
    x = np.zeros(256, np.float32)
    x[0] = 31 / 16
    x[1:7] = np.array([2.5, -2.5, 0.5, -0.5, 1.5, -1.5], np.float32) / 16
    blk = orc.quantize(Q6_K, x)[0]
    assert blk[0] == 0x00 and blk[1] == 0x2C
    q = orc.dequantize_f64(Q6_K, blk, 256) * 16
    np.testing.assert_array_equal(q[:7], [31, 3, -3, 1, -1, 2, -2])
    assert np.all(q[7:] == 0)


# --------------------------------------------------------------------------
# fp16 converters: numpy's float16 cast is IEEE round-to-nearest-even
# --------------------------------------------------------------------------

def _f16_sweep():
    """fp32 inputs for the fp16 converters: every positive fp32 whose exponent
    lies in the window where fp16 rounding is non-trivial (2^-26 <= x < 2^16,
    all 2^23 mantissas of each of those 42 binades), plus seeded samples of
    the negatives, of the underflow region (incl. fp32 subnormals) and of the
    overflow region."""
    n = 1 << 23
    for e in range(101, 143):
        u = np.arange(e << 23, (e << 23) + n, dtype=np.uint32)
        yield u.view(np.float32)
    g = np.random.Generator(np.random.PCG64(1234))
    yield (g.integers(0, 1 << 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
           | np.uint32(0x80000000)).view(np.float32)
    yield g.integers(0, 101 << 23, size=1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)
    yield g.integers(143 << 23, 0x7F800001, size=1 << 20, dtype=np.uint64).astype(np.uint32).view(np.float32)


def test_f16_rn_sweep_vs_numpy():
    for x in _f16_sweep():
        got = orc.f16_rn(x)
        with np.errstate(over="ignore"):  # values past the fp16 range round to inf
            ref = x.astype(np.float16).view(np.uint16)
        nan = np.isnan(x)
        assert np.array_equal(got[~nan], ref[~nan])
        assert np.all((got[nan] & 0x7C00) == 0x7C00) and np.all((got[nan] & 0x3FF) != 0)


def test_f16_rn_special_values():
    x = np.array([0.0, -0.0, 1.0, 65504.0, 65519.99, 65520.0, 2.0 ** -24, 2.0 ** -25,
                  2.0 ** -25 * 1.0000001, 2.0 ** -14, 1e-30, -np.inf, 3.5 / 7], np.float32)
    with np.errstate(over="ignore"):  # 65520 rounds to inf
        ref = x.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(orc.f16_rn(x), ref)


def test_f16_ru_sweep_properties():
    """Round toward +inf: the result is >= v, and the next fp16 value below the
    result is < v (so it is the least fp16 value >= v)."""
    for x in _f16_sweep():
        x = x[np.isfinite(x)]
        h = orc.f16_ru(x)
        r = h.view(np.float16).astype(np.float32)
        assert np.all((r >= x) | (np.isinf(r) & (r > 0)))
        pos = (h & 0x8000) == 0
        pred = np.where(pos & (h != 0), h - 1, np.where(pos, 0x8001, h + 1)).astype(np.uint16)
        below = pred.view(np.float16).astype(np.float32)
        assert np.all(below < x)


def test_f16_ru_spot_values():
    assert orc.f16_ru(np.array([1.0], np.float32))[0] == 0x3C00
    assert orc.f16_ru(np.array([1.0000001], np.float32))[0] == 0x3C01
    assert orc.f16_ru(np.array([-1.0000001], np.float32))[0] == 0xBC00
    assert orc.f16_ru(np.array([1e-30], np.float32))[0] == 0x0001
    assert orc.f16_ru(np.array([70000.0], np.float32))[0] == 0x7C00
    assert orc.f16_ru(np.array([-70000.0], np.float32))[0] == 0xFBFF


# --------------------------------------------------------------------------
# Round-trip bounds (|x - x_hat| <= half the step) on the workload
# distributions and the degenerate blocks
# --------------------------------------------------------------------------

def _blocks_zoo(be, seed=1):
    g = inputs.rng(seed)
    rows = [
        inputs.normal(g, (64, 8 * be), 0.02),               # N(0, 0.02^2) weights
        inputs.outlier_weights(g, 16, 8 * be, frac=0.01),   # row spread + outliers
        inputs.normal(g, (16, 8 * be)),                     # N(0, 1) activations
        np.abs(inputs.normal(g, (4, 8 * be))),              # all positive
        -np.abs(inputs.normal(g, (4, 8 * be))),             # all negative
        np.full((2, 8 * be), 0.37, np.float32),             # all equal
        np.full((2, 8 * be), -2.5, np.float32),
        np.zeros((2, 8 * be), np.float32),                  # all zero
        inputs.normal(g, (4, 8 * be), 1e-6),                # tiny sigma: subnormal fp16 scales
        inputs.normal(g, (4, 8 * be), 1e-9),
    ]
    x = np.concatenate([r.reshape(-1, be) for r in rows])
    # a block with one huge outlier
    x[3, 5] = 40.0
    return np.ascontiguousarray(x.reshape(-1))


@pytest.mark.parametrize("t", [Q4_0, Q8_0, Q8_K, Q6_K])
def test_roundtrip_symmetric(t):
    be, bb = orc.block_elems(t), orc.block_bytes(t)
    x = _blocks_zoo(be)
    q = orc.quantize(t, x)
    xh = orc.dequantize(t, q, x.size).reshape(-1, be)
    xb = x.reshape(-1, be)
    if t == Q8_K:
        d = q[:, :4].copy().view(np.float32)[:, 0].astype(np.float64)
    else:
        d = q[:, :2].copy().view(np.float16)[:, 0].astype(np.float64)
    x64 = xb.astype(np.float64)
    err = np.abs(x64 - xh)
    amax = np.abs(xb).max(axis=1).astype(np.float64)
    # Within the code range the nearest code is at most d/2 away; a value
    # beyond the extreme code (possible when the fp16 scale rounded down, or
    # underflowed to 0 for a tiny block) is clipped, adding its excess.
    top_pos = {Q4_0: 7.0, Q6_K: 31.0}.get(t, 127.0) * d
    top_neg = {Q4_0: 8.0, Q6_K: 32.0}.get(t, 127.0) * d
    top = np.where(x64 >= 0, top_pos[:, None], top_neg[:, None])
    excess = np.maximum(0.0, np.abs(x64) - top)
    assert np.all(err <= d[:, None] / 2 * (1 + 1e-6) + excess + 1e-7 * amax[:, None])
    # with a normal fp16 scale the clipped excess is only the scale's rounding
    normal = d >= 2.0 ** -14
    assert np.all(excess[normal] <= amax[normal, None] * 2.0 ** -10)
    # max|x| maps to the extreme code for the 8-bit formats
    if t in (Q8_0, Q8_K):
        off = 2 if t == Q8_0 else 4
        codes = q[:, off:off + be].view(np.int8)
        nz = d >= (2.0 ** -14 if t == Q8_0 else 1e-30)   # normal scales only
        i = np.abs(xb).argmax(axis=1)
        assert np.all(np.abs(codes[np.arange(len(i)), i][nz]) == 127)
    if t == Q8_K:
        codes = q[:, 4:260].view(np.int8).astype(np.int32)
        bs = q[:, 260:276].copy().view(np.int16).astype(np.int32)
        np.testing.assert_array_equal(bs, codes.reshape(-1, 8, 32).sum(axis=2))
    if t == Q6_K:
        # codes read straight from the bytes: with a normal fp16 scale max|x|
        # maps to +-31 and code 0 (q = -32) never occurs; a zero block stores 32
        lo = np.stack([q[:, 2:130] & 15, q[:, 2:130] >> 4], axis=2).reshape(-1, 256)
        hi = np.stack([(q[:, 130:194] >> (2 * k)) & 3 for k in range(4)], axis=2).reshape(-1, 256)
        c = (lo | (hi << 4)).astype(np.int64)
        np.testing.assert_array_equal(c - 32, np.round(xh / np.where(d == 0, 1, d)[:, None]))
        nz = d >= 2.0 ** -14
        i = np.abs(xb).argmax(axis=1)
        assert np.all(np.abs(c[np.arange(len(i)), i][nz] - 32) == 31)
        assert np.all(c[d == 0] == 32)
        assert c[nz].min() >= 1


def _q4k_fields(q):
    """Decode d, dmin and the 6-bit fields of Q4_K blocks straight from the bytes."""
    d = q[:, 0:2].copy().view(np.float16)[:, 0].astype(np.float64)
    dmin = q[:, 2:4].copy().view(np.float16)[:, 0].astype(np.float64)
    v = np.zeros(len(q), dtype=object)
    for i in range(12):
        v = v + (q[:, 4 + i].astype(object) << (8 * i))
    f = np.array([[(int(vv) >> (6 * k)) & 63 for k in range(16)] for vv in v], np.int64)
    return d, dmin, f[:, :8], f[:, 8:]


@pytest.mark.parametrize("t,qmax", [(Q4_K, 15), (Q5_K, 31)])
def test_roundtrip_q4_k(t, qmax):
    x = _blocks_zoo(256)
    q = orc.quantize(t, x)
    xh = orc.dequantize(t, q, x.size).reshape(-1, 8, 32).astype(np.float64)
    xb = x.reshape(-1, 8, 32).astype(np.float64)
    d, dmin, sc, m = _q4k_fields(q)
    step = d[:, None] * sc
    err = np.abs(xb - xh)
    scale = np.abs(xb).max(axis=(1, 2))
    bound = step / 2 * (1 + 1e-6) + 1e-6 * scale[:, None] + 1e-30
    assert np.all(err <= bound[:, :, None])
    # the reconstruction is d*sc*q - dmin*m: recover q and check it is an integer in [0, qmax]
    with np.errstate(invalid="ignore", divide="ignore"):
        qq = (xh + (dmin[:, None] * m)[:, :, None]) / step[:, :, None]
    ok = step > 0
    assert np.all(np.abs(qq[ok] - np.round(qq[ok])) < 1e-3)
    assert np.all((np.round(qq[ok]) >= 0) & (np.round(qq[ok]) <= qmax))
    if t == Q5_K:
        # the codes straight from the bytes (low nibbles and the fifth-bit
        # plane as the format defines them) are the recovered codes
        e = np.arange(256)
        nib = np.where(e % 2 == 1, q[:, 16 + e // 2] >> 4, q[:, 16 + e // 2] & 15).astype(np.int64)
        j, tt, i, p = e // 32, (e % 32) // 8, (e % 8) // 2, e % 2
        hb = (q[:, 144 + 4 * j + i] >> (2 * tt + p)) & 1
        codes = (nib | (hb.astype(np.int64) << 4)).reshape(-1, 8, 32)
        np.testing.assert_array_equal(codes[ok], np.round(qq[ok]).astype(np.int64))


def _k_fields(q):
    """d, dmin and the 6-bit fields of Q4_K / Q5_K blocks, from the bytes."""
    return _q4k_fields(q)


def _sub_sse(x, xh):
    """Squared reconstruction error per sub-block, float64: [blocks, 8]."""
    return ((x.reshape(-1, 8, 32).astype(np.float64) - xh.reshape(-1, 8, 32)) ** 2).sum(axis=2)


@pytest.mark.parametrize("t", [Q4_K, Q5_K])
def test_errmin_never_worse_and_same_format(t):
    """The error-minimizing encoder keeps the min/max fit's d and dmin (bytes
    0..3) and never reconstructs a sub-block worse than the min/max fit
    (float64 error, up to the fp32 rounding of the encoder's own measure)."""
    x = np.concatenate([_blocks_zoo(256), inputs.outlier_weights(inputs.rng(5), 32, 2048, frac=0.01).reshape(-1)])
    a, b = orc.quantize(t, x), orc.quantize(t, x, errmin=True)
    assert a.shape == b.shape
    np.testing.assert_array_equal(a[:, :4], b[:, :4])
    ea = _sub_sse(x, orc.dequantize_f64(t, a, x.size))
    eb = _sub_sse(x, orc.dequantize_f64(t, b, x.size))
    assert np.all(eb <= ea * (1 + 1e-5) + 1e-30)
    assert eb.sum() < 0.9 * ea.sum()  # and it does find better pairs on these inputs


def _round_half_away(v):
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


@pytest.mark.parametrize("t,qmax", [(Q4_K, 15), (Q5_K, 31)])
def test_errmin_window_bruteforce(t, qmax):
    """Brute force of the search's definition, in float64: for every
    sub-block, every (sc, m) within 4 of the min/max fit's pair (clipped to
    0..63) with its nearest codes; the encoder's choice lies in that window
    and is its minimum up to fp32 rounding."""
    x = inputs.outlier_weights(inputs.rng(6), 4, 512, frac=0.02).reshape(-1)
    a, b = orc.quantize(t, x), orc.quantize(t, x, errmin=True)
    d, dmin, sc0, m0 = _k_fields(a)
    _, _, sc1, m1 = _k_fields(b)
    eb = _sub_sse(x, orc.dequantize_f64(t, b, x.size))
    xb = x.reshape(-1, 8, 32).astype(np.float64)
    for blk in range(xb.shape[0]):
        for j in range(8):
            assert abs(sc1[blk, j] - sc0[blk, j]) <= 4 and abs(m1[blk, j] - m0[blk, j]) <= 4
            best = np.inf
            for sc in range(max(0, sc0[blk, j] - 4), min(63, sc0[blk, j] + 4) + 1):
                for m in range(max(0, m0[blk, j] - 4), min(63, m0[blk, j] + 4) + 1):
                    step, base = d[blk] * sc, -dmin[blk] * m
                    qv = np.zeros(32) if step == 0 else np.clip(_round_half_away((xb[blk, j] - base) / step), 0, qmax)
                    best = min(best, ((xb[blk, j] - (step * qv + base)) ** 2).sum())
            assert eb[blk, j] <= best * (1 + 1e-5) + 1e-30


def test_errmin_hand_case():
    """A sub-block on the grid of step 2^-8 * 5 (codes 0..15, min 0) whose
    largest element sits a hair above 15 steps: the min/max fit rounds the
    scale up to sc = 6 (every other element then falls between codes), while
    sc = 5 reconstructs all but that element exactly.  Sub-block 1 fixes
    d = 2^-8 (range 945/256)."""
    x = np.zeros(256, np.float32)
    c = np.array([0, 15, 3, 8, 1, 12, 7, 4] * 4, np.float32)
    x[0:32] = c * 5 / 256
    x[1] = np.float32(75.01 / 256)
    x[32:64] = np.arange(32, dtype=np.float32) * 945 / 256 / 31
    a, b = orc.quantize(Q4_K, x), orc.quantize(Q4_K, x, errmin=True)
    d, _, sc0, _ = _k_fields(a)
    _, _, sc1, _ = _k_fields(b)
    assert d[0] == 2.0 ** -8 and sc0[0, 0] == 6 and sc1[0, 0] == 5
    xh = orc.dequantize_f64(Q4_K, b, 256)
    others = np.r_[0, 2:32]
    np.testing.assert_array_equal(xh[others], x[others].astype(np.float64))
    assert _sub_sse(x, xh)[0, 0] < 1e-3 * _sub_sse(x, orc.dequantize_f64(Q4_K, a, 256))[0, 0]


def test_nonfinite_rejected():
    x = np.zeros(32, np.float32)
    x[3] = np.nan
    with pytest.raises(ValueError):
        orc.quantize(Q8_0, x)


# --------------------------------------------------------------------------
# The product: brute force in float64 on tiny inputs, and exact integer cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("wtype", [Q4_0, Q8_0, Q4_K, Q6_K, Q5_K])
@pytest.mark.parametrize("rows,cols,batch", [(1, 256, 1), (5, 512, 3), (7, 1024, 2)])
def test_matmul_ref_vs_bruteforce(wtype, rows, cols, batch):
    atype = orc.ACT_TYPE[wtype]
    g = inputs.rng(100 + rows)
    W = inputs.outlier_weights(g, rows, cols, frac=0.01)
    X = inputs.normal(g, (batch, cols))
    Wq = orc.quantize(wtype, W)
    Xq = orc.quantize(atype, X)
    Wd = orc.dequantize_f64(wtype, Wq, W.size).reshape(rows, cols)
    Xd = orc.dequantize_f64(atype, Xq, X.size).reshape(batch, cols)
    # the fp32 reconstruction is the exact one rounded once
    np.testing.assert_array_equal(orc.dequantize(wtype, Wq, W.size).reshape(rows, cols),
                                  Wd.astype(np.float32))
    # the brute-force double dot of dequantized values, by a naive loop ...
    naive = np.zeros((batch, rows))
    for b in range(batch):
        for r in range(rows):
            s = 0.0
            for i in range(cols):
                s += Wd[r, i] * Xd[b, i]
            naive[b, r] = s
    # ... and by numpy's float64 matmul
    lib = Xd @ Wd.T
    y, T = orc.matmul_ref(wtype, Wq, Xq, rows, cols, batch)
    assert np.all(T > 0)
    np.testing.assert_allclose(y, naive, rtol=0, atol=1e-12 * T.max())
    np.testing.assert_allclose(y, lib, rtol=0, atol=1e-12 * T.max())


def _q8_0_blocks_d1(codes):
    """Q8_0 blocks with fp16 scale 1.0 (0x3C00) holding the given int8 codes."""
    nb = codes.size // 32
    q = np.zeros((nb, 34), np.uint8)
    q[:, 0] = 0x00
    q[:, 1] = 0x3C
    q[:, 2:] = codes.reshape(nb, 32).astype(np.int8).view(np.uint8)
    return q


def test_integer_special_case_q8_0():
    """With every scale 1, the product is a pure integer matvec: numpy int64."""
    g = inputs.rng(7)
    rows, cols, batch = 9, 512, 4
    Wc = g.integers(-127, 128, size=(rows, cols))
    Xc = g.integers(-127, 128, size=(batch, cols))
    y, _ = orc.matmul_ref(Q8_0, _q8_0_blocks_d1(Wc), _q8_0_blocks_d1(Xc), rows, cols, batch)
    np.testing.assert_array_equal(y, (Xc @ Wc.T).astype(np.float64))
    s = orc.block_sums(Q8_0, _q8_0_blocks_d1(Wc), _q8_0_blocks_d1(Xc), rows, cols, batch)
    ref = (Xc.reshape(batch, 1, cols // 32, 32) * Wc.reshape(1, rows, cols // 32, 32)).sum(-1)
    np.testing.assert_array_equal(s, ref)


def test_integer_special_case_q4_0():
    """Q4_0 with scale 1: codes c in [0, 15] stand for c - 8."""
    g = inputs.rng(8)
    rows, cols, batch = 6, 256, 3
    C = g.integers(0, 16, size=(rows, cols))
    Xc = g.integers(-127, 128, size=(batch, cols))
    nb = cols // 32
    Wq = np.zeros((rows * nb, 18), np.uint8)
    Wq[:, 1] = 0x3C
    Cb = C.reshape(rows * nb, 32)
    Wq[:, 2:] = (Cb[:, 0::2] | (Cb[:, 1::2] << 4)).astype(np.uint8)
    y, _ = orc.matmul_ref(Q4_0, Wq, _q8_0_blocks_d1(Xc), rows, cols, batch)
    np.testing.assert_array_equal(y, (Xc @ (C - 8).T).astype(np.float64))


def test_integer_special_case_q4_k():
    """Q4_K with d = dmin = 1 and a Q8_K scale of 1: y = sum sc*q*a - m*a exactly."""
    g = inputs.rng(9)
    rows, cols, batch = 4, 512, 2
    nsb = cols // 256
    Q = g.integers(0, 16, size=(rows, cols))
    SC = g.integers(0, 64, size=(rows, nsb, 8))
    M = g.integers(0, 64, size=(rows, nsb, 8))
    A = g.integers(-127, 128, size=(batch, cols))
    Wq = np.zeros((rows, nsb, 144), np.uint8)
    Wq[:, :, 1] = 0x3C
    Wq[:, :, 3] = 0x3C
    for r in range(rows):
        for s in range(nsb):
            v = 0
            for k in range(8):
                v |= int(SC[r, s, k]) << (6 * k)
                v |= int(M[r, s, k]) << (6 * (k + 8))
            Wq[r, s, 4:16] = np.frombuffer(v.to_bytes(12, "little"), np.uint8)
            qb = Q[r, 256 * s:256 * (s + 1)]
            Wq[r, s, 16:] = (qb[0::2] | (qb[1::2] << 4)).astype(np.uint8)
    Xq = np.zeros((batch, nsb, 276), np.uint8)
    Xq[:, :, 0:4] = np.frombuffer(np.float32(1.0).tobytes(), np.uint8)
    Ab = A.reshape(batch, nsb, 256)
    Xq[:, :, 4:260] = Ab.astype(np.int8).view(np.uint8)
    Xq[:, :, 260:276] = Ab.reshape(batch, nsb, 8, 32).sum(-1).astype(np.int16).view(np.uint8)
    # dense reconstruction in integers: w = sc*q - m
    Wint = (SC.repeat(32, axis=2).reshape(rows, cols) * Q - M.repeat(32, axis=2).reshape(rows, cols))
    y, _ = orc.matmul_ref(Q4_K, Wq.reshape(rows, -1), Xq.reshape(batch, -1), rows, cols, batch)
    np.testing.assert_array_equal(y, (A @ Wint.T).astype(np.float64))
    s = orc.block_sums(Q4_K, Wq.reshape(rows, -1), Xq.reshape(batch, -1), rows, cols, batch)
    S1 = np.einsum("rsk,brski->brs", SC, Q.reshape(1, rows, nsb, 8, 32) * Ab.reshape(batch, 1, nsb, 8, 32))
    S2 = np.einsum("rsk,bsk->brs", M, Ab.reshape(batch, nsb, 8, 32).sum(-1))
    np.testing.assert_array_equal(s[..., 0], S1)
    np.testing.assert_array_equal(s[..., 1], S2)


def test_integer_special_case_q6_k():
    """Q6_K with d = 1 and a Q8_K scale of 1: codes c in [0, 63] stand for c - 32,
    so y and the per-block sums are a pure integer product (numpy int64).  The
    blocks are packed here from the format definition, independently of the
    oracle's encoder."""
    g = inputs.rng(9)
    rows, cols, batch = 5, 768, 3
    nb = cols // 256
    C = g.integers(0, 64, size=(rows, cols))
    Xc = g.integers(-127, 128, size=(batch, cols))
    Cb = C.reshape(rows * nb, 256)
    Wq = np.zeros((rows * nb, 194), np.uint8)
    Wq[:, 1] = 0x3C                                          # fp16 1.0
    Wq[:, 2:130] = ((Cb[:, 0::2] & 15) | ((Cb[:, 1::2] & 15) << 4)).astype(np.uint8)
    top = Cb >> 4
    Wq[:, 130:194] = (top[:, 0::4] | (top[:, 1::4] << 2) | (top[:, 2::4] << 4) |
                      (top[:, 3::4] << 6)).astype(np.uint8)
    Xb = Xc.reshape(batch * nb, 256)
    Xq = np.zeros((batch * nb, 276), np.uint8)
    Xq[:, 0:4] = np.frombuffer(np.float32(1.0).tobytes(), np.uint8)
    Xq[:, 4:260] = Xb.astype(np.int8).view(np.uint8)
    Xq[:, 260:276] = Xb.reshape(-1, 8, 32).sum(-1).astype(np.int16).view(np.uint8)
    y, _ = orc.matmul_ref(Q6_K, Wq.reshape(rows, -1), Xq.reshape(batch, -1), rows, cols, batch)
    np.testing.assert_array_equal(y, (Xc @ (C - 32).T).astype(np.float64))
    s = orc.block_sums(Q6_K, Wq.reshape(rows, -1), Xq.reshape(batch, -1), rows, cols, batch)
    ref = (Xc.reshape(batch, 1, nb, 256) * (C - 32).reshape(1, rows, nb, 256)).sum(-1)
    np.testing.assert_array_equal(s, ref)


def test_integer_special_case_q5_k():
    """Q5_K with d = dmin = 1 and a Q8_K scale of 1: codes q in [0, 31], so
    y = sum (sc*q - m)*a and the sums S1 = sum_j sc_j s_j, S2 = sum_j m_j t_j
    are pure integers (numpy int64).  The blocks are packed here from the
    format definition (low nibbles in the Q4_0 order; fifth bit of element
    32j + 8t + 2i + p in bit 2t + p of byte 144 + 4j + i), independently of the
    oracle's encoder."""
    g = inputs.rng(10)
    rows, cols, batch = 4, 512, 3
    nsb = cols // 256
    Q = g.integers(0, 32, size=(rows, cols))
    SC = g.integers(0, 64, size=(rows, nsb, 8))
    M = g.integers(0, 64, size=(rows, nsb, 8))
    A = g.integers(-127, 128, size=(batch, cols))
    Wq = np.zeros((rows, nsb, 176), np.uint8)
    Wq[:, :, 1] = 0x3C
    Wq[:, :, 3] = 0x3C
    for r in range(rows):
        for s in range(nsb):
            v = 0
            for k in range(8):
                v |= int(SC[r, s, k]) << (6 * k)
                v |= int(M[r, s, k]) << (6 * (k + 8))
            Wq[r, s, 4:16] = np.frombuffer(v.to_bytes(12, "little"), np.uint8)
            qb = Q[r, 256 * s:256 * (s + 1)]
            Wq[r, s, 16:144] = ((qb[0::2] & 15) | ((qb[1::2] & 15) << 4)).astype(np.uint8)
            for e in range(256):
                if qb[e] >> 4:
                    j, t, i, p = e // 32, (e % 32) // 8, (e % 8) // 2, e % 2
                    Wq[r, s, 144 + 4 * j + i] |= 1 << (2 * t + p)
    Xq = np.zeros((batch, nsb, 276), np.uint8)
    Xq[:, :, 0:4] = np.frombuffer(np.float32(1.0).tobytes(), np.uint8)
    Ab = A.reshape(batch, nsb, 256)
    Xq[:, :, 4:260] = Ab.astype(np.int8).view(np.uint8)
    Xq[:, :, 260:276] = Ab.reshape(batch, nsb, 8, 32).sum(-1).astype(np.int16).view(np.uint8)
    Wint = (SC.repeat(32, axis=2).reshape(rows, cols) * Q - M.repeat(32, axis=2).reshape(rows, cols))
    y, _ = orc.matmul_ref(Q5_K, Wq.reshape(rows, -1), Xq.reshape(batch, -1), rows, cols, batch)
    np.testing.assert_array_equal(y, (A @ Wint.T).astype(np.float64))
    s = orc.block_sums(Q5_K, Wq.reshape(rows, -1), Xq.reshape(batch, -1), rows, cols, batch)
    S1 = np.einsum("rsk,brski->brs", SC, Q.reshape(1, rows, nsb, 8, 32) * Ab.reshape(batch, 1, nsb, 8, 32))
    S2 = np.einsum("rsk,bsk->brs", M, Ab.reshape(batch, nsb, 8, 32).sum(-1))
    np.testing.assert_array_equal(s[..., 0], S1)
    np.testing.assert_array_equal(s[..., 1], S2)


def test_tolerance_scale_is_sum_of_magnitudes():
    """T is at least |y| (triangle inequality) and equals |y| when every term
    has the same sign (all-positive weights and activations, Q8_0 x Q8_0)."""
    g = inputs.rng(11)
    W = np.abs(inputs.normal(g, (3, 256)))
    X = np.abs(inputs.normal(g, (2, 256)))
    y, T = orc.matmul_ref(Q8_0, orc.quantize(Q8_0, W), orc.quantize(Q8_0, X), 3, 256, 2)
    np.testing.assert_allclose(T, np.abs(y), rtol=1e-15)
    W2 = inputs.normal(g, (3, 256))
    y2, T2 = orc.matmul_ref(Q8_0, orc.quantize(Q8_0, W2), orc.quantize(Q8_0, X), 3, 256, 2)
    assert np.all(T2 >= np.abs(y2))


@pytest.mark.parametrize("t", [Q4_0, Q8_0, Q4_K, Q8_K, Q6_K, Q5_K])
def test_multithreaded_quantize_equals_blockwise(t):
    """The row-parallel quantizer used for timing is the pinned one, row by row."""
    be = orc.block_elems(t)
    x = inputs.outlier_weights(inputs.rng(17), 33, 4 * be, frac=0.01)
    np.testing.assert_array_equal(orc.quantize_rows_mt(t, x, 4), orc.quantize(t, x))


# --------------------------------------------------------------------------
# Quantized KV cache: append is the block encoding written at one position;
# the scores are the dot of dequantized keys and dequantized query
# --------------------------------------------------------------------------

@pytest.mark.parametrize("t", [Q8_0, Q4_0])
def test_kv_append_writes_one_row_per_head(t):
    g = inputs.rng(7)
    n_heads, capacity, head_dim = 3, 32, 64
    cache = np.full((n_heads, capacity, head_dim // 32 * orc.block_bytes(t)), 0xA5, np.uint8)
    before = cache.copy()
    x = inputs.normal(g, (n_heads, head_dim))
    orc.kv_append(t, x, cache, 5)
    for h in range(n_heads):
        # the row round-trips within half a step of its block scale ...
        xd = orc.dequantize_f64(t, cache[h, 5], head_dim)
        for b in range(head_dim // 32):
            blk = x[h, 32 * b:32 * b + 32].astype(np.float64)
            d = np.abs(blk).max() / (127.0 if t == Q8_0 else 7.0)
            # the fp16 rounding of d moves a step by at most 2^-11 relative
            assert np.all(np.abs(xd[32 * b:32 * b + 32] - blk) <= d * (0.5 + 2.0 ** -10))
        # ... and every other row is untouched
        np.testing.assert_array_equal(np.delete(cache[h], 5, axis=0), np.delete(before[h], 5, axis=0))


@pytest.mark.parametrize("t", [Q8_0, Q4_0])
def test_kv_scores_vs_bruteforce(t):
    g = inputs.rng(8)
    n_heads, capacity, head_dim, n_pos = 3, 64, 96, 37
    cache = np.zeros((n_heads, capacity, head_dim // 32 * orc.block_bytes(t)), np.uint8)
    # per-head scale spread so a head mix-up cannot hide
    for p in range(n_pos):
        orc.kv_append(t, inputs.normal(g, (n_heads, head_dim)) * np.array([[0.5], [1.0], [4.0]]), cache, p)
    q = inputs.normal(g, (n_heads, head_dim)) * np.array([[3.0], [0.25], [1.0]])
    S, T = orc.kv_scores_ref(t, cache, q, n_pos)
    for h in range(n_heads):
        K = np.stack([orc.dequantize_f64(t, cache[h, p], head_dim) for p in range(n_pos)])
        qd = orc.dequantize_f64(Q8_0, orc.quantize(Q8_0, q[h]), head_dim)
        naive = np.array([sum(K[p, i] * qd[i] for i in range(head_dim)) for p in range(n_pos)])
        assert np.all(T[h] > 0)
        np.testing.assert_allclose(S[h], naive, rtol=0, atol=1e-12 * T[h].max())
