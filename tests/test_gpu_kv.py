"""GPU parity of the quantized KV cache ("llama.cpp 推理引擎" §3.7.3) against
the CPU oracle: the appended cache bytes bit-identical (and every other row
untouched), the scores within 1e-4 * sum|block terms| per output, and the
same scores as the GEMV of one head's rows."""
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


def filled_cache(t, n_heads, capacity, head_dim, n_fill, seed):
    """Oracle and GPU caches filled by appending n_fill positions (keys with a
    per-head scale spread and 0.1% outliers); unwritten rows hold 0xA5."""
    g = inputs.rng(seed)
    row_bytes = head_dim // 32 * orc.block_bytes(t)
    ref = np.full((n_heads, capacity, row_bytes), 0xA5, np.uint8)
    cache = dev(ref)
    scale = np.exp(g.uniform(np.log(0.25), np.log(4.0), (n_heads, 1))).astype(np.float32)
    for p in range(n_fill):
        x = inputs.normal(g, (n_heads, head_dim)) * scale
        hot = g.random(x.shape) < 0.001
        x = np.where(hot, 10.0 * x, x).astype(np.float32)
        orc.kv_append(t, x, ref, p)
        gq.gq_kv_append(t, dev(x), cache, n_heads, head_dim, capacity, p)
    return ref, cache


@pytest.mark.parametrize("t", [Q8_0, Q4_0])
@pytest.mark.parametrize("n_heads,capacity,head_dim", [(4, 64, 128), (3, 96, 64), (2, 32, 256), (5, 64, 32)])
def test_kv_append_bytes(t, n_heads, capacity, head_dim):
    ref, cache = filled_cache(t, n_heads, capacity, head_dim, n_fill=7, seed=capacity + head_dim)
    # and one position out of order, near the end of the cache
    g = inputs.rng(99)
    x = inputs.normal(g, (n_heads, head_dim))
    orc.kv_append(t, x, ref, capacity - 1)
    gq.gq_kv_append(t, dev(x), cache, n_heads, head_dim, capacity, capacity - 1)
    assert host(cache).tobytes() == ref.tobytes()


@pytest.mark.parametrize("t", [Q8_0, Q4_0])
@pytest.mark.parametrize("n_heads,capacity,head_dim,n_pos",
                         [(4, 64, 128, 1), (4, 64, 128, 31), (4, 64, 128, 64), (3, 320, 64, 289),
                          (2, 288, 256, 257), (6, 32, 32, 20), (1, 512, 96, 511)])
def test_kv_scores_vs_oracle(t, n_heads, capacity, head_dim, n_pos):
    ref, cache = filled_cache(t, n_heads, capacity, head_dim, n_fill=n_pos, seed=7 * n_pos + head_dim)
    g = inputs.rng(n_pos)
    q = inputs.normal(g, (n_heads, head_dim)) * 2.0
    S, T = orc.kv_scores_ref(t, ref, q, n_pos)
    s = host(gq.kv_scores(t, cache, dev(q), n_pos))
    assert s.shape == (n_heads, n_pos)
    assert_close(s, S, T)


@pytest.mark.parametrize("t", [Q8_0, Q4_0])
def test_kv_scores_equal_gemv_of_one_head(t):
    """Head h's scores are the product of its first n_pos key rows with q[h]
    (the GEMV path of the library) within the same bound."""
    n_heads, capacity, head_dim, n_pos = 2, 256, 256, 200
    ref, cache = filled_cache(t, n_heads, capacity, head_dim, n_fill=n_pos, seed=3)
    g = inputs.rng(4)
    q = inputs.normal(g, (n_heads, head_dim))
    s = host(gq.kv_scores(t, cache, dev(q), n_pos))
    S, T = orc.kv_scores_ref(t, ref, q, n_pos)
    for h in range(n_heads):
        W = cache[h, :n_pos].contiguous()
        y = host(gq.matmul_f32(t, W, dev(q[h:h + 1]), n_pos, head_dim, 1))
        assert_close(y[0], S[h], T[h])
        assert_close(s[h], S[h], T[h])


def test_kv_scores_full_size_sampled():
    """A 7B-shape cache (32 heads x 4096 positions x 128) in the launch shape
    the bench times, checked on sampled positions."""
    t, n_heads, capacity, head_dim = Q8_0, 32, 4096, 128
    g = inputs.rng(11)
    keys = torch.randn(capacity, n_heads, head_dim, device="cuda")
    cache = gq.kv_cache(t, n_heads, capacity, head_dim)
    for p in range(capacity):
        gq.gq_kv_append(t, keys[p], cache, n_heads, head_dim, capacity, p)
    q = inputs.normal(g, (n_heads, head_dim))
    s = host(gq.kv_scores(t, cache, dev(q), capacity))
    ch = host(cache)
    pick = g.choice(capacity, 24, replace=False)
    for h in (0, 13, 31):
        S, T = orc.kv_scores_ref(t, ch[h:h + 1, pick], q[h:h + 1], len(pick))
        assert_close(s[h, pick], S[0], T[0])
    # the cache bytes themselves: the appended rows equal the oracle's encoding
    kh = host(keys)
    for p in pick[:4]:
        np.testing.assert_array_equal(ch[:, p], orc.quantize(t, kh[p]).reshape(n_heads, -1))


def test_bounded_wait_runs_out_and_device_stays_usable():
    """Failure detection without a fault: with the test switch on, one warp
    per CTA arms its transfer barrier for its key span but issues no copy;
    its short bounded wait runs out with nothing in flight, the status word
    says so, and the next (normal) call on the same context is correct."""
    t, n_heads, capacity, head_dim, n_pos = Q8_0, 2, 64, 128, 64
    ref, cache = filled_cache(t, n_heads, capacity, head_dim, n_fill=n_pos, seed=5)
    q = inputs.normal(inputs.rng(6), (n_heads, head_dim))
    assert gq.gq_device_status(reset=True) == 0
    gq.gq_debug_kv_timeout(True)
    try:
        gq.kv_scores(t, cache, dev(q), n_pos)
        torch.cuda.synchronize()
        word = gq.gq_device_status(reset=True)
    finally:
        gq.gq_debug_kv_timeout(False)
    assert word & (1 << 2), word  # the KV transfer-timeout bit
    s = host(gq.kv_scores(t, cache, dev(q), n_pos))
    S, T = orc.kv_scores_ref(t, ref, q, n_pos)
    assert_close(s, S, T)
    assert gq.gq_device_status(reset=True) == 0
