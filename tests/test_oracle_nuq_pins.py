"""Pins of the NUQ (Lloyd-Max) oracle against facts fixed outside the oracle.

Source: "KVQuant-NUQ" (VeloxQuant-MLX docs), How it works: quantile-seeded
Lloyd-Max levels, nearest-level codes, rank-based outlier isolation; Max's
optimal quantizer for the Gaussian is the classical fixed point of the same
iteration.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def distortion64(x, lev):
    x = x.astype(np.float64)
    lev = np.asarray(lev, dtype=np.float64)
    return float(np.min((x[:, None] - lev[None, :]) ** 2, axis=1).sum())


def test_outlier_count_rounds_half_up():
    # k = floor(f * n + 0.5) with f the fp32 config value, evaluated in double
    assert oracle.outlier_count(0.01, 4095) == 41     # 40.95 + 0.5
    assert oracle.outlier_count(0.01, 128) == 1       # 1.28 + 0.5
    assert oracle.outlier_count(0.01, 49) == 0        # 0.49 + 0.5
    assert oracle.outlier_count(0.25, 2) == 1         # exactly 0.5 + 0.5: half rounds up
    assert oracle.outlier_count(0.25, 6) == 2         # 1.5 + 0.5
    assert oracle.outlier_count(0.25, 5) == 1         # 1.25 + 0.5
    assert oracle.outlier_count(0.0, 4095) == 0
    # 0.01 is not exact in binary: fp32(0.01) * 50 = 0.49999999..., so k = 0
    assert oracle.outlier_count(0.01, 50) == 0


def test_quantile_init_positions():
    # level i = sorted[floor((2i+1) n / (2L))]
    lev, _, nf = oracle.nuq_fit(np.arange(16, dtype=np.float32)[::-1].copy(), 8, 0)
    assert nf == 16 and lev.tolist() == [1, 3, 5, 7, 9, 11, 13, 15]
    lev, _, _ = oracle.nuq_fit(np.arange(10, dtype=np.float32), 4, 0)
    assert lev.tolist() == [1, 3, 6, 8]               # floor(10/8), floor(30/8), floor(50/8), floor(70/8)


def test_r32_order_differs_from_sequential():
    # lane 0 holds positions 0 and 32 (1e8 - 1e8 = 0), lane 1 holds the 1.0:
    # R32 gives 1.0, a sequential fp32 sum gives 0.0
    x = np.zeros(64, dtype=np.float32)
    x[0], x[1], x[32] = 1e8, 1.0, -1e8
    assert oracle.r32_sum(x) == 1.0
    seq = np.float32(0)
    for v in x:
        seq = np.float32(seq + v)
    assert seq == 0.0


def test_lloyd_distortion_never_increases():
    g = np.random.default_rng(7)
    x = g.standard_t(4.0, size=2000).astype(np.float32)
    prev = None
    for it in range(0, 12):
        lev, _, _ = oracle.nuq_fit(x, 8, it)
        d = distortion64(x, lev)
        if prev is not None:
            assert d <= prev * (1 + 1e-6), (it, d, prev)
        prev = d
        assert np.all(np.diff(lev) >= 0), lev     # levels stay sorted


def test_few_distinct_values_reconstruct_exactly():
    g = np.random.default_rng(3)
    vals = np.array([-2.5, -0.75, 0.125, 1.0, 3.5], dtype=np.float32)   # fp16-exact
    x = g.choice(vals, size=300).astype(np.float32)
    _, lut, _ = oracle.nuq_fit(x, 8, 8)
    codes = oracle.nuq_assign(x, lut)
    assert np.array_equal(f16(lut)[codes], x)


def test_max_gaussian_eight_level_optimum():
    # Max (1960): the 8-level MSE-optimal quantizer of N(0,1) has outputs
    # +-0.2451, +-0.7560, +-1.3439, +-2.1519
    x = np.random.default_rng(11).standard_normal(200_000).astype(np.float32)
    lev, _, _ = oracle.nuq_fit(x, 8, 80)
    want = np.array([-2.1519, -1.3439, -0.7560, -0.2451, 0.2451, 0.7560, 1.3439, 2.1519])
    assert np.max(np.abs(lev - want)) < 0.03, lev


def test_nuq_beats_uniform_on_laplacian():
    # the page reports a much lower error than the uniform grid at 3 bits on
    # Laplacian data; require at least a factor of 2
    x = np.random.default_rng(5).laplace(size=20_000).astype(np.float32)
    _, lut, _ = oracle.nuq_fit(x, 8, 8)
    mse_nuq = np.mean((f16(lut)[oracle.nuq_assign(x, lut)] - x) ** 2)
    s = (x.max() - x.min()) / 7.0
    uni = x.min() + s * np.clip(np.rint((x - x.min()) / s), 0, 7)
    mse_uni = np.mean((uni - x) ** 2)
    assert mse_nuq < 0.5 * mse_uni, (mse_nuq, mse_uni)


@pytest.mark.parametrize("n,k", [(128, 1), (4095, 41), (50, 7), (9, 9)])
def test_outliers_are_exactly_the_top_k_by_rank(n, k):
    g = np.random.default_rng(n)
    x = np.round(g.standard_normal(n) * 4).astype(np.float32)   # many ties in |x|
    mask = oracle.topk_abs(x, k)
    assert mask.sum() == k
    want = sorted(range(n), key=lambda i: (-abs(float(x[i])), i))[:k]
    assert sorted(np.flatnonzero(mask).tolist()) == sorted(want)


def test_constant_vector_takes_the_lowest_indices():
    mask = oracle.topk_abs(np.full(20, 3.0, dtype=np.float32), 4)
    assert np.flatnonzero(mask).tolist() == [0, 1, 2, 3]


def test_zero_fraction_is_plain_nuq():
    x = np.random.default_rng(9).standard_t(4.0, size=500).astype(np.float32)
    flag, lut, codes = oracle.nuq_vector(x, 3, 8, 0.0)
    assert not flag.any()
    _, lut2, _ = oracle.nuq_fit(x, 8, 8)
    assert np.array_equal(lut, lut2) and np.array_equal(codes, oracle.nuq_assign(x, lut2))


def test_outliers_leave_the_fit():
    x = np.random.default_rng(2).standard_normal(400).astype(np.float32)
    x[17] = 1e4
    flag, lut, _ = oracle.nuq_vector(x, 3, 8, 0.01)   # k = 4
    assert flag[17] and flag.sum() == 4
    _, lut2, _ = oracle.nuq_fit(x, 8, 8, exclude=flag)
    assert np.array_equal(lut, lut2)
    assert f16(lut).max() < 10


def test_codes_are_the_nearest_fp16_level():
    g = np.random.default_rng(4)
    x = g.standard_t(4.0, size=3000).astype(np.float32)
    _, lut, _ = oracle.nuq_fit(x, 8, 8)
    lev = f16(lut)
    codes = oracle.nuq_assign(x, lut)
    dist = np.abs(x[:, None] - lev[None, :])           # fp32, as the definition
    want = np.argmin(dist, axis=1)                     # first minimum = lower index on ties
    assert np.array_equal(codes, want)


# ---- decode-time keys ("KVQuant-NUQ" page, Dense-and-Sparse outlier isolation:
# decode keys against the per-channel threshold frozen at prefill) ----------------

def _nuq_w(S, d=64, n_sink=1, frac=0.05):
    import workloads as W
    return W.NUQ.with_(batch=1, n_kv_heads=2, n_q_heads=8, head_dim=d, seq=S, kv_dtype="f32", n_sink=n_sink,
                       extra={"lloyd_iters": 8, "outlier_frac": frac})


def test_frozen_threshold_is_the_kth_magnitude():
    from oracle import cache as OC
    rng = np.random.default_rng(7)
    P, d = 101, 64
    w = _nuq_w(P, d)
    x = rng.standard_normal((1, 2, P, d)).astype(np.float32)
    thr = OC.nuq_key_thresholds(w, x, P)
    k = oracle.outlier_count(0.05, P - 1)
    assert k == 5
    for h in range(2):
        for c in range(d):
            col = [abs(float(v)) for v in x[0, h, 1:P, c]]
            assert sum(1 for m in col if m >= thr[0, h, c]) == k
            assert float(thr[0, h, c]) == sorted(col, reverse=True)[k - 1]
    # no prefill outliers: nothing is an outlier at decode either
    assert np.all(np.isinf(OC.nuq_key_thresholds(_nuq_w(P, d, frac=0.0), x, P)))


def test_reappended_prefill_tokens_reproduce_the_prefill():
    # a decode copy of a prefill key gets the prefill's code, and the threshold
    # test picks exactly the prefill's rank outliers (distinct magnitudes)
    from oracle import cache as OC
    rng = np.random.default_rng(8)
    P, d, ns = 90, 64, 1
    S = P + (P - ns)
    w = _nuq_w(S, d, n_sink=ns)
    x = np.zeros((1, 2, S, d), dtype=np.float32)
    x[:, :, :P] = rng.standard_normal((1, 2, P, d))
    x[:, :, P:] = x[:, :, ns:P]
    nt = OC.quantize_nuq_stream(w, x, True, P, S)
    nq = P - ns
    assert nt.outlier[:, :, :nq].sum() == 2 * d * oracle.outlier_count(0.05, nq)
    assert np.array_equal(nt.codes[:, :, nq:], nt.codes[:, :, :nq])
    assert np.array_equal(nt.outlier[:, :, nq:], nt.outlier[:, :, :nq])
    assert np.array_equal(nt.xhat[:, :, nq:], nt.xhat[:, :, :nq])


def test_key_side_channel_cap_drops_the_latest_entries():
    from oracle import cache as OC
    rng = np.random.default_rng(9)
    P, d, S = 60, 64, 100
    w = _nuq_w(S, d)
    x = (rng.standard_normal((1, 2, S, d)) * 1.5).astype(np.float32)
    free = OC.quantize_nuq_stream(w, x, True, P, S)
    n_pre = int(free.outlier[0, 0, :P - 1].sum())
    n_dec = int(free.outlier[0, 0, P - 1:].sum())
    assert n_dec > 10
    cap = n_pre + n_dec - 7
    capped = OC.quantize_nuq_stream(w, x, True, P, S, nnz_cap=cap)
    assert int(capped.outlier[0, 0].sum()) == cap
    # the 7 dropped are the last 7 decode outliers in token-major, channel order
    t, c = np.nonzero(free.outlier[0, 0, P - 1:])
    dropped = set(zip(t[-7:].tolist(), c[-7:].tolist()))
    t2, c2 = np.nonzero(free.outlier[0, 0, P - 1:] & ~capped.outlier[0, 0, P - 1:])
    assert set(zip(t2.tolist(), c2.tolist())) == dropped
    # a dropped outlier keeps the level of its code
    lev = capped.lut[0, 0].view(np.float16).astype(np.float32)
    for (ti, ci) in dropped:
        assert capped.xhat[0, 0, P - 1 + ti, ci] == lev[ci, capped.codes[0, 0, P - 1 + ti, ci]]
    # a cap below the prefill's own entries stores no decode outlier
    none = OC.quantize_nuq_stream(w, x, True, P, S, nnz_cap=n_pre - 1)
    assert not none.outlier[:, :, P - 1:].any()


def test_value_tokens_are_fitted_independently():
    # per-token value tables: a token's table and codes do not depend on the others
    from oracle import cache as OC
    rng = np.random.default_rng(10)
    S, d = 12, 64
    w = _nuq_w(S, d)
    x = rng.standard_normal((1, 2, S, d)).astype(np.float32)
    full = OC.quantize_nuq_stream(w, x, False, 5, S)
    for t in (1, 6, 11):
        one = OC.quantize_nuq(w, np.ascontiguousarray(x[:, :, [0, t]]), False, 2)
        assert np.array_equal(one.lut[:, :, 0], full.lut[:, :, t - 1])
        assert np.array_equal(one.codes[:, :, 0], full.codes[:, :, t - 1])
