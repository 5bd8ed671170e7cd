"""Pins of the oracle's grouped value fit and key refit blocks.

Source: "KVQuant-NUQ" (VeloxQuant-MLX docs), Configuration reference:
kvquant_group_size (how many elements share one fit) and
kvquant_refit_interval (key levels fitted anew after N decode steps), with How
it works (quantile-seeded Lloyd-Max, rank outliers per token) and Quantization
axes (keys per channel, values per token).

Readings pinned here:
  * a value token's channels split into groups of g consecutive channels, each
    fitted on its own values with its own table; the outliers are ranked over
    the whole token;
  * key tables belong to blocks of N quantized slots on the slot grid; blocks
    the prefill reaches keep the prefill's tables, and a block of decode keys
    gets tables fitted on its own N keys once its last slot arrives.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def f16(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def _w(S, d=128, n_sink=1, frac=0.0, iters=8, **extra):
    import workloads as W
    ex = {"lloyd_iters": iters, "outlier_frac": frac}
    ex.update(extra)
    return W.NUQ.with_(batch=1, n_kv_heads=1, n_q_heads=4, head_dim=d, seq=S, kv_dtype="f32", n_sink=n_sink,
                       n_recent=extra.get("refit_interval", 0), extra=ex)


def test_group_of_the_whole_vector_is_the_plain_fit():
    rng = np.random.default_rng(3)
    for bits in (2, 3, 4):
        x = rng.standard_t(4, 128).astype(np.float32)
        f1, l1, c1 = oracle.nuq_vector(x, bits, 8, 0.03)
        f2, l2, c2 = oracle.nuq_vector_grouped(x, bits, 8, 0.03, 128)
        assert np.array_equal(f1, f2) and np.array_equal(l1, l2[0]) and np.array_equal(c1, c2)


def test_hand_worked_groups():
    # group G holds 100 G + 0, 1, ..., 31.  Quantile seeds of 32 values and 4
    # levels sit at sorted positions floor((2i+1) 32 / 8) = 4, 12, 20, 28; one
    # Lloyd sweep moves them to the cell means 4, 12.5, 20.5, 28 (boundary
    # values go to the lower level: cells 0..8, 9..16, 17..24, 25..31), which
    # is a fixed point.  A fit over the whole token would seed at 16, 48, 80, 112.
    x = np.concatenate([100.0 * G + np.arange(32) for G in range(4)]).astype(np.float32)
    _, lut0, _ = oracle.nuq_vector_grouped(x, 2, 0, 0.0, 32)
    _, lut8, codes = oracle.nuq_vector_grouped(x, 2, 8, 0.0, 32)
    for G in range(4):
        assert f16(lut0[G]).tolist() == [100 * G + 4, 100 * G + 12, 100 * G + 20, 100 * G + 28]
        assert f16(lut8[G]).tolist() == [100 * G + 4, 100 * G + 12.5, 100 * G + 20.5, 100 * G + 28]
        # codes: 0..8 -> 0, 9..16 -> 1, 17..24 -> 2, 25..31 -> 3
        assert codes[32 * G:32 * G + 32].tolist() == [0] * 9 + [1] * 8 + [2] * 8 + [3] * 7
    # d = 64 in two groups, 16-bit levels of each group within its own range
    _, lut, _ = oracle.nuq_vector_grouped(x[:64], 3, 8, 0.0, 32)
    assert f16(lut[0]).max() <= 31 and f16(lut[1]).min() >= 100


def test_outliers_are_ranked_over_the_whole_token():
    # k = floor(0.03 * 128 + 0.5) = 4 outliers; the four largest magnitudes all
    # sit in group 2, so group 2 loses four values to the side channel and the
    # other groups none (a per-group top-k would take one from each group)
    rng = np.random.default_rng(5)
    x = rng.uniform(-1, 1, 128).astype(np.float32)
    x[[70, 75, 80, 90]] = [50.0, -60.0, 70.0, -80.0]
    flag, lut, codes = oracle.nuq_vector_grouped(x, 3, 8, 0.03, 32)
    assert flag.sum() == 4 and set(np.flatnonzero(flag).tolist()) == {70, 75, 80, 90}
    # group 2's table is fitted without them: its levels stay inside the other values' range
    lev = f16(lut[2])
    assert lev.max() <= 1.0 and lev.min() >= -1.0


def test_each_group_is_the_fit_of_its_slice():
    rng = np.random.default_rng(11)
    for g, bits in ((32, 3), (64, 2), (16, 4)):
        x = (rng.standard_t(4, 128) * np.repeat(rng.uniform(0.5, 4, 128 // g), g)).astype(np.float32)
        flag, lut, codes = oracle.nuq_vector_grouped(x, bits, 8, 0.02, g)
        assert flag.sum() == oracle.outlier_count(0.02, 128)
        for G in range(128 // g):
            sl = slice(G * g, G * g + g)
            lev, lut16, _ = oracle.nuq_fit(x[sl], 1 << bits, 8, exclude=flag[sl])
            assert np.array_equal(lut[G], lut16), (g, G)
            assert np.array_equal(codes[sl], oracle.nuq_assign(x[sl], lut16))


def test_group_distortion_never_increases_across_sweeps():
    rng = np.random.default_rng(13)
    x = rng.standard_t(3, 128).astype(np.float32)
    prev = None
    for it in range(8):
        _, lut, _ = oracle.nuq_vector_grouped(x, 2, it, 0.0, 32)
        # distortion of each group against its fp32-rounded-to-fp16 levels is
        # dominated by the fit; compare the fp32 Lloyd levels instead
        d = []
        for G in range(4):
            lev, _, _ = oracle.nuq_fit(x[32 * G:32 * G + 32], 4, it)
            d.append(float(np.min((x[32 * G:32 * G + 32, None].astype(np.float64) - lev[None, :]) ** 2, axis=1).sum()))
            assert np.array_equal(lut[G], oracle.nuq_fit(x[32 * G:32 * G + 32], 4, it)[1])
        if prev is not None:
            assert all(a <= b * (1 + 1e-6) for a, b in zip(d, prev))
        prev = d


def test_grouped_value_cache_dequantizes_through_its_groups():
    from oracle import cache as OC
    rng = np.random.default_rng(17)
    w = _w(20, group_size=32, frac=0.01)
    x = np.zeros((1, 1, 20, 128), dtype=np.float32)
    x[...] = rng.standard_normal((20, 128)) * np.repeat([0.1, 1.0, 10.0, 100.0], 32)
    nv = OC.quantize_nuq(w, x, False, 20)
    assert nv.lut.shape == (1, 1, 19, 4 * 8)
    for t in range(19):
        lev = f16(nv.lut[0, 0, t]).reshape(4, 8)
        for c in range(128):
            if not nv.outlier[0, 0, t, c]:
                assert nv.xhat[0, 0, t, c] == lev[c // 32, nv.codes[0, 0, t, c]]
    # a group's reconstruction error follows its own scale
    err = np.abs(nv.xhat[0, 0] - x[0, 0, 1:]).reshape(19, 4, 32).max(axis=(0, 2))
    assert err[0] < 0.2 and err[3] > err[0]


def test_refit_blocks_follow_the_slot_grid():
    # N = 128; a prefill of P = 100 tokens with one sink has 99 quantized slots,
    # so it reaches block 0 only: slots 99..127 are coded with the prefill's
    # tables.  Block 1 (slots 128..255) is decode keys only: its tables are
    # fitted on its own keys once slot 255 arrives.  Block 2 is incomplete.
    from oracle import cache as OC
    rng = np.random.default_rng(19)
    N, P, S = 128, 100, 300
    w = _w(S, refit_interval=N, frac=0.02)
    x = np.zeros((1, 1, S, 128), dtype=np.float32)
    x[0, 0, :1 + 128] = rng.uniform(-1, 1, (129, 128))           # slots 0..127 (and the sink)
    x[0, 0, 1 + 128:1 + 256] = 1000 + rng.uniform(-1, 1, (128, 128))
    x[0, 0, 1 + 256:] = -500 + rng.uniform(-1, 1, (S - 257, 128))
    nk = OC.quantize_nuq_stream(w, x, True, P, S)
    pre = OC.quantize_nuq(w, x, True, P)
    assert nk.n_coded == 256
    assert np.array_equal(nk.blk_lut[0, 0, 0], pre.lut[0, 0])
    lev1 = f16(nk.blk_lut[0, 0, 1])
    assert lev1.min() >= 999 and lev1.max() <= 1001                # fitted on block 1 alone
    # the prefill's block: decode slots take the prefill's levels
    for s in range(99, 128):
        for c in range(0, 128, 17):
            want = oracle.nuq_assign(x[0, 0, 1 + s, c:c + 1], pre.lut[0, 0, c])[0]
            assert nk.codes[0, 0, s, c] == want
    # block 1's rank outliers: exactly floor(0.02 * 128 + 0.5) = 3 per channel
    assert np.all(nk.outlier[0, 0, 128:256].sum(axis=0) == 3)
    # slots of the incomplete block are not coded yet
    assert np.isnan(nk.xhat[0, 0, 256:]).all() and not np.isnan(nk.xhat[0, 0, :256]).any()


def test_refit_block_is_a_prefill_of_its_keys():
    from oracle import cache as OC
    rng = np.random.default_rng(23)
    N, P, S = 128, 300, 700
    w = _w(S, refit_interval=N, frac=0.01, n_sink=4)
    x = rng.standard_t(4, (1, 1, S, 128)).astype(np.float32)
    nk = OC.quantize_nuq_stream(w, x, True, P, S)
    pq = P - 4
    b0 = -(-pq // N)                       # 3: blocks 0..2 hold the prefill's tables
    assert nk.n_coded == 5 * N
    for b in range(b0):
        assert np.array_equal(nk.blk_lut[:, :, b], OC.quantize_nuq(w, x, True, P).lut)
    for b in range(b0, 5):
        one = OC.quantize_nuq(w, x, True, 4 + (b + 1) * N, t0=4 + b * N)
        assert np.array_equal(nk.blk_lut[:, :, b], one.lut)
        assert np.array_equal(nk.codes[:, :, b * N:(b + 1) * N], one.codes)
        assert np.array_equal(nk.outlier[:, :, b * N:(b + 1) * N], one.outlier)


def test_refit_zero_keeps_the_frozen_tables():
    from oracle import cache as OC
    rng = np.random.default_rng(29)
    w0 = _w(260, frac=0.02)
    x = rng.standard_normal((1, 1, 260, 128)).astype(np.float32)
    a = OC.quantize_nuq_stream(w0, x, True, 60, 260)
    assert a.blk_lut is None and not np.isnan(a.xhat).any()
    pre = OC.quantize_nuq(w0, x, True, 60)
    assert np.array_equal(a.lut, pre.lut)
