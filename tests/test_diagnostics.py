"""The bench's synthetic diagnostics without a GPU: the library's analytic
symbol model against the oracle's, and the pieces that turn a quantized cache
into D-Quant's Table 1 quantities (codes read back from packed records, entropy,
Coding Gain, Normal Gap, the rotation used for NMSE), each pinned against the
oracle's packers, closed forms or the oracle's own rotation."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def lib():
    from quantized_decode_attention_gb300 import build
    build.build()
    from quantized_decode_attention_gb300 import _lib
    return _lib.load()


@pytest.mark.parametrize("n,M", [(128, 8), (1024, 8), (1024, 6), (64, 3), (2, 2), (4096, 16)])
def test_symbol_probs_match_the_oracle(lib, n, M):
    """D-Quant Sec. 4.2: the unsharpened order-statistics model, by the library
    (tail integrals of the maximum) and by the oracle (its density), agree and
    sum to one; the model is symmetric about the middle level."""
    import oracle
    from quantized_decode_attention_gb300 import symbol_probs
    p = np.array(symbol_probs(n, M))
    ref = oracle.DqTable(n, M, alpha=1.0).prob
    np.testing.assert_allclose(p, ref, rtol=0, atol=1e-12)
    assert abs(p.sum() - 1.0) < 1e-12
    np.testing.assert_allclose(p, p[::-1], rtol=0, atol=1e-12)


def test_symbol_probs_refuses_bad_arguments(lib):
    from quantized_decode_attention_gb300 import DQError, symbol_probs
    for n, M in ((0, 8), (128, 1), (128, 17)):
        with pytest.raises(DQError):
            symbol_probs(n, M)


@pytest.mark.parametrize("bits,d", [(2, 64), (2, 128), (3, 128), (4, 64), (4, 128)])
def test_codes_of_records_reads_back_every_code(bits, d):
    """Each record, key row or value pair, holds exactly the codes the oracle
    packed into it (as a multiset: the diagnostic only counts codes).  The codes
    are skewed per channel, so pairing the two planes of a 3-bit code wrongly
    changes the counts."""
    import bench
    from oracle import cache as OC
    rng = np.random.default_rng(7 + bits)
    codes = rng.integers(0, 1 << bits, size=(2, 3, 10, d)).astype(np.uint8)
    codes[..., : d // 3] = rng.integers(0, 2, size=codes[..., : d // 3].shape)
    codes[..., d // 3: d // 2] = (1 << bits) - 1
    rk = OC.pack_k(codes, bits)
    got = bench.codes_of_records(rk, bits).reshape(-1, d)
    np.testing.assert_array_equal(np.sort(got, axis=1), np.sort(codes.reshape(-1, d), axis=1))
    rv = OC.pack_v(codes, bits)
    got = bench.codes_of_records(rv, bits).reshape(-1, 2 * d)
    pairs = codes.reshape(2, 3, 5, 2 * d)
    np.testing.assert_array_equal(np.sort(got, axis=1), np.sort(pairs.reshape(-1, 2 * d), axis=1))


def test_coding_stats_closed_forms():
    """Coding Gain = log2 M - H and Normal Gap = CE - H (D-Quant Sec. 3): a histogram
    proportional to the model has no gap; a uniform histogram has no gain and a gap
    equal to the model's mean code length minus log2 M; a worked example."""
    import bench
    p = np.array([0.1, 0.2, 0.4, 0.2, 0.1])
    s = bench.coding_stats(p * 1000, p)
    assert abs(s["normal_gap"]) < 1e-12
    H = -(p * np.log2(p)).sum()
    assert abs(s["entropy"] - H) < 1e-12 and abs(s["coding_gain"] - (np.log2(5) - H)) < 1e-12
    u = bench.coding_stats(np.ones(5), p)
    assert abs(u["coding_gain"]) < 1e-12
    assert abs(u["normal_gap"] - (-np.log2(p).mean() - np.log2(5))) < 1e-12
    w = bench.coding_stats(np.array([1, 1, 2, 0]), np.array([0.25, 0.25, 0.25, 0.25]))
    assert abs(w["entropy"] - 1.5) < 1e-12 and abs(w["coding_gain"] - 0.5) < 1e-12
    assert abs(w["normal_gap"] - 0.5) < 1e-12


def test_hadamard_rows_is_the_oracle_rotation():
    import bench
    import oracle
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 128)).astype(np.float32)
    np.testing.assert_allclose(bench.hadamard_rows(x), oracle.rotate_hadamard_rows(x), rtol=0, atol=2e-6)


def test_preprocessing_row_reads_a_whole_cache_buffer():
    """The bench hands preprocessing_row a cache's entire code buffer, flat, as the
    library lays it out ([unit][slot][record], value records holding token pairs).
    Built here from the oracle's packed records of real 3-bit codes, that buffer
    gives exactly the oracle codes' histogram, and the row's NMSE is the plain one."""
    import bench
    import oracle
    import workloads as W
    from oracle import cache as OC
    w = W.LLAMA.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=128, n_sink=0, n_recent=0, meta_dtype="f32", bits=3)
    k, v = W.make_kv(w)
    p = oracle.DqTable(w.head_dim, 8, alpha=1.0).prob
    for key, bits in ((True, k), (False, v)):
        qt = OC.quantize_tensor(w, bits, key, w.seq)
        flat = (OC.pack_k(qt.codes, 3) if key else OC.pack_v(qt.codes, 3)).reshape(-1)
        x = bench.hadamard_rows(W.bf16_bits_to_f32(bits).astype(np.float64))
        xhat = qt.xhat.astype(np.float64)
        row = bench.preprocessing_row("k" if key else "v", "hadamard", x, xhat, flat,
                                      3 * w.head_dim // 8 if key else 3 * w.head_dim // 4, p)
        ref = bench.coding_stats(np.bincount(qt.codes.ravel(), minlength=8), p)
        for f in ("entropy", "coding_gain", "normal_gap"):
            assert row[f] == ref[f], f
        assert row["nmse"] == float(((x - xhat) ** 2).sum() / (x * x).sum())


def test_preprocessing_table_on_oracle_caches():
    """D-Quant Table 1's quantities computed the bench's way on oracle-quantized
    Llama-shaped keys (per-channel means, outlier channels): rotating spreads the
    outlier channels and removing the mean centres the keys, so key NMSE falls at
    each step, and the rotated keys sit far closer to the normal model than the raw
    ones.  Values (already Gaussian) keep a small gap either way, and every Normal
    Gap is non-negative (Gibbs)."""
    import bench
    import oracle
    import workloads as W
    from oracle import cache as OC
    w0 = W.LLAMA.with_(batch=1, seq=256, n_sink=0, n_recent=0, meta_dtype="f32", bits=3)
    k, v = W.make_kv(w0)
    p = oracle.DqTable(w0.head_dim, 8, alpha=1.0).prob
    res = {}
    for name, rot, mean in (("raw", "none", False), ("hadamard", "hadamard", False), ("mean", "hadamard", True)):
        w = w0.with_(rot_k=rot, rot_v=rot, mean_k=mean)
        for key, bits in ((True, k), (False, v)):
            qt = OC.quantize_tensor(w, bits, key, w.seq)
            x = W.bf16_bits_to_f32(bits).astype(np.float64)
            x = bench.hadamard_rows(x) if rot == "hadamard" else x
            err = x - qt.xhat.astype(np.float64)
            packed = OC.pack_k(qt.codes, 3) if key else OC.pack_v(qt.codes, 3)
            hist = np.bincount(bench.codes_of_records(packed, 3), minlength=8)
            np.testing.assert_array_equal(hist, np.bincount(qt.codes.ravel(), minlength=8))
            st = bench.coding_stats(hist, p)
            st["nmse"] = float((err * err).sum() / (x * x).sum())
            res[("k" if key else "v", name)] = st
    assert res[("k", "raw")]["nmse"] > res[("k", "hadamard")]["nmse"] > res[("k", "mean")]["nmse"]
    assert res[("k", "hadamard")]["normal_gap"] < 0.25 * res[("k", "raw")]["normal_gap"]
    for key in res:
        assert res[key]["normal_gap"] >= 0.0 and 0.0 < res[key]["coding_gain"] < 3.0, key
    assert res[("v", "raw")]["normal_gap"] < 0.05 and res[("v", "hadamard")]["normal_gap"] < 0.05
