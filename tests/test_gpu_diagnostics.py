"""The bench's diagnostics measured through the library, checked against the
oracle on the same tokens.

D-Quant Sec. 3, Table 1 (NMSE, empirical entropy, Coding Gain, Normal Gap of
an 8-level per-token grid, raw / after the Hadamard rotation / after also
removing the key channel mean): bench.preprocessing_effect reads the codes
out of the library's own cache buffers and dequantizes through the library;
the same statistics from the oracle's quantization must be identical, since
the codes and dequantized values are bit-exact."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def test_preprocessing_table_equals_the_oracle():
    import bench
    import workloads as W
    from oracle import cache as OC
    from quantized_decode_attention_gb300 import symbol_probs
    batch, seq = 1, 256
    res = bench.preprocessing_effect(batch=batch, seq=seq)
    got = {(r["tensor"], r["preprocessing"]): r for r in res["rows"]}
    assert len(got) == 5
    p = np.array(symbol_probs(128, 8))
    w0 = W.LLAMA.with_(batch=batch, seq=seq, n_sink=0, n_recent=0, meta_dtype="f32", bits=3)
    k, v = W.make_kv(W.LLAMA.with_(batch=batch, seq=seq))
    for name, rot, mean in (("raw", "none", False), ("hadamard", "hadamard", False),
                            ("hadamard+mean", "hadamard", True)):
        w = w0.with_(rot_k=rot, rot_v=rot, mean_k=mean)
        for key, bits in ((True, k), (False, v)):
            tag = ("k" if key else "v", name)
            if tag not in got:
                continue
            qt = OC.quantize_tensor(w, bits, key, seq)
            x = W.bf16_bits_to_f32(bits).astype(np.float64)
            x = bench.hadamard_rows(x) if rot == "hadamard" else x
            err = x - qt.xhat.astype(np.float64)
            want = bench.coding_stats(np.bincount(qt.codes.ravel(), minlength=8), p)
            for f in ("entropy", "coding_gain", "normal_gap"):
                assert got[tag][f] == want[f], (tag, f, got[tag][f], want[f])
            assert got[tag]["nmse"] == float((err * err).sum() / (x * x).sum()), tag


def test_drift_statistics_of_the_library_containers_equal_the_oracle():
    """D-Quant App. C (drift makes only sparse, local corrections): the library
    counts, while it encodes, the symbols drift moved off the nearest level of
    their stream's final fp16 grid and the largest move; on the same tokens
    the oracle's Algorithm 1 gives its symbols and their nearest levels, and
    the counts must agree exactly (moves of at most one level, a few percent
    of the symbols)."""
    import oracle
    import workloads as W
    from helpers import cfg_for, to_device
    from oracle import cache as OC
    from quantized_decode_attention_gb300 import KVCache
    extra = dict(W.DQUANT.extra)
    w = W.DQUANT.with_(batch=1, n_kv_heads=8, n_q_heads=32, seq=256, n_recent=16, extra=extra)
    S = w.seq
    k, v = W.make_kv(w)
    cache = KVCache.allocate(cfg_for(w))
    cache.quantize(to_device(k, w.kv_dtype), to_device(v, w.kv_dtype))
    cache.check()
    got = cache.drift_stats()
    assert cache.drift_stats() == {f"{t}_{f}": 0 for t in "kv" for f in ("changed", "coded", "max_move")}
    tk, tv = OC.dq_tables(w)
    for t, x_bits, key, tab, cb in (("k", k, True, tk, extra["container_k"]), ("v", v, False, tv, extra["container_v"])):
        dt = OC.quantize_dquant(w, x_bits, key, S)
        changed, move = 0, 0
        for b in range(dt.x.shape[0]):
            for p in range(dt.x.shape[1]):
                r = oracle.dq_encode_stream(dt.x[b, p], tab, cb)
                assert np.array_equal(r["m"], dt.m[b, p])
                dlt = np.abs(r["m"].astype(int) - r["m_near"].astype(int))
                changed += int((dlt > 0).sum())
                move = max(move, int(dlt.max()))
        assert got[f"{t}_coded"] == dt.m.size, (t, got)
        assert got[f"{t}_changed"] == changed, (t, got, changed)
        assert got[f"{t}_max_move"] == move <= 1, (t, got, move)
        assert 0 < changed < 0.1 * dt.m.size
    cache.close()
