"""GPU parity of the non-uniform (Lloyd-Max) scheme against the oracle.

"KVQuant-NUQ" (VeloxQuant-MLX docs): per-channel key tables and per-token value
tables fit at prefill, rank-based outliers in an fp16 side channel, sinks kept
exact.  Tables, codes, side channel and 16-bit regions must match bit for bit.
"""
import numpy as np
import pytest

import workloads as W
from oracle import cache as OC

from helpers import cfg_for, nuq_views, to_device

pytestmark = pytest.mark.gpu

CASES = {
    # a 3-bit cache of the KVQuant shape, Student-t data; several 64-token blocks and a ragged tail
    "nuq3-d128": W.NUQ.with_(batch=1, n_kv_heads=2, n_q_heads=8, seq=300),
    # 2-bit, d64, a recent window as well as the sink
    "nuq2-d64-recent": W.NUQ.with_(batch=2, n_kv_heads=1, n_q_heads=4, head_dim=64, seq=200, bits=2, n_recent=16),
    # 4-bit, no sink
    "nuq4-d128-nosink": W.NUQ.with_(batch=1, n_kv_heads=1, n_q_heads=4, seq=130, bits=4, n_sink=0),
    # plain NUQ (no outliers) and no Lloyd sweeps (quantile seeds only)
    "nuq3-frac0-iters0": W.NUQ.with_(batch=1, n_kv_heads=1, n_q_heads=4, seq=97,
                                     extra={"outlier_frac": 0.0, "lloyd_iters": 0}),
    # bf16 input: side-channel values are rounded to fp16
    "nuq3-bf16": W.NUQ.with_(batch=1, n_kv_heads=1, n_q_heads=4, seq=150, kv_dtype="bf16"),
    # value tables per 32-channel group (Configuration reference, kvquant_group_size)
    "nuq3-group32": W.NUQ.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=300,
                                extra={"lloyd_iters": 8, "outlier_frac": 0.01, "group_size": 32}),
    "nuq4-group32-bf16": W.NUQ.with_(batch=1, n_kv_heads=1, n_q_heads=4, seq=200, bits=4, kv_dtype="bf16",
                                     extra={"lloyd_iters": 8, "outlier_frac": 0.02, "group_size": 32}),
    "nuq2-group32": W.NUQ.with_(batch=1, n_kv_heads=2, n_q_heads=8, seq=170, bits=2,
                                extra={"lloyd_iters": 8, "outlier_frac": 0.01, "group_size": 32}),
}


def _compare(w, got, qcap, k, v, nk, nv, S):
    """Tables, codes, side channels and 16-bit regions of a cache of length S."""
    nq = S - w.n_sink
    if nk.blk_lut is not None:   # key refit blocks: the coded slots and the tables of their blocks
        N = w.extra["refit_interval"]
        nc = nk.n_coded
        assert np.array_equal(got["lut_k_blk"][:, :, :-(-nc // N)], nk.blk_lut[:, :, :-(-nc // N)])
        assert np.array_equal(got["codes_k"][:, :, :nc], OC.pack_k(nk.codes[:, :, :nc], w.bits))
    else:
        assert np.array_equal(got["lut_k"], nk.lut)
        assert np.array_equal(got["codes_k"][:, :, :nq], OC.pack_k(nk.codes, w.bits))
    assert np.array_equal(got["lut_v"][:, :, :nq], nv.lut)
    pv = OC.pack_v(nv.codes, w.bits)
    full = nq // 2
    assert np.array_equal(got["codes_v"][:, :, :full], pv[:, :, :full])
    if nq % 2:  # the last record holds one token: compare its half only
        half = got["codes_v"][:, :, full].view(np.uint16).reshape(w.batch, w.n_kv_heads, -1, 2)[..., 0]
        want = pv[:, :, full].view(np.uint16).reshape(w.batch, w.n_kv_heads, -1, 2)[..., 0]
        assert np.array_equal(half, want)
    kk = OC.nuq_key_outliers_csr(nk, qcap, got["col_k"].shape[-1]) if "rowptr" in got else None
    if kk is not None:
        rp, col, val = kk
        assert np.array_equal(got["rowptr"][:, :, :qcap + 1], rp)
        for b in range(w.batch):
            for h in range(w.n_kv_heads):
                n_nz = rp[b, h, -1]
                assert np.array_equal(got["col_k"][b, h, :n_nz], col[b, h, :n_nz])
                assert np.array_equal(got["val_k"][b, h, :n_nz], val[b, h, :n_nz])
    else:
        assert not nk.outlier.any()
    if "col_v" in got:
        col, val = OC.nuq_value_outliers(nv, qcap, got["col_v"].shape[-1])
        assert np.array_equal(got["col_v"][:, :, :nq], col[:, :, :nq])
        assert np.array_equal(got["val_v"][:, :, :nq], val[:, :, :nq])
    else:
        assert not nv.outlier.any()
    for slot, bits in OC.raw_regions(w, k[:, :, :S], S).items():
        assert np.array_equal(got["raw_k"][:, :, slot], bits), slot
    for slot, bits in OC.raw_regions(w, v[:, :, :S], S).items():
        assert np.array_equal(got["raw_v"][:, :, slot // 2, :, slot & 1], bits), slot


@pytest.mark.parametrize("name", list(CASES))
def test_nuq_prefill_is_bit_exact(name):
    import torch
    from quantized_decode_attention_gb300 import KVCache
    w = CASES[name]
    S = w.seq
    k, v = W.make_kv(w)
    cache = KVCache.allocate(cfg_for(w))
    cache.quantize(to_device(k, w.kv_dtype), to_device(v, w.kv_dtype))
    torch.cuda.synchronize()
    cache.check()
    got, qcap = nuq_views(w, cache, S)
    nk = OC.quantize_nuq(w, k, True, S)
    nv = OC.quantize_nuq(w, v, False, S)
    _compare(w, got, qcap, k, v, nk, nv, S)
    if "thr_k" in got:
        assert np.array_equal(got["thr_k"], OC.nuq_key_thresholds(w, k, S))


# Decode-time appends: keys against the tables and thresholds frozen at the
# prefill, values fitted per token; one token at a time and in batches.
STREAM = {
    "nuq3-d128": (W.NUQ.with_(batch=1, n_kv_heads=2, n_q_heads=8, seq=300), [200] + [1] * 40 + [60]),
    "nuq2-d64-recent": (W.NUQ.with_(batch=2, n_kv_heads=1, n_q_heads=4, head_dim=64, seq=200, bits=2,
                                    n_recent=16), [120, 1, 1, 1, 77]),
    "nuq4-bf16-nosink": (W.NUQ.with_(batch=1, n_kv_heads=1, n_q_heads=4, seq=180, bits=4, kv_dtype="bf16",
                                     n_sink=0), [100, 1, 79]),
    # key refit blocks of 128 slots (Configuration reference, kvquant_refit_interval)
    # with grouped values: the prefill reaches blocks 0-1; single tokens fill
    # block 2 partway, a 300-token append completes blocks 2 and 3, single
    # tokens then complete block 4
    "nuq3-refit128-group32": (W.NUQ.with_(batch=1, n_kv_heads=2, n_q_heads=8, seq=650, n_recent=128,
                                          extra={"lloyd_iters": 8, "outlier_frac": 0.01, "group_size": 32,
                                                 "refit_interval": 128}),
                              [200] + [1] * 60 + [300] + [1] * 90),
    # the prefill ends on a block boundary (256 quantized slots = blocks 0-1), so
    # the first appended key already waits for block 2; 2 bits, one KV head
    "nuq2-refit128-aligned": (W.NUQ.with_(batch=1, n_kv_heads=1, n_q_heads=4, seq=520, bits=2, n_recent=128,
                                          extra={"lloyd_iters": 8, "outlier_frac": 0.02, "refit_interval": 128}),
                              [257] + [1] * 5 + [250] + [8]),
    # refit alone (whole-token values), 4 bits, bf16, no sink; blocks of 256
    "nuq4-refit256-bf16": (W.NUQ.with_(batch=2, n_kv_heads=1, n_q_heads=4, seq=700, bits=4, kv_dtype="bf16",
                                       n_sink=0, n_recent=256,
                                       extra={"lloyd_iters": 8, "outlier_frac": 0.02, "refit_interval": 256}),
                           [100, 1, 1, 300, 298]),
}


def _stream_cache(w, steps, k, v, check_at):
    """Fill a cache by the given calls; yields (cache, P, S) after each call whose end is in check_at."""
    from quantized_decode_attention_gb300 import KVCache
    cache = KVCache.allocate(cfg_for(w))
    pos = 0
    for n in steps:
        cache.quantize(to_device(k[:, :, pos:pos + n], w.kv_dtype), to_device(v[:, :, pos:pos + n], w.kv_dtype),
                       pos0=pos)
        pos += n
        if pos in check_at:
            yield cache, steps[0], pos
    cache.close()


@pytest.mark.parametrize("name", list(STREAM))
def test_nuq_appends_match_oracle(name):
    import torch
    from helpers import out_to_np
    w, steps = STREAM[name]
    k, v = W.make_kv(w)
    q = W.make_q(w)
    qd = to_device(q, "f32")
    dt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[w.out_dtype]
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=dt, device="cuda")
    mid = steps[0] + sum(steps[1:-1])
    for cache, P, S in _stream_cache(w, steps, k, v, (mid, w.seq)):
        torch.cuda.synchronize()
        cache.check()
        got, qcap = nuq_views(w, cache, w.seq)
        nnz = got["col_k"].shape[-1] if "col_k" in got else None
        nk = OC.quantize_nuq_stream(w, k[:, :, :S], True, P, S, nnz)
        nv = OC.quantize_nuq_stream(w, v[:, :, :S], False, P, S)
        if S == w.seq:
            assert nk.outlier[:, :, P - w.n_sink:].any()  # decode keys did meet the threshold
        _compare(w, got, qcap, k, v, nk, nv, S)
        assert np.array_equal(got["thr_k"], OC.nuq_key_thresholds(w, k, P))
        if "pq" in got:
            assert np.all(got["pq"] == P - w.n_sink)
        cache.attention(qd, out, S)
        torch.cuda.synchronize()
        cache.check()
        ref = OC.attention(w, q, k[:, :, :S], v[:, :, :S], S, nk, nv)
        assert np.all(np.abs(out_to_np(out) - ref) <= _out_tol(w, ref)), (S, float(np.max(np.abs(out_to_np(out) - ref))))
        out2 = torch.empty_like(out)  # the allocation-free entry point reads the same tables
        cache.attention_noalloc(qd, out2, S)
        torch.cuda.synchronize()
        assert np.all(np.abs(out_to_np(out2) - ref) <= _out_tol(w, ref)), S


def test_nuq_key_side_channel_overflow():
    """Decode keys four times the prefill's scale overflow the side channel: the
    cache reports it, and keeps exactly the first entries that fit."""
    import torch
    from quantized_decode_attention_gb300 import DQError
    from helpers import out_to_np
    w = W.NUQ.with_(batch=1, n_kv_heads=2, n_q_heads=8, seq=260, n_recent=0)
    P = 60
    k, v = W.make_kv(w)
    kf = W.bits_to_f32(k, w.kv_dtype).copy()
    kf[:, :, P:] *= 4.0
    k = W.to_dtype_bits(kf, w.kv_dtype)
    q = W.make_q(w)
    for cache, P_, S in _stream_cache(w, [P, 100, 100], k, v, (w.seq,)):
        torch.cuda.synchronize()
        with pytest.raises(DQError):
            cache.check()
        got, qcap = nuq_views(w, cache, w.seq)
        nnz = got["col_k"].shape[-1]
        nk = OC.quantize_nuq_stream(w, k, True, P, S, nnz)
        nv = OC.quantize_nuq_stream(w, v, False, P, S)
        assert np.all(nk.outlier.sum(axis=(2, 3)) == nnz)   # the channel is full in every unit
        _compare(w, got, qcap, k, v, nk, nv, S)
        out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float16, device="cuda")
        cache.attention(to_device(q, "f32"), out, S)
        torch.cuda.synchronize()
        ref = OC.attention(w, q, k, v, S, nk, nv)
        assert np.all(np.abs(out_to_np(out) - ref) <= _out_tol(w, ref))


def test_nuq_append_without_quantized_prefill_is_refused():
    import torch
    from quantized_decode_attention_gb300 import KVCache, DQError
    w = CASES["nuq3-d128"]            # one sink
    k, v = W.make_kv(w)
    cache = KVCache.allocate(cfg_for(w))
    cache.quantize(to_device(k[:, :, :1], w.kv_dtype), to_device(v[:, :, :1], w.kv_dtype))
    with pytest.raises(DQError):
        cache.quantize(to_device(k[:, :, 1:2], w.kv_dtype), to_device(v[:, :, 1:2], w.kv_dtype), pos0=1)
    torch.cuda.synchronize()
    cache.close()


def _out_tol(w, ref):
    # 2e-3 for the arithmetic, plus rounding of the output to its 16-bit type
    ulp = 2.0 ** -8 if w.out_dtype == "bf16" else (2.0 ** -11 if w.out_dtype == "f16" else 0.0)
    return 2e-3 + ulp * np.abs(ref)


@pytest.mark.parametrize("name", list(CASES))
def test_nuq_attention_matches_oracle(name):
    import torch
    from quantized_decode_attention_gb300 import KVCache
    from helpers import out_to_np
    w = CASES[name]
    S = w.seq
    k, v = W.make_kv(w)
    q = W.make_q(w)
    cache = KVCache.allocate(cfg_for(w))
    cache.quantize(to_device(k, w.kv_dtype), to_device(v, w.kv_dtype))
    dt = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}[w.out_dtype]
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=dt, device="cuda")
    qd = to_device(q, "f32")
    cache.attention(qd, out, S)
    torch.cuda.synchronize()
    cache.check()
    got = out_to_np(out)
    nk = OC.quantize_nuq(w, k, True, S)
    nv = OC.quantize_nuq(w, v, False, S)
    ref = OC.attention(w, q, k, v, S, nk, nv)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= _out_tol(w, ref)), float(np.max(np.abs(got - ref)))
    # the allocation-free entry point computes the same
    out2 = torch.empty_like(out)
    cache.attention_noalloc(qd, out2, S)
    torch.cuda.synchronize()
    assert np.all(np.abs(out_to_np(out2) - ref) <= _out_tol(w, ref))
