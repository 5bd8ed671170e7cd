"""Parity at the benchmark's full sizes, on sampled (batch, KV head) units.

The caches and calls are the ones the benchmark times:
- the Llama-3-8B-shaped decode layer (batch 16, 32 query / 8 KV heads, d128,
  8192 bf16 tokens, 4 sinks + 128 recent) at 2, 3 and 4 bits, prefilled, then
  the benchmark's step -- one token re-appended at position 8191 and attention
  over 8192 tokens in one dq_decode_step -- replayed from a CUDA graph, with
  bf16 outputs and, at 2 bits, fp32 outputs held to 2e-3 exactly;
- the KVQuant NUQ cache (batch 8, 4096 fp16 Student-t tokens, 3 bits, 1 sink,
  1 % outliers), prefilled, attention over 4096 tokens from a CUDA graph.
The oracle recomputes a few units one by one.  Their records, metadata, tables
and side channels must match bit for bit, and the outputs of their query heads
must be within the attention tolerance (2e-3 plus the output's own rounding).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from oracle import cache as OC

from helpers import cfg_for, expected_buffers, lib_views, nuq_views, out_to_np, to_device

pytestmark = pytest.mark.gpu

LLAMA_UNITS = [(0, 0), (7, 3), (15, 7)]
NUQ_UNITS = [(0, 0), (3, 5), (7, 7)]


def _tol(ref, out_dtype):
    ulp = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11}.get(out_dtype, 0.0)
    return 2e-3 + ulp * np.abs(ref)


def _graph_replay(fn):
    """Run fn(stream) once eagerly, then capture it in a CUDA graph and replay it."""
    import torch
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fn(s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn(s)
        g.replay()
        s.synchronize()
    return g


@pytest.fixture(scope="module")
def llama_inputs():
    w = W.LLAMA
    k, v = W.make_kv(w)
    kn, vn = W.make_new_token(w)
    q = W.make_q(w)
    return w, k, v, kn, vn, q


@pytest.mark.parametrize("bits,out_dtype", [(2, "bf16"), (3, "bf16"), (4, "bf16"), (2, "f32")])
def test_llama_full_size_sampled_units(llama_inputs, bits, out_dtype):
    import torch
    from quantized_decode_attention_gb300 import KVCache
    w0, k, v, kn, vn, q = llama_inputs
    w = w0.with_(bits=bits, out_dtype=out_dtype)
    S = w.seq
    cache = KVCache.allocate(cfg_for(w), zero=False)
    cache.quantize(to_device(k, "bf16"), to_device(v, "bf16"), pos0=0)
    kn_d, vn_d, q_d = to_device(kn, "bf16"), to_device(vn, "bf16"), to_device(q, "f32")
    td = torch.float32 if out_dtype == "f32" else torch.bfloat16
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=td, device="cuda")

    def step(s):
        cache.decode_step(kn_d, vn_d, q_d, out, S, stream=s.cuda_stream)

    _graph_replay(step)
    cache.check()
    got_out = out_to_np(out)
    got = lib_views(w, cache, S)
    # the cache the calls describe: token S-1 replaced by the new one (it lies
    # in the recent window at prefill, so the frozen key mean is unchanged)
    kf, vf = k.copy(), v.copy()
    kf[:, :, S - 1], vf[:, :, S - 1] = kn[:, :, 0], vn[:, :, 0]
    nq = S - w.n_sink
    w1 = w.with_(batch=1, n_kv_heads=1, n_q_heads=w.group)
    for b, h in LLAMA_UNITS:
        ku, vu = kf[b:b + 1, h:h + 1], vf[b:b + 1, h:h + 1]
        qk = oracle.quantize_tensor(w1, ku, True, S)
        qv = oracle.quantize_tensor(w1, vu, False, S)
        exp = expected_buffers(w1, qk, qv, nq)
        assert np.array_equal(got["codes_k"][b, h, :nq], exp["codes_k"][0, 0]), (b, h)
        assert np.array_equal(got["codes_v"][b, h, :nq // 2], exp["codes_v"][0, 0, :nq // 2]), (b, h)
        assert np.array_equal(got["meta_k"][b, h, :nq], exp["meta_k"][0, 0]), (b, h)
        assert np.array_equal(got["meta_v"][b, h, :nq], exp["meta_v"][0, 0]), (b, h)
        assert np.array_equal(got["mean_k"][b, h].view(np.uint32), qk.mu[0, 0].view(np.uint32)), (b, h)
        assert np.array_equal(got["raw_k"][b, h, w.n_sink + (S - 1) % w.n_recent], kn[b, h, 0])
        qu = q[b:b + 1, h * w.group:(h + 1) * w.group]
        ref = oracle.attention(w1, qu, ku, vu, S, qk, qv)[0]
        g = got_out[b, h * w.group:(h + 1) * w.group]
        assert np.all(np.abs(g - ref) <= _tol(ref, w.out_dtype)), (b, h, float(np.max(np.abs(g - ref))))
    assert np.all(np.isfinite(got_out))
    cache.close()


def test_nuq_full_size_sampled_units():
    import torch
    from quantized_decode_attention_gb300 import KVCache
    w = W.NUQ
    S = w.seq
    k, v = W.make_kv(w)
    q = W.make_q(w)
    cache = KVCache.allocate(cfg_for(w), zero=False)
    cache.quantize(to_device(k, w.kv_dtype), to_device(v, w.kv_dtype), pos0=0)
    q_d = to_device(q, "f32")
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float16, device="cuda")
    _graph_replay(lambda s: cache.attention(q_d, out, S, stream=s.cuda_stream))
    cache.check()
    got_out = out_to_np(out)
    got, qcap = nuq_views(w, cache, S)
    nq = S - w.n_sink
    w1 = w.with_(batch=1, n_kv_heads=1, n_q_heads=w.group)
    for b, h in NUQ_UNITS:
        ku, vu = k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1]
        nk = OC.quantize_nuq(w1, ku, True, S)
        nv = OC.quantize_nuq(w1, vu, False, S)
        assert np.array_equal(got["lut_k"][b, h], nk.lut[0, 0]), (b, h)
        assert np.array_equal(got["lut_v"][b, h, :nq], nv.lut[0, 0]), (b, h)
        assert np.array_equal(got["codes_k"][b, h, :nq], OC.pack_k(nk.codes, w.bits)[0, 0]), (b, h)
        pv = OC.pack_v(nv.codes, w.bits)[0, 0]
        assert np.array_equal(got["codes_v"][b, h, :nq // 2], pv[:nq // 2]), (b, h)
        rp, col, val = OC.nuq_key_outliers_csr(nk, qcap, got["col_k"].shape[-1])
        assert np.array_equal(got["rowptr"][b, h, :qcap + 1], rp[0, 0]), (b, h)
        n_nz = int(rp[0, 0, -1])
        assert n_nz == w.head_dim * oracle.outlier_count(0.01, nq)
        assert np.array_equal(got["col_k"][b, h, :n_nz], col[0, 0, :n_nz]), (b, h)
        assert np.array_equal(got["val_k"][b, h, :n_nz], val[0, 0, :n_nz]), (b, h)
        cv, vv = OC.nuq_value_outliers(nv, qcap, got["col_v"].shape[-1])
        assert np.array_equal(got["col_v"][b, h, :nq], cv[0, 0, :nq]), (b, h)
        assert np.array_equal(got["val_v"][b, h, :nq], vv[0, 0, :nq]), (b, h)
        qu = q[b:b + 1, h * w.group:(h + 1) * w.group]
        ref = OC.attention(w1, qu, ku, vu, S, nk, nv)[0]
        g = got_out[b, h * w.group:(h + 1) * w.group]
        assert np.all(np.abs(g - ref) <= _tol(ref, w.out_dtype)), (b, h, float(np.max(np.abs(g - ref))))
    assert np.all(np.isfinite(got_out))
    cache.close()


DQ_BATCHES = [0, 31]


def test_dquant_full_size_sampled_sequences():
    """The D-Quant cache of the benchmark (batch 32, 8 KV heads, 16384 bf16
    tokens, 128 recent; keys 8 levels in 331 bytes, values 6 levels in 231
    bytes): containers, metadata and window means of two sequences bit for bit,
    and their 32 query heads' outputs within the attention tolerance."""
    import torch
    from quantized_decode_attention_gb300 import KVCache
    w = W.DQUANT
    S = w.seq
    k, v = W.make_kv(w)
    q = W.make_q(w)
    cache = KVCache.allocate(cfg_for(w), zero=False)
    cache.quantize(to_device(k, "bf16"), to_device(v, "bf16"), pos0=0)
    q_d = to_device(q, "f32")
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    _graph_replay(lambda s: cache.attention(q_d, out, S, stream=s.cuda_stream))
    cache.check()
    got_out = out_to_np(out)
    from helpers import dquant_views
    got, qcap = dquant_views(w, cache, S)
    nq = S - w.n_sink
    w1 = w.with_(batch=1)
    for b in DQ_BATCHES:
        kb, vb = k[b:b + 1], v[b:b + 1]
        dk = OC.quantize_dquant(w1, kb, True, S)
        dv = OC.quantize_dquant(w1, vb, False, S)
        assert not dk.flags.any() and not dv.flags.any()
        assert np.array_equal(got["codes_k"][b, :nq], dk.container[0]), b
        assert np.array_equal(got["codes_v"][b, :nq], dv.container[0]), b
        assert np.array_equal(got["meta_k"][b, :nq, 0], dk.s16[0]) and np.array_equal(got["meta_k"][b, :nq, 1], dk.o16[0])
        assert np.array_equal(got["meta_v"][b, :nq, 0], dv.s16[0]) and np.array_equal(got["meta_v"][b, :nq, 1], dv.o16[0])
        nw = dk.mean_q.shape[1]
        assert np.array_equal(got["mean_q"][b, :nw], dk.mean_q[0])
        assert np.array_equal(got["mean_sc"][b, :nw], dk.mean_sc[0])
        ref = OC.attention(w1, q[b:b + 1], kb, vb, S, dk, dv)[0]
        assert np.all(np.abs(got_out[b] - ref) <= _tol(ref, "bf16")), (b, float(np.max(np.abs(got_out[b] - ref))))
    assert np.all(np.isfinite(got_out))
    cache.close()


QWEN_UNITS = [(0, 0), (3, 7)]


def test_qwen_long_full_size_sampled_units():
    """The Qwen3-8B-shaped long-context cache (batch 4, 32 query / 8 KV heads,
    131072 bf16 tokens, dense key transform with compensated queries, 2-bit
    grid clipped to the 0.1 / 99.9 % quantiles): the new token re-appended at
    the last position and attention over 131072 tokens from one CUDA graph;
    two units' records bit for bit and their heads' outputs within tolerance."""
    import torch
    from quantized_decode_attention_gb300 import KVCache
    w = W.QWEN_LONG.with_(seq=131072)
    S = w.seq
    k, v = W.make_kv(w)
    kn, vn = W.make_new_token(w)
    q = W.make_q(w)
    T, Qc = W.dense_transform(w)
    cache = KVCache.allocate(cfg_for(w), zero=False)
    cache.tensors["k_transform"].view(torch.float32).copy_(torch.from_numpy(T).reshape(-1))
    cache.tensors["q_comp"].view(torch.float32).copy_(torch.from_numpy(Qc).reshape(-1))
    cache.quantize(to_device(k, "bf16"), to_device(v, "bf16"), pos0=0)
    kn_d, vn_d, q_d = to_device(kn, "bf16"), to_device(vn, "bf16"), to_device(q, "f32")
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")

    def step(s):
        cache.quantize(kn_d, vn_d, pos0=S - 1, stream=s.cuda_stream)
        cache.attention(q_d, out, S, stream=s.cuda_stream)

    _graph_replay(step)
    cache.check()
    got_out = out_to_np(out)
    got = lib_views(w, cache, S)
    w1 = w.with_(batch=1, n_kv_heads=1, n_q_heads=w.group)
    for b, h in QWEN_UNITS:
        ku = k[b:b + 1, h:h + 1].copy()
        vu = v[b:b + 1, h:h + 1].copy()
        ku[:, :, S - 1], vu[:, :, S - 1] = kn[b:b + 1, h:h + 1, 0], vn[b:b + 1, h:h + 1, 0]
        qk = oracle.quantize_tensor(w1, ku, True, S, T=T[h:h + 1])
        qv = oracle.quantize_tensor(w1, vu, False, S)
        exp = expected_buffers(w1, qk, qv, S)
        assert np.array_equal(got["codes_k"][b, h, :S], exp["codes_k"][0, 0]), (b, h)
        assert np.array_equal(got["codes_v"][b, h, :S // 2], exp["codes_v"][0, 0, :S // 2]), (b, h)
        assert np.array_equal(got["meta_k"][b, h, :S], exp["meta_k"][0, 0]), (b, h)
        assert np.array_equal(got["meta_v"][b, h, :S], exp["meta_v"][0, 0]), (b, h)
        qu = q[b:b + 1, h * w.group:(h + 1) * w.group]
        ref = oracle.attention(w1, qu, ku, vu, S, qk, qv, q_comp=Qc[h:h + 1])[0]
        g = got_out[b, h * w.group:(h + 1) * w.group]
        assert np.all(np.abs(g - ref) <= _tol(ref, w.out_dtype)), (b, h, float(np.max(np.abs(g - ref))))
    assert np.all(np.isfinite(got_out))
    cache.close()
