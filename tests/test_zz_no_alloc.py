"""The allocation-free decode-attention entry point.

Some callers cannot let a library allocate device memory (engines that hand
out all memory from their own pool, decode loops that must not trigger the
synchronization cudaMalloc/cudaFree can cause, fixed memory budgets).  For them
dq_decode_attention_noalloc keeps its split workspace in a static device array.
These tests call it through the C ABI and check it against the context-based
entry point; this file is collected last on purpose.
"""
import ctypes as C

import numpy as np
import pytest

import workloads as W
from helpers import cfg_for, to_device


def _lib():
    import __graft_entry__
    __graft_entry__.build()
    from quantized_decode_attention_gb300 import _lib as B
    return B, B.load()


@pytest.mark.gpu
def test_noalloc_matches_context_entry_point_on_two_calls():
    import torch
    B, lib = _lib()
    from quantized_decode_attention_gb300 import KVCache
    w = W.LLAMA.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=409)
    S = 409
    k, v = W.make_kv(w)
    cache = KVCache.allocate(cfg_for(w, max_seq=S, out_dtype="f32"))
    cache.quantize(to_device(k, "bf16"), to_device(v, "bf16"))
    cache.check()
    stream = torch.cuda.current_stream().cuda_stream
    bufs = cache.buffers()
    for call in range(2):
        q = to_device(W.make_q(w, salt=call), "f32")
        ref = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
        got = torch.full_like(ref, float("nan"))
        cache.attention(q, ref, S)
        st = lib.dq_decode_attention_noalloc(C.byref(cache.cfg), C.byref(bufs), q.data_ptr(), got.data_ptr(),
                                             S, w.head_dim ** -0.5, stream)
        assert st == 0, lib.dq_last_error()
        torch.cuda.synchronize()
        err = (got - ref).abs().max().item()
        assert np.isfinite(err) and err <= 2e-3, (call, err)
    cache.check()
    cache.close()


def test_noalloc_refuses_configs_beyond_its_scratch():
    B, lib = _lib()
    from quantized_decode_attention_gb300 import make_config
    cfg = make_config(batch=4097, n_kv_heads=8, n_q_heads=32, head_dim=128, max_seq=1024)
    b = B.Buffers()
    for n in B.BUFFER_NAMES:
        setattr(b, n, 0x10000)
    st = lib.dq_decode_attention_noalloc(C.byref(cfg), C.byref(b), 0x20000, 0x30000, 100, 0.1, None)
    assert st == 1
    assert b"allocation-free limit" in lib.dq_last_error()


def _noalloc(lib, cache, q, out, S, stream):
    b = cache.buffers()
    return lib.dq_decode_attention_noalloc(C.byref(cache.cfg), C.byref(b), q.data_ptr(), out.data_ptr(), S,
                                           cache.cfg.head_dim ** -0.5, stream)


@pytest.mark.gpu
def test_noalloc_dense_transform_matches_context_and_oracle():
    # a dense (learned) key transform with clipping: the queries are
    # compensated inside the kernel, since this entry point has no workspace
    # for the compensated copy the context-based call keeps
    import torch
    import oracle
    from helpers import out_to_np
    B, lib = _lib()
    from quantized_decode_attention_gb300 import KVCache
    w = W.QWEN_LONG.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=400, n_sink=2, n_recent=16)
    S = w.seq
    k, v = W.make_kv(w)
    q = W.make_q(w)
    T, Qc = W.dense_transform(w)
    cache = KVCache.allocate(cfg_for(w, max_seq=S, out_dtype="f32"))
    cache.tensors["k_transform"].view(torch.float32).copy_(torch.from_numpy(T).reshape(-1))
    cache.tensors["q_comp"].view(torch.float32).copy_(torch.from_numpy(Qc).reshape(-1))
    cache.quantize(to_device(k, w.kv_dtype), to_device(v, w.kv_dtype))
    cache.check()
    qd = to_device(q, "f32")
    ref = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    got = torch.full_like(ref, float("nan"))
    cache.attention(qd, ref, S)
    st = _noalloc(lib, cache, qd, got, S, torch.cuda.current_stream().cuda_stream)
    assert st == 0, lib.dq_last_error()
    cache.check()
    assert float((got - ref).abs().max()) <= 1e-5, float((got - ref).abs().max())
    qk = oracle.quantize_tensor(w, k, True, S, T=T)
    qv = oracle.quantize_tensor(w, v, False, S)
    want = oracle.attention(w, q, k, v, S, qk, qv, q_comp=Qc)
    err = np.abs(out_to_np(got) - want).max()
    assert err <= 2e-3, float(err)
    cache.close()


@pytest.mark.gpu
def test_noalloc_admits_batch_256_and_refuses_batch_1024():
    # 256 sequences x 8 KV heads at head_dim 128 (2048 units, four record
    # slots each) fit the static scratch; 1024 x 8 (8192 units) do not, and
    # are refused on the host with the partials message before any launch.
    # Real, zeroed buffers back both configs all the same.
    import torch
    B, lib = _lib()
    from quantized_decode_attention_gb300 import KVCache
    stream = torch.cuda.current_stream().cuda_stream
    S = 2048
    w = W.LLAMA.with_(batch=256, seq=S)
    g = torch.Generator(device="cuda").manual_seed(7)
    cache = KVCache.allocate(cfg_for(w, max_seq=S, out_dtype="f32"))
    shape = (w.batch, w.n_kv_heads, S, w.head_dim)
    kd = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    vd = torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)
    cache.quantize(kd, vd)
    del kd, vd
    qd = torch.randn((w.batch, w.n_q_heads, w.head_dim), generator=g, device="cuda")
    ref = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    got = torch.full_like(ref, float("nan"))
    cache.attention(qd, ref, S)
    st = _noalloc(lib, cache, qd, got, S, stream)
    assert st == 0, lib.dq_last_error()
    cache.check()
    # both calls hand chunks to warps as they free up; over 2048 tokens and a
    # million outputs the differently ordered fp32 sums part by a few 1e-5 at
    # most, while a lost or doubled record would move outputs by 1e-2 or more
    assert float((got - ref).abs().max()) <= 2e-4, float((got - ref).abs().max())
    cache.close()

    big = KVCache.allocate(cfg_for(W.LLAMA.with_(batch=1024, seq=S), max_seq=S, out_dtype="f32"))
    q = torch.zeros((1024, w.n_q_heads, w.head_dim), device="cuda")
    out = torch.zeros_like(q)
    st = _noalloc(lib, big, q, out, S, stream)
    assert st == 1
    assert b"split partials need" in lib.dq_last_error()
    torch.cuda.synchronize()
    big.close()
