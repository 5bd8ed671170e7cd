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
