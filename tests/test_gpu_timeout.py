"""A bounded device wait that runs out.

Every wait in the kernels here gives up after a time limit, latches a status
bit and lets the kernel return, so that a lost arrival cannot hang the GPU.
This test makes such a wait run out on purpose -- on a barrier nothing arrives
at, in a kernel of its own, with a 2 ms limit -- and checks that dq_check
reports DQ_ETIMEOUT once, that the status is cleared after the report, and that
the context stays usable: the stale per-unit record count the expired kernel
leaves behind is cleared before the next attention call, whose output then
matches the call made before the timeout and the oracle.  No fault and no
hang is involved."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import cfg_for, out_to_np, to_device

pytestmark = pytest.mark.gpu

TOL = 2e-3
REORDER = 1e-5


def test_expired_wait_reports_timeout_and_the_context_recovers():
    import torch
    from quantized_decode_attention_gb300 import DQError, KVCache
    from quantized_decode_attention_gb300 import _lib as B
    lib = B.load()
    w = W.LLAMA.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=300)
    S = w.seq
    k, v = W.make_kv(w)
    q = W.make_q(w)
    cache = KVCache.allocate(cfg_for(w, max_seq=S, out_dtype="f32"))
    cache.quantize(to_device(k, "bf16"), to_device(v, "bf16"))
    cache.check()
    qd = to_device(q, "f32")
    before = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    cache.attention(qd, before, S)
    cache.check()

    stream = torch.cuda.current_stream().cuda_stream
    assert lib.dq_test_expire_wait(cache.ctx, 2_000_000, stream) == 0, lib.dq_last_error()
    with pytest.raises(DQError) as e:
        cache.check()
    assert e.value.name == "DQ_ETIMEOUT", str(e.value)
    cache.check()  # reported once, then cleared

    for i in range(2):
        after = torch.full_like(before, float("nan"))
        cache.attention(qd, after, S)
        cache.check()
        assert float((after - before).abs().max()) <= REORDER, (i, float((after - before).abs().max()))
    qk = oracle.quantize_tensor(w, k, True, S)
    qv = oracle.quantize_tensor(w, v, False, S)
    want = oracle.attention(w, q, k, v, S, qk, qv)
    err = np.abs(out_to_np(after) - want).max()
    assert err <= TOL, float(err)
    cache.close()
