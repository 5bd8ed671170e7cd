"""The fused decode step (dq_decode_step) against its definition: an append of
token seq_len - 1 followed by decode attention over seq_len tokens.

Every cache buffer after each step must equal, byte for byte, what the two
separate calls leave behind, the step's output must agree with theirs to fp32
summation-order noise (the attention kernel hands its chunks to warps as they
free up, so the order in which partial sums meet varies from run to run), and
both must lie within the attention bound of the oracle.  Cases cover the one-launch path
(affine caches with a recent window: 2, 3 and 4 bits, head_dim 64, a dense key
transform with clipping, the ring wrapping around) and the two-call path a
cache without a recent window takes."""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import cfg_for, out_to_np, to_device

pytestmark = pytest.mark.gpu

TOL = 2e-3
REORDER = 1e-5  # two fp32 sums of the same O(1) terms in different orders

CASES = {
    "llama2": W.LLAMA.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=400),
    "llama3": W.LLAMA.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=400, bits=3),
    "llama4": W.LLAMA.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=400, bits=4),
    "d64-2bit": W.LLAMA.with_(batch=2, n_kv_heads=2, n_q_heads=8, head_dim=64, seq=400, n_sink=2, n_recent=32),
    "dense-clip": W.QWEN_LONG.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=400, n_sink=2, n_recent=16),
    "no-recent": W.LLAMA.with_(batch=1, n_kv_heads=2, n_q_heads=8, seq=400, bits=4, n_sink=1, n_recent=0),
    "quest": W.LLAMA.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=400, grid="quest"),
}


def _cache(w, max_seq, T=None, Qc=None):
    import torch
    from quantized_decode_attention_gb300 import KVCache
    c = KVCache.allocate(cfg_for(w, max_seq=max_seq, out_dtype="f32"))
    if T is not None:
        c.tensors["k_transform"].view(torch.float32).copy_(torch.from_numpy(T).reshape(-1))
        c.tensors["q_comp"].view(torch.float32).copy_(torch.from_numpy(Qc).reshape(-1))
    return c


@pytest.mark.parametrize("name", list(CASES))
def test_decode_step_equals_append_then_attention(name):
    import torch
    w = CASES[name]
    S0, n_steps, max_seq = 300, 7, 512
    k, v = W.make_kv(w, seq=S0 + n_steps)
    q = W.make_q(w)
    T = Qc = None
    if w.rot_k == "dense":
        T, Qc = W.dense_transform(w)
    dt = w.kv_dtype
    fused, ref = _cache(w, max_seq, T, Qc), _cache(w, max_seq, T, Qc)
    for c in (fused, ref):
        c.quantize(to_device(k[:, :, :S0], dt), to_device(v[:, :, :S0], dt), pos0=0)
        c.check()
    qd = to_device(q, "f32")
    out_f = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    out_r = torch.empty_like(out_f)
    for i in range(n_steps):
        t = S0 + i
        kn, vn = to_device(k[:, :, t:t + 1], dt), to_device(v[:, :, t:t + 1], dt)
        fused.decode_step(kn, vn, qd, out_f, t + 1)
        ref.quantize(kn, vn, pos0=t)
        ref.attention(qd, out_r, t + 1)
        fused.check()
        ref.check()
        for n, tf in fused.tensors.items():
            if tf is None or n in ("k_transform", "q_comp"):
                continue
            assert torch.equal(tf, ref.tensors[n]), (name, i, n)
        assert float((out_f - out_r).abs().max()) <= REORDER, (name, i, float((out_f - out_r).abs().max()))
    # the last step against the oracle: the same tokens appended one at a time
    # on the frozen prefill mean
    S = S0 + n_steps
    qk0 = oracle.quantize_tensor(w, k[:, :, :S0], True, S0, T=T)
    qv0 = oracle.quantize_tensor(w, v[:, :, :S0], False, S0)
    qk1 = oracle.quantize_tensor(w, k[:, :, S0:S], True, S, mu_frozen=qk0.mu, pos0=S0, T=T)
    qv1 = oracle.quantize_tensor(w, v[:, :, S0:S], False, S, pos0=S0)
    cat = lambda a0, a1: oracle.QuantTensor(*(np.concatenate([x, y], 2) for x, y in
                                              ((a0.codes, a1.codes), (a0.s, a1.s), (a0.o, a1.o))), a0.mu,
                                            np.concatenate([a0.xhat, a1.xhat], 2))
    want = oracle.attention(w, q, k[:, :, :S], v[:, :, :S], S, cat(qk0, qk1), cat(qv0, qv1), q_comp=Qc)
    err = np.abs(out_to_np(out_f) - want).max()
    assert err <= TOL, (name, float(err))
    fused.close()
    ref.close()
