"""GPU parity of the affine path against the CPU oracle, through the C ABI.

Bit-exact: packed key/value records, fp16/fp32 scale-offset, the fp32 key
channel mean, the 16-bit sink/recent slots and the dequantized fp32 values.
Attention: max-abs error <= 2e-3 against the fp64 oracle on the same
quantized cache (fp32 output); a bf16 output may add its own rounding, at
most half a bf16 ulp of the result (<= 2^-8 |y|).
"""
import numpy as np
import pytest

import oracle
import workloads as W
from helpers import cfg_for, expected_buffers, lib_views, out_to_np, to_device

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def small(w, **kw):
    return w.with_(**kw)


CASES = {
    "tiny": (W.TINY, 128),
    "llama2-ragged": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=409), 409),
    "llama3-ragged": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=409, bits=3), 409),
    "llama4-ragged": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=409, bits=4), 409),
    "llama2-short": (small(W.LLAMA, batch=1, n_kv_heads=2, n_q_heads=8, seq=100), 100),
    "llama2-meta32": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=409, meta_dtype="f32"), 409),
    # the QuEST grid ("WUSH-KV", evaluation) on the same caches
    "llama2-quest": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=409, grid="quest"), 409),
    "llama3-quest": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=409, bits=3, grid="quest"), 409),
    "llama4-quest-meta32": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=409, bits=4, grid="quest",
                                  meta_dtype="f32"), 409),
    "d64-quest": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, head_dim=64, seq=300, n_sink=2,
                        n_recent=32, grid="quest"), 300),
    "qwen-dense-quest": (small(W.QWEN_LONG, batch=2, n_kv_heads=2, n_q_heads=8, seq=333, clip=0.0,
                               grid="quest"), 333),
    "llama3-meta32": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=409, bits=3, meta_dtype="f32"), 409),
    "llama2-g2": (small(W.LLAMA, batch=2, n_kv_heads=4, n_q_heads=8, seq=257), 257),
    "qwen-dense-clip": (small(W.QWEN_LONG, batch=2, n_kv_heads=2, n_q_heads=8, seq=333), 333),
    "d64-bf16-2bit": (small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, head_dim=64, seq=300, n_sink=2,
                            n_recent=32), 300),
    "fp16-novrot": (small(W.LLAMA, batch=1, n_kv_heads=2, n_q_heads=8, seq=290, kv_dtype="f16", rot_v="none",
                          bits=4, n_sink=1, n_recent=0), 290),
}


def run_case(w, S, out_dtype="f32"):
    import torch
    from quantized_decode_attention_gb300 import KVCache
    k, v = W.make_kv(w, seq=S)
    q = W.make_q(w)
    T = Qc = None
    if w.rot_k == "dense":
        T, Qc = W.dense_transform(w)
    cache = KVCache.allocate(cfg_for(w, max_seq=S, out_dtype=out_dtype))
    if T is not None:
        cache.tensors["k_transform"].view(torch.float32).copy_(torch.from_numpy(T).reshape(-1))
        cache.tensors["q_comp"].view(torch.float32).copy_(torch.from_numpy(Qc).reshape(-1))
    cache.quantize(to_device(k, w.kv_dtype), to_device(v, w.kv_dtype), pos0=0)
    cache.check()
    return cache, k, v, q, T, Qc


@pytest.mark.parametrize("name", list(CASES))
def test_quantize_bit_exact(name):
    import torch
    w, S = CASES[name]
    cache, k, v, q, T, Qc = run_case(w, S)
    qk = oracle.quantize_tensor(w, k, True, S, T=T)
    qv = oracle.quantize_tensor(w, v, False, S)
    nq = S - w.n_sink
    exp = expected_buffers(w, qk, qv, nq)
    got = lib_views(w, cache, S)
    assert np.array_equal(got["codes_k"][:, :, :nq], exp["codes_k"])
    npair = nq // 2
    assert np.array_equal(got["codes_v"][:, :, :npair], exp["codes_v"][:, :, :npair])
    if nq % 2:
        for b in range(w.batch):
            for h in range(w.n_kv_heads):
                cg = oracle.unpack_v_token(got["codes_v"][b, h, npair], w.head_dim, w.bits, 0)
                assert np.array_equal(cg, qv.codes[b, h, nq - 1])
    assert np.array_equal(got["meta_k"][:, :, :nq], exp["meta_k"])
    assert np.array_equal(got["meta_v"][:, :, :nq], exp["meta_v"])
    if w.mean_k:
        assert np.array_equal(got["mean_k"].view(np.uint32), qk.mu.view(np.uint32))
    # 16-bit regions
    for which, x in (("raw_k", k), ("raw_v", v)):
        reg = oracle.raw_regions(w, x, S)
        for slot, bits16 in reg.items():
            if which == "raw_k":
                g = got[which][:, :, slot]
            else:
                g = got[which][:, :, slot >> 1, :, slot & 1]
            assert np.array_equal(g, bits16), (which, slot)
    # dequantize export, bit-exact fp32
    for which, qt in ((0, qk), (1, qv)):
        out = torch.empty((w.batch, w.n_kv_heads, nq, w.head_dim), dtype=torch.float32, device="cuda")
        cache.dequantize(which, 0, nq, out)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy().view(np.uint32), qt.xhat.view(np.uint32)), which
    cache.close()


@pytest.mark.parametrize("name", list(CASES))
@pytest.mark.parametrize("out_dtype", ["f32", "bf16"])
def test_attention_parity(name, out_dtype):
    import torch
    w, S = CASES[name]
    cache, k, v, q, T, Qc = run_case(w, S, out_dtype=out_dtype)
    qk = oracle.quantize_tensor(w, k, True, S, T=T)
    qv = oracle.quantize_tensor(w, v, False, S)
    td = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[out_dtype]
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=td, device="cuda")
    # the recent ring holds the latest tokens of the last write, so shorter
    # lengths are only meaningful without a recent window
    lens = {S} if w.n_recent else {S, max(1, S - 37), min(S, w.n_sink + 1), 1}
    for seq_len in sorted(lens):
        cache.attention(to_device(q, "f32"), out, seq_len)
        cache.check()
        ref = oracle.attention(w, q, k, v, seq_len, qk, qv, q_comp=Qc)
        got = out_to_np(out)
        err = np.abs(got - ref)
        bound = TOL + (2.0 ** -8 * np.abs(ref) if out_dtype == "bf16" else 0.0)
        assert np.all(err <= bound), (seq_len, float(err.max()))
    cache.close()


def test_append_decode_tokens():
    """Prefill, then append tokens one at a time with the frozen mean; the codes of
    appended tokens, the recent ring and attention after each append match."""
    import torch
    from quantized_decode_attention_gb300 import KVCache
    w = small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=400)
    S0, n_new = 300, 6
    k, v = W.make_kv(w, seq=S0 + n_new)
    q = W.make_q(w)
    cache = KVCache.allocate(cfg_for(w, max_seq=512, out_dtype="f32"))
    cache.quantize(to_device(k[:, :, :S0], "bf16"), to_device(v[:, :, :S0], "bf16"), pos0=0)
    qk0 = oracle.quantize_tensor(w, k[:, :, :S0], True, S0)
    qv0 = oracle.quantize_tensor(w, v[:, :, :S0], False, S0)
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    for i in range(n_new):
        t = S0 + i
        cache.quantize(to_device(k[:, :, t:t + 1], "bf16"), to_device(v[:, :, t:t + 1], "bf16"), pos0=t)
        S = t + 1
        qk1 = oracle.quantize_tensor(w, k[:, :, S0:S], True, S, mu_frozen=qk0.mu, pos0=S0)
        qv1 = oracle.quantize_tensor(w, v[:, :, S0:S], False, S, pos0=S0)
        qk = oracle.QuantTensor(*(np.concatenate([a, b], 2) for a, b in
                                  ((qk0.codes, qk1.codes), (qk0.s, qk1.s), (qk0.o, qk1.o))), qk0.mu,
                                np.concatenate([qk0.xhat, qk1.xhat], 2))
        qv = oracle.QuantTensor(*(np.concatenate([a, b], 2) for a, b in
                                  ((qv0.codes, qv1.codes), (qv0.s, qv1.s), (qv0.o, qv1.o))), qv0.mu,
                                np.concatenate([qv0.xhat, qv1.xhat], 2))
        got = lib_views(w, cache, 512)
        slot = t - w.n_sink
        assert np.array_equal(got["codes_k"][:, :, slot], oracle.pack_k(qk.codes[:, :, slot:slot + 1], w.bits)[:, :, 0])
        assert np.array_equal(got["raw_k"][:, :, w.n_sink + t % w.n_recent], k[:, :, t])
        cache.attention(to_device(q, "f32"), out, S)
        cache.check()
        ref = oracle.attention(w, q, k[:, :, :S], v[:, :, :S], S, qk, qv)
        assert np.abs(out_to_np(out) - ref).max() <= TOL
    cache.close()


def test_nonfinite_input_is_reported():
    from quantized_decode_attention_gb300 import DQError, KVCache
    w = small(W.LLAMA, batch=1, n_kv_heads=2, n_q_heads=8, seq=64, n_sink=0, n_recent=0)
    k, v = W.make_kv(w)
    k = k.copy()
    k[0, 1, 5, 3] = 0x7FC0  # bf16 NaN
    cache = KVCache.allocate(cfg_for(w))
    cache.quantize(to_device(k, "bf16"), to_device(v, "bf16"))
    with pytest.raises(DQError) as e:
        cache.check()
    assert e.value.name == "DQ_ENONFINITE"
    cache.check()  # cleared
    cache.close()


def test_unquantized_16bit_cache():
    """Every token a 16-bit slot (n_sink = the whole sequence): the cache holds the
    inputs as given and attention is exact to fp32 rounding."""
    import torch
    from quantized_decode_attention_gb300 import KVCache
    w = small(W.LLAMA, batch=2, n_kv_heads=2, n_q_heads=8, seq=300, n_sink=300, n_recent=0)
    k, v = W.make_kv(w)
    q = W.make_q(w)
    cache = KVCache.allocate(cfg_for(w, out_dtype="f32"))
    cache.quantize(to_device(k, "bf16"), to_device(v, "bf16"))
    rcap = -(-300 // 16) * 16
    raw_k = cache.tensors["raw_k"].cpu().numpy().view(np.uint16).reshape(w.batch, w.n_kv_heads, rcap, w.head_dim)
    assert np.array_equal(raw_k[:, :, :300], k)
    out = torch.empty((w.batch, w.n_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    cache.attention(to_device(q, "f32"), out, 300)
    cache.check()
    qk = oracle.quantize_tensor(w, k, True, 300)
    qv = oracle.quantize_tensor(w, v, False, 300)
    ref = oracle.attention(w, q, k, v, 300, qk, qv)
    assert np.abs(out_to_np(out) - ref).max() <= TOL
    cache.close()
