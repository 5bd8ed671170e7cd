"""The C ABI without a GPU: the library builds, loads and exports every entry
point include/dq.h declares; buffer sizes and host-side validation."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from quantized_decode_attention_gb300 import build
    build.build()
    from quantized_decode_attention_gb300 import _lib
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "dq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dq_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"dq_quantize_kv", "dq_decode_attention", "dq_free", "dq_kv_sizes", "dq_check"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def _llama(**kw):
    from quantized_decode_attention_gb300 import make_config
    args = dict(batch=16, n_kv_heads=8, n_q_heads=32, head_dim=128, max_seq=8192, bits=2, n_sink=4, n_recent=128)
    args.update(kw)
    return make_config(**args)


def test_sizes_llama_layout(lib):
    from quantized_decode_attention_gb300 import kv_sizes
    for bits in (2, 3, 4):
        s = kv_sizes(_llama(bits=bits))
        U, qcap, rcap = 128, 8192, 144
        assert qcap % 16 == 0 and (8192 - 4) <= qcap
        assert s["codes_k"] == U * qcap * 128 * bits // 8
        assert s["codes_v"] == U * qcap * 128 * bits // 8
        assert s["meta_k"] == s["meta_v"] == U * qcap * 4
        assert s["mean_k"] == U * 128 * 4
        assert s["raw_k"] == s["raw_v"] == U * rcap * 128 * 2
        assert s["lut_k"] == 0 and s["k_transform"] == 0


def test_accounting_int2_fp16_meta_is_2_25_bpv(lib):
    """D-Quant Sec. 3.1: INT2 with an fp16 scale and zero point per 128 values is 2.25 BPV."""
    from quantized_decode_attention_gb300 import kv_sizes
    s = kv_sizes(_llama(n_sink=0, n_recent=0, mean_k=False, max_seq=16 * 1000))
    values = 128 * 16 * 1000 * 128   # U * tokens * d
    assert (s["codes_k"] + s["meta_k"]) * 8 / values == pytest.approx(2.25)


def test_validation_errors_without_gpu(lib):
    from quantized_decode_attention_gb300 import _lib
    P = C.c_void_p
    bad = [(_llama(n_q_heads=33), 1), (_llama(head_dim=96), 3), (_llama(bits=5), 1),
           (_llama(n_q_heads=64), 3)]
    for cfg, want in bad:
        arr = (C.c_size_t * _lib.NUM_BUFFERS)()
        assert lib.dq_kv_sizes(C.byref(cfg), arr) == want, lib.dq_last_error()
    cfg = _llama()
    ctx = P()
    b = _lib.Buffers()
    # NULL inputs are rejected before any device work
    assert lib.dq_quantize_kv(C.byref(ctx), C.byref(cfg), C.byref(b), None, None, 0, 1, None) == 1
    # a misaligned buffer pointer is rejected on the host
    for n in _lib.BUFFER_NAMES:
        setattr(b, n, 0x10000)
    b.codes_k = 0x10008
    assert lib.dq_quantize_kv(C.byref(ctx), C.byref(cfg), C.byref(b), 0x20000, 0x30000, 0, 1, None) == 2
    assert b"codes_k" in lib.dq_last_error()
    b.codes_k = 0x10000
    # token range beyond max_seq
    assert lib.dq_quantize_kv(C.byref(ctx), C.byref(cfg), C.byref(b), 0x20000, 0x30000, 8190, 5, None) == 1
    assert lib.dq_decode_attention(C.byref(ctx), C.byref(cfg), C.byref(b), 0x20000, 0x30000, 0, 0.1, None) == 1
    assert lib.dq_decode_attention(C.byref(ctx), C.byref(cfg), C.byref(b), 0x20008, 0x30000, 10, 0.1, None) == 2
    assert not ctx  # no context was created by failing calls
    lib.dq_free(None)
    assert lib.dq_check(None, None) == 0
    assert lib.dq_status_name(7) == b"DQ_ENONFINITE"
