"""The bench's algorithmic bytes (the numerator of every roofline fraction it
reports), recomputed from the library's own buffer sizes: per quantized slot,
the cache records of dq_kv_sizes divided by their slot capacity, times the
slots a call at full length reads, plus the 16-bit regions, q and out."""
import os
import sys

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


def _qo(w):
    B, Hq, d = w.batch, w.n_q_heads, w.head_dim
    return B * Hq * d * 4 + B * Hq * d * 2          # q fp32 in, out bf16


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_affine_bytes_from_buffer_sizes(lib, bits):
    import bench
    import workloads as W
    from helpers import cfg_for
    from quantized_decode_attention_gb300 import kv_sizes
    w = W.LLAMA.with_(bits=bits)
    S, U, d = w.seq, w.batch * w.n_kv_heads, w.head_dim
    sz = kv_sizes(cfg_for(w))
    qcap = sz["codes_k"] // (U * d * bits // 8)
    assert qcap >= S - w.n_sink and qcap % 64 == 0
    per_slot = (sz["codes_k"] + sz["codes_v"] + sz["meta_k"] + sz["meta_v"]) // (U * qcap)
    n_raw = w.n_sink + w.n_recent
    expect = U * (S - n_raw) * per_slot + sz["mean_k"] + U * n_raw * d * 2 * 2 + _qo(w)
    assert bench.algorithmic_bytes(w, bits, S)["total"] == expect
    # the figures the bench reports at the Llama-3-8B shape: 83.39 / 116.40 / 149.42 MB
    assert round(expect / 1e6, 2) == {2: 83.39, 3: 116.40, 4: 149.42}[bits]


def test_dquant_bytes_from_buffer_sizes(lib):
    import bench
    import workloads as W
    from helpers import cfg_for
    from quantized_decode_attention_gb300 import kv_sizes
    for w in (W.DQUANT, W.DQUANT_196):
        S, B, U, d = w.seq, w.batch, w.batch * w.n_kv_heads, w.head_dim
        sz = kv_sizes(cfg_for(w))
        qcap = sz["meta_k"] // (B * 4)
        per_slot = (sz["codes_k"] + sz["codes_v"] + sz["meta_k"] + sz["meta_v"]) // (B * qcap)
        assert per_slot == w.extra["container_k"] + w.extra["container_v"] + 8
        n_q = S - w.n_sink - w.n_recent
        windows = -(-n_q // 128)
        mean = sz["mean_k"] // (qcap // 128) * windows          # one INT8 record per window read
        expect = B * n_q * per_slot + mean + U * (w.n_sink + w.n_recent) * d * 2 * 2 + _qo(w)
        assert bench.dquant_algorithmic_bytes(w, S)["total"] == expect


def test_nuq_bytes_from_buffer_sizes(lib):
    """Codes and value tables per slot and the key tables from the buffer sizes;
    the side channels at their nominal counts (k per key channel by rank, k_v per
    value token) with 4 bytes an entry, and one row pointer per slot."""
    import bench
    import workloads as W
    from helpers import cfg_for
    from quantized_decode_attention_gb300 import kv_sizes
    w = W.NUQ
    S, U, d, L = w.seq, w.batch * w.n_kv_heads, w.head_dim, 1 << w.bits
    sz = kv_sizes(cfg_for(w))
    qcap = sz["lut_v"] // (U * L * 2)
    n_q = S - w.n_sink
    per_slot = (sz["codes_k"] + sz["codes_v"] + sz["lut_v"]) // (U * qcap)
    kk = int(0.01 * n_q + 0.5)                   # outliers per key channel (41 at 4095 tokens)
    kv = int(0.01 * d + 0.5)                     # per value token (1 at d = 128)
    side = U * (d * kk * 4 + (n_q + 1) * 4) + U * n_q * kv * 4
    expect = U * n_q * per_slot + sz["lut_k"] + side + U * w.n_sink * d * 2 * 2 + _qo(w)
    assert bench.nuq_algorithmic_bytes(w, S)["total"] == expect


def test_nuq_group_refit_bytes_from_buffer_sizes(lib):
    """The grouped / refit variant: value tables per slot from the buffer sizes
    (four per token), one key table set per refit block of the quantized
    tokens read (the buffer holds one per block of the capacity, plus the
    prefill counts), the 16-bit recent window besides the sink."""
    import bench
    from helpers import cfg_for
    from quantized_decode_attention_gb300 import kv_sizes
    w = bench.NUQ_GROUP_REFIT
    S, U, d, L = w.seq, w.batch * w.n_kv_heads, w.head_dim, 1 << w.bits
    sz = kv_sizes(cfg_for(w))
    qcap = sz["codes_k"] // (U * d * w.bits // 8)
    n_q = S - w.n_sink - w.n_recent
    per_slot = (sz["codes_k"] + sz["codes_v"] + sz["lut_v"]) // (U * qcap)
    assert sz["lut_v"] == U * qcap * 4 * L * 2
    blocks = -(-qcap // 128)
    assert sz["lut_k"] == U * blocks * d * L * 2 + U * 4
    kk = int(0.01 * n_q + 0.5)
    kv = int(0.01 * d + 0.5)
    side = U * (d * kk * 4 + (n_q + 1) * 4) + U * n_q * kv * 4
    tables_k = U * (-(-n_q // 128)) * d * L * 2
    expect = U * n_q * per_slot + tables_k + side + U * (w.n_sink + w.n_recent) * d * 2 * 2 + _qo(w)
    assert bench.nuq_algorithmic_bytes(w, S)["total"] == expect
