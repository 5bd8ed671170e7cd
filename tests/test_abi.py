"""The C ABI without a GPU: the library builds, loads and exports every entry
point include/dq.h declares; buffer sizes and host-side validation."""
import ctypes as C
import os
import re

import numpy as np
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
    # the fused decode step: NULL inputs, a step without a prefilled token, a
    # step past max_seq, a misaligned new token
    step = lambda kn, vn, q, seq: lib.dq_decode_step(C.byref(ctx), C.byref(cfg), C.byref(b), kn, vn, q, 0x30000,
                                                     seq, 0.1, None)
    assert step(None, 0x40000, 0x20000, 10) == 1
    assert step(0x50000, 0x40000, 0x20000, 1) == 1
    assert step(0x50000, 0x40000, 0x20000, 8193) == 1
    assert step(0x50008, 0x40000, 0x20000, 10) == 2
    assert not ctx  # no context was created by failing calls
    lib.dq_free(None)
    assert lib.dq_check(None, None) == 0
    assert lib.dq_test_expire_wait(None, 1000, None) == 1  # needs a context with a workspace
    assert lib.dq_status_name(7) == b"DQ_ENONFINITE"
    assert lib.dq_status_name(8) == b"DQ_ETIMEOUT"


def _dquant(**kw):
    from quantized_decode_attention_gb300 import make_config
    args = dict(batch=32, n_kv_heads=8, n_q_heads=32, head_dim=128, max_seq=16384, scheme="rans",
                rot_k="hadamard", rot_v="none", mean_k=True, n_recent=128, levels_k=8, levels_v=6,
                container_k=331, container_v=231)
    args.update(kw)
    return make_config(**args)


def test_sizes_dquant_layout(lib):
    """D-Quant Sec. 5.1: 331- and 231-byte containers per 1024-value stream with fp16
    (s, o) and an INT8 window mean are 2.68 + 1.84 = 2.26 bits per value on average."""
    from quantized_decode_attention_gb300 import kv_sizes
    s = kv_sizes(_dquant())
    B, qcap, n = 32, 16384, 1024
    assert s["codes_k"] == B * qcap * 331 and s["codes_v"] == B * qcap * 231
    assert s["meta_k"] == s["meta_v"] == B * qcap * 4
    assert s["mean_k"] == B * (qcap // 128) * (n + 16)
    assert s["lut_k"] == 0 and s["ol_col_k"] == 0
    bpv = (s["codes_k"] + s["codes_v"] + s["meta_k"] + s["meta_v"] + s["mean_k"]) * 8 / (2 * B * qcap * n)
    assert bpv == pytest.approx(2.26, abs=0.005)


def test_sizes_dquant_196(lib):
    """D-Quant Sec. 5 ("lower storage budget"): the same 8 / 6 levels at 1.96 bits
    per value.  The sizes the library reports give that budget, and both
    containers hold the cheapest coding of a stream (the model's most probable
    symbol in every position, plus the 32-bit state) with room to spare."""
    import oracle
    import workloads as W
    from quantized_decode_attention_gb300 import kv_sizes
    e = W.DQUANT_196.extra
    s = kv_sizes(_dquant(container_k=e["container_k"], container_v=e["container_v"]))
    B, qcap, n = 32, 16384, 1024
    bpv = (s["codes_k"] + s["codes_v"] + s["meta_k"] + s["meta_v"] + s["mean_k"]) * 8 / (2 * B * qcap * n)
    assert bpv == pytest.approx(1.96, abs=0.005)
    assert bpv == pytest.approx(W.dquant_bits_per_value(W.DQUANT_196), abs=1e-3)
    for M, C in ((8, e["container_k"]), (6, e["container_v"])):
        t = oracle.DqTable(n, M, alpha=1.4)
        cheapest = min(-np.log2(f / 256.0) for f in t.f) * n + 32
        assert cheapest < 8 * C


def test_dquant_model_matches_the_oracle(lib):
    import oracle
    from quantized_decode_attention_gb300._lib import rans_model
    for H, Mk, Mv, Ck, Cv in ((8, 8, 6, 331, 231), (2, 16, 4, 172, 100), (1, 3, 2, 60, 40)):
        cfg = _dquant(n_kv_heads=H, n_q_heads=4 * H, levels_k=Mk, levels_v=Mv, container_k=Ck, container_v=Cv)
        for which, M in ((0, Mk), (1, Mv)):
            f, c = rans_model(cfg, which)
            t = oracle.DqTable(H * 128, M, alpha=1.4)
            assert f == t.f.tolist() and c == t.c.tolist(), (H, M)


def test_dquant_infeasible_container_is_refused(lib):
    """16 levels at 2.26 bits per value cannot fit: the cheapest symbol costs more."""
    from quantized_decode_attention_gb300 import DQError, kv_sizes
    with pytest.raises(DQError) as e:
        kv_sizes(_dquant(levels_k=16, container_k=289))
    assert e.value.status == 4   # DQ_EINFEASIBLE
    kv_sizes(_dquant(levels_k=16, container_k=343))


def test_dquant_validation(lib):
    from quantized_decode_attention_gb300 import DQError, kv_sizes
    for bad in (dict(head_dim=64), dict(n_kv_heads=3, n_q_heads=12), dict(levels_k=17), dict(container_v=4),
                dict(meta_dtype="f32"), dict(rot_k="dense")):
        with pytest.raises(DQError):
            kv_sizes(_dquant(**bad))


def test_dquant_feasible_alphabet_matches_the_oracle(lib):
    """D-Quant App. C (Fig. 6 left): the largest alphabet whose cheapest stream fits
    a container, by the library (as the bench reports it) and by the oracle's own
    symbol model (cheapest symbol cost times n against B = 8C - 32 bits).  The
    entropy-coded container holds at least the levels of fixed-width coding at the
    same rate, and the default 8 / 6 levels lie inside the region at the key and
    value payloads of the 2.26-bit point (331 and 231 bytes)."""
    import oracle
    sys_path_bench()
    import bench
    n = 1024
    got = bench.feasible_alphabet(n)
    for row in got:
        C = row["container_bytes"]
        feas = [M for M in range(2, 17)
                if int(oracle.DqTable(n, M, alpha=1.4).r.min()) * n <= oracle.dq_budget_fx(C)]
        assert row["entropy_coded_levels"] == (max(feas) if feas else None), row
        assert row["entropy_coded_levels"] >= row["fixed_width_levels"], row
    for M, C in ((8, 331), (6, 231)):
        assert int(oracle.DqTable(n, M, alpha=1.4).r.min()) * n <= oracle.dq_budget_fx(C)


def sys_path_bench():
    import os
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)


def test_ablation_reference_is_exact_attention():
    """The D-Quant ablation (Sec. 5.4, Fig. 4) scores each setting against exact
    attention over the unquantized tokens.  That reference, as the bench computes
    it, equals the oracle's fp64 attention on the same bf16 / fp16 tokens, unit by
    unit, with query head h reading KV head floor(h Hkv / Hq)."""
    import oracle
    import workloads as W
    sys_path_bench()
    import bench
    for dt in ("bf16", "f16"):
        w = W.DQUANT.with_(batch=2, n_kv_heads=2, n_q_heads=8, seq=70, kv_dtype=dt)
        k, v = W.make_kv(w)
        q = W.make_q(w)
        got = bench.exact_attention(q, k, v, dt)
        K = oracle.raw16_to_f64(k, dt)
        V = oracle.raw16_to_f64(v, dt)
        G = w.n_q_heads // w.n_kv_heads
        for b in range(w.batch):
            for h in range(w.n_kv_heads):
                ref = oracle.attention_f64(q[b, h * G:(h + 1) * G], K[b, h], V[b, h], w.head_dim ** -0.5)
                np.testing.assert_allclose(got[b, h * G:(h + 1) * G], ref, rtol=1e-12, atol=1e-13)


def test_ablation_settings_feasibility(lib):
    """Every setting of the three ablation axes fits its containers by the symbol
    model, except 16 value levels in 231 bytes: the cheapest 16-level symbol costs
    more than the 1.77 bits per value that container leaves (the dash of D-Quant
    Table 2), which the bench reports as infeasible."""
    import oracle
    sys_path_bench()
    import bench
    n = 1024
    fits = lambda M, C: int(oracle.DqTable(n, M, alpha=1.4).r.min()) * n <= oracle.dq_budget_fx(C)
    for mk, mv in bench.ABL_LEVELS:
        assert fits(mk, 331) and (fits(mv, 231) == (mv != 16)), (mk, mv)
    for ck, cv in bench.ABL_BUDGETS:
        assert fits(8, ck) and fits(6, cv), (ck, cv)
    for ck in bench.ABL_KEY_BYTES:
        assert fits(8, ck) and fits(6, bench.ABL_PAIR_BYTES - ck), ck


def test_quest_step_factor_matches_the_oracle(lib):
    # the library derives alpha_b on its own (bisection on the derivative of the
    # Gaussian error); the oracle by golden-section search on the error itself
    import oracle
    from quantized_decode_attention_gb300 import _lib
    for bits in range(1, 9):
        assert _lib.quest_step(bits) == np.float32(oracle.quest_step_factor(bits)), bits
    c = C.c_float()
    assert lib.dq_quest_step(0, C.byref(c)) == 1 and lib.dq_quest_step(2, None) == 1


def test_quest_grid_validation(lib):
    from quantized_decode_attention_gb300 import _lib, make_config
    arr = (C.c_size_t * _lib.NUM_BUFFERS)()
    base = dict(batch=2, n_kv_heads=2, n_q_heads=8, head_dim=128, max_seq=512, n_sink=4, n_recent=16)
    ref = (C.c_size_t * _lib.NUM_BUFFERS)()
    assert lib.dq_kv_sizes(C.byref(make_config(**base)), ref) == 0
    assert lib.dq_kv_sizes(C.byref(make_config(**base, grid_k="quest")), arr) == 0
    assert list(arr) == list(ref)  # same layout: the grid only picks s and o
    assert lib.dq_kv_sizes(C.byref(make_config(**base, grid_k="quest", clip_k=0.99)), arr) == 1
    cfg = make_config(**base)
    cfg.k.grid = 2
    assert lib.dq_kv_sizes(C.byref(cfg), arr) == 1
    nuq = make_config(**{**base, "n_recent": 0}, scheme="nuq", rot_k="none", rot_v="none", mean_k=False, bits=3)
    nuq.k.grid = 1
    assert lib.dq_kv_sizes(C.byref(nuq), arr) == 3


def test_nuq_group_and_refit_layout_and_validation(lib):
    # KVQuant-NUQ, Configuration reference: value tables per group of 32
    # channels, key tables per refit block of N quantized slots
    from quantized_decode_attention_gb300 import _lib, make_config
    arr = (C.c_size_t * _lib.NUM_BUFFERS)()
    names = _lib.BUFFER_NAMES
    base = dict(batch=2, n_kv_heads=2, n_q_heads=8, head_dim=128, max_seq=1025, kv_dtype="f16", n_sink=1,
                scheme="nuq", rot_k="none", rot_v="none", mean_k=False, bits=3)
    U, d, L, qcap = 4, 128, 8, 1024
    assert lib.dq_kv_sizes(C.byref(make_config(**base)), arr) == 0
    plain = dict(zip(names, list(arr)))
    assert plain["lut_k"] == U * d * L * 2 and plain["lut_v"] == U * qcap * L * 2
    assert lib.dq_kv_sizes(C.byref(make_config(**base, group_size_v=32)), arr) == 0
    grp = dict(zip(names, list(arr)))
    assert grp["lut_v"] == U * qcap * 4 * L * 2 and grp["lut_k"] == plain["lut_k"]
    assert lib.dq_kv_sizes(C.byref(make_config(**base, group_size_v=128)), arr) == 0
    assert dict(zip(names, list(arr)))["lut_v"] == plain["lut_v"]
    assert lib.dq_kv_sizes(C.byref(make_config(**{**base, "n_recent": 256}, refit_k=256)), arr) == 0
    ref = dict(zip(names, list(arr)))
    assert ref["lut_k"] == U * 4 * d * L * 2 + U * 4        # 4 blocks of 256 slots, then the prefill counts
    assert ref["codes_k"] == plain["codes_k"] and ref["lut_v"] == plain["lut_v"]
    bad = [
        (dict(group_size_v=16), 3), (dict(group_size_v=64), 3),              # only 0, 32 or head_dim
        (dict(refit_k=100, n_recent=128), 1), (dict(refit_k=-128, n_recent=128), 1),
        (dict(refit_k=128), 3),                                                # the window must hold a block
        (dict(refit_k=128, n_recent=128, kv_dtype="f32"), 3),                  # 16-bit keys read back
        (dict(refit_k=128, n_recent=128, head_dim=64, bits=2), 3),
        (dict(group_size_v=32, head_dim=64, bits=2), 3),
    ]
    for kw, status in bad:
        cfg = make_config(**{**base, **kw})
        assert lib.dq_kv_sizes(C.byref(cfg), arr) == status, kw
    cfg = make_config(**base)
    cfg.k.group_size = 32                                                      # keys span their tokens
    assert lib.dq_kv_sizes(C.byref(cfg), arr) == 3
    cfg = make_config(**{**base, "n_recent": 128})
    cfg.v.refit_interval = 128                                                 # refits are for keys
    assert lib.dq_kv_sizes(C.byref(cfg), arr) == 1
    aff = make_config(batch=2, n_kv_heads=2, n_q_heads=8, head_dim=128, max_seq=512)
    aff.v.group_size = 32                                                      # non-uniform scheme only
    assert lib.dq_kv_sizes(C.byref(aff), arr) == 1
