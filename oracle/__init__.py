"""CPU oracle for quantized decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The CUDA library never does, and
this package never imports the CUDA library: the two share nothing but the
seeded input generators in ``workloads.py``.

The arithmetic lives in plain C (``affine.c``, ``format.c``, ``nuq.c``, ``rans.c``), compiled with
``-O2 -ffp-contract=off`` into ``liboracle.so``; this module only marshals
arguments and assembles whole-cache buffers from per-token C results.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = ["affine.c", "format.c", "nuq.c", "rans.c"]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so from the C sources next to this file."""
    srcs = [os.path.join(_HERE, s) for s in _SRCS if os.path.exists(os.path.join(_HERE, s))]
    newest = max(os.path.getmtime(s) for s in srcs)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-fopenmp", "-o", tmp] + srcs + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = np.ctypeslib.ndpointer
_f32 = _P(dtype=np.float32, flags="C_CONTIGUOUS")
_f64 = _P(dtype=np.float64, flags="C_CONTIGUOUS")
_u8 = _P(dtype=np.uint8, flags="C_CONTIGUOUS")


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB_PATH)
            L.or_f32_to_f16.restype = C.c_uint16
            L.or_f32_to_f16.argtypes = [C.c_float]
            L.or_f16_to_f32.restype = C.c_float
            L.or_f16_to_f32.argtypes = [C.c_uint16]
            L.or_fwht_f32.argtypes = [_f32, C.c_int]
            L.or_fwht_f64.argtypes = [_f64, C.c_int]
            L.or_hadamard_scale.restype = C.c_float
            L.or_hadamard_scale.argtypes = [C.c_int]
            L.or_rotate_hadamard.argtypes = [_f32, _f32, C.c_int]
            L.or_rotate_dense.argtypes = [_f32, _f32, _f32, C.c_int]
            L.or_quantile_pos.argtypes = [C.c_double, C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_float)]
            L.or_affine_quantize.argtypes = [_f32, C.c_int, C.c_int, C.c_int, C.c_double, C.c_float, _u8,
                                             C.POINTER(C.c_float), C.POINTER(C.c_float)]
            L.or_quest_mse.restype = C.c_double
            L.or_quest_mse.argtypes = [C.c_double, C.c_int]
            L.or_quest_alpha_exact.restype = C.c_double
            L.or_quest_alpha_exact.argtypes = [C.c_int]
            L.or_quest_alpha.restype = C.c_double
            L.or_quest_alpha.argtypes = [C.c_int]
            L.or_quest_step_factor.restype = C.c_float
            L.or_quest_step_factor.argtypes = [C.c_int]
            L.or_quest_rms.restype = C.c_float
            L.or_quest_rms.argtypes = [_f32, C.c_int]
            L.or_affine_dequant.argtypes = [_u8, C.c_int, C.c_float, C.c_float, C.c_void_p, _f32]
            L.or_quantize_unit.argtypes = [_f32, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_int,
                                           C.c_int, C.c_int, _f32, C.c_int, C.c_int, C.c_double,
                                           C.c_float, C.c_int, _u8, _f32, _f32, C.c_void_p]
            L.or_dequant_f64.argtypes = [_u8, _f32, _f32, C.c_void_p, C.c_int, C.c_int, C.c_int, _f64]
            L.or_attention_f64.argtypes = [_f64, _f64, _f64, C.c_int, C.c_int, C.c_int, C.c_double, _f64]
            L.or_k_row_bytes.restype = C.c_int
            L.or_k_row_bytes.argtypes = [C.c_int, C.c_int]
            L.or_v_pair_bytes.restype = C.c_int
            L.or_v_pair_bytes.argtypes = [C.c_int, C.c_int]
            L.or_pack_k_row.argtypes = [_u8, C.c_int, C.c_int, _u8]
            L.or_unpack_k_row.argtypes = [_u8, C.c_int, C.c_int, _u8]
            L.or_pack_v_token.argtypes = [_u8, C.c_int, C.c_int, C.c_int, C.c_void_p]
            L.or_unpack_v_token.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, _u8]
            L.or_raw_v_index.restype = C.c_long
            L.or_raw_v_index.argtypes = [C.c_int, C.c_int, C.c_int]
            L.or_raw_slot.restype = C.c_int
            L.or_raw_slot.argtypes = [C.c_long, C.c_int, C.c_int]
            _u16 = _P(dtype=np.uint16, flags="C_CONTIGUOUS")
            L.or_topk_abs.argtypes = [_f32, C.c_int, C.c_int, _u8]
            L.or_outlier_count.restype = C.c_int
            L.or_outlier_count.argtypes = [C.c_float, C.c_int]
            L.or_r32_sum.restype = C.c_float
            L.or_r32_sum.argtypes = [_f32, C.c_int]
            L.or_nuq_fit.restype = C.c_int
            L.or_nuq_fit.argtypes = [_f32, C.c_void_p, C.c_int, C.c_int, C.c_int, _f32, C.c_void_p]
            L.or_nuq_assign.argtypes = [_f32, C.c_int, _u16, C.c_int, _u8]
            L.or_nuq_vector.restype = C.c_int
            L.or_nuq_vector.argtypes = [_f32, C.c_int, C.c_int, C.c_int, C.c_float, _u8, _u16, _u8]
            L.or_nuq_vector_grouped.restype = C.c_int
            L.or_nuq_vector_grouped.argtypes = [_f32, C.c_int, C.c_int, C.c_int, C.c_int, C.c_float, _u8, _u16, _u8]
            _i32 = _P(dtype=np.int32, flags="C_CONTIGUOUS")
            _i64 = _P(dtype=np.int64, flags="C_CONTIGUOUS")
            L.or_dq_expected_max.restype = C.c_double
            L.or_dq_expected_max.argtypes = [C.c_int]
            L.or_dq_table.restype = C.c_int
            L.or_dq_table.argtypes = [C.c_int, C.c_int, C.c_double, C.c_int, _i32, _i32, _f64]
            L.or_dq_costs.argtypes = [_i32, C.c_int, C.c_int, _i64]
            L.or_dq_pow2_table.argtypes = [_f32]
            L.or_dq_drift.restype = C.c_int
            L.or_dq_drift.argtypes = [_f32, C.c_int, C.c_float, C.c_float, _i64, C.c_int, C.c_longlong, _f32,
                                      _u8, C.POINTER(C.c_longlong)]
            L.or_dq_refit.argtypes = [_f32, _u8, C.c_int, C.POINTER(C.c_float), C.POINTER(C.c_float)]
            L.or_rans_encode.restype = C.c_int
            L.or_rans_encode.argtypes = [_u8, C.c_int, _i32, _i32, C.c_int, C.c_int, _u8]
            L.or_rans_decode.restype = C.c_int
            L.or_rans_decode.argtypes = [_u8, C.c_int, C.c_int, _i32, _i32, C.c_int, C.c_int, _u8,
                                         C.POINTER(C.c_uint32), C.POINTER(C.c_int)]
            L.or_dq_encode_stream.restype = C.c_int
            L.or_dq_encode_stream.argtypes = [_f32, C.c_int, C.c_int, C.c_int, _i32, _i32, C.c_int, _i64, _f32,
                                              _u8, C.POINTER(C.c_uint16), C.POINTER(C.c_uint16), _u8, C.c_void_p]
            L.or_dq_window_mean.argtypes = [_f32, C.c_int, C.c_int, _P(dtype=np.int8, flags="C_CONTIGUOUS"),
                                            C.POINTER(C.c_uint16), _f32]
            L.or_dq_encode_streams.argtypes = [_f32, C.c_int, C.c_int, C.c_int, C.c_int, _i32, _i32, C.c_int, _i64,
                                               _f32, _u8, _u16, _u16, _u8, _i32]
            L.or_rotate_hadamard_rows.argtypes = [_f32, _f32, C.c_long, C.c_int]
            _lib = L
        return _lib


# ---------------------------------------------------------------------------
# thin per-step wrappers (used by the pin tests)
# ---------------------------------------------------------------------------

def f32_to_f16_bits(x) -> np.ndarray:
    L = lib()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([L.or_f32_to_f16(float(v)) for v in x], dtype=np.uint16)


def f16_bits_to_f32(h) -> np.ndarray:
    L = lib()
    h = np.asarray(h, dtype=np.uint16).ravel()
    return np.array([L.or_f16_to_f32(int(v)) for v in h], dtype=np.float32)


def fwht(x: np.ndarray) -> np.ndarray:
    x = np.array(x, dtype=np.float32 if np.asarray(x).dtype != np.float64 else np.float64, copy=True)
    fn = lib().or_fwht_f64 if x.dtype == np.float64 else lib().or_fwht_f32
    fn(x, x.shape[-1])
    return x


def rotate_hadamard(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    lib().or_rotate_hadamard(x, y, x.shape[-1])
    return y


def rotate_hadamard_rows(x: np.ndarray) -> np.ndarray:
    """The normalized Hadamard rotation of every row (last axis) of x."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    d = x.shape[-1]
    lib().or_rotate_hadamard_rows(x, y, x.size // d, d)
    return y


def rotate_dense(T: np.ndarray, x: np.ndarray) -> np.ndarray:
    T = np.ascontiguousarray(T, dtype=np.float32)
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    lib().or_rotate_dense(T, x, y, x.shape[-1])
    return y


def hadamard_scale(d: int) -> float:
    return float(lib().or_hadamard_scale(d))


def quantile_pos(kappa: float, n: int):
    i = C.c_int()
    f = C.c_float()
    lib().or_quantile_pos(kappa, n, C.byref(i), C.byref(f))
    return i.value, f.value


def affine_quantize(x: np.ndarray, bits: int, meta_f16: bool, clip: float = 0.0, quest: bool = False):
    """One token's codes and stored (s, o): min/max grid, quantile clip, or the
    QuEST grid (quest=True)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.zeros(x.shape[-1], dtype=np.uint8)
    s, o = C.c_float(), C.c_float()
    qc = quest_step_factor(bits) if quest else 0.0
    lib().or_affine_quantize(x, x.shape[-1], bits, int(meta_f16), clip, qc, codes, C.byref(s), C.byref(o))
    return codes, np.float32(s.value), np.float32(o.value)


def quest_mse(alpha: float, levels: int) -> float:
    """Mean squared error on N(0,1) of the symmetric grid clipped at +-alpha."""
    return float(lib().or_quest_mse(alpha, levels))


def quest_alpha(bits: int, exact: bool = False) -> float:
    """The MSE-optimal Gaussian clip alpha_b (rounded to 4 decimals unless exact)."""
    return float(lib().or_quest_alpha_exact(bits) if exact else lib().or_quest_alpha(bits))


def quest_step_factor(bits: int) -> float:
    """fp32 c_b = 2 alpha_b / 2^bits (s = c_b * RMS)."""
    return float(lib().or_quest_step_factor(bits))


def quest_rms(x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return float(lib().or_quest_rms(x, x.shape[-1]))


def affine_dequant(codes, s, o, mu=None) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[-1], dtype=np.float32)
    mu_p = None
    if mu is not None:
        mu = np.ascontiguousarray(mu, dtype=np.float32)
        mu_p = mu.ctypes.data_as(C.c_void_p)
    lib().or_affine_dequant(codes, codes.shape[-1], float(s), float(o), mu_p, out)
    return out


def pack_k_row(codes, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    d = codes.shape[-1]
    row = np.zeros(lib().or_k_row_bytes(d, bits), dtype=np.uint8)
    lib().or_pack_k_row(codes, d, bits, row)
    return row


def unpack_k_row(row, d: int, bits: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    out = np.zeros(d, dtype=np.uint8)
    lib().or_unpack_k_row(row, d, bits, out)
    return out


def pack_v_token(codes, bits: int, e: int, rec: np.ndarray) -> None:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    assert rec.flags.c_contiguous and rec.dtype == np.uint8
    lib().or_pack_v_token(codes, codes.shape[-1], bits, e, rec.ctypes.data_as(C.c_void_p))


def unpack_v_token(rec, d: int, bits: int, e: int) -> np.ndarray:
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    out = np.zeros(d, dtype=np.uint8)
    lib().or_unpack_v_token(rec.ctypes.data_as(C.c_void_p), d, bits, e, out)
    return out


def raw_slot(t: int, n_sink: int, n_recent: int) -> int:
    return lib().or_raw_slot(t, n_sink, n_recent)


def topk_abs(x, k: int) -> np.ndarray:
    """Rank-based top-k by |x| (ties to the lower index) -> bool mask."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flag = np.zeros(x.size, dtype=np.uint8)
    lib().or_topk_abs(x, x.size, int(k), flag)
    return flag.astype(bool)


def outlier_count(f: float, n: int) -> int:
    return int(lib().or_outlier_count(float(f), int(n)))


def r32_sum(x) -> float:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return float(lib().or_r32_sum(x, x.size))


def nuq_fit(x, levels: int, iters: int, exclude=None):
    """Lloyd-Max levels of the non-excluded values: (fp32 levels, fp16 bits, n_fit)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    lev = np.zeros(levels, dtype=np.float32)
    lut = np.zeros(levels, dtype=np.uint16)
    ex = None
    if exclude is not None:
        ex = np.ascontiguousarray(exclude, dtype=np.uint8)
    nf = lib().or_nuq_fit(x, None if ex is None else ex.ctypes.data_as(C.c_void_p), x.size, levels, iters, lev,
                          lut.ctypes.data_as(C.c_void_p))
    return lev, lut, nf


def nuq_assign(x, lut16) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    lut16 = np.ascontiguousarray(lut16, dtype=np.uint16)
    codes = np.zeros(x.size, dtype=np.uint8)
    lib().or_nuq_assign(x, x.size, lut16, lut16.size, codes)
    return codes


def nuq_vector(x, bits: int, iters: int, frac: float):
    """One vector: (outlier mask, fp16 table, codes)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flag = np.zeros(x.size, dtype=np.uint8)
    lut = np.zeros(1 << bits, dtype=np.uint16)
    codes = np.zeros(x.size, dtype=np.uint8)
    lib().or_nuq_vector(x, x.size, bits, iters, float(frac), flag, lut, codes)
    return flag.astype(bool), lut, codes


def nuq_vector_grouped(x, bits: int, iters: int, frac: float, group: int):
    """One vector fitted per group of `group` elements: (outlier mask, fp16
    tables [n / group, 2^bits], codes); outliers ranked over the whole vector."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if group <= 0 or x.size % group:
        raise ValueError("group must divide the vector")
    flag = np.zeros(x.size, dtype=np.uint8)
    lut = np.zeros((x.size // group, 1 << bits), dtype=np.uint16)
    codes = np.zeros(x.size, dtype=np.uint8)
    lib().or_nuq_vector_grouped(x, x.size, group, bits, iters, float(frac), flag, lut, codes)
    return flag.astype(bool), lut, codes


# ---- D-Quant container (rans.c) ---------------------------------------------

class DqTable:
    """Frequency table of one tensor: f, c (int32), fixed-point costs r (int64),
    the unsharpened bin probabilities, and the prob precision p."""

    def __init__(self, n: int, M: int, alpha: float = 1.4, p: int = 8):
        self.n, self.M, self.alpha, self.p = n, M, alpha, p
        self.f = np.zeros(M, dtype=np.int32)
        self.c = np.zeros(M, dtype=np.int32)
        self.prob = np.zeros(M, dtype=np.float64)
        if lib().or_dq_table(n, M, float(alpha), p, self.f, self.c, self.prob) != 0:
            raise ValueError("no valid frequency table")
        self.r = np.zeros(M, dtype=np.int64)
        lib().or_dq_costs(self.f, M, p, self.r)

    @classmethod
    def from_freqs(cls, f, p: int = 8) -> "DqTable":
        """A table with given frequencies (summing to 2^p), for hand-worked cases."""
        t = cls.__new__(cls)
        t.n, t.M, t.alpha, t.p = 0, len(f), 1.0, p
        t.f = np.ascontiguousarray(f, dtype=np.int32)
        t.c = np.concatenate([[0], np.cumsum(t.f)[:-1]]).astype(np.int32)
        t.prob = t.f / float(1 << p)
        t.r = np.zeros(t.M, dtype=np.int64)
        lib().or_dq_costs(t.f, t.M, p, t.r)
        return t


def dq_expected_max(n: int) -> float:
    return float(lib().or_dq_expected_max(n))


def dq_pow2_table() -> np.ndarray:
    F = np.zeros(512, dtype=np.float32)
    lib().or_dq_pow2_table(F)
    return F


def dq_budget_fx(C_bytes: int) -> int:
    """B * 2^16 with B = 8C - 32 (sigma = a 32-bit state)."""
    return (8 * C_bytes - 32) * 65536


def dq_drift(x, s: float, o: float, tab: DqTable, C_bytes: int | None = None, F=None, budget_fx=None):
    """Drift assignment: (symbols, integer cost, feasible).  The budget is that of a
    C_bytes container, or budget_fx (bits * 2^16) directly."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    F = dq_pow2_table() if F is None else F
    m = np.zeros(x.size, dtype=np.uint8)
    cost = C.c_longlong(0)
    bfx = dq_budget_fx(C_bytes) if budget_fx is None else int(budget_fx)
    ok = lib().or_dq_drift(x, x.size, float(s), float(o), tab.r, tab.M, bfx, F, m, C.byref(cost))
    return m, int(cost.value), bool(ok)


def dq_refit(x, m, s: float, o: float):
    x = np.ascontiguousarray(x, dtype=np.float32)
    m = np.ascontiguousarray(m, dtype=np.uint8)
    sc, oc = C.c_float(s), C.c_float(o)
    lib().or_dq_refit(x, m, x.size, C.byref(sc), C.byref(oc))
    return float(sc.value), float(oc.value)


def rans_encode(m, tab: DqTable, C_bytes: int):
    """(container bytes, emitted byte count or -1 on overflow)."""
    m = np.ascontiguousarray(m, dtype=np.uint8)
    out = np.zeros(C_bytes, dtype=np.uint8)
    pushed = lib().or_rans_encode(m, m.size, tab.f, tab.c, tab.p, C_bytes, out)
    return out, int(pushed)


def rans_decode(container, n: int, tab: DqTable):
    """(symbols, final state, bytes consumed after the state); raises if the
    decoder would read past the container."""
    pay = np.ascontiguousarray(container, dtype=np.uint8)
    m = np.zeros(n, dtype=np.uint8)
    xf, used = C.c_uint32(0), C.c_int(0)
    if lib().or_rans_decode(pay, pay.size, n, tab.f, tab.c, tab.M, tab.p, m, C.byref(xf), C.byref(used)) != 0:
        raise ValueError("decoder ran past the container")
    return m, int(xf.value), int(used.value)


def dq_encode_stream(x, tab: DqTable, C_bytes: int, F=None):
    """Algorithm 1 on one stream: dict(container, s16, o16, m, m_near, flags)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    F = dq_pow2_table() if F is None else F
    cont = np.zeros(C_bytes, dtype=np.uint8)
    m = np.zeros(x.size, dtype=np.uint8)
    mn = np.zeros(x.size, dtype=np.uint8)
    s16, o16 = C.c_uint16(0), C.c_uint16(0)
    flags = lib().or_dq_encode_stream(x, x.size, tab.M, C_bytes, tab.f, tab.c, tab.p, tab.r, F, cont,
                                      C.byref(s16), C.byref(o16), m, mn.ctypes.data_as(C.c_void_p))
    return {"container": cont, "s16": int(s16.value), "o16": int(o16.value), "m": m, "m_near": mn,
            "flags": int(flags)}


def dq_encode_streams(X, tab: DqTable, C_bytes: int, F=None):
    """Algorithm 1 on each row of X [ns, n]: (containers [ns, C], s16 [ns], o16 [ns],
    symbols [ns, n], flags [ns])."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    ns, n = X.shape
    F = dq_pow2_table() if F is None else F
    cont = np.zeros((ns, C_bytes), dtype=np.uint8)
    s16 = np.zeros(ns, dtype=np.uint16)
    o16 = np.zeros(ns, dtype=np.uint16)
    m = np.zeros((ns, n), dtype=np.uint8)
    flags = np.zeros(ns, dtype=np.int32)
    if ns:
        lib().or_dq_encode_streams(X, ns, n, tab.M, C_bytes, tab.f, tab.c, tab.p, tab.r, F, cont, s16, o16, m,
                                   flags)
    return cont, s16, o16, m, flags


def dq_window_mean(y):
    """y [n_tok, n] fp32 -> (int8 q [n], fp16 scale bits, dequantized mean [n] fp32)."""
    y = np.ascontiguousarray(y, dtype=np.float32)
    n_tok, n = y.shape
    q = np.zeros(n, dtype=np.int8)
    mu = np.zeros(n, dtype=np.float32)
    sc = C.c_uint16(0)
    lib().or_dq_window_mean(y, n_tok, n, q, C.byref(sc), mu)
    return q, int(sc.value), mu


def attention_f64(q: np.ndarray, K: np.ndarray, V: np.ndarray, sm_scale: float) -> np.ndarray:
    """q [G,d], K/V [S,d] -> out [G,d], all fp64."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    G, d = q.shape
    out = np.zeros((G, d), dtype=np.float64)
    lib().or_attention_f64(q, K, V, G, K.shape[0], d, sm_scale, out)
    return out


from .cache import *  # noqa: E402,F401,F403  (whole-cache assembly)
