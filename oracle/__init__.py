"""CPU oracle for quantized decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The CUDA library never does, and
this package never imports the CUDA library: the two share nothing but the
seeded input generators in ``workloads.py``.

The arithmetic lives in plain C (``affine.c``, ``format.c``, ``nuq.c``), compiled with
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
            L.or_affine_quantize.argtypes = [_f32, C.c_int, C.c_int, C.c_int, C.c_double, _u8,
                                             C.POINTER(C.c_float), C.POINTER(C.c_float)]
            L.or_affine_dequant.argtypes = [_u8, C.c_int, C.c_float, C.c_float, C.c_void_p, _f32]
            L.or_quantize_unit.argtypes = [_f32, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_int,
                                           C.c_int, C.c_int, _f32, C.c_int, C.c_int, C.c_double,
                                           C.c_int, _u8, _f32, _f32, C.c_void_p]
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


def affine_quantize(x: np.ndarray, bits: int, meta_f16: bool, clip: float = 0.0):
    x = np.ascontiguousarray(x, dtype=np.float32)
    codes = np.zeros(x.shape[-1], dtype=np.uint8)
    s, o = C.c_float(), C.c_float()
    lib().or_affine_quantize(x, x.shape[-1], bits, int(meta_f16), clip, codes, C.byref(s), C.byref(o))
    return codes, np.float32(s.value), np.float32(o.value)


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
