"""ctypes binding of libdq (include/dq.h): argument marshalling only.

Every step of the quantize / attention path runs in the CUDA library; this
module only builds the C structs, hands over raw device pointers of torch
tensors and the current CUDA stream, and turns status codes into exceptions.
There is no CPU fallback: if libdq.so is missing, loading raises.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libdq.so")

DQ_F32, DQ_F16, DQ_BF16 = 0, 1, 2
DQ_AFFINE, DQ_NUQ, DQ_RANS = 0, 1, 2
DQ_ROT_NONE, DQ_ROT_HADAMARD, DQ_ROT_DENSE = 0, 1, 2
STATUS = ["DQ_OK", "DQ_EINVAL", "DQ_EALIGN", "DQ_EUNSUPPORTED", "DQ_EINFEASIBLE", "DQ_ENOMEM",
          "DQ_ECUDA", "DQ_ENONFINITE", "DQ_ETIMEOUT"]
DTYPES = {"f32": DQ_F32, "f16": DQ_F16, "bf16": DQ_BF16}
ROTS = {"none": DQ_ROT_NONE, "hadamard": DQ_ROT_HADAMARD, "dense": DQ_ROT_DENSE}
SCHEMES = {"affine": DQ_AFFINE, "nuq": DQ_NUQ, "rans": DQ_RANS}
GRIDS = {"minmax": 0, "quest": 1}


class TensorCfg(C.Structure):
    _fields_ = [("scheme", C.c_int), ("bits", C.c_int), ("levels", C.c_int), ("container_bytes", C.c_int),
                ("rot", C.c_int), ("mean", C.c_int), ("clip", C.c_float), ("grid", C.c_int),
                ("lloyd_iters", C.c_int), ("outlier_frac", C.c_float), ("group_size", C.c_int),
                ("refit_interval", C.c_int)]


class Config(C.Structure):
    _fields_ = [("batch", C.c_int), ("n_kv_heads", C.c_int), ("n_q_heads", C.c_int), ("head_dim", C.c_int),
                ("max_seq", C.c_int), ("kv_dtype", C.c_int), ("meta_dtype", C.c_int), ("out_dtype", C.c_int),
                ("k", TensorCfg), ("v", TensorCfg), ("n_sink", C.c_int), ("n_recent", C.c_int),
                ("rans_alpha", C.c_float), ("rans_prob_bits", C.c_int)]


BUFFER_NAMES = ["codes_k", "codes_v", "meta_k", "meta_v", "mean_k", "lut_k", "lut_v", "raw_k", "raw_v",
                "ol_rowptr_k", "ol_col_k", "ol_val_k", "ol_rowptr_v", "ol_col_v", "ol_val_v",
                "k_transform", "q_comp"]
NUM_BUFFERS = len(BUFFER_NAMES)


class Buffers(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in BUFFER_NAMES]


class DQError(RuntimeError):
    def __init__(self, status: int, msg: str):
        self.status = status
        self.name = STATUS[status] if 0 <= status < len(STATUS) else f"status {status}"
        super().__init__(f"{self.name}: {msg}")


_lib = None
_lib_path = LIB_PATH


def use_checked_build() -> None:
    """Make this process load the bounds-checked build (libdq_checked.so, built
    with quantized_decode_attention_gb300.build.build(checked=True)) instead of
    libdq.so.  Call before the library is first loaded."""
    global _lib_path
    if _lib is not None:
        raise RuntimeError("the library is already loaded in this process")
    _lib_path = os.path.join(os.path.dirname(LIB_PATH), "libdq_checked.so")


def load() -> C.CDLL:
    """Load libdq.so (built by quantized_decode_attention_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_lib_path):
        raise RuntimeError(f"{_lib_path} is not built; run quantized_decode_attention_gb300.build.build()")
    L = C.CDLL(_lib_path)
    P = C.c_void_p
    L.dq_kv_sizes.argtypes = [C.POINTER(Config), C.POINTER(C.c_size_t)]
    L.dq_quantize_kv.argtypes = [C.POINTER(P), C.POINTER(Config), C.POINTER(Buffers), P, P, C.c_longlong,
                                 C.c_longlong, P]
    L.dq_decode_attention.argtypes = [C.POINTER(P), C.POINTER(Config), C.POINTER(Buffers), P, P,
                                      C.c_longlong, C.c_float, P]
    L.dq_decode_step.argtypes = [C.POINTER(P), C.POINTER(Config), C.POINTER(Buffers), P, P, P, P,
                                 C.c_longlong, C.c_float, P]
    L.dq_dequantize_kv.argtypes = [C.POINTER(P), C.POINTER(Config), C.POINTER(Buffers), C.c_int,
                                   C.c_longlong, C.c_longlong, P, P]
    L.dq_decode_attention_noalloc.argtypes = [C.POINTER(Config), C.POINTER(Buffers), P, P, C.c_longlong,
                                              C.c_float, P]
    L.dq_decode_attention_noalloc.restype = C.c_int
    L.dq_check.argtypes = [P, P]
    L.dq_test_expire_wait.argtypes = [P, C.c_ulonglong, P]
    L.dq_test_checked_probe.argtypes = [P, P]
    L.dq_drift_stats.argtypes = [P, P, C.POINTER(C.c_ulonglong)]
    L.dq_free.argtypes = [P]
    L.dq_free.restype = None
    L.dq_last_error.restype = C.c_char_p
    L.dq_status_name.restype = C.c_char_p
    L.dq_status_name.argtypes = [C.c_int]
    L.dq_rans_model.argtypes = [C.POINTER(Config), C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_int),
                                C.POINTER(C.c_int)]
    L.dq_symbol_probs.argtypes = [C.c_int, C.c_int, C.POINTER(C.c_double)]
    L.dq_quest_step.argtypes = [C.c_int, C.POINTER(C.c_float)]
    for f in ("dq_kv_sizes", "dq_quantize_kv", "dq_decode_attention", "dq_decode_step", "dq_dequantize_kv", "dq_check",
              "dq_test_expire_wait", "dq_test_checked_probe", "dq_rans_model", "dq_symbol_probs",
              "dq_quest_step", "dq_drift_stats"):
        getattr(L, f).restype = C.c_int
    _lib = L
    return L


def rans_model(cfg: Config, which: int):
    """(f, c) of the symbol model of keys (which=0) or values (which=1)."""
    M = C.c_int(0)
    f = (C.c_int * 16)()
    c = (C.c_int * 16)()
    _raise(load().dq_rans_model(C.byref(cfg), which, C.byref(M), f, c))
    return list(f[:M.value]), list(c[:M.value])


def symbol_probs(n: int, levels: int):
    """Unsharpened level probabilities of the Gaussian order-statistics model
    for streams of n values on a per-token grid of `levels` levels."""
    p = (C.c_double * 16)()
    _raise(load().dq_symbol_probs(n, levels, p))
    return list(p[:levels])


def quest_step(bits: int) -> float:
    """The QuEST grid's step factor c_b (a token's scale is c_b * RMS)."""
    c = C.c_float()
    _raise(load().dq_quest_step(bits, C.byref(c)))
    return c.value


def _raise(st: int):
    if st != 0:
        raise DQError(st, load().dq_last_error().decode())


def make_config(*, batch, n_kv_heads, n_q_heads, head_dim, max_seq, kv_dtype="bf16", meta_dtype="f16",
                out_dtype="bf16", bits=2, bits_v=None, rot_k="hadamard", rot_v="hadamard", mean_k=True,
                clip_k=0.0, clip_v=None, grid_k="minmax", grid_v=None, n_sink=0, n_recent=0, scheme="affine",
                lloyd_iters=8,
                outlier_frac=0.01, group_size_v=0, refit_k=0, levels_k=8, levels_v=6, container_k=331, container_v=231,
                rans_alpha=1.4) -> Config:
    c = Config()
    c.batch, c.n_kv_heads, c.n_q_heads, c.head_dim, c.max_seq = batch, n_kv_heads, n_q_heads, head_dim, max_seq
    c.kv_dtype, c.meta_dtype, c.out_dtype = DTYPES[kv_dtype], DTYPES[meta_dtype], DTYPES[out_dtype]
    c.k.scheme = c.v.scheme = SCHEMES[scheme]
    c.k.bits, c.v.bits = bits, bits if bits_v is None else bits_v
    c.k.rot, c.v.rot = ROTS[rot_k], ROTS[rot_v]
    c.k.mean, c.v.mean = int(bool(mean_k)), 0
    c.k.clip = clip_k
    c.v.clip = clip_k if clip_v is None else clip_v
    c.k.grid = GRIDS[grid_k]
    c.v.grid = GRIDS[grid_k if grid_v is None else grid_v]
    c.n_sink, c.n_recent = n_sink, n_recent
    if scheme == "nuq":
        c.k.lloyd_iters = c.v.lloyd_iters = lloyd_iters
        c.k.outlier_frac = c.v.outlier_frac = outlier_frac
        c.v.group_size = group_size_v
        c.k.refit_interval = refit_k
    c.rans_alpha, c.rans_prob_bits = rans_alpha, 8
    if scheme == "rans":
        c.k.levels, c.v.levels = levels_k, levels_v
        c.k.container_bytes, c.v.container_bytes = container_k, container_v
    return c


def kv_sizes(cfg: Config):
    arr = (C.c_size_t * NUM_BUFFERS)()
    _raise(load().dq_kv_sizes(C.byref(cfg), arr))
    return dict(zip(BUFFER_NAMES, list(arr)))


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) or None
    return int(stream) or None


@dataclass
class KVCache:
    """Device buffers of one cache (torch uint8 tensors) plus the library context.

    torch provides the memory and the stream; the library does all the work.
    """
    cfg: Config
    tensors: dict
    ctx: C.c_void_p

    @classmethod
    def allocate(cls, cfg: Config, device="cuda", zero: bool = True):
        import torch
        sizes = kv_sizes(cfg)
        alloc = torch.zeros if zero else torch.empty
        tensors = {n: (alloc(s, dtype=torch.uint8, device=device) if s else None) for n, s in sizes.items()}
        return cls(cfg, tensors, C.c_void_p())

    def buffers(self) -> Buffers:
        """The C struct of buffer pointers, built once: the tensors never move
        (their contents are written in place)."""
        b = getattr(self, "_bufs", None)
        if b is None:
            b = Buffers()
            for n in BUFFER_NAMES:
                setattr(b, n, _ptr(self.tensors.get(n)))
            self._bufs = b
        return b

    def quantize(self, k, v, pos0: int = 0, stream=None):
        """k, v: device tensors [B, Hkv, n_tok, d] (kv dtype) -> writes the cache."""
        n_tok = k.shape[2]
        b = self.buffers()
        _raise(load().dq_quantize_kv(C.byref(self.ctx), C.byref(self.cfg), C.byref(b), _ptr(k), _ptr(v),
                                     pos0, n_tok, _stream(stream)))

    def attention(self, q, out, seq_len: int, sm_scale: float | None = None, stream=None):
        """q: fp32 [B, Hq, d]; out: [B, Hq, d] in the out dtype (device tensors)."""
        if sm_scale is None:
            sm_scale = self.cfg.head_dim ** -0.5
        b = self.buffers()
        _raise(load().dq_decode_attention(C.byref(self.ctx), C.byref(self.cfg), C.byref(b), _ptr(q), _ptr(out),
                                          seq_len, sm_scale, _stream(stream)))

    def decode_step(self, k_new, v_new, q, out, seq_len: int, sm_scale: float | None = None, stream=None):
        """Append token seq_len - 1 (k_new, v_new: [B, Hkv, 1, d] in the kv dtype)
        and attend over seq_len tokens (q fp32 [B, Hq, d], out [B, Hq, d])."""
        if sm_scale is None:
            sm_scale = self.cfg.head_dim ** -0.5
        b = self.buffers()
        _raise(load().dq_decode_step(C.byref(self.ctx), C.byref(self.cfg), C.byref(b), _ptr(k_new), _ptr(v_new),
                                     _ptr(q), _ptr(out), seq_len, sm_scale, _stream(stream)))

    def attention_noalloc(self, q, out, seq_len: int, sm_scale: float | None = None, stream=None):
        """Same result as attention(), through the entry point that allocates nothing
        (its split workspace is a static device array inside the library)."""
        if sm_scale is None:
            sm_scale = self.cfg.head_dim ** -0.5
        b = self.buffers()
        _raise(load().dq_decode_attention_noalloc(C.byref(self.cfg), C.byref(b), _ptr(q), _ptr(out), seq_len,
                                                  sm_scale, _stream(stream)))

    def dequantize(self, which: int, slot0: int, n: int, out, stream=None):
        b = self.buffers()
        _raise(load().dq_dequantize_kv(C.byref(self.ctx), C.byref(self.cfg), C.byref(b), which, slot0, n,
                                       _ptr(out), _stream(stream)))

    def clone_shared(self) -> "KVCache":
        """A copy of the cache buffers that shares this cache's context (workspace).
        Calls on the two must be ordered on one stream; only the owner frees it."""
        c = KVCache(self.cfg, {n: (t.clone() if t is not None else None) for n, t in self.tensors.items()},
                    self.ctx)
        c._borrowed = True
        return c

    def detach(self):
        """Forget a borrowed context without freeing it."""
        self.ctx = C.c_void_p()

    def drift_stats(self, stream=None) -> dict:
        """Entropy-coded caches: drift statistics since the last read (and clear)."""
        out = (C.c_ulonglong * 6)()
        _raise(load().dq_drift_stats(self.ctx, _stream(stream), out))
        return {"k_changed": out[0], "k_coded": out[1], "k_max_move": out[2],
                "v_changed": out[3], "v_coded": out[4], "v_max_move": out[5]}

    def check(self, stream=None):
        _raise(load().dq_check(self.ctx, _stream(stream)))

    def close(self):
        if getattr(self, "_borrowed", False):
            self.detach()
            return
        if self.ctx:
            load().dq_free(self.ctx)
            self.ctx = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
