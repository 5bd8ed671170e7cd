"""Seeded synthetic inputs and the workload table.

This module only draws random inputs and names the workload shapes.  It holds
none of the quantization or attention arithmetic, so both the CPU oracle and
the CUDA path can take their inputs from here without sharing any method code.

Every tensor is drawn from numpy's PCG64 generator seeded with
``config_index * 1000 + tensor_id`` (tensor ids below), so the same arrays can
be rebuilt anywhere.  16-bit inputs are returned as ``uint16`` bit patterns
(numpy has no bfloat16); ``f32_to_bf16_bits`` rounds to nearest-even.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

# tensor ids used in the seeds
TID_K, TID_V, TID_Q, TID_KMEAN, TID_KOUTLIER, TID_QNEW, TID_KNEW, TID_VNEW = 1, 2, 3, 4, 5, 6, 7, 8
TID_SIGMA_K, TID_SIGMA_Q = 9, 10


@dataclass(frozen=True)
class Workload:
    """Shape and quantizer settings of one synthetic decode-attention workload."""
    name: str
    index: int                 # config index (seed base)
    batch: int
    n_kv_heads: int
    n_q_heads: int
    head_dim: int
    seq: int
    kv_dtype: str              # "f32" | "f16" | "bf16"
    scheme: str = "affine"     # "affine" | "nuq" | "rans"
    bits: int = 4
    meta_dtype: str = "f16"    # "f16" | "f32"
    rot_k: str = "hadamard"    # "none" | "hadamard" | "dense"
    rot_v: str = "hadamard"
    mean_k: bool = True
    clip: float = 0.0          # 0 = min/max; else two-sided quantile kappa
    grid: str = "minmax"       # affine grid: "minmax" (or the kappa clip) | "quest"
    n_sink: int = 0
    n_recent: int = 0
    k_dist: str = "normal"     # "normal" | "llama" | "student4" | "cov"
    v_dist: str = "normal"
    out_dtype: str = "bf16"
    extra: dict = field(default_factory=dict)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads


TINY = Workload("tiny", 1, batch=1, n_kv_heads=1, n_q_heads=1, head_dim=64, seq=128,
                kv_dtype="f32", bits=4, meta_dtype="f32", out_dtype="f32")
LLAMA = Workload("llama3-8b-decode", 2, batch=16, n_kv_heads=8, n_q_heads=32, head_dim=128,
                 seq=8192, kv_dtype="bf16", bits=2, meta_dtype="f16", n_sink=4, n_recent=128,
                 k_dist="llama")
NUQ = Workload("kvquant-nuq", 3, batch=8, n_kv_heads=8, n_q_heads=32, head_dim=128, seq=4096,
               kv_dtype="f16", scheme="nuq", bits=3, rot_k="none", rot_v="none", mean_k=False,
               n_sink=1, k_dist="student4", v_dist="student4", out_dtype="f16")
QWEN_LONG = Workload("qwen3-8b-long", 4, batch=4, n_kv_heads=8, n_q_heads=32, head_dim=128,
                     seq=32768, kv_dtype="bf16", bits=2, rot_k="dense", rot_v="none",
                     mean_k=False, clip=0.999, k_dist="cov")
DQUANT = Workload("dquant-rans", 5, batch=32, n_kv_heads=8, n_q_heads=32, head_dim=128,
                  seq=16384, kv_dtype="bf16", scheme="rans", rot_k="hadamard", rot_v="none",
                  n_recent=128, meta_dtype="f16",
                  extra={"levels_k": 8, "levels_v": 6, "container_k": 331, "container_v": 231,
                         "alpha": 1.4, "mean_window": 128})

# D-Quant at 1.96 bits per value with the same 8 / 6 levels (D-Quant Sec. 5,
# "lower storage budget"; Fig. 4 middle): the 2.26-bit payloads scaled in
# proportion, keys 8 levels in 286 bytes and values 6 levels in 200 bytes
DQUANT_196 = DQUANT.with_(name="dquant-rans-1.96bpv",
                          extra={**DQUANT.extra, "container_k": 286, "container_v": 200})

WORKLOADS = {w.name: w for w in (TINY, LLAMA, NUQ, QWEN_LONG, DQUANT, DQUANT_196)}


def dquant_bits_per_value(w: Workload) -> float:
    """Storage of a D-Quant cache per quantized value: containers, fp16 (s, o)
    per stream, and the keys' INT8 window mean with its fp16 scale per 128 tokens."""
    n = w.n_kv_heads * w.head_dim
    e = w.extra
    mean = (n + 2) / e.get("mean_window", 128) if w.mean_k else 0.0
    return ((e["container_k"] + 4 + mean) + (e["container_v"] + 4)) * 8 / (2 * n)


def rng(index: int, tid: int, salt: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(index * 1000 + tid + 1_000_003 * salt))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bfloat16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = ((u >> 16) & 1) + 0x7FFF
    return ((u + r) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def to_dtype_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Cast fp32 samples to the workload's storage dtype ('f32' stays float32)."""
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def bits_to_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.asarray(x, dtype=np.float32)
    if dtype == "f16":
        return np.asarray(x, dtype=np.uint16).view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f32(np.asarray(x, dtype=np.uint16))
    raise ValueError(dtype)


def _draw(w: Workload, tid: int, dist: str, shape, salt: int = 0) -> np.ndarray:
    g = rng(w.index, tid, salt)
    if dist == "normal":
        return g.standard_normal(shape, dtype=np.float32)
    if dist == "student4":
        return g.standard_t(4.0, size=shape).astype(np.float32)
    raise ValueError(dist)


def llama_channel_stats(w: Workload):
    """Per-(kv head, channel) means ~N(0, 2) and the ~1% of channels scaled x10."""
    mu = (rng(w.index, TID_KMEAN).standard_normal((w.n_kv_heads, w.head_dim)) * np.sqrt(2.0)).astype(np.float32)
    n_pairs = w.n_kv_heads * w.head_dim
    n_out = int(np.floor(0.01 * n_pairs + 0.5))
    pick = rng(w.index, TID_KOUTLIER).choice(n_pairs, size=n_out, replace=False)
    scale = np.ones(n_pairs, dtype=np.float32)
    scale[pick] = 10.0
    return mu, scale.reshape(w.n_kv_heads, w.head_dim)


def cov_factor(w: Workload, tid: int) -> np.ndarray:
    """A per-kv-head covariance factor A (Sigma = A A^T / d + 0.1 I) for 'cov' keys/queries."""
    d = w.head_dim
    a = rng(w.index, tid).standard_normal((w.n_kv_heads, d, d))
    sig = np.einsum("hij,hkj->hik", a, a) / d + 0.1 * np.eye(d)[None]
    return np.linalg.cholesky(sig).astype(np.float64)


def make_kv(w: Workload, seq: Optional[int] = None, batch: Optional[int] = None, salt: int = 0):
    """Raw K and V as [B, Hkv, S, d] arrays in the workload's storage dtype."""
    S = w.seq if seq is None else seq
    B = w.batch if batch is None else batch
    shape = (B, w.n_kv_heads, S, w.head_dim)
    if w.k_dist == "llama":
        k = _draw(w, TID_K, "normal", shape, salt)
        mu, sc = llama_channel_stats(w)
        k += mu[None, :, None, :]
        k *= sc[None, :, None, :]
    elif w.k_dist == "cov":
        L = cov_factor(w, TID_SIGMA_K).astype(np.float32)
        z = _draw(w, TID_K, "normal", shape, salt)
        k = np.empty_like(z)
        for h in range(w.n_kv_heads):          # k = L z per (sequence, token): a BLAS product per head
            k[:, h] = z[:, h] @ L[h].T
    else:
        k = _draw(w, TID_K, w.k_dist, shape, salt)
    v = _draw(w, TID_V, w.v_dist, shape, salt)
    return to_dtype_bits(k, w.kv_dtype), to_dtype_bits(v, w.kv_dtype)


def make_q(w: Workload, batch: Optional[int] = None, salt: int = 0) -> np.ndarray:
    """Decode queries [B, Hq, d] in fp32 (cov workloads: q ~ N(0, Sigma_Q) per kv group)."""
    B = w.batch if batch is None else batch
    z = rng(w.index, TID_Q, salt).standard_normal((B, w.n_q_heads, w.head_dim), dtype=np.float32)
    if w.k_dist == "cov":
        L = cov_factor(w, TID_SIGMA_Q).astype(np.float32)
        kvh = np.arange(w.n_q_heads) // w.group
        z = np.einsum("hij,bhj->bhi", L[kvh], z).astype(np.float32)
    return z


def make_new_token(w: Workload, batch: Optional[int] = None, salt: int = 0):
    """One new decode token's K and V, [B, Hkv, 1, d], same distributions as the cache."""
    return make_kv(w, seq=1, batch=batch, salt=10_000 + salt)


def _sylvester(d: int) -> np.ndarray:
    H = np.ones((1, 1))
    while H.shape[0] < d:
        H = np.block([[H, H], [H, -H]])
    return H


def dense_transform(w: Workload, gamma: float = 1e-2):
    """Synthetic dense key transform T and its query compensation T^{-T}, per KV head.

    Stands in for a calibrated transform: built from the synthetic key and query
    covariances as c * (Hn) * Lambda^(-1/4) * U^T * L^T, with L the Cholesky factor of
    the damped query covariance, U Lambda U^T = L^T (damped key covariance) L, and c
    chosen so that ||T||_F = sqrt(d).  Returns float32 arrays [Hkv, d, d].
    """
    d = w.head_dim
    Lk = cov_factor(w, TID_SIGMA_K)
    Lq = cov_factor(w, TID_SIGMA_Q)
    Hn = _sylvester(d) / np.sqrt(d)
    Ts, Qs = [], []
    for h in range(w.n_kv_heads):
        SK = Lk[h] @ Lk[h].T
        SQ = Lq[h] @ Lq[h].T
        L = np.linalg.cholesky(SQ + gamma * np.trace(SQ) / d * np.eye(d))
        M = SK + gamma * np.trace(SK) / d * np.eye(d)
        lam, U = np.linalg.eigh(L.T @ M @ L)
        T = Hn @ np.diag(lam ** -0.25) @ U.T @ L.T
        T *= np.sqrt(d) / np.linalg.norm(T)
        Ts.append(T)
        Qs.append(np.linalg.inv(T).T)
    return np.stack(Ts).astype(np.float32), np.stack(Qs).astype(np.float32)
