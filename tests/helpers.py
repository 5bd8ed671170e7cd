"""Test-side glue: workload -> library config, uploads, and oracle expectations."""
from __future__ import annotations

import numpy as np

import oracle
import workloads as W


def cfg_for(w: W.Workload, max_seq: int | None = None, out_dtype: str | None = None):
    from quantized_decode_attention_gb300 import make_config
    return make_config(batch=w.batch, n_kv_heads=w.n_kv_heads, n_q_heads=w.n_q_heads, head_dim=w.head_dim,
                       max_seq=max_seq or w.seq, kv_dtype=w.kv_dtype, meta_dtype=w.meta_dtype,
                       out_dtype=out_dtype or w.out_dtype, bits=w.bits, rot_k=w.rot_k, rot_v=w.rot_v,
                       mean_k=w.mean_k, clip_k=w.clip, clip_v=w.clip, grid_k=w.grid, n_sink=w.n_sink,
                       n_recent=w.n_recent,
                       scheme=w.scheme, lloyd_iters=w.extra.get("lloyd_iters", 8),
                       outlier_frac=w.extra.get("outlier_frac", 0.01),
                       group_size_v=w.extra.get("group_size", 0), refit_k=w.extra.get("refit_interval", 0),
                       levels_k=w.extra.get("levels_k", 8), levels_v=w.extra.get("levels_v", 6),
                       container_k=w.extra.get("container_k", 331), container_v=w.extra.get("container_v", 231),
                       rans_alpha=w.extra.get("alpha", 1.4))


def to_device(arr: np.ndarray, dtype: str):
    import torch
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(arr, dtype=np.float32)).cuda()
    t = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.uint16).view(np.int16)).cuda()
    return t.view(torch.float16 if dtype == "f16" else torch.bfloat16)


def out_to_np(t) -> np.ndarray:
    import torch
    return t.float().cpu().numpy().astype(np.float64) if t.dtype != torch.float32 else t.cpu().numpy().astype(np.float64)


def dense_inputs(w: W.Workload):
    T, Qc = W.dense_transform(w)
    return T, Qc


def oracle_cache(w: W.Workload, k, v, S, T=None):
    qk = oracle.quantize_tensor(w, k, True, S, T=T)
    qv = oracle.quantize_tensor(w, v, False, S)
    return qk, qv


def expected_buffers(w: W.Workload, qk, qv, nq: int):
    """Packed records / meta the library must hold for quantized slots [0, nq)."""
    exp = {
        "codes_k": oracle.pack_k(qk.codes[:, :, :nq], w.bits),
        "codes_v": oracle.pack_v(qv.codes[:, :, :nq], w.bits),
    }
    if w.meta_dtype == "f16":
        exp["meta_k"] = oracle.meta_f16_bits(qk.s[:, :, :nq], qk.o[:, :, :nq])
        exp["meta_v"] = oracle.meta_f16_bits(qv.s[:, :, :nq], qv.o[:, :, :nq])
    else:
        exp["meta_k"] = np.stack([qk.s[:, :, :nq], qk.o[:, :, :nq]], -1).view(np.uint32)
        exp["meta_v"] = np.stack([qv.s[:, :, :nq], qv.o[:, :, :nq]], -1).view(np.uint32)
    return exp


def lib_views(w: W.Workload, cache, max_seq: int):
    """Reshape the library's byte buffers into [U-major] numpy views."""
    B, H, d = w.batch, w.n_kv_heads, w.head_dim
    qcap = -(-(max_seq - w.n_sink) // 64) * 64
    rcap = -(-(w.n_sink + w.n_recent) // 16) * 16
    rowk = d * w.bits // 8
    t = {n: (x.cpu().numpy() if x is not None else None) for n, x in cache.tensors.items()}
    mb = 2 if w.meta_dtype == "f16" else 4
    out = {
        "codes_k": t["codes_k"].reshape(B, H, qcap, rowk),
        "codes_v": t["codes_v"].reshape(B, H, qcap // 2, 2 * rowk),
        "meta_k": t["meta_k"].view(np.uint16 if mb == 2 else np.uint32).reshape(B, H, qcap, 2),
        "meta_v": t["meta_v"].view(np.uint16 if mb == 2 else np.uint32).reshape(B, H, qcap, 2),
    }
    if t["mean_k"] is not None:
        out["mean_k"] = t["mean_k"].view(np.float32).reshape(B, H, d)
    if rcap:
        out["raw_k"] = t["raw_k"].view(np.uint16).reshape(B, H, rcap, d)
        out["raw_v"] = t["raw_v"].view(np.uint16).reshape(B, H, rcap // 2, d, 2)
    return out


def nuq_views(w: W.Workload, cache, S: int):
    """Reshape a non-uniform cache's byte buffers into [B, H, ...] numpy views."""
    from quantized_decode_attention_gb300 import kv_sizes
    B, H, d, L = w.batch, w.n_kv_heads, w.head_dim, 1 << w.bits
    qcap = -(-(S - w.n_sink) // 64) * 64
    rcap = -(-(w.n_sink + w.n_recent) // 16) * 16
    rowk = d * w.bits // 8
    t = {n: (x.cpu().numpy() if x is not None else None) for n, x in cache.tensors.items()}
    sizes = kv_sizes(cache.cfg)
    gv = d // (w.extra.get("group_size", 0) or d)
    N = w.extra.get("refit_interval", 0) or 0
    v = {
        "codes_k": t["codes_k"].reshape(B, H, qcap, rowk),
        "codes_v": t["codes_v"].reshape(B, H, qcap // 2, 2 * rowk),
        "lut_v": t["lut_v"].view(np.uint16).reshape(B, H, qcap, gv * L),
    }
    if N:  # key tables per refit block, then the prefill's quantized slot count per unit
        nbk = -(-qcap // N)
        tab = t["lut_k"][:B * H * nbk * d * L * 2]
        v["lut_k_blk"] = tab.view(np.uint16).reshape(B, H, nbk, d, L)
        v["pq"] = t["lut_k"][B * H * nbk * d * L * 2:].view(np.int32).reshape(B, H)
    else:
        v["lut_k"] = t["lut_k"].view(np.uint16).reshape(B, H, d, L)
    if t["ol_rowptr_k"] is not None:
        v["rowptr"] = t["ol_rowptr_k"].view(np.int32).reshape(B, H, -1)
        v["col_k"] = t["ol_col_k"].view(np.uint16).reshape(B, H, -1)
        v["val_k"] = t["ol_val_k"].view(np.uint16).reshape(B, H, -1)
    if t["ol_col_v"] is not None:
        v["col_v"] = t["ol_col_v"].view(np.uint16).reshape(B, H, qcap, -1)
        v["val_v"] = t["ol_val_v"].view(np.uint16).reshape(B, H, qcap, -1)
    if rcap:
        v["raw_k"] = t["raw_k"].view(np.uint16).reshape(B, H, rcap, d)
        v["raw_v"] = t["raw_v"].view(np.uint16).reshape(B, H, rcap // 2, d, 2)
    if t["meta_k"] is not None:  # frozen per-channel key outlier thresholds, fp32
        v["thr_k"] = t["meta_k"].view(np.float32).reshape(B, H, d)
    assert sizes["meta_v"] == 0 and sizes["mean_k"] == 0
    return v, qcap


def dquant_views(w: W.Workload, cache, S: int):
    """Reshape an entropy-coded cache's byte buffers into [B, ...] numpy views."""
    B, H, d = w.batch, w.n_kv_heads, w.head_dim
    n = H * d
    qcap = -(-(S - w.n_sink) // 128) * 128
    rcap = -(-(w.n_sink + w.n_recent) // 16) * 16
    t = {nm: (x.cpu().numpy() if x is not None else None) for nm, x in cache.tensors.items()}
    v = {
        "codes_k": t["codes_k"].reshape(B, qcap, w.extra["container_k"]),
        "codes_v": t["codes_v"].reshape(B, qcap, w.extra["container_v"]),
        "meta_k": t["meta_k"].view(np.uint16).reshape(B, qcap, 2),
        "meta_v": t["meta_v"].view(np.uint16).reshape(B, qcap, 2),
    }
    if t["mean_k"] is not None:
        rec = t["mean_k"].reshape(B, qcap // 128, n + 16)
        v["mean_q"] = rec[:, :, :n].view(np.int8)
        v["mean_sc"] = np.ascontiguousarray(rec[:, :, n:n + 2]).view(np.uint16)[..., 0]
    if rcap:
        v["raw_k"] = t["raw_k"].view(np.uint16).reshape(B, H, rcap, d)
        v["raw_v"] = t["raw_v"].view(np.uint16).reshape(B, H, rcap // 2, d, 2)
    return v, qcap
