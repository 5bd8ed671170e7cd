"""Whole-cache assembly on top of the C oracle -- TEST INFRASTRUCTURE ONLY.

Builds, for a workload and raw K/V, the bytes every cache buffer must hold
(packed records, scale/offset, key channel mean, 16-bit sink and recent
regions) and the fp64 decode-attention output.  The per-token arithmetic is
the C code in ``affine.c``/``format.c``; this module only loops over units and
tokens and places results at the addresses the format specifies.

Token regions ("KVQuant-NUQ" page, Attention Sink-Aware quantization; "D-Quant"
page, Sec. 5.1 implementation details: the most recent 128 tokens in BF16):
  * tokens t < n_sink are kept exact in 16-bit (raw slot t);
  * every token t >= n_sink is quantized into quantized slot t - n_sink;
  * the latest n_recent tokens are also kept exact in 16-bit, in raw slot
    n_sink + (t mod n_recent); attention at length S reads them raw and reads
    the quantized slots only for tokens in [n_sink, S - n_recent).
  * the key channel mean is taken at prefill over [n_sink, S - n_recent).
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np

import workloads as W

from . import lib, nuq_assign, outlier_count, pack_k_row, pack_v_token

_ROT = {"none": 0, "hadamard": 1, "dense": 2}


def _f32_input(bits: np.ndarray, dtype: str) -> np.ndarray:
    return np.ascontiguousarray(W.bits_to_f32(bits, dtype), dtype=np.float32)


def raw16_bits(bits: np.ndarray, dtype: str) -> np.ndarray:
    """What a raw region stores: the 16-bit input as is; fp32 input as binary16."""
    if dtype in ("f16", "bf16"):
        return np.asarray(bits, dtype=np.uint16)
    from . import f32_to_f16_bits
    return f32_to_f16_bits(np.asarray(bits, dtype=np.float32)).reshape(np.shape(bits))


def raw16_to_f64(bits16: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return W.bf16_bits_to_f32(bits16).astype(np.float64)
    return np.asarray(bits16, dtype=np.uint16).view(np.float16).astype(np.float64)


def raw_dtype(dtype: str) -> str:
    return "bf16" if dtype == "bf16" else "f16"


@dataclass
class QuantTensor:
    """Oracle result for one tensor (K or V) of the whole cache."""
    codes: np.ndarray     # [B, H, Sq, d] uint8, natural channel order
    s: np.ndarray         # [B, H, Sq] float32 stored scale (after fp16 rounding if any)
    o: np.ndarray         # [B, H, Sq] float32 stored offset
    mu: np.ndarray        # [B, H, d] float32 (zeros when no mean)
    xhat: np.ndarray      # [B, H, Sq, d] float32 dequantized, rotated space (+mu)


def quantize_tensor(w: W.Workload, x_bits: np.ndarray, is_key: bool, S: int,
                    T: np.ndarray | None = None, mu_frozen: np.ndarray | None = None,
                    pos0: int = 0) -> QuantTensor:
    """Quantize tokens [max(pos0, n_sink), pos0 + n) of x_bits [B,H,n,d].

    pos0 == 0 is a prefill: the key mean is computed over [n_sink, S - n_recent).
    pos0 > 0 appends with the frozen mean ``mu_frozen``.
    """
    L = lib()
    B, H, n, d = x_bits.shape
    x = _f32_input(x_bits, w.kv_dtype)
    bits = w.bits
    rot = _ROT[w.rot_k if is_key else w.rot_v]
    mean = bool(w.mean_k) and is_key
    meta_f16 = 1 if w.meta_dtype == "f16" else 0
    qc = float(L.or_quest_step_factor(bits)) if w.grid == "quest" else 0.0  # QuEST grid step factor
    q_t0 = max(0, w.n_sink - pos0)
    nq = n - q_t0
    codes = np.zeros((B, H, nq, d), dtype=np.uint8)
    s = np.zeros((B, H, nq), dtype=np.float32)
    o = np.zeros((B, H, nq), dtype=np.float32)
    xhat = np.zeros((B, H, nq, d), dtype=np.float32)
    mu = np.zeros((B, H, d), dtype=np.float32)
    for b in range(B):
        for h in range(H):
            xu = np.ascontiguousarray(x[b, h])
            Tp = None
            if rot == 2:
                Tu = np.ascontiguousarray(T[h], dtype=np.float32)
                Tp = Tu.ctypes.data_as(C.c_void_p)
            mode = 0
            mu_u = np.zeros(d, dtype=np.float32)
            if mean:
                if pos0 == 0:
                    mode = 1
                else:
                    mode = 2
                    mu_u[:] = mu_frozen[b, h]
            m_t0 = w.n_sink - pos0
            m_t1 = S - w.n_recent - pos0
            m_t0, m_t1 = max(0, m_t0), max(0, m_t1)
            if m_t1 < m_t0:
                m_t1 = m_t0
            cu = np.zeros((nq, d), dtype=np.uint8)
            su = np.zeros(nq, dtype=np.float32)
            ou = np.zeros(nq, dtype=np.float32)
            xh = np.zeros((nq, d), dtype=np.float32)
            L.or_quantize_unit(xu, n, d, rot, Tp, mode, m_t0, m_t1, mu_u, bits, meta_f16,
                               float(np.float32(w.clip)), qc, q_t0, cu, su, ou, xh.ctypes.data_as(C.c_void_p))
            codes[b, h], s[b, h], o[b, h], xhat[b, h], mu[b, h] = cu, su, ou, xh, mu_u
    return QuantTensor(codes, s, o, mu, xhat)


@dataclass
class NuqTensor:
    """Oracle result for one tensor under the non-uniform (Lloyd-Max) scheme.

    "KVQuant-NUQ" page, Quantization axes: keys get one table per channel over
    the quantized tokens, values one table per token over its channels (per
    group of channels with a group size, Configuration reference); the
    outliers of each vector (exactly k by rank) keep their fp16 value."""
    codes: np.ndarray     # [B, H, Sq, d] uint8 nearest-level codes (outliers included)
    lut: np.ndarray       # keys [B, H, d, L]; values [B, H, Sq, G * L] (G tables per token): fp16 bits
    outlier: np.ndarray   # [B, H, Sq, d] bool
    val16: np.ndarray     # [B, H, Sq, d] uint16: fp16 bits of the input (outlier values)
    xhat: np.ndarray      # [B, H, Sq, d] float32: table value, or the outlier's fp16 value (NaN: not yet coded)
    blk_lut: np.ndarray | None = None  # keys with a refit interval: [B, H, NB, d, L] tables per slot block
    n_coded: int | None = None         # keys with a refit interval: slots [0, n_coded) are coded


def _value_group(w: W.Workload) -> int:
    g = w.extra.get("group_size", 0)
    return w.head_dim if g in (0, None) else g


def quantize_nuq(w: W.Workload, x_bits: np.ndarray, is_key: bool, S: int, t0: int | None = None) -> NuqTensor:
    """Prefill of tokens [t0, S) of x_bits [B,H,S,d] under the NUQ scheme (t0
    defaults to n_sink).  Values are fitted per token, per group of channels
    when the workload sets a group size; keys per channel over all the tokens."""
    from . import nuq_vector, nuq_vector_grouped
    B, H, n, d = x_bits.shape
    x = _f32_input(x_bits, w.kv_dtype)[:, :, (w.n_sink if t0 is None else t0):S]
    nq = x.shape[2]
    L = 1 << w.bits
    iters, frac = w.extra.get("lloyd_iters", 8), w.extra.get("outlier_frac", 0.01)
    g = _value_group(w)
    codes = np.zeros((B, H, nq, d), dtype=np.uint8)
    out = np.zeros((B, H, nq, d), dtype=bool)
    lut = np.zeros((B, H, d, L) if is_key else (B, H, nq, (d // g) * L), dtype=np.uint16)
    for b in range(B):
        for h in range(H):
            if is_key:
                for c in range(d):
                    fl, lu, co = nuq_vector(np.ascontiguousarray(x[b, h, :, c]), w.bits, iters, frac)
                    codes[b, h, :, c], out[b, h, :, c], lut[b, h, c] = co, fl, lu
            else:
                for t in range(nq):
                    fl, lu, co = nuq_vector_grouped(np.ascontiguousarray(x[b, h, t]), w.bits, iters, frac, g)
                    codes[b, h, t], out[b, h, t], lut[b, h, t] = co, fl, lu.reshape(-1)
    # fp16 rounding (RNE) as a library primitive; the oracle's own binary16
    # conversion is pinned against the same numpy cast
    val16 = x.astype(np.float16).view(np.uint16)
    levels = lut.view(np.float16).astype(np.float32)
    if is_key:
        tab = np.take_along_axis(levels[:, :, None, :, :], codes[..., None].astype(np.int64), axis=-1)[..., 0]
    else:
        grp = np.repeat(np.arange(d // g), g)[None, None, None, :]        # table of each channel
        idx = (grp * L + codes).astype(np.int64)
        tab = np.take_along_axis(levels, idx.reshape(B, H, nq, d), axis=-1)
    xhat = np.where(out, val16.view(np.float16).astype(np.float32), tab).astype(np.float32)
    return NuqTensor(codes, lut, out, val16, xhat)


def nuq_key_thresholds(w: W.Workload, x_bits: np.ndarray, P: int) -> np.ndarray:
    """Per-channel key outlier thresholds frozen at a prefill of P tokens, fp32 [B, H, d].

    "KVQuant-NUQ" page, Dense-and-Sparse outlier isolation: a decode key column
    has one sample, so it is screened against a threshold fixed at prefill.
    Reading: the threshold of a channel is the magnitude of its k-th largest
    |x| over the prefill's quantized tokens [n_sink, P), k the prefill's rank
    count, i.e. the smallest magnitude the prefill sent to the side channel;
    +inf when k = 0 (no decode outliers)."""
    x = _f32_input(x_bits, w.kv_dtype)[:, :, w.n_sink:P]
    k = outlier_count(w.extra.get("outlier_frac", 0.01), x.shape[2])
    B, H, _, d = x.shape
    if k == 0:
        return np.full((B, H, d), np.inf, dtype=np.float32)
    mags = -np.sort(-np.abs(x), axis=2)            # descending along tokens
    return np.ascontiguousarray(mags[:, :, k - 1, :], dtype=np.float32)


def quantize_nuq_stream(w: W.Workload, x_bits: np.ndarray, is_key: bool, P: int, S: int,
                        nnz_cap: int | None = None) -> NuqTensor:
    """Tokens [n_sink, S) of a cache filled by a prefill of P tokens (P > n_sink)
    and then appends of tokens [P, S).

    "KVQuant-NUQ" page, Quantization axes and Dense-and-Sparse outlier isolation:
    values are fitted per token, so an appended value is quantized exactly as at
    prefill.  Keys keep the per-channel tables of the prefill; an appended key
    takes the nearest level of its channel's table and is an outlier when
    |x| >= the channel's frozen threshold (nuq_key_thresholds).  The key side
    channel holds nnz_cap entries per (sequence, head), filled in token order and
    channel order; an outlier that finds it full is not stored and keeps its level.

    Configuration reference, kvquant_refit_interval N > 0 (keys): the key tables
    belong to blocks of N quantized slots (slot = token - n_sink).  Every block
    the prefill reaches keeps the prefill's tables, and its decode keys are
    coded as above.  A block of decode keys only is refitted when its last slot
    arrives: per channel, rank outliers and a Lloyd fit over the block's own N
    keys, exactly as a prefill of those N tokens; until then its keys are not
    coded (they are read from the 16-bit recent window)."""
    if not is_key:
        return quantize_nuq(w, x_bits, False, S)
    N = w.extra.get("refit_interval", 0) or 0
    pre = quantize_nuq(w, x_bits, True, P)
    B, H, _, d = x_bits.shape
    L = 1 << w.bits
    ns = w.n_sink
    pq, sq = P - ns, S - ns                      # prefill's and cache's quantized slot counts
    imm = sq if N == 0 else min(sq, -(-pq // N) * N)   # slots coded with the prefill's tables
    thr = nuq_key_thresholds(w, x_bits, P)
    x = _f32_input(x_bits, w.kv_dtype)[:, :, P:ns + imm]
    nd = x.shape[2]
    codes = np.zeros((B, H, nd, d), dtype=np.uint8)
    for b in range(B):
        for h in range(H):
            for c in range(d):
                codes[b, h, :, c] = nuq_assign(np.ascontiguousarray(x[b, h, :, c]), pre.lut[b, h, c])
    out = np.abs(x) >= thr[:, :, None, :]
    val16 = x.astype(np.float16).view(np.uint16)
    levels = pre.lut.view(np.float16).astype(np.float32)
    tab = np.take_along_axis(levels[:, :, None, :, :], codes[..., None].astype(np.int64), axis=-1)[..., 0]
    xhat = np.where(out, val16.view(np.float16).astype(np.float32), tab).astype(np.float32)
    parts = [(codes, out, val16, xhat)]
    blk_lut, n_coded = None, None
    if N > 0:
        nb = -(-max(sq, 1) // N)
        blk_lut = np.zeros((B, H, nb, d, L), dtype=np.uint16)
        for blk in range(-(-pq // N)):
            blk_lut[:, :, blk] = pre.lut
        blk = -(-pq // N)
        while (blk + 1) * N <= sq:               # complete blocks of decode keys
            t0 = ns + blk * N
            one = quantize_nuq(w, x_bits, True, t0 + N, t0=t0)
            blk_lut[:, :, blk] = one.lut
            parts.append((one.codes, one.outlier, one.val16, one.xhat))
            blk += 1
        n_coded = blk * N if blk > -(-pq // N) else imm
        left = sq - n_coded                      # slots waiting for their block
        if left > 0:
            z = np.zeros((B, H, left, d), dtype=np.uint8)
            parts.append((z, np.zeros(z.shape, bool), np.zeros(z.shape, np.uint16),
                          np.full(z.shape, np.nan, np.float32)))
    codes = np.concatenate([pre.codes] + [p[0] for p in parts], 2)
    out = np.concatenate([pre.outlier] + [p[1] for p in parts], 2)
    val16 = np.concatenate([pre.val16] + [p[2] for p in parts], 2)
    xhat = np.concatenate([pre.xhat] + [p[3] for p in parts], 2)
    if nnz_cap is not None:                      # decode entries in slot order while the channel has room
        for b in range(B):
            for h in range(H):
                room = nnz_cap - int(pre.outlier[b, h].sum())
                flat = out[b, h, pq:].reshape(-1)            # slot-major, channels ascending
                idx = np.flatnonzero(flat)
                cut = idx[max(room, 0):]
                flat[cut] = False
                out[b, h, pq:] = flat.reshape(out[b, h, pq:].shape)
                # an entry that found no room keeps its level
                tt, cc = np.unravel_index(cut, (sq - pq, d))
                for t_, c_ in zip(tt, cc):
                    xhat[b, h, pq + t_, c_] = _nuq_key_level(w, pre, blk_lut, b, h, pq + t_, c_, codes, N)
    return NuqTensor(codes, pre.lut, out, val16, xhat, blk_lut, n_coded)


def _nuq_key_level(w, pre, blk_lut, b, h, slot, c, codes, N):
    lut = pre.lut[b, h, c] if N == 0 else blk_lut[b, h, slot // N, c]
    return np.float32(lut.view(np.float16)[codes[b, h, slot, c]])


def nuq_key_outliers_csr(nt: NuqTensor, qcap: int, nnz_cap: int):
    """Key side channel by token: rowptr [B,H,qcap+1] int32, col/val [B,H,nnz_cap]
    uint16 (channel, fp16 bits), a token's entries in channel order."""
    B, H, nq, d = nt.outlier.shape
    rowptr = np.zeros((B, H, qcap + 1), dtype=np.int32)
    col = np.zeros((B, H, nnz_cap), dtype=np.uint16)
    val = np.zeros((B, H, nnz_cap), dtype=np.uint16)
    for b in range(B):
        for h in range(H):
            cnt = nt.outlier[b, h].sum(axis=1)
            rowptr[b, h, 1:nq + 1] = np.cumsum(cnt)
            rowptr[b, h, nq + 1:] = rowptr[b, h, nq]
            tt, cc = np.nonzero(nt.outlier[b, h])          # row-major: tokens ascending, channels ascending
            col[b, h, :len(cc)] = cc
            val[b, h, :len(cc)] = nt.val16[b, h, tt, cc]
    return rowptr, col, val


def nuq_value_outliers(nt: NuqTensor, qcap: int, k: int):
    """Value side channel, exactly k per token: col/val [B,H,qcap,k] in channel order."""
    B, H, nq, d = nt.outlier.shape
    col = np.zeros((B, H, qcap, k), dtype=np.uint16)
    val = np.zeros((B, H, qcap, k), dtype=np.uint16)
    for b in range(B):
        for h in range(H):
            for t in range(nq):
                cc = np.flatnonzero(nt.outlier[b, h, t])
                col[b, h, t, :len(cc)] = cc
                val[b, h, t, :len(cc)] = nt.val16[b, h, t, cc]
    return col, val


@dataclass
class DqTensor:
    """D-Quant cache of one tensor (all KV heads of a token form one stream).

    container [B, Sq, C] uint8; s16, o16 [B, Sq] uint16 fp16 bits; m [B, Sq, n]
    symbols (n = Hkv * d, head-major); flags [B, Sq] (1 = over budget, 2 =
    container overflow); keys also carry the windowed mean: mean_q [B, Wn, n]
    int8, mean_sc [B, Wn] fp16 bits, mu_hat [B, Wn, n] fp32 (window = 128
    quantized slots); x [B, Sq, n] fp32 holds the coded stream values (rotated,
    keys less their window mean)."""
    container: np.ndarray
    s16: np.ndarray
    o16: np.ndarray
    m: np.ndarray
    flags: np.ndarray
    mean_q: np.ndarray | None = None
    mean_sc: np.ndarray | None = None
    mu_hat: np.ndarray | None = None
    x: np.ndarray | None = None


def dq_tables(w: W.Workload):
    """(key table, value table) of a D-Quant workload."""
    from . import DqTable
    n = w.n_kv_heads * w.head_dim
    a = w.extra.get("alpha", 1.4)
    return (DqTable(n, w.extra.get("levels_k", 8), alpha=a), DqTable(n, w.extra.get("levels_v", 6), alpha=a))


def quantize_dquant(w: W.Workload, x_bits: np.ndarray, is_key: bool, S: int) -> DqTensor:
    """Prefill of tokens [n_sink, S) of x_bits [B,Hkv,S,d] under D-Quant
    (Algorithm 1 per stream; keys rotated and windowed-mean removed)."""
    from . import dq_encode_streams, dq_window_mean, rotate_hadamard_rows
    B, H, _, d = x_bits.shape
    n = H * d
    ns = w.n_sink
    nq = S - ns
    x = _f32_input(x_bits, w.kv_dtype)[:, :, ns:S]                 # [B,H,nq,d]
    rot = w.rot_k if is_key else w.rot_v
    if rot == "hadamard":
        x = rotate_hadamard_rows(x)
    streams = np.ascontiguousarray(x.transpose(0, 2, 1, 3).reshape(B, nq, n))
    tk, tv = dq_tables(w)
    tab = tk if is_key else tv
    C_bytes = w.extra.get("container_k" if is_key else "container_v")
    mean_q = mean_sc = mu_hat = None
    if is_key and w.mean_k:
        Wl = w.extra.get("mean_window", 128)
        nw = -(-nq // Wl)
        mean_q = np.zeros((B, nw, n), dtype=np.int8)
        mean_sc = np.zeros((B, nw), dtype=np.uint16)
        mu_hat = np.zeros((B, nw, n), dtype=np.float32)
        for b in range(B):
            for wi in range(nw):
                q8, sc, mh = dq_window_mean(streams[b, wi * Wl:(wi + 1) * Wl])
                mean_q[b, wi], mean_sc[b, wi], mu_hat[b, wi] = q8, sc, mh
        widx = np.arange(nq) // Wl
        streams = (streams - mu_hat[:, widx]).astype(np.float32)   # fp32 subtraction
    cont, s16, o16, m, flags = dq_encode_streams(streams.reshape(B * nq, n), tab, C_bytes)
    return DqTensor(cont.reshape(B, nq, C_bytes), s16.reshape(B, nq), o16.reshape(B, nq), m.reshape(B, nq, n),
                    flags.reshape(B, nq), mean_q, mean_sc, mu_hat, streams)


def dquant_dequant_f64(w: W.Workload, dt: DqTensor, is_key: bool) -> np.ndarray:
    """Dequantized quantized tokens in the raw space, fp64 [B, Hkv, Sq, d]:
    x^ = s m + o (+ the dequantized window mean for keys), rotated back."""
    B, nq, n = dt.m.shape
    H, d = w.n_kv_heads, w.head_dim
    s = dt.s16.view(np.float16).astype(np.float64)
    o = dt.o16.view(np.float16).astype(np.float64)
    x = s[..., None] * dt.m.astype(np.float64) + o[..., None]
    if dt.mu_hat is not None:
        Wl = w.extra.get("mean_window", 128)
        x = x + dt.mu_hat[:, np.arange(nq) // Wl].astype(np.float64)
    x = x.reshape(B, nq, H, d).transpose(0, 2, 1, 3)
    if (w.rot_k if is_key else w.rot_v) == "hadamard":
        # the normalized Hadamard transform is its own inverse (fp64, exact +-1 entries)
        Hm = np.array([[1.0]])
        while Hm.shape[0] < d:
            Hm = np.block([[Hm, Hm], [Hm, -Hm]])
        x = x @ (Hm / np.sqrt(d))
    return np.ascontiguousarray(x)


def pack_k(codes: np.ndarray, bits: int) -> np.ndarray:
    """[..., n, d] codes -> [..., n, row_bytes] key records."""
    lead = codes.shape[:-1]
    flat = codes.reshape(-1, codes.shape[-1])
    rows = np.stack([pack_k_row(c, bits) for c in flat]) if len(flat) else np.zeros((0, 1), np.uint8)
    return rows.reshape(*lead, -1)


def pack_v(codes: np.ndarray, bits: int) -> np.ndarray:
    """[B, H, n, d] codes -> [B, H, ceil(n/2), pair_bytes] value pair records.
    The second half of a trailing odd pair is left zero."""
    B, H, n, d = codes.shape
    pb = lib().or_v_pair_bytes(d, bits)
    out = np.zeros((B, H, (n + 1) // 2, pb), dtype=np.uint8)
    for b in range(B):
        for h in range(H):
            for t in range(n):
                rec = out[b, h, t // 2]
                pack_v_token(codes[b, h, t], bits, t & 1, rec)
    return out


def meta_f16_bits(s: np.ndarray, o: np.ndarray) -> np.ndarray:
    """[..., n] scale/offset (already binary16 values) -> [..., n, 2] uint16 bits."""
    return np.stack([s.astype(np.float16).view(np.uint16), o.astype(np.float16).view(np.uint16)], -1)


def raw_regions(w: W.Workload, x_bits: np.ndarray, S: int, pos0: int = 0):
    """Raw slots written by tokens [pos0, pos0+n): returns {slot: bits16[B,H,d]}.
    Only tokens that are sinks or among the last n_recent of length S are kept."""
    B, H, n, d = x_bits.shape
    r16 = raw16_bits(x_bits, w.kv_dtype)
    out = {}
    for i in range(n):
        t = pos0 + i
        if t < w.n_sink:
            out[t] = r16[:, :, i]
        elif w.n_recent > 0 and t >= S - w.n_recent:
            out[w.n_sink + (t % w.n_recent)] = r16[:, :, i]
    return out


def attention(w: W.Workload, q: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, S: int,
              qk: QuantTensor, qv: QuantTensor, sm_scale: float | None = None,
              q_comp: np.ndarray | None = None, units=None) -> np.ndarray:
    """fp64 decode attention over a cache of length S.

    q [B,Hq,d] fp32.  k_bits/v_bits [B,Hkv,S,d] are the raw tokens (used as stored
    in the 16-bit regions).  qk/qv hold the quantized tokens [n_sink, S).  Quantized
    tokens are dequantized in fp64 from codes and metadata and mapped back to the raw
    space.  Returns out [B,Hq,d] fp64 (entries of units not listed stay zero).
    """
    L = lib()
    B, Hkv, _, d = k_bits.shape
    G = w.n_q_heads // w.n_kv_heads
    if sm_scale is None:
        sm_scale = 1.0 / np.sqrt(d)
    ns, nr = w.n_sink, w.n_recent
    n_s = min(S, ns)
    q_hi = max(n_s, S - nr)           # quantized tokens [n_s, q_hi)
    rdt = raw_dtype(w.kv_dtype)
    out = np.zeros((B, w.n_q_heads, d), dtype=np.float64)
    if units is None:
        units = [(b, h) for b in range(B) for h in range(Hkv)]
    for (b, h) in units:
        K = np.zeros((S, d), dtype=np.float64)
        V = np.zeros((S, d), dtype=np.float64)
        # 16-bit regions, as stored
        kr = raw16_to_f64(raw16_bits(k_bits[b, h, :S], w.kv_dtype), rdt)
        vr = raw16_to_f64(raw16_bits(v_bits[b, h, :S], w.kv_dtype), rdt)
        K[:n_s], V[:n_s] = kr[:n_s], vr[:n_s]
        K[q_hi:S], V[q_hi:S] = kr[q_hi:S], vr[q_hi:S]
        nq = q_hi - n_s
        if nq > 0 and isinstance(qk, DqTensor):
            K[n_s:q_hi] = dquant_dequant_f64(w, qk, True)[b, h, :nq]
            V[n_s:q_hi] = dquant_dequant_f64(w, qv, False)[b, h, :nq]
        elif nq > 0 and isinstance(qk, NuqTensor):
            K[n_s:q_hi] = qk.xhat[b, h, :nq].astype(np.float64)
            V[n_s:q_hi] = qv.xhat[b, h, :nq].astype(np.float64)
        elif nq > 0:
            for X, qt, key in ((K, qk, True), (V, qv, False)):
                rot = _ROT[w.rot_k if key else w.rot_v]
                cu = np.ascontiguousarray(qt.codes[b, h, :nq])
                su = np.ascontiguousarray(qt.s[b, h, :nq])
                ou = np.ascontiguousarray(qt.o[b, h, :nq])
                mu_p = None
                if key and w.mean_k:
                    mu_u = np.ascontiguousarray(qt.mu[b, h])
                    mu_p = mu_u.ctypes.data_as(C.c_void_p)
                deq = np.zeros((nq, d), dtype=np.float64)
                L.or_dequant_f64(cu, su, ou, mu_p, nq, d, 1 if rot == 1 else 0, deq)
                if rot == 2:
                    # keys live in the transformed space: q~ = Tinv^T q, so map k back
                    # with k_raw[j] = sum_i Tinv^T[i][j] k~[i] (fp64 on the fp32 matrix).
                    deq = deq @ q_comp[h].astype(np.float64)
                X[n_s:q_hi] = deq
        qg = q[b, h * G:(h + 1) * G].astype(np.float64)
        out[b, h * G:(h + 1) * G] = _attn(L, qg, K, V, sm_scale)
    return out


def _attn(L, q, K, V, sm_scale):
    G, d = q.shape
    o = np.zeros((G, d), dtype=np.float64)
    L.or_attention_f64(np.ascontiguousarray(q), np.ascontiguousarray(K), np.ascontiguousarray(V),
                       G, K.shape[0], d, float(sm_scale), o)
    return o


__all__ = ["QuantTensor", "quantize_tensor", "NuqTensor", "quantize_nuq", "nuq_key_outliers_csr",
           "nuq_key_thresholds", "quantize_nuq_stream",
           "DqTensor", "dq_tables", "quantize_dquant", "dquant_dequant_f64",
           "nuq_value_outliers", "pack_k", "pack_v", "meta_f16_bits", "raw_regions",
           "attention", "raw16_bits", "raw16_to_f64", "raw_dtype"]
