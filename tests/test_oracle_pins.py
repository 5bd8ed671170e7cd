"""Pins of the CPU oracle against things other than itself (no GPU).

Each test ties one oracle step to a library routine, a closed form, a
hand-computed example or a brute force, so that a dropped term, a wrong sign,
a wrong index or a transposed operand in the oracle fails here.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
import workloads as W


# ---------------------------------------------------------------- fp16 ----

def test_f32_to_f16_matches_numpy_rne():
    g = np.random.default_rng(1)
    vals = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * 10.0 ** g.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e6, -1e6, np.inf, -np.inf,
                  2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -26, 6.1e-5, 1.0 + 2.0 ** -11,
                  1.0 + 3 * 2.0 ** -11, 2049.0, 2051.0], dtype=np.float32),
    ]).astype(np.float32)
    ours = oracle.f32_to_f16_bits(vals)
    with np.errstate(over="ignore"):
        ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(ours, ref)
    nan = oracle.f32_to_f16_bits(np.array([np.nan], np.float32))[0]
    assert (nan & 0x7C00) == 0x7C00 and (nan & 0x3FF) != 0


def test_f16_to_f32_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f32(bits)
    ref = bits.view(np.float16).astype(np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(ours[fin].view(np.uint32), ref[fin].view(np.uint32))
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


# ------------------------------------------------------------- Hadamard ----

@pytest.mark.parametrize("d", [2, 4, 8, 16, 32, 64, 128])
def test_fwht_matches_sylvester_matrix(d):
    H = scipy.linalg.hadamard(d).astype(np.float64)
    x = np.random.default_rng(d).standard_normal(d)
    assert np.allclose(oracle.fwht(x), H @ x, rtol=0, atol=1e-12)
    # columns: FWHT(e_i) == H[:, i] exactly, in fp32 too
    for i in range(d):
        e = np.zeros(d, np.float32)
        e[i] = 1
        assert np.array_equal(oracle.fwht(e), H[:, i].astype(np.float32))


@pytest.mark.parametrize("d", [64, 128])
def test_fwht_orthogonality_exact(d):
    # H H^T = d I, and applying the transform twice gives d*x exactly for small ints
    H = np.stack([oracle.fwht(np.eye(d, dtype=np.float32)[i]) for i in range(d)])
    assert np.array_equal(H @ H.T, d * np.eye(d, dtype=np.float32))
    x = np.random.default_rng(7).integers(-8, 9, d).astype(np.float32)
    assert np.array_equal(oracle.fwht(oracle.fwht(x)), d * x)


@pytest.mark.parametrize("d", [64, 128])
def test_normalized_rotation_involution_and_parseval(d):
    x = np.random.default_rng(3).standard_normal(d).astype(np.float32)
    y = oracle.rotate_hadamard(x)
    H = scipy.linalg.hadamard(d) / math.sqrt(d)
    assert np.allclose(y, H @ x.astype(np.float64), atol=2e-6)
    assert np.allclose(oracle.rotate_hadamard(y), x, atol=3e-6)
    assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-5 * np.linalg.norm(x)
    assert oracle.hadamard_scale(64) == 0.125


def test_dense_transform_matches_matmul():
    d = 128
    g = np.random.default_rng(4)
    T = g.standard_normal((d, d)).astype(np.float32)
    x = g.standard_normal(d).astype(np.float32)
    assert np.allclose(oracle.rotate_dense(T, x), T.astype(np.float64) @ x, rtol=1e-5, atol=1e-4)
    # a permutation matrix moves values exactly
    P = np.eye(d, dtype=np.float32)[g.permutation(d)]
    assert np.array_equal(oracle.rotate_dense(P, x), P @ x)


# --------------------------------------------------------------- affine ----

def test_affine_hand_example_round_half_even():
    # grid o=0, s=1 (b=2, min 0, max 3): half-way values round to the even level
    x = np.array([0.0, 0.5, 1.5, 2.5, 3.0, 1.49, 2.51, 0.51], np.float32)
    codes, s, o = oracle.affine_quantize(x, 2, meta_f16=False)
    assert (s, o) == (1.0, 0.0)
    assert codes.tolist() == [0, 0, 2, 2, 3, 1, 3, 1]


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_affine_fp32_meta_error_bound_and_ends(bits):
    g = np.random.default_rng(bits)
    for _ in range(50):
        x = g.standard_normal(128).astype(np.float32) * g.uniform(0.01, 50)
        codes, s, o = oracle.affine_quantize(x, bits, meta_f16=False)
        L = 2 ** bits
        assert s == np.float32(np.float32(x.max() - x.min()) / np.float32(L - 1))
        assert o == x.min()
        xh = oracle.affine_dequant(codes, s, o)
        assert np.all(np.abs(x.astype(np.float64) - xh) <= s / 2 * (1 + 1e-5) + 1e-6 * np.abs(x).max())
        assert codes[np.argmin(x)] == 0 and codes[np.argmax(x)] == L - 1
        # brute force: the code is a nearest level (ties allowed)
        lev = o + s * np.arange(L, dtype=np.float64)
        dist = np.abs(x[:, None].astype(np.float64) - lev[None])
        best = dist.min(1)
        got = dist[np.arange(128), codes]
        assert np.all(got <= best + 1e-6 * s)


@pytest.mark.parametrize("bits", [2, 4])
def test_affine_fp16_meta_bound(bits):
    g = np.random.default_rng(10 + bits)
    for _ in range(50):
        x = (g.standard_normal(128) * 3 + g.standard_normal()).astype(np.float32)
        codes, s16, o16 = oracle.affine_quantize(x, bits, meta_f16=True)
        L = 2 ** bits
        s32 = np.float32(np.float32(x.max() - x.min()) / np.float32(L - 1))
        o32 = x.min()
        assert s16 == np.float16(s32) and o16 == np.float16(o32)
        xh = oracle.affine_dequant(codes, s16, o16).astype(np.float64)
        bound = s16 / 2 + abs(o32 - o16) + (L - 1) * abs(float(s32) - float(s16)) + 1e-5
        assert np.all(np.abs(x - xh) <= bound)


def test_affine_constant_vector():
    x = np.full(128, 1.7, np.float32)
    codes, s, o = oracle.affine_quantize(x, 2, meta_f16=False)
    assert s == 0 and np.all(codes == 0) and np.array_equal(oracle.affine_dequant(codes, s, o), x)


def test_percentile_clip_matches_numpy_quantile():
    g = np.random.default_rng(5)
    for _ in range(20):
        x = g.standard_t(3, 128).astype(np.float32)
        codes, s, o = oracle.affine_quantize(x, 2, meta_f16=False, clip=0.999)
        lo, hi = np.quantile(x.astype(np.float64), [0.001, 0.999], method="linear")
        assert abs(o - lo) <= 1e-5 * max(1, abs(lo))
        assert abs(s * 3 - (hi - lo)) <= 1e-4 * max(1, hi - lo)
        assert codes[np.argmax(x)] == 3 and codes[np.argmin(x)] == 0
    i, f = oracle.quantile_pos(0.999, 128)
    assert i == 126 and abs(f - 0.873) < 1e-6


def test_mean_removal_is_the_channel_mean():
    w = W.TINY.with_(n_sink=2, n_recent=8)
    k, _ = W.make_kv(w, seq=64)
    qt = oracle.quantize_tensor(w, k, True, 64)
    y = np.stack([oracle.rotate_hadamard(k[0, 0, t]) for t in range(64)]).astype(np.float64)
    ref = y[2:64 - 8].mean(0)
    assert np.allclose(qt.mu[0, 0], ref, atol=1e-5)
    # sinks and recent tokens are excluded from the mean: changing them leaves it unchanged
    k2 = k.copy()
    k2[0, 0, :2] += 100
    k2[0, 0, 56:] -= 50
    qt2 = oracle.quantize_tensor(w, k2, True, 64)
    assert np.array_equal(qt.mu, qt2.mu)
    assert np.array_equal(qt.codes[0, 0, :54], qt2.codes[0, 0, :54])


# -------------------------------------------------------------- packing ----

def test_pack_k_hand_built_bytes():
    c = np.zeros(128, np.uint8)
    c[0], c[8], c[1], c[16], c[2] = 5, 10, 3, 7, 9
    row = oracle.pack_k_row(c, 4)
    exp = np.zeros(64, np.uint8)
    exp[0], exp[2], exp[1], exp[16] = 0xA5, 0x03, 0x07, 0x09
    assert np.array_equal(row, exp)
    c2 = np.zeros(128, np.uint8)
    c2[0], c2[8], c2[16], c2[1] = 1, 2, 3, 3
    row2 = oracle.pack_k_row(c2, 2)
    exp2 = np.zeros(32, np.uint8)
    exp2[0] = 1 | (2 << 2) | (3 << 4)
    exp2[2] = 3
    assert np.array_equal(row2, exp2)


def test_pack_v_hand_built_bytes():
    rec = np.zeros(64, np.uint8)
    c0 = np.zeros(128, np.uint8)
    c0[0], c0[8], c0[16], c0[1] = 1, 2, 3, 2
    c1 = np.zeros(128, np.uint8)
    c1[0] = 3
    oracle.pack_v_token(c0, 2, 0, rec)
    oracle.pack_v_token(c1, 2, 1, rec)
    exp = np.zeros(64, np.uint8)
    exp[0] = 1 | (2 << 2) | (3 << 4)
    exp[2] = 3
    exp[8] = 2
    assert np.array_equal(rec, exp)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_roundtrip_and_bijection(d, bits):
    if bits == 3 and d == 64:
        pytest.skip("3-bit records need d = 128")
    g = np.random.default_rng(d + bits)
    for _ in range(20):
        c = g.integers(0, 2 ** bits, d).astype(np.uint8)
        assert np.array_equal(oracle.unpack_k_row(oracle.pack_k_row(c, bits), d, bits), c)
        rec = np.zeros(2 * d * bits // 8, np.uint8)
        c2 = g.integers(0, 2 ** bits, d).astype(np.uint8)
        oracle.pack_v_token(c, bits, 0, rec)
        oracle.pack_v_token(c2, bits, 1, rec)
        assert np.array_equal(oracle.unpack_v_token(rec, d, bits, 0), c)
        assert np.array_equal(oracle.unpack_v_token(rec, d, bits, 1), c2)
    # every record bit is used by exactly one (channel, bit) pair
    full = np.full(d, 2 ** bits - 1, np.uint8)
    assert np.unpackbits(oracle.pack_k_row(full, bits)).sum() == d * bits
    seen = np.zeros(d * bits, np.int64)
    for ch in range(d):
        for k in range(bits):
            c = np.zeros(d, np.uint8)
            c[ch] = 1 << k
            bitsv = np.unpackbits(oracle.pack_k_row(c, bits), bitorder="little")
            assert bitsv.sum() == 1
            seen[np.argmax(bitsv)] += 1
    assert np.all(seen == 1)


# ------------------------------------------------------------ attention ----

def test_attention_matches_torch_sdpa():
    g = np.random.default_rng(11)
    G, S, d = 4, 300, 64
    q = g.standard_normal((G, d))
    K = g.standard_normal((S, d))
    V = g.standard_normal((S, d))
    out = oracle.attention_f64(q, K, V, 1 / math.sqrt(d))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None, :], torch.from_numpy(K)[None, None].expand(1, G, S, d),
        torch.from_numpy(V)[None, None].expand(1, G, S, d)).numpy()[0, :, 0]
    assert np.allclose(out, ref, atol=1e-12)
    # a different scale is honored
    out2 = oracle.attention_f64(q, K, V, 0.3)
    ref2 = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, :, None, :], torch.from_numpy(K)[None, None].expand(1, G, S, d),
        torch.from_numpy(V)[None, None].expand(1, G, S, d), scale=0.3).numpy()[0, :, 0]
    assert np.allclose(out2, ref2, atol=1e-12)


def test_attention_special_cases():
    g = np.random.default_rng(12)
    d = 32
    q = g.standard_normal((2, d))
    V = g.standard_normal((50, d))
    K = np.tile(g.standard_normal(d), (50, 1))       # all-equal keys -> mean of V
    assert np.allclose(oracle.attention_f64(q, K, V, 0.2), np.tile(V.mean(0), (2, 1)), atol=1e-12)
    assert np.allclose(oracle.attention_f64(q, K[:1], V[:1], 0.2), np.tile(V[0], (2, 1)), atol=1e-14)
    # permuting the tokens changes nothing
    K2 = g.standard_normal((50, d))
    p = g.permutation(50)
    assert np.allclose(oracle.attention_f64(q, K2, V, 0.2), oracle.attention_f64(q, K2[p], V[p], 0.2), atol=1e-13)


def test_dequant_f64_inverse_rotation_and_fold_identities():
    """Eq. (7)-(9) of the D-Quant page: the affine terms fold into q.k and P.V."""
    g = np.random.default_rng(13)
    d, n = 128, 40
    codes = g.integers(0, 4, (n, d)).astype(np.uint8)
    s = g.uniform(0.1, 2, n).astype(np.float32)
    o = g.uniform(-3, 0, n).astype(np.float32)
    mu = g.standard_normal(d).astype(np.float32)
    import ctypes as C
    L = oracle.lib()
    out = np.zeros((n, d))
    L.or_dequant_f64(codes, s, o, mu.ctypes.data_as(C.c_void_p), n, d, 1, out)
    H = scipy.linalg.hadamard(d) / math.sqrt(d)
    rot = o[:, None].astype(np.float64) + s[:, None].astype(np.float64) * codes + mu[None].astype(np.float64)
    assert np.allclose(out, rot @ H.T, atol=1e-12)
    q = g.standard_normal(d)
    lhs = rot @ q
    rhs = s * (codes @ q) + o * q.sum() + q @ mu
    assert np.allclose(lhs, rhs, atol=1e-12)
    a = g.uniform(0, 1, n)
    assert np.allclose(a @ (o[:, None] + s[:, None] * codes.astype(np.float64)),
                       (a * s) @ codes + (a * o).sum(), atol=1e-12)


# --------------------------------------------------------------- regions ----

def test_raw_regions_sinks_exact_and_recent_ring():
    w = W.LLAMA.with_(batch=1, n_kv_heads=1, n_q_heads=4, seq=300)
    k, _ = W.make_kv(w)
    S = 300
    reg = oracle.raw_regions(w, k, S)
    assert sorted(reg) == list(range(4)) + sorted(4 + (t % 128) for t in range(S - 128, S))
    for t in range(4):
        assert np.array_equal(reg[t], k[:, :, t])        # bit-exact sink rows
    for t in range(S - 128, S):
        assert np.array_equal(reg[4 + t % 128], k[:, :, t])
    assert oracle.raw_slot(299, 4, 128) == 4 + 299 % 128
    # n_sink = 0: no sink slots at all
    reg0 = oracle.raw_regions(w.with_(n_sink=0, n_recent=0), k, S)
    assert reg0 == {}


def test_three_bit_key_row_hand_built_bytes():
    # d = 128, 3 bits: a 32-byte 2-bit plane, then a 16-byte 1-bit plane whose
    # field f sits at bit P(f) of its half: P = 2, 4, 6, 8, 10, 12, 14, 0, 3,
    # 5, 7, 9, 11, 13, 15, 1.  Channel c -> field idx = tig*16 + 2i + sub
    # (tig = (c >> 1) & 3, i = c >> 4, sub = (c >> 3) & 1), half c & 1.
    codes = np.zeros(128, np.uint8)
    # bit 2 only: channel -> (idx, half): 0 -> (0, 0) P 2; 1 -> (0, 1) P 2;
    # 8 -> (1, 0) P 4; 56 -> (7, 0) P 0; 120 -> (15, 0) P 1; 64 -> (8, 0) P 3;
    # 65 -> (8, 1) P 3; 2 -> (16, 0): second 1-bit word, P 2
    for c in (0, 1, 8, 56, 120, 64, 65, 2):
        codes[c] = 4
    codes[3] = 3            # (16, 1): 2-bit plane word 2, field 0, half 1 -> byte 10 = 0b11
    exp = np.zeros(48, np.uint8)
    exp[32] = 0x04 | 0x10 | 0x01 | 0x02 | 0x08   # half 0 of 1-bit word 0: bits 2, 4, 0, 1, 3
    exp[34] = 0x04 | 0x08                          # half 1 of 1-bit word 0: bits 2, 3
    exp[36] = 0x04                                 # 1-bit word 1, bit 2
    exp[10] = 0x03
    row = oracle.pack_k_row(codes, 3)
    assert np.array_equal(row, exp), np.flatnonzero(row != exp)
    assert np.array_equal(oracle.unpack_k_row(row, 128, 3), codes)
