"""Pins of the D-Quant oracle (fixed-size rANS container with Drift) against
facts fixed outside the oracle.

Source: "D-Quant: Driftable Entropy Coding for KV Cache Quantization" --
Sec. 4.2 Eq. (3)-(4) (container budget, token-wise affine grid, Gaussian
order-statistics model), Sec. 4.3 Eq. (5)-(6) (Drift), Sec. 4.4 (sharpening),
App. A Algorithms 1-2 (encoder, decoder), App. C (drift moves symbols by at
most one level).  The rANS coder is Duda (2013), cited on the page.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "rans_hand.json")
L_STATE = 1 << 23


# ---- probability model ------------------------------------------------------

@pytest.mark.parametrize("n,want,tol", [
    (1, 0.0, 1e-12),
    (2, 1.0 / math.sqrt(math.pi), 1e-9),              # closed form
    (3, 3.0 / (2.0 * math.sqrt(math.pi)), 1e-9),      # closed form
    (5, 1.16296, 2e-5),                                # tabulated expected maxima of N(0,1) samples
    (10, 1.53875, 2e-5),
    (100, 2.50759, 2e-5),
])
def test_expected_max_of_normals(n, want, tol):
    assert abs(oracle.dq_expected_max(n) - want) < tol


def test_bin_probabilities_match_a_library_integration():
    scipy = pytest.importorskip("scipy")
    from scipy import integrate, stats
    n, M = 1024, 8
    dens = lambda x: x * n * stats.norm.pdf(x) * stats.norm.cdf(x) ** (n - 1)
    a = integrate.quad(dens, -12, 12, limit=400, points=[2.0, 3.0, 4.0])[0]
    assert abs(oracle.dq_expected_max(n) - a) < 1e-8
    u = -a + 2 * a * np.arange(M) / (M - 1)
    edges = np.concatenate([[-np.inf], (u[1:] + u[:-1]) / 2, [np.inf]])
    p = np.diff(stats.norm.cdf(edges))
    t = oracle.DqTable(n, M, alpha=1.4)
    assert np.allclose(t.prob, p, atol=1e-10)


@pytest.mark.parametrize("M", [2, 3, 4, 6, 8, 12, 16])
@pytest.mark.parametrize("alpha", [1.0, 1.4])
def test_frequency_table_is_a_valid_symmetric_model(M, alpha):
    t = oracle.DqTable(1024, M, alpha=alpha)
    assert t.f.sum() == 256 and t.f.min() >= 1
    assert np.array_equal(t.c, np.concatenate([[0], np.cumsum(t.f)[:-1]]))
    assert abs(t.prob.sum() - 1.0) < 1e-12
    assert np.allclose(t.prob, t.prob[::-1], atol=1e-12)
    # the model is symmetric; only the one frequency that absorbed the rounding
    # shortfall may break the mirror
    assert (t.f != t.f[::-1]).sum() <= 2
    # sharpening never flattens: the central symbols are at least as likely
    assert t.f[M // 2] >= t.f[0]
    # fixed-point costs round -log2(f/256) up to 1/65536 of a bit
    exact = (8.0 - np.log2(t.f)) * 65536.0
    assert np.all(t.r >= exact - 1e-9) and np.all(t.r < exact + 1.0)


def test_costs_of_power_of_two_frequencies_are_exact():
    f = [128, 64, 32, 16, 8, 4, 2, 1, 1]
    t = oracle.DqTable.from_freqs(f)
    assert t.r.tolist() == [65536 * k for k in (1, 2, 3, 4, 5, 6, 7, 8, 8)]


def test_paper_operating_point_bits_per_value():
    # 331-byte keys (+ an INT8 mean of 1024 channels per 128 tokens) and 231-byte
    # values, per 1024-value stream: 2.68 and 1.84 bits per value, 2.26 on average
    n = 1024
    # with fp16 (s, o) per stream: (331 + 4 + 8) * 8 / 1024 = 2.68, (231 + 4) * 8 / 1024 = 1.84
    assert round((331 + 4 + n / 128) * 8 / n, 2) == 2.68
    assert round((231 + 4) * 8 / n, 2) == 1.84
    assert round(((331 + 4 + n / 128) + (231 + 4)) * 8 / (2 * n), 2) == 2.26


def test_sixteen_levels_do_not_fit_2p26_bits():
    # the cheapest 16-level symbol costs more than a 289-byte container allows
    t = oracle.DqTable(1024, 16)
    assert 1024 * t.r.min() > oracle.dq_budget_fx(289)
    assert 1024 * t.r.min() <= oracle.dq_budget_fx(343)


# ---- rANS container ---------------------------------------------------------

def test_hand_worked_containers():
    g = json.load(open(GOLDEN))
    for case in g["cases"]:
        t = oracle.DqTable.from_freqs(case["f"])
        assert t.c.tolist() == case["c"]
        m = np.array(case["symbols"], dtype=np.uint8)
        cont, pushed = oracle.rans_encode(m, t, case["C"])
        assert pushed == case["emitted"], case["name"]
        assert cont.tolist() == case["container"], case["name"]
        dm, xf, used = oracle.rans_decode(cont, m.size, t)
        assert np.array_equal(dm, m) and xf == L_STATE and used == pushed


def _random_table(g, M):
    while True:
        f = g.integers(1, 60, size=M)
        f = np.maximum(1, np.round(f * 256 / f.sum())).astype(int)
        f[np.argmax(f)] += 256 - f.sum()
        if f.min() >= 1:
            return oracle.DqTable.from_freqs(f)


@pytest.mark.parametrize("seed", range(6))
def test_round_trip_and_information_identity(seed):
    g = np.random.default_rng(seed)
    M = int(g.integers(2, 17))
    t = _random_table(g, M)
    n = int(g.integers(1, 700))
    p = t.f / 256.0
    m = g.choice(M, size=n, p=p).astype(np.uint8)
    info = float(np.sum(-np.log2(t.f[m] / 256.0)))
    C = 4 + int(info / 8) + 64
    cont, pushed = oracle.rans_encode(m, t, C)
    assert pushed >= 0
    dm, xf, used = oracle.rans_decode(cont, n, t)
    assert np.array_equal(dm, m)
    assert xf == L_STATE and used == pushed          # the decoder ends where the encoder began
    assert np.all(cont[4 + pushed:] == 0)
    x_final = int(cont[0]) | int(cont[1]) << 8 | int(cont[2]) << 16 | int(cont[3]) << 24
    bits = 8 * pushed + math.log2(x_final) - 23
    # each step scales the state by 256/f within a factor (1 +- 2^-15)
    assert abs(bits - info) <= n * math.log2(1 + 2.0 ** -15) + 1e-9


def test_uniform_frequencies_cost_exactly_k_bits():
    t = oracle.DqTable.from_freqs([64, 64, 64, 64])    # 2 bits per symbol
    g = np.random.default_rng(3)
    for n in (1, 3, 4, 13, 64):
        m = g.integers(0, 4, size=n).astype(np.uint8)
        cont, pushed = oracle.rans_encode(m, t, 64)
        x_final = int.from_bytes(bytes(cont[:4]), "little")
        assert 8 * pushed + math.log2(x_final) - 23 == pytest.approx(2 * n, abs=n * 1e-4)
        # the state holds 23..31 bits, so 2n - 8 < 8 * bytes <= 2n
        assert pushed == n // 4


# ---- Drift ------------------------------------------------------------------

def _grid(s, o, M):
    return np.array([np.float32(o) + np.float32(s) * np.float32(m) for m in range(M)], dtype=np.float32)


def _minmax(x, M):
    lo, hi = np.float32(x.min()), np.float32(x.max())
    return np.float32((hi - lo) / np.float32(M - 1)), lo


@pytest.mark.parametrize("seed", range(5))
def test_drift_is_optimal_for_its_own_rate_brute_force(seed):
    g = np.random.default_rng(100 + seed)
    n, M = 5, 4
    t = oracle.DqTable(n, M, alpha=1.4)
    x = g.standard_normal(n).astype(np.float32)
    s, o = _minmax(x, M)
    grid = _grid(s, o, M).astype(np.float64)
    xs = x.astype(np.float64)
    allm = np.array(list(itertools.product(range(M), repeat=n)))
    dist = ((xs[None, :] - grid[allm]) ** 2).sum(1)
    cost = t.r[allm].sum(1)
    lo_b, hi_b = int(cost.min()), int(cost.max())
    for budget in np.linspace(lo_b - 1000, hi_b + 1000, 25).astype(np.int64):
        m, c, ok = oracle.dq_drift(x, s, o, t, budget_fx=int(budget))
        assert c == int(t.r[m].sum())
        if budget < lo_b:
            assert not ok
            continue
        assert ok and c <= budget
        d = float(((xs - grid[m]) ** 2).sum())
        # no assignment that spends at most as many bits has lower distortion
        better = dist[(cost <= c)].min()
        assert d <= better + 1e-6 * max(1.0, better), (budget, d, better)


def test_drift_distortion_falls_as_the_budget_grows():
    g = np.random.default_rng(8)
    t = oracle.DqTable(1024, 8)
    x = g.standard_normal(1024).astype(np.float32)
    s, o = _minmax(x, 8)
    grid = _grid(s, o, 8).astype(np.float64)
    prev = None
    for C in range(200, 420, 10):
        m, c, ok = oracle.dq_drift(x, s, o, t, C)
        d = float(((x.astype(np.float64) - grid[m]) ** 2).sum())
        if ok:
            assert c <= oracle.dq_budget_fx(C)
        if prev is not None:
            assert d <= prev + 1e-9
        prev = d


def test_drift_is_nearest_rounding_when_that_fits():
    g = np.random.default_rng(9)
    t = oracle.DqTable(1024, 8)
    x = g.standard_normal(1024).astype(np.float32)
    s, o = _minmax(x, 8)
    grid = _grid(s, o, 8)
    near = np.argmin(np.abs(x[:, None] - grid[None, :]), axis=1)
    assert int(t.r[near].sum()) <= oracle.dq_budget_fx(1000)
    m, _, ok = oracle.dq_drift(x, s, o, t, 1000)
    assert ok and np.array_equal(m, near)


# ---- Refit ------------------------------------------------------------------

def test_refit_recovers_an_exact_line():
    g = np.random.default_rng(4)
    m = g.integers(0, 8, size=1024).astype(np.uint8)
    x = (np.float32(-1.5) + np.float32(0.25) * m.astype(np.float32)).astype(np.float32)
    s, o = oracle.dq_refit(x, m, 9.0, 9.0)
    assert s == 0.25 and o == -1.5


def test_refit_is_least_squares():
    g = np.random.default_rng(5)
    x = g.standard_normal(1024).astype(np.float32)
    m = np.clip(np.rint((x + 3) / 0.8), 0, 7).astype(np.uint8)
    s, o = oracle.dq_refit(x, m, 0.0, 0.0)
    A = np.stack([m.astype(np.float64), np.ones(1024)], 1)
    ls, lo = np.linalg.lstsq(A, x.astype(np.float64), rcond=None)[0]
    assert abs(s - ls) < 1e-5 and abs(o - lo) < 1e-5


def test_refit_keeps_a_degenerate_fit():
    x = np.random.default_rng(6).standard_normal(64).astype(np.float32)
    m = np.full(64, 3, dtype=np.uint8)
    assert oracle.dq_refit(x, m, 0.5, -0.25) == (0.5, -0.25)


# ---- windowed INT8 key mean -------------------------------------------------

def test_window_mean_exact_and_bounded():
    g = np.random.default_rng(7)
    n = 1024
    mu = (g.integers(-64, 64, size=n) / 16.0).astype(np.float32)   # dyadic: sums are exact
    y = np.repeat(mu[None, :], 128, 0)
    q, sc16, mu_hat = oracle.dq_window_mean(y)
    sc = float(np.array([sc16], dtype=np.uint16).view(np.float16)[0])
    assert sc == float(np.float16(np.float32(np.abs(mu).max()) / np.float32(127)))
    assert np.abs(q.astype(int)).max() == 127
    assert np.all(np.abs(mu_hat.astype(np.float64) - mu) <= sc / 2 * (1 + 1e-3))
    q0, s0, m0 = oracle.dq_window_mean(np.zeros((5, n), dtype=np.float32))
    assert s0 == 0 and not q0.any() and not m0.any()


# ---- Algorithm 1 end to end -------------------------------------------------

@pytest.mark.parametrize("M,C", [(8, 331), (6, 231)])
def test_streams_fill_their_containers_and_decode(M, C):
    g = np.random.default_rng(M)
    t = oracle.DqTable(1024, M)
    F = oracle.dq_pow2_table()
    changed = []
    for _ in range(20):
        x = g.standard_normal(1024).astype(np.float32)
        r = oracle.dq_encode_stream(x, t, C, F)
        assert r["flags"] == 0
        m, xf, used = oracle.rans_decode(r["container"], 1024, t)
        assert np.array_equal(m, r["m"]) and xf == L_STATE and 4 + used <= C
        # drift only makes local corrections: no symbol moves more than one level
        assert np.abs(r["m"].astype(int) - r["m_near"].astype(int)).max() <= 1
        changed.append(np.mean(r["m"] != r["m_near"]))
    assert np.mean(changed) < 0.2


def test_key_streams_drift_less_than_value_streams():
    g = np.random.default_rng(11)
    F = oracle.dq_pow2_table()
    fr = {}
    for M, C in ((8, 331), (6, 231)):
        t = oracle.DqTable(1024, M)
        fr[M] = np.mean([np.mean((lambda r: r["m"] != r["m_near"])(
            oracle.dq_encode_stream(g.standard_normal(1024).astype(np.float32), t, C, F))) for _ in range(20)])
    assert fr[8] < fr[6]


def test_constant_stream():
    t = oracle.DqTable(1024, 8)
    x = np.full(1024, 0.75, dtype=np.float32)
    r = oracle.dq_encode_stream(x, t, 331)
    assert r["flags"] == 0 and r["s16"] == 0
    assert float(np.array([r["o16"]], dtype=np.uint16).view(np.float16)[0]) == 0.75
    assert np.all(r["m"] == np.argmax(t.f))     # every value takes the cheapest symbol


@pytest.mark.parametrize("M, C, frac_max", [(8, 331, 0.02), (6, 231, 0.12), (8, 286, 0.10), (6, 200, 0.14)])
def test_drift_makes_sparse_local_corrections(M, C, frac_max):
    """D-Quant App. C ("Drift makes only sparse, local corrections"): against the
    nearest level on the final grid, drift changes a small share of the symbols
    and moves none by more than one level.  Standard-normal streams of 1024
    values at the 2.26- and 1.96-bit containers (the page measures 0.75 % of
    key and 5.00 % of value symbols on real caches)."""
    rng = np.random.default_rng(123)
    t = oracle.DqTable(1024, M, alpha=1.4)
    changed = 0
    for _ in range(200):
        r = oracle.dq_encode_stream(rng.standard_normal(1024).astype(np.float32), t, C)
        assert r["flags"] == 0
        d = np.abs(r["m"].astype(int) - r["m_near"].astype(int))
        assert d.max() <= 1
        changed += int((d > 0).sum())
    assert changed / (200 * 1024) < frac_max


# ---- Algorithm 1 as a sequence of steps -------------------------------------

ALG1 = os.path.join(os.path.dirname(__file__), "golden", "alg1_hand.json")


def _f16_bits(v: float) -> int:
    return int(np.array([v], dtype=np.float16).view(np.uint16)[0])


def _f16_val(bits: int) -> float:
    return float(np.array([bits], dtype=np.uint16).view(np.float16)[0])


def _lstsq(x, m):
    A = np.stack([np.asarray(m, np.float64), np.ones(len(x))], 1)
    return np.linalg.lstsq(A, np.asarray(x, np.float64), rcond=None)[0]


def test_algorithm1_hand_worked_stream():
    """App. A Algorithm 1 on a stream worked by hand (tests/golden/alg1_hand.json):
    FitMinMax, Drift, Refit, fp16 s and o, Drift, then the coder.  The fixture's
    own steps are checked with a library least-squares solve and numpy's fp16
    rounding, and each plausible wrong order (no refit, no second Drift, fp16
    before the first Drift) is shown to give a different stream."""
    d = json.load(open(ALG1))
    x = np.array(d["x"], dtype=np.float32)
    M, C = d["M"], d["container"]
    t = oracle.DqTable.from_freqs(d["freqs"])
    r = oracle.dq_encode_stream(x, t, C)
    want_s16, want_o16 = d["step4_fp16"]["s16_bits"], d["step4_fp16"]["o16_bits"]
    assert r["flags"] == 0
    assert (r["s16"], r["o16"]) == (want_s16, want_o16)
    assert r["m"].tolist() == d["step5_drift_symbols"]
    m, xf, _ = oracle.rans_decode(r["container"], x.size, t)
    assert m.tolist() == d["step5_drift_symbols"] and xf == L_STATE

    # the fixture is consistent with the page's steps
    s0 = (np.float32(x.max()) - np.float32(x.min())) / np.float32(M - 1)
    assert float(s0) == d["step1_fitminmax"]["s"] and float(x.min()) == d["step1_fitminmax"]["o"]
    grid0 = np.float32(0.0) + s0 * np.arange(M, dtype=np.float32)
    assert np.argmin(np.abs(x[:, None] - grid0[None, :]), 1).tolist() == d["step2_drift_symbols"]
    ls, lo = _lstsq(x, d["step2_drift_symbols"])
    assert abs(ls - d["step3_refit"]["s"]) < 1e-12 and abs(lo - d["step3_refit"]["o"]) < 1e-12
    assert (_f16_bits(ls), _f16_bits(lo)) == (want_s16, want_o16)
    g16 = np.float32(_f16_val(want_o16)) + np.float32(_f16_val(want_s16)) * np.arange(M, dtype=np.float32)
    assert np.argmin(np.abs(x[:, None] - g16[None, :]), 1).tolist() == d["step5_drift_symbols"]

    # each wrong order, run through the oracle's own (separately pinned) steps
    m1, _, _ = oracle.dq_drift(x, float(s0), 0.0, t, C)
    assert m1.tolist() == d["step2_drift_symbols"]
    assert _f16_bits(float(s0)) != want_s16                                   # Refit dropped
    assert m1.tolist() != d["step5_drift_symbols"]                            # second Drift dropped
    mA, _, _ = oracle.dq_drift(x, _f16_val(_f16_bits(float(s0))), 0.0, t, C)  # fp16 before the first Drift
    sA, oA = oracle.dq_refit(x, mA, 0.0, 0.0)
    assert (_f16_bits(sA), _f16_bits(oA)) != (want_s16, want_o16)
    w = d["wrong_orders"]
    assert _f16_val(_f16_bits(float(s0))) == w["no_refit_s16"]
    assert (_f16_val(_f16_bits(sA)), _f16_val(_f16_bits(oA))) == (w["fp16_before_first_drift"]["s16"],
                                                                    w["fp16_before_first_drift"]["o16"])


def test_algorithm1_final_symbols_are_drift_on_the_fp16_refit_grid():
    """With a budget that binds (Drift moves symbols away from nearest rounding),
    the stream's s and o are the fp16 least-squares fit to the first Drift's
    symbols on the min/max grid, and its symbols are Drift on that fp16 grid
    (App. A Algorithm 1, lines FitMinMax to the second Drift)."""
    t = oracle.DqTable(64, 8)
    F = oracle.dq_pow2_table()
    rng = np.random.default_rng(21)
    C, checked, bound = 22, 0, 0
    for _ in range(20):
        x = rng.standard_normal(64).astype(np.float32)
        s0 = (np.float32(x.max()) - np.float32(x.min())) / np.float32(7)
        o0 = np.float32(x.min())
        grid = o0 + s0 * np.arange(8, dtype=np.float32)
        near = np.argmin(np.abs(x[:, None] - grid[None, :]), 1)
        m1, _, ok1 = oracle.dq_drift(x, float(s0), float(o0), t, C, F)
        bound += not np.array_equal(m1, near)
        ls, lo = _lstsq(x, m1)
        # skip a sample whose fp64 fit sits within fp32 noise of an fp16 rounding boundary
        if any(abs(float(np.float16(v)) - v) > 0.49 * abs(float(np.spacing(np.float16(v)))) for v in (ls, lo)):
            continue
        r = oracle.dq_encode_stream(x, t, C, F)
        assert r["flags"] == 0
        assert (r["s16"], r["o16"]) == (_f16_bits(ls), _f16_bits(lo))
        m2, _, _ = oracle.dq_drift(x, _f16_val(r["s16"]), _f16_val(r["o16"]), t, C, F)
        assert np.array_equal(r["m"], m2)
        checked += 1
    assert checked >= 15 and bound == 20


# ---- whole-cache assembly ----------------------------------------------------

def _hadamard(d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    return scipy_linalg.hadamard(d).astype(np.float64)


def test_dquant_key_streams_are_head_major_rows_minus_the_window_mean():
    """Stream assembly of the key cache (Sec. 4.2: one token's key over all KV
    heads forms a stream; keys are rotated and lose a windowed channel mean).
    Keys are built so that the rotated rows are known dyadic values y = z + c_w,
    with z summing to zero over each 128-token window and c_w a window constant
    exactly representable as INT8 times 2^-6.  The oracle's window means must
    then be exactly c_w and its streams exactly the head-major concatenation of
    z, which is checked by encoding those streams directly."""
    H, d, ns, nq = 2, 64, 2, 300
    S = ns + nq
    n = H * d
    rng = np.random.default_rng(31)
    Hm = _hadamard(d)
    nw = -(-nq // 128)
    kq = rng.integers(-126, 127, size=(nw, n))
    kq[:, 0] = 127                                      # max |mu| = 127 * 2^-6: the scale is exactly 2^-6
    kq[:, 1] = -127
    c = kq * 2.0 ** -6                                  # window constants [nw, n]
    z = np.zeros((nq, n))
    for w0 in range(0, nq, 128):                        # zero-sum pairs inside every window
        cnt = min(128, nq - w0)
        for t in range(w0, w0 + cnt - 1, 2):
            v = rng.integers(-64, 65, size=n) * 2.0 ** -5
            z[t], z[t + 1] = v, -v
    y = z + c[np.arange(nq) // 128]                     # rotated, stream order [nq, H*d]
    yh = y.reshape(nq, H, d).transpose(1, 0, 2)         # [H, nq, d]
    # the raw key whose normalized Hadamard rotation (H/8 at d = 64) is y, exactly
    kraw = np.zeros((1, H, S, d), dtype=np.float32)
    kraw[0, :, ns:] = (yh @ Hm) / 8.0
    kraw[0, :, :ns] = rng.standard_normal((H, ns, d)).astype(np.float32)   # sinks: outside every stream
    w = __import__("workloads").DQUANT.with_(batch=1, n_kv_heads=H, n_q_heads=4 * H, head_dim=d, seq=S,
                                             kv_dtype="f32", n_sink=ns, n_recent=0,
                                             extra={**__import__("workloads").DQUANT.extra,
                                                    "container_k": 64, "container_v": 48})
    dt = oracle.quantize_dquant(w, kraw, True, S)
    assert np.array_equal(dt.mean_q[0].astype(np.int64), kq)
    assert np.all(dt.mean_sc[0] == _f16_bits(2.0 ** -6))
    assert np.array_equal(dt.mu_hat[0].astype(np.float64), c)
    tk, _ = oracle.cache.dq_tables(w)
    cont, s16, o16, m, flags = oracle.dq_encode_streams(z.astype(np.float32), tk, 64)
    assert np.array_equal(dt.container[0], cont) and np.array_equal(dt.m[0], m)
    assert np.array_equal(dt.s16[0], s16) and np.array_equal(dt.o16[0], o16)
    assert np.array_equal(dt.flags[0], flags)
    # values: no rotation, no mean, the same head-major assembly of the raw rows
    vraw = np.zeros((1, H, S, d), dtype=np.float32)
    vraw[0, :, ns:] = yh
    dv = oracle.quantize_dquant(w, vraw, False, S)
    _, tv = oracle.cache.dq_tables(w)
    cont, s16, o16, m, _ = oracle.dq_encode_streams(y.astype(np.float32), tv, 48)
    assert dv.mean_q is None
    assert np.array_equal(dv.container[0], cont) and np.array_equal(dv.m[0], m)


def test_dquant_dequant_is_eq7_then_the_inverse_rotation():
    """Dequantization (App. A Eq. (7)): k^ = s m + o + mu per stream value, then
    the stream is split into heads and rotated back with the normalized Hadamard
    matrix from scipy (its own inverse)."""
    import workloads as W
    H, d, ns, nq = 2, 64, 1, 260
    S = ns + nq
    w = W.DQUANT.with_(batch=2, n_kv_heads=H, n_q_heads=4 * H, head_dim=d, seq=S, kv_dtype="bf16", n_sink=ns,
                       n_recent=0, extra={**W.DQUANT.extra, "container_k": 64, "container_v": 48})
    k, v = W.make_kv(w)
    Hn = _hadamard(d) / np.sqrt(d)
    for is_key, x in ((True, k), (False, v)):
        dt = oracle.quantize_dquant(w, x, is_key, S)
        s = dt.s16.view(np.float16).astype(np.float64)
        o = dt.o16.view(np.float16).astype(np.float64)
        want = np.zeros((2, H, nq, d))
        for b in range(2):
            for t in range(nq):
                vals = s[b, t] * dt.m[b, t].astype(np.float64) + o[b, t]
                if is_key:
                    vals = vals + dt.mu_hat[b, t // 128].astype(np.float64)
                for h in range(H):
                    row = vals[h * d:(h + 1) * d]
                    want[b, h, t] = Hn @ row if is_key else row
        got = oracle.dquant_dequant_f64(w, dt, is_key)
        assert np.abs(got - want).max() < 1e-12
        # and the result is close to the input it encodes (a 2-3 bit grid)
        xin = W.bits_to_f32(x, w.kv_dtype)[:, :, ns:S].astype(np.float64)
        assert np.sqrt(np.mean((got - xin) ** 2)) < 0.5
