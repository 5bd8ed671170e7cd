"""Pins of the oracle's QuEST grid ("WUSH-KV: KV Cache Quantization with
Data-Adaptive Transforms", evaluation: the QuEST integer quantizer, per token,
symmetric, clipped from the group RMS; the near-optimality result assumes
Gaussian tails).

The reading: 2^b levels symmetric about zero with step s = 2 alpha_b RMS / 2^b,
alpha_b the clip that minimizes the mean squared error of that grid on a
standard normal.  These tests tie the oracle's alpha_b, its error model and
its per-token arithmetic to things the mathematics fixes: the closed form at
one bit, an independent numerical minimization with scipy's integrator, the
classical optimal uniform-quantizer steps for a Gaussian, a Monte-Carlo error,
exact hand-worked tokens, and the RMS within fp32 rounding.
"""
import math

import numpy as np
import pytest

import oracle


def test_one_bit_clip_is_twice_the_mean_absolute_value():
    # two levels at +-alpha/2: the best level is E|X| = sqrt(2/pi), and the
    # error is 1 - 2/pi
    a = oracle.quest_alpha(1, exact=True)
    assert abs(a - 2.0 * math.sqrt(2.0 / math.pi)) < 1e-7
    assert abs(oracle.quest_mse(a, 2) - (1.0 - 2.0 / math.pi)) < 1e-12


def test_error_model_and_clip_against_scipy_integration():
    integrate = pytest.importorskip("scipy.integrate")
    optimize = pytest.importorskip("scipy.optimize")
    stats = pytest.importorskip("scipy.stats")

    def mse(alpha, L):  # the grid's error by numerical integration, cell by cell
        D = 2 * alpha / L
        tot = 0.0
        for k in range(L):
            a = -np.inf if k == 0 else -alpha + k * D
            b = np.inf if k == L - 1 else -alpha + (k + 1) * D
            c = -alpha + (k + 0.5) * D
            tot += integrate.quad(lambda x: (x - c) ** 2 * stats.norm.pdf(x), a, b, epsabs=1e-13, epsrel=1e-12)[0]
        return tot

    for bits in (2, 3, 4):
        L = 1 << bits
        for alpha in (1.0, 2.0, 3.0):
            assert abs(oracle.quest_mse(alpha, L) - mse(alpha, L)) < 1e-9, (bits, alpha)
        best = optimize.minimize_scalar(lambda a: mse(a, L), bounds=(0.5, 5.0), method="bounded",
                                        options={"xatol": 1e-9}).x
        assert abs(oracle.quest_alpha(bits, exact=True) - best) < 2e-5, (bits, best)


@pytest.mark.parametrize("bits,step,err", [(2, 0.9957, 0.1188), (3, 0.5860, 0.03744), (4, 0.3352, 0.01154)])
def test_clip_matches_the_optimal_uniform_gaussian_quantizer(bits, step, err):
    # the classical optimal uniform quantizer for N(0,1) with 4, 8, 16 levels
    # (step and mean squared error, four significant figures): alpha = step * L / 2
    L = 1 << bits
    a = oracle.quest_alpha(bits, exact=True)
    assert abs(2 * a / L - step) < 6e-5
    assert abs(oracle.quest_mse(a, L) - err) < 6e-5 * max(1.0, err / 1e-2)
    # a minimum: nudging the clip either way costs error
    assert oracle.quest_mse(a * 1.01, L) > oracle.quest_mse(a, L) < oracle.quest_mse(a * 0.99, L)
    # the stored constant: alpha rounded to 4 decimals, c_b = fp32(2 alpha / L)
    assert oracle.quest_alpha(bits) == round(a, 4)
    assert oracle.quest_step_factor(bits) == np.float32(2 * round(a, 4) / L)


def test_rms_is_the_root_mean_square_within_fp32_rounding():
    rng = np.random.default_rng(7)
    for d in (64, 128):
        for _ in range(50):
            x = (rng.standard_normal(d) * rng.uniform(0.01, 100)).astype(np.float32)
            exact = math.sqrt(float(np.mean(x.astype(np.float64) ** 2)))
            assert abs(oracle.quest_rms(x) - exact) <= 2e-6 * exact
    assert oracle.quest_rms(np.zeros(128, np.float32)) == 0.0
    assert oracle.quest_rms(np.full(128, -3.0, np.float32)) == 3.0


def test_hand_worked_token_two_bits():
    # x = +-1 alternating: RMS = 1 exactly, so s = fp16(c_2) with c_2 = fp32(0.9957)
    # = 2039 * 2^-11 after fp16 rounding; o = fp16(-1.5 s) = -1529 * 2^-10;
    # x = +1 sits 2.504 steps above o -> code 3; x = -1 0.495 steps -> code 0
    x = np.array([1.0, -1.0] * 64, dtype=np.float32)
    codes, s, o = oracle.affine_quantize(x, 2, True, quest=True)
    assert s == np.float32(2039 * 2.0 ** -11)
    assert o == np.float32(-1529 * 2.0 ** -10)
    assert list(codes[:4]) == [3, 0, 3, 0] and set(codes.tolist()) == {0, 3}
    # without fp16 rounding o is exactly -1.5 s
    codes, s, o = oracle.affine_quantize(x, 2, False, quest=True)
    assert s == np.float32(0.9957) and o == np.float32(-1.5) * s
    # values past the clip fall to the outer codes; a zero token stores s = 0
    y = np.zeros(128, np.float32)
    y[0], y[1] = 1000.0, -1000.0
    codes, s, o = oracle.affine_quantize(y, 3, True, quest=True)
    assert codes[0] == 7 and codes[1] == 0 and codes[2] in (3, 4)
    codes, s, o = oracle.affine_quantize(np.zeros(128, np.float32), 4, True, quest=True)
    assert s == 0.0 and not codes.any()


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_monte_carlo_error_matches_the_model(bits):
    # Gaussian tokens through the grid (fp32 s and o): the per-element squared
    # error over sigma^2 approaches the model's error at alpha_b (the per-token
    # RMS estimate moves the clip by a few percent, a second-order effect at
    # the optimum)
    rng = np.random.default_rng(11 + bits)
    L = 1 << bits
    errs = []
    for t in range(400):
        sigma = rng.uniform(0.1, 10.0)
        x = (rng.standard_normal(128) * sigma).astype(np.float32)
        codes, s, o = oracle.affine_quantize(x, bits, False, quest=True)
        xh = oracle.affine_dequant(codes, s, o)
        errs.append(np.mean((xh.astype(np.float64) - x) ** 2) / sigma ** 2)
    model = oracle.quest_mse(oracle.quest_alpha(bits), L)
    assert abs(np.mean(errs) / model - 1.0) < 0.06, (np.mean(errs), model)
