"""Pins for the oracle's standalone skinny GEMM + fused consumer (CPU only).

oracle.model.gemm_consumer restates the consumer of a K-split GEMM (blog post
"Embodied inference acceleration: first ask how old the observation is", section
"Static quantisation changes the work between two GEMMs": the GEMM's dequantised
product plus bias feeds a gated residual, x <- x + gate * y, whose result is
normalised by AdaRMSNorm and quantised with a static scale for the next GEMM;
section "Small-M GEMM": the product is the sum of the K slices' partials).

Each check pins it to something other than its own formula:
  * gate = 0 leaves x bit-identical, and a constant row then quantises to a
    value known in closed form (c / sqrt(c^2 + eps) * (1 + scale) + shift lands
    on a point of the E4M3 grid);
  * A = 0 makes the product vanish, so y equals the bias exactly;
  * integer A, W and bias with unit scales give y exactly, checked against a
    brute-force scalar loop;
  * x = 0 and A = 0 with a constant bias: the residual output is a constant row,
    so q is the closed form above (the norm is taken after the residual);
  * a planted mistake (gate applied before the bias, bias dropped, gate ignored,
    scale used without the 1 +, the norm taken of the pre-residual x) fails at
    least one of the checks above.
"""
import math

import numpy as np

from oracle import codecs as C
from oracle import model as O


def _weight(codes, scale=1.0):
    return O.PreparedWeight(np.asarray(codes, np.float64), scale, "fp8")


def _check_gate_zero(fn):
    """gate = 0: x_out == x bit for bit; constant rows c quantise to the closed form."""
    M, K, N, eps = 3, 16, 32, 1e-6
    rng = np.random.default_rng(11)
    a = C.e4m3(rng.standard_normal((M, K)))
    w = _weight(C.e4m3(rng.standard_normal((N, K))))
    x = np.full((M, N), 3.0)
    x[1] = -3.0
    bias = rng.standard_normal(N)
    gate = np.zeros(N)
    scale, shift = np.full(N, 1.0), np.full(N, 0.5)
    _, x_out, q = fn(a, 1.0, w, bias, x, gate, scale, shift, 1.0, eps)
    if not np.array_equal(x_out, x):
        return "gate = 0 changed x"
    # x_hat = +-3 / sqrt(9 + eps) = +-(1 - 5.6e-8); h = x_hat * 2 + 0.5 -> 2.5 or -1.5,
    # both on the E4M3 grid and far (> 1e-7) from any rounding boundary
    xh = 3.0 / math.sqrt(9.0 + eps)
    want = np.empty((M, N))
    want[:] = C.e4m3(np.array([xh * 2.0 + 0.5]))[0]
    want[1] = C.e4m3(np.array([-xh * 2.0 + 0.5]))[0]
    if not (want[0, 0] == 2.5 and want[1, 0] == -1.5):
        return "closed-form grid points moved"
    if not np.array_equal(q, want):
        return "q of constant rows differs from the closed form"
    return None


def _check_zero_activation(fn):
    """A = 0: y == bias exactly and x_out == x + gate * bias."""
    M, K, N = 4, 32, 16
    rng = np.random.default_rng(12)
    w = _weight(C.e4m3(rng.standard_normal((N, K))), 0.37)
    bias = rng.standard_normal(N)
    x = rng.standard_normal((M, N))
    gate = rng.standard_normal(N)
    y, x_out, _ = fn(np.zeros((M, K)), 0.5, w, bias, x, gate, np.zeros(N), np.zeros(N), 1.0, 1e-6)
    if not np.array_equal(y, np.broadcast_to(bias, (M, N))):
        return "A = 0 does not give y = bias"
    if not np.array_equal(x_out, x + gate * bias):
        return "A = 0 does not give x + gate * bias"
    return None


def _check_integer_exact(fn):
    """Integer A, W, bias with unit scales: y exact, against a scalar loop."""
    M, K, N = 3, 24, 8
    rng = np.random.default_rng(13)
    a = rng.integers(-3, 4, (M, K)).astype(np.float64)
    wc = rng.integers(-3, 4, (N, K)).astype(np.float64)
    bias = rng.integers(-5, 6, N).astype(np.float64)
    x = rng.integers(-4, 5, (M, N)).astype(np.float64)
    gate = rng.integers(-2, 3, N).astype(np.float64)
    y, x_out, _ = fn(a, 1.0, _weight(wc), bias, x, gate, np.zeros(N), np.zeros(N), 1.0, 1e-6)
    want_y = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += a[m, k] * wc[n, k]
            want_y[m, n] = acc + bias[n]
    if not np.array_equal(y, want_y):
        return "integer product + bias is not exact"
    want_x = np.array([[x[m, n] + gate[n] * want_y[m, n] for n in range(N)] for m in range(M)])
    if not np.array_equal(x_out, want_x):
        return "integer gated residual is not exact"
    return None


def _check_norm_after_residual(fn):
    """x = 0, A = 0, bias = 3, gate = 1: the residual makes every row the constant 3,
    whose normalised, modulated value 2.5 (closed form above) is what q must hold."""
    M, K, N, eps = 2, 16, 32, 1e-6
    w = _weight(np.ones((N, K)))
    _, x_out, q = fn(np.zeros((M, K)), 1.0, w, np.full(N, 3.0), np.zeros((M, N)), np.ones(N),
                     np.full(N, 1.0), np.full(N, 0.5), 1.0, eps)
    if not np.array_equal(x_out, np.full((M, N), 3.0)):
        return "x + gate * bias is not the constant row"
    if not np.array_equal(q, np.full((M, N), 2.5)):
        return "q is not the normalised residual output"
    return None


CHECKS = (_check_gate_zero, _check_zero_activation, _check_integer_exact, _check_norm_after_residual)


def failures(fn):
    return [msg for msg in (chk(fn) for chk in CHECKS) if msg]


def test_oracle_gemm_consumer_passes_its_pins():
    assert failures(O.gemm_consumer) == []


# ---------------------------------------------------------------- planted mistakes

def _gate_before_bias(a, s_a, w, bias, x, gate, scale, shift, s_q, eps, act_fmt="fp8"):
    y = O.gemm(a, s_a, w)
    x_out = np.asarray(x, np.float64) + np.asarray(gate) * y + np.asarray(bias)
    return y + bias, x_out, O.quant_codes(O.ada_norm(x_out, scale, shift, eps), s_q, act_fmt)


def _bias_dropped(a, s_a, w, bias, x, gate, scale, shift, s_q, eps, act_fmt="fp8"):
    y = O.gemm(a, s_a, w)
    x_out = np.asarray(x, np.float64) + np.asarray(gate) * y
    return y, x_out, O.quant_codes(O.ada_norm(x_out, scale, shift, eps), s_q, act_fmt)


def _gate_ignored(a, s_a, w, bias, x, gate, scale, shift, s_q, eps, act_fmt="fp8"):
    y = O.gemm(a, s_a, w) + np.asarray(bias)
    x_out = np.asarray(x, np.float64) + y
    return y, x_out, O.quant_codes(O.ada_norm(x_out, scale, shift, eps), s_q, act_fmt)


def _scale_without_one(a, s_a, w, bias, x, gate, scale, shift, s_q, eps, act_fmt="fp8"):
    y = O.gemm(a, s_a, w) + np.asarray(bias)
    x_out = np.asarray(x, np.float64) + np.asarray(gate) * y
    h = O.rms_norm(x_out, eps) * np.asarray(scale) + np.asarray(shift)
    return y, x_out, O.quant_codes(h, s_q, act_fmt)


def _norm_of_input(a, s_a, w, bias, x, gate, scale, shift, s_q, eps, act_fmt="fp8"):
    y = O.gemm(a, s_a, w) + np.asarray(bias)
    x_out = np.asarray(x, np.float64) + np.asarray(gate) * y
    return y, x_out, O.quant_codes(O.ada_norm(x, scale, shift, eps), s_q, act_fmt)


def test_planted_mistakes_fail_a_pin():
    for bad in (_gate_before_bias, _bias_dropped, _gate_ignored, _scale_without_one, _norm_of_input):
        assert failures(bad), f"{bad.__name__} passed every pin"
