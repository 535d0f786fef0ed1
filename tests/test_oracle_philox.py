"""Pins for the oracle's counter-based noise (CPU only).

- the round structure, key schedule and output order: the W = 64 instantiation of
  the same code equals numpy's Philox4x64-10 bit generator (a library routine)
  for several keys and counters; the W = 32 instantiation used for the noise
  differs only in its multipliers and Weyl constants;
- the Weyl constants: against the golden ratio and sqrt(3) to 60 digits
  (decimal arithmetic, an independent method);
- Box-Muller: closed-form special cases (radius 1 at u = e^-1/2; angles 0,
  1/4, 1/2 of a turn) and the moments of a large sample;
- the chunk layout: element i comes from block i // 4, word i % 4 (brute force on
  a ragged 3 x 5 chunk).
"""
from decimal import Decimal, getcontext

import numpy as np
import pytest

from oracle import philox as X


def test_weyl_constants_closed_form():
    getcontext().prec = 60
    phi_m1 = (Decimal(5).sqrt() - 1) / 2
    r3_m1 = Decimal(3).sqrt() - 1
    for w in (32, 64):
        g, r = X.weyl_constants(w)
        assert g == int(phi_m1 * (1 << w))
        assert r == int(r3_m1 * (1 << w))


@pytest.mark.parametrize("key,ctr", [((0, 0), (0, 0, 0, 0)), ((1, 2), (3, 4, 5, 6)),
                                     ((0xDEADBEEF12345678, 0x0123456789ABCDEF), (2 ** 64 - 3, 7, 0, 2 ** 63))])
def test_philox4x64_equals_numpy(key, ctr):
    """numpy's Philox4x64-10 advances its 256-bit counter before each block."""
    g = np.random.Philox(key=np.array(key, dtype=np.uint64), counter=np.array(ctr, dtype=np.uint64))
    got = [int(v) for v in g.random_raw(8)]
    c = list(ctr)
    want = []
    for _ in range(2):
        # 256-bit increment, word 0 least significant
        for i in range(4):
            c[i] = (c[i] + 1) & (2 ** 64 - 1)
            if c[i]:
                break
        want += list(X.philox(tuple(c), key, w=64))
    assert got == want


def test_philox4x32_is_a_bijection_sample():
    """Distinct counters under one key give distinct blocks (Philox is a bijection)."""
    seen = {X.philox((b, 0, 5, 9), (11, 13)) for b in range(2000)}
    assert len(seen) == 2000


def test_box_muller_closed_forms():
    # u_a = e^(-1/2) gives radius sqrt(-2 ln u_a) = 1
    wa = np.array([round(np.exp(-0.5) * 2.0 ** 32 - 0.5)] * 3, dtype=np.uint32)
    wb = np.array([0, 2 ** 30, 2 ** 31], dtype=np.uint32)   # angle 0, a quarter, a half turn
    z0, z1 = X.box_muller(wa, wb)
    np.testing.assert_allclose(z0, [1.0, 0.0, -1.0], atol=1e-8)
    np.testing.assert_allclose(z1, [0.0, 1.0, 0.0], atol=1e-8)


def test_noise_moments():
    z = np.concatenate([X.decision_noise(7, c, 50, 32).ravel() for c in range(20)])   # 32,000 samples
    n = z.size
    assert abs(z.mean()) < 4.0 / np.sqrt(n)
    assert abs(z.var() - 1.0) < 4.0 * np.sqrt(2.0 / n)
    assert abs(np.mean(z ** 4) - 3.0) < 0.15   # Gaussian kurtosis


def test_noise_layout_brute_force():
    seed, counter = 0x1234_5678_9ABC_DEF0, 0xFEDC_BA98_7654_3210
    z = X.decision_noise(seed, counter, 3, 5)
    k = (seed & 0xFFFFFFFF, seed >> 32)
    for i in range(15):
        b, j = divmod(i, 4)
        w = X.philox((b, 0, counter & 0xFFFFFFFF, counter >> 32), k)
        ua = (w[j & 2] + 0.5) / 2.0 ** 32
        ub = (w[(j & 2) + 1] + 0.5) / 2.0 ** 32
        r = np.sqrt(-2.0 * np.log(ua))
        want = r * (np.cos(2 * np.pi * ub) if j % 2 == 0 else np.sin(2 * np.pi * ub))
        assert z.ravel()[i] == want


def test_streams_differ():
    a = X.decision_noise(1, 0, 4, 8)
    assert np.array_equal(a, X.decision_noise(1, 0, 4, 8))
    assert not np.allclose(a, X.decision_noise(1, 1, 4, 8))
    assert not np.allclose(a, X.decision_noise(2, 0, 4, 8))
