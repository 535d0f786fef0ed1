"""Counter-based Gaussian noise for a decision (test infrastructure only: used by
tests/ and bench.py's CPU baseline, never by the product path).

Philox4xW-R (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
1, 2, 3", SC'11, section 3.2 "Philox"), written from the paper's definition:

* state: four W-bit words (x0, x1, x2, x3), key: two W-bit words (k0, k1);
* one round: (hi0, lo0) = M0 * x0 and (hi1, lo1) = M1 * x2 as 2W-bit products,
  then x <- (hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0);
* the key is bumped by the Weyl constants between rounds:
  (k0, k1) <- (k0 + W0, k1 + W1) mod 2^W;
* W0 and W1 are the fractional parts of the golden ratio and of sqrt(3), scaled
  by 2^W and truncated; M0, M1 are the paper's multipliers (table 2 of the
  paper: Philox4x32 0xD2511F53, 0xCD9E8D57; Philox4x64 0xD2E7470EE14C6C93,
  0xCA5A826395121157).

The decision's noise (the device generator implements the same mapping):
element i of the row-major [M][A] chunk comes from Philox4x32-10 block b = i // 4
with counter (b, 0, counter_lo, counter_hi) and key (seed_lo, seed_hi); words
(w0, w1) give elements 4b, 4b+1 and (w2, w3) give 4b+2, 4b+3 by Box-Muller
(Box and Muller, "A note on the generation of random normal deviates", 1958):
u = (w + 1/2) / 2^32, z_even = sqrt(-2 ln u_a) cos(2 pi u_b),
z_odd = sqrt(-2 ln u_a) sin(2 pi u_b).
"""
from __future__ import annotations

import math

import numpy as np

MULTIPLIERS = {32: (0xD2511F53, 0xCD9E8D57), 64: (0xD2E7470EE14C6C93, 0xCA5A826395121157)}


def weyl_constants(w: int) -> tuple[int, int]:
    """floor(2^w * (phi - 1)) and floor(2^w * (sqrt(3) - 1)) with exact integer roots."""
    one = 1 << w
    golden = (math.isqrt(5 << (2 * w)) - one) // 2   # (sqrt(5) - 1) / 2 = phi - 1
    root3 = math.isqrt(3 << (2 * w)) - one
    return golden, root3


def philox(ctr: tuple[int, int, int, int], key: tuple[int, int], w: int = 32, rounds: int = 10) -> tuple[int, ...]:
    """One Philox4xW block: four W-bit output words for a counter and a key."""
    mask = (1 << w) - 1
    m0, m1 = MULTIPLIERS[w]
    w0, w1 = weyl_constants(w)
    x0, x1, x2, x3 = (c & mask for c in ctr)
    k0, k1 = (k & mask for k in key)
    for r in range(rounds):
        if r:
            k0, k1 = (k0 + w0) & mask, (k1 + w1) & mask
        p0, p1 = m0 * x0, m1 * x2
        x0, x1, x2, x3 = ((p1 >> w) ^ x1 ^ k0), p1 & mask, ((p0 >> w) ^ x3 ^ k1), p0 & mask
    return x0, x1, x2, x3


def split64(v: int) -> tuple[int, int]:
    v &= (1 << 64) - 1
    return v & 0xFFFFFFFF, v >> 32


def raw_blocks(seed: int, counter: int, nblocks: int) -> np.ndarray:
    """[nblocks][4] uint32 words of the decision stream (seed, counter)."""
    k = split64(seed)
    c_lo, c_hi = split64(counter)
    out = np.empty((nblocks, 4), dtype=np.uint32)
    for b in range(nblocks):
        out[b] = philox((b, 0, c_lo, c_hi), k)
    return out


def box_muller(wa: np.ndarray, wb: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Two standard normals per pair of 32-bit words, in float64."""
    ua = (wa.astype(np.float64) + 0.5) / 2.0 ** 32
    ub = (wb.astype(np.float64) + 0.5) / 2.0 ** 32
    r = np.sqrt(-2.0 * np.log(ua))
    return r * np.cos(2.0 * np.pi * ub), r * np.sin(2.0 * np.pi * ub)


def decision_noise(seed: int, counter: int, M: int, A: int) -> np.ndarray:
    """The [M][A] float64 noise chunk of decision stream (seed, counter)."""
    n = M * A
    words = raw_blocks(seed, counter, (n + 3) // 4)
    z0, z1 = box_muller(words[:, 0], words[:, 1])
    z2, z3 = box_muller(words[:, 2], words[:, 3])
    z = np.stack([z0, z1, z2, z3], axis=1).reshape(-1)
    return z[:n].reshape(M, A)
