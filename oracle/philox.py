"""Philox4x32-10 and the Box-Muller normal map, in plain numpy (oracle side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source of the generator: J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw,
"Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), the Philox-4x32
S-box/P-box round and its Weyl key schedule.  The pages this library follows
only ask for Gaussian noise N(0, sigma^2 C^2 I) added once to the clipped sum
("Privacy-Preserving Machine Learning", section "Differentially private
stochastic gradient descent", phase 4; "Differential Privacy in Fine-Tuning
(DP-SGD)", "Calibrated Gaussian Noise Addition"); the choice of generator and
of the words-to-normal map is this library's reading, stated below.

Round (one of ten), on counter (c0, c1, c2, c3) and key (k0, k1):
    hi0:lo0 = M0 * c0          (full 64-bit product of two 32-bit words)
    hi1:lo1 = M1 * c2
    (c0, c1, c2, c3) <- (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0)
and between rounds the key is bumped by the Weyl constants (W0, W1), mod 2^32.

Coordinate k of the noise vector (reading of the pages' silence):
    key     = (seed mod 2^32, seed div 2^32)
    counter = (j mod 2^32, j div 2^32, step mod 2^32, step div 2^32), j = k div 4
    words x0..x3 of block j feed two Box-Muller pairs:
        (x0, x1) -> z[4j],   z[4j+1]
        (x2, x3) -> z[4j+2], z[4j+3]
    u1 = ((xa >> 8) + 1) * 2^-24   in (0, 1]   (log u1 is always finite)
    u2 = (xb >> 8) * 2^-24          in [0, 1)
    r  = sqrt(-2 ln u1);  z_first = r cos(2 pi u2);  z_second = r sin(2 pi u2)
All of this is evaluated in float64 here.

Pins (tests/test_oracle_philox.py): raw words against cuRAND's host-side
Philox4_32_10 generator (an independent implementation, called through its
public API); closed-form special values of the uniform and Box-Muller maps;
mean / variance / Kolmogorov-Smirnov statistics against N(0, 1); the RMS norm
closed form sigma*C*sqrt(d) of "Privacy-Preserving Machine Learning", section
"The privacy-utility trade-off in modern LLMs".
"""

from __future__ import annotations

import numpy as np

# Philox-4x32 multipliers and Weyl key increments (Salmon et al., SC'11).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
PHILOX_ROUNDS = 10

_MASK32 = np.uint64(0xFFFFFFFF)


def _mulhilo(m: int, x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Full 32x32 -> 64-bit product, split into (high word, low word)."""
    prod = np.uint64(m) * x.astype(np.uint64)
    return prod >> np.uint64(32), prod & _MASK32


def philox4x32_10(counter: np.ndarray, key: tuple[int, int]) -> np.ndarray:
    """Apply the ten-round Philox-4x32 bijection.

    counter : uint32-valued array of shape [n, 4] (any integer dtype)
    key     : pair of 32-bit ints
    returns : uint32 array [n, 4]
    """
    c = np.asarray(counter, dtype=np.uint64) & _MASK32
    c0, c1, c2, c3 = c[:, 0], c[:, 1], c[:, 2], c[:, 3]
    k0 = int(key[0]) & 0xFFFFFFFF
    k1 = int(key[1]) & 0xFFFFFFFF
    for rnd in range(PHILOX_ROUNDS):
        if rnd > 0:
            k0 = (k0 + PHILOX_W0) & 0xFFFFFFFF
            k1 = (k1 + PHILOX_W1) & 0xFFFFFFFF
        hi0, lo0 = _mulhilo(PHILOX_M0, c0)
        hi1, lo1 = _mulhilo(PHILOX_M1, c2)
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1,
                          hi0 ^ c3 ^ np.uint64(k1), lo0)
    return np.stack([c0, c1, c2, c3], axis=1).astype(np.uint32)


def noise_key(seed: int) -> tuple[int, int]:
    seed = int(seed) & 0xFFFFFFFFFFFFFFFF
    return seed & 0xFFFFFFFF, seed >> 32


def noise_counters(step: int, j0: int, nblocks: int) -> np.ndarray:
    """Counters of Philox blocks j0 .. j0+nblocks-1 for one optimizer step."""
    step = int(step) & 0xFFFFFFFFFFFFFFFF
    j = np.arange(j0, j0 + nblocks, dtype=np.uint64)
    ctr = np.empty((nblocks, 4), dtype=np.uint64)
    ctr[:, 0] = j & _MASK32
    ctr[:, 1] = j >> np.uint64(32)
    ctr[:, 2] = step & 0xFFFFFFFF
    ctr[:, 3] = step >> 32
    return ctr


def raw_blocks(seed: int, step: int, j0: int, nblocks: int) -> np.ndarray:
    """Philox words of blocks j0.. for (seed, step): uint32 [nblocks, 4]."""
    return philox4x32_10(noise_counters(step, j0, nblocks), noise_key(seed))


def uniform_open0(x: np.ndarray) -> np.ndarray:
    """u1 = ((x >> 8) + 1) / 2^24, in (0, 1], float64 (exact)."""
    return ((np.asarray(x, dtype=np.uint64) >> np.uint64(8)) + np.uint64(1)).astype(np.float64) * 2.0 ** -24


def uniform_closed0(x: np.ndarray) -> np.ndarray:
    """u2 = (x >> 8) / 2^24, in [0, 1), float64 (exact)."""
    return (np.asarray(x, dtype=np.uint64) >> np.uint64(8)).astype(np.float64) * 2.0 ** -24


def box_muller(xa: np.ndarray, xb: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Two standard normals from two 32-bit words (float64)."""
    u1 = uniform_open0(xa)
    u2 = uniform_closed0(xb)
    r = np.sqrt(-2.0 * np.log(u1))
    theta = 2.0 * np.pi * u2
    return r * np.cos(theta), r * np.sin(theta)


def normals(seed: int, step: int, k0: int, n: int) -> np.ndarray:
    """z[k0 .. k0+n-1] of the noise stream of (seed, step), float64."""
    if n <= 0:
        return np.zeros(0, dtype=np.float64)
    j0 = k0 // 4
    j1 = (k0 + n - 1) // 4
    w = raw_blocks(seed, step, j0, j1 - j0 + 1)
    za, zb = box_muller(w[:, 0], w[:, 1])
    zc, zd = box_muller(w[:, 2], w[:, 3])
    z = np.stack([za, zb, zc, zd], axis=1).reshape(-1)
    off = k0 - 4 * j0
    return z[off:off + n]


def normals_at(seed: int, step: int, ks: np.ndarray) -> np.ndarray:
    """z at arbitrary coordinates ks (int array), float64."""
    ks = np.asarray(ks, dtype=np.int64)
    if ks.size == 0:
        return np.zeros(0, dtype=np.float64)
    j = (ks // 4).astype(np.uint64)
    step = int(step) & 0xFFFFFFFFFFFFFFFF
    ctr = np.empty((ks.size, 4), dtype=np.uint64)
    ctr[:, 0] = j & _MASK32
    ctr[:, 1] = j >> np.uint64(32)
    ctr[:, 2] = step & 0xFFFFFFFF
    ctr[:, 3] = step >> 32
    w = philox4x32_10(ctr, noise_key(seed))
    lane = ks % 4
    first = (lane % 2) == 0
    pair = lane // 2
    xa = np.where(pair == 0, w[:, 0], w[:, 2])
    xb = np.where(pair == 0, w[:, 1], w[:, 3])
    za, zb = box_muller(xa, xb)
    return np.where(first, za, zb)
