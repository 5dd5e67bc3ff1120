"""Pins for the oracle's Philox4x32-10 stream and Box-Muller normals (CPU only).

The raw words are pinned to cuRAND's host-side Philox4_32_10 generator, an
implementation independent of the oracle, called through its public API: its
output block b (for a generation of at least 2^16 blocks) is the Philox block
with counter (b div 2^16, 0, b mod 2^16, 0) and key = the 64-bit seed; a
generator offset reaches the second counter word.  The normal map is pinned
by closed-form special values and by its distribution.
"""

import ctypes
import ctypes.util
import json
import math
import os

import numpy as np
import pytest
from scipy import stats

from oracle import philox


def _curand():
    candidates = ["/usr/local/cuda/lib64/libcurand.so", ctypes.util.find_library("curand")]
    for path in candidates:
        if not path:
            continue
        try:
            return ctypes.CDLL(path)
        except OSError:
            continue
    pytest.skip("libcurand not available")


def _curand_words(lib, seed, nwords, offset=0):
    gen = ctypes.c_void_p()
    assert lib.curandCreateGeneratorHost(ctypes.byref(gen), 161) == 0  # PHILOX4_32_10
    try:
        assert lib.curandSetPseudoRandomGeneratorSeed(gen, ctypes.c_ulonglong(seed)) == 0
        if offset:
            assert lib.curandSetGeneratorOffset(gen, ctypes.c_ulonglong(offset)) == 0
        out = np.zeros(nwords, dtype=np.uint32)
        assert lib.curandGenerate(gen, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(nwords)) == 0
    finally:
        lib.curandDestroyGenerator(gen)
    return out.reshape(-1, 4)


@pytest.mark.parametrize("seed", [0, 1, 0x0123456789ABCDEF, 0xFFFFFFFFFFFFFFFF])
def test_raw_words_match_curand_host(seed):
    lib = _curand()
    nthreads = 1 << 16
    nblocks = 3 * nthreads
    ref = _curand_words(lib, seed, 4 * nblocks)
    b = np.arange(nblocks, dtype=np.uint64)
    ctr = np.zeros((nblocks, 4), dtype=np.uint64)
    ctr[:, 0] = b // nthreads
    ctr[:, 2] = b % nthreads
    ours = philox.philox4x32_10(ctr, philox.noise_key(seed))
    assert np.array_equal(ours, ref)


def test_raw_words_high_counter_word_match_curand():
    lib = _curand()
    seed = 0x0123456789ABCDEF
    j, s = 2 ** 32 + 3, 5
    ref = _curand_words(lib, seed, 8, offset=4 * (j * 65536 + s))
    # oracle's own (seed, step, block) addressing: step -> counter word 2
    assert np.array_equal(philox.raw_blocks(seed, s, j, 1)[0], ref[0])
    assert np.array_equal(philox.raw_blocks(seed, s + 1, j, 1)[0], ref[1])


def test_step_high_word_and_key_change_stream():
    a = philox.raw_blocks(7, 3, 0, 8)
    assert not np.array_equal(a, philox.raw_blocks(7, 3 + (1 << 32), 0, 8))
    assert not np.array_equal(a, philox.raw_blocks(7 + (1 << 32), 3, 0, 8))
    assert not np.array_equal(a, philox.raw_blocks(7, 4, 0, 8))


def test_uniform_maps_closed_form():
    x = np.array([0, 0xFF, 0x100, 0x80000000, 0xFFFFFFFF], dtype=np.uint32)
    u1 = philox.uniform_open0(x)
    u2 = philox.uniform_closed0(x)
    assert u1.tolist() == [2.0 ** -24, 2.0 ** -24, 2 * 2.0 ** -24, 0.5 + 2.0 ** -24, 1.0]
    assert u2.tolist() == [0.0, 0.0, 2.0 ** -24, 0.5, 1.0 - 2.0 ** -24]
    # both are exact in float32
    assert np.array_equal(u1.astype(np.float32).astype(np.float64), u1)
    assert np.array_equal(u2.astype(np.float32).astype(np.float64), u2)


def test_box_muller_special_values():
    rmax = math.sqrt(48.0 * math.log(2.0))      # u1 = 2^-24
    za, zb = philox.box_muller(np.array([0], np.uint32), np.array([0], np.uint32))
    assert za[0] == pytest.approx(rmax, abs=1e-15) and zb[0] == 0.0
    za, zb = philox.box_muller(np.array([0xFFFFFFFF], np.uint32), np.array([0x12345678], np.uint32))
    assert za[0] == 0.0 and zb[0] == 0.0          # u1 = 1 -> r = 0
    za, zb = philox.box_muller(np.array([0], np.uint32), np.array([0x40000000], np.uint32))
    assert abs(za[0]) < 1e-15 and zb[0] == pytest.approx(rmax, abs=1e-15)   # theta = pi/2
    za, zb = philox.box_muller(np.array([0], np.uint32), np.array([0x80000000], np.uint32))
    assert za[0] == pytest.approx(-rmax, abs=1e-15) and abs(zb[0]) < 1e-14  # theta = pi
    # u1 = e^-1/2 gives r = 1 up to the 2^-24 quantisation of u1
    x = np.uint32(int(round(math.exp(-0.5) * 2 ** 24 - 1)) << 8)
    za, _ = philox.box_muller(np.array([x]), np.array([0], np.uint32))
    assert za[0] == pytest.approx(1.0, abs=1e-6)


def test_pairing_of_words_into_coordinates():
    w = philox.raw_blocks(11, 2, 5, 1)[0]
    z = philox.normals(11, 2, 20, 4)
    za, zb = philox.box_muller(w[0:1], w[1:2])
    zc, zd = philox.box_muller(w[2:3], w[3:4])
    assert z.tolist() == [za[0], zb[0], zc[0], zd[0]]
    ks = np.array([21, 20, 23, 22, 1 << 40], dtype=np.int64)
    zat = philox.normals_at(11, 2, ks)
    assert zat[:4].tolist() == [zb[0], za[0], zd[0], zc[0]]
    assert zat[4] == philox.normals(11, 2, 1 << 40, 1)[0]
    # unaligned slices agree with the aligned stream
    full = philox.normals(3, 1, 0, 64)
    assert np.array_equal(philox.normals(3, 1, 7, 30), full[7:37])


def test_normal_distribution():
    n = 1 << 21
    z = philox.normals(0, 0, 0, n)
    assert abs(z.mean()) < 5.0 / math.sqrt(n)
    assert abs(z.var() - 1.0) < 5.0 * math.sqrt(2.0 / n)
    assert stats.kstest(z, "norm").pvalue > 1e-4
    tail = np.mean(np.abs(z) > 3.0)
    assert abs(tail - 2 * stats.norm.sf(3.0)) < 6 * math.sqrt(2 * stats.norm.sf(3.0) / n)
    # first and second member of a pair are uncorrelated
    zz = z.reshape(-1, 2)
    assert abs(np.corrcoef(zz[:, 0], zz[:, 1])[0, 1]) < 5.0 / math.sqrt(n / 2)


def test_noise_rms_closed_form(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "noise_rms.json")))
    for case in g["cases"]:
        rms = g["sigma_c"] * math.sqrt(case["d"])
        assert round(rms, 2) == case["printed_sum_rms"]
        assert round(g["learning_rate"] * rms / g["normalizer"], 2) == case["printed_step_rms"]
    # empirical: ||sigma C z|| over P coordinates is sigma C sqrt(P) within a few 1/sqrt(2P)
    P, sc = 1_000_000, 0.8 * 0.5
    z = philox.normals(5, 9, 0, P)
    ratio = np.linalg.norm(sc * z) / (sc * math.sqrt(P))
    assert abs(ratio - 1.0) < 5.0 / math.sqrt(2 * P)
