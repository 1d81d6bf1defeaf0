"""Pins of the oracle's Philox4x32-10 uniforms (oracle/philox.py).

* The generator's published known-answer vectors (tests/golden).
* The round structure (word permutation, key schedule, round count) at 64-bit
  width against an independent implementation: numpy's own Philox bit
  generator (Philox4x64-10).
* The draw layout (seed, offset, row, slot) -> (key, counter) -> u, through
  the same known-answer vectors: their words are all distinct, so a swapped
  or misplaced word changes the answer.
* The uniforms' distribution: Kolmogorov-Smirnov and chi-square on 10^6
  draws, the 2^-24 grid, no correlation between neighbouring draws or calls.
"""
import os

import numpy as np
import pytest
from scipy import stats

from oracle import philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def _kat():
    rows = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        rows.append((w[0:4], w[4:6], w[6:10]))
    assert len(rows) == 3
    return rows


@pytest.mark.parametrize("i", range(3))
def test_known_answers_plain_integers(i):
    ctr, key, want = _kat()[i]
    assert list(philox.philox_block(ctr, key)) == want


def test_known_answers_vectorised():
    kat = _kat()
    ctr = np.array([c for c, _, _ in kat], dtype=np.uint64)
    key = np.array([k for _, k, _ in kat], dtype=np.uint64)
    got = philox.philox4x32_10(ctr, key)
    np.testing.assert_array_equal(got, np.array([w for _, _, w in kat], dtype=np.uint64))


# Philox4x64-10's constants (the same paper's table for N = 4, W = 64)
M64 = (0xD2E7470EE14C6C93, 0xCA5A826395121157)
W64 = (0x9E3779B97F4A7C15, 0xBB67AE8584CAA73B)


@pytest.mark.parametrize("key,ctr0", [((3, 5), 7), ((0, 0), 0), ((2 ** 64 - 1, 12345), 2 ** 40)])
def test_round_structure_matches_numpy_philox4x64(key, ctr0):
    """numpy.random.Philox increments its 256-bit counter before each block
    and emits the block's four words; the plain-integer rounds at W = 64 must
    give the same stream."""
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                          counter=np.array([ctr0, 0, 0, 0], dtype=np.uint64))
    raw = [int(v) for v in bg.random_raw(12)]
    for blk in range(3):
        words = philox.philox_block((ctr0 + 1 + blk, 0, 0, 0), key, M64, W64, bits=64)
        assert list(words) == raw[4 * blk:4 * blk + 4]


def _layout_args(ctr, key):
    """(seed, offset, row, slot) whose draw uses counter ctr and key key."""
    return key[0] | key[1] << 32, ctr[2] | ctr[3] << 32, ctr[0], ctr[1]


@pytest.mark.parametrize("i", range(3))
def test_draw_layout_through_known_answers(i):
    ctr, key, want = _kat()[i]
    seed, offset, row, slot = _layout_args(ctr, key)
    u = (want[0] >> 8) * 2.0 ** -24
    assert philox.uniform_at(seed, offset, row, slot) == u
    c, k = philox.draw_counter_key(seed, offset, row, slot)
    assert [int(v) for v in c] == ctr
    assert [int(v) for v in k] == key
    assert (philox.philox4x32_10(c, k)[0] >> np.uint64(8)) * 2.0 ** -24 == u


def test_uniforms_array_matches_single_draws():
    seed, offset = 0x0123456789ABCDEF, 2 ** 33 + 17
    u = philox.uniforms(seed, offset, 9, 7)
    for r in range(9):
        for s in range(7):
            assert u[r, s] == philox.uniform_at(seed, offset, r, s)


def test_uniform_distribution():
    u = philox.uniforms(2024, 5, 1000, 1000).ravel()      # 10^6 draws
    assert np.all((u >= 0) & (u < 1))
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))   # the 2^-24 grid
    assert np.all(u.astype(np.float32).astype(np.float64) == u)
    assert stats.kstest(u, "uniform").pvalue > 1e-4
    counts = np.bincount((u * 256).astype(np.int64), minlength=256)
    assert stats.chisquare(counts).pvalue > 1e-4
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / u.size)


def test_neighbouring_draws_uncorrelated():
    n = 1000
    u = philox.uniforms(77, 0, n, n)
    lim = 5 / np.sqrt(u.size)
    assert abs(np.corrcoef(u[:-1].ravel(), u[1:].ravel())[0, 1]) < lim        # rows
    assert abs(np.corrcoef(u[:, :-1].ravel(), u[:, 1:].ravel())[0, 1]) < lim  # slots
    v = philox.uniforms(77, 1, n, n)                                           # next call
    assert abs(np.corrcoef(u.ravel(), v.ravel())[0, 1]) < 5 / np.sqrt(u.size)
    w = philox.uniforms(78, 0, n, n)                                           # next seed
    assert abs(np.corrcoef(u.ravel(), w.ravel())[0, 1]) < 5 / np.sqrt(u.size)


def test_row_and_slot_are_not_interchangeable():
    u = philox.uniforms(9, 3, 64, 64)
    assert not np.array_equal(u, u.T)


def test_seed_and_offset_range():
    philox.uniform_at(2 ** 64 - 1, 2 ** 64 - 1, 0, 0)
    with pytest.raises(ValueError):
        philox.uniform_at(2 ** 64, 0, 0, 0)
    with pytest.raises(ValueError):
        philox.uniforms(0, -1, 1, 1)
