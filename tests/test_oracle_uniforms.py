"""Pins of the oracle's counter-based uniforms.

* Philox4x64-10 through numpy reproduces the published known-answer vectors
  (tests/golden/philox4x64_10_kat.txt, Random123 / SC'11).
* The counter convention: u_acc / u_smp of node n come from the block at
  counter (n + 1, b, offset, 0), words 0 and 1, top 24 bits.
"""
import os

import numpy as np
import pytest

from oracle import philox_block, uniforms_for


def _kat(golden_dir):
    rows = []
    with open(os.path.join(golden_dir, "philox4x64_10_kat.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            w = [int(x, 16) for x in line.split()]
            rows.append((w[0:4], w[4:6], w[6:10]))
    assert len(rows) == 3
    return rows


def test_numpy_philox_matches_published_kat(golden_dir):
    for ctr, key, expect in _kat(golden_dir):
        # numpy pre-increments word 0 (with carry) before each block, so seed
        # one below the wanted counter.
        c = (ctr[0] + (ctr[1] << 64) + (ctr[2] << 128) + (ctr[3] << 192) - 1) \
            % (1 << 256)
        words = [(c >> (64 * i)) & ((1 << 64) - 1) for i in range(4)]
        g = np.random.Philox(key=np.array(key, dtype=np.uint64),
                             counter=np.array(words, dtype=np.uint64))
        got = [int(x) for x in g.random_raw(4)]
        assert got == expect


def test_philox_block_counter_convention():
    # philox_block takes the counter that is actually hashed.
    w = philox_block(7, (3, 5, 11, 0))
    g = np.random.Philox(key=np.array([7, 0], dtype=np.uint64),
                         counter=np.array([2, 5, 11, 0], dtype=np.uint64))
    assert [int(x) for x in w] == [int(x) for x in g.random_raw(4)]
    with pytest.raises(ValueError):
        philox_block(7, (0, 1, 2, 0))


def test_large_seed_is_exact():
    # a seed above 2^53 must reach the generator unchanged
    seed = (1 << 63) + 12345
    w = philox_block(seed, (1, 0, 0, 0))
    g = np.random.Philox(key=np.array([seed, 0], dtype=np.uint64),
                         counter=np.zeros(4, dtype=np.uint64))
    assert [int(x) for x in w] == [int(x) for x in g.random_raw(4)]
    w2 = philox_block(seed + 1, (1, 0, 0, 0))
    assert [int(x) for x in w] != [int(x) for x in w2]


def test_uniforms_layout_and_grid():
    seed, off, b = 1234, 9, 3
    ua, us = uniforms_for(seed, off, b, 6)
    for n in range(6):
        w = philox_block(seed, (n + 1, b, off, 0))
        assert ua[n] == (int(w[0]) >> 40) / 2.0 ** 24
        assert us[n] == (int(w[1]) >> 40) / 2.0 ** 24
    assert np.all((ua >= 0) & (ua < 1)) and np.all((us >= 0) & (us < 1))
    # on the 2^-24 grid, hence exact in fp32
    assert np.all(ua * 2 ** 24 == np.floor(ua * 2 ** 24))
    assert np.all(ua.astype(np.float32).astype(np.float64) == ua)


def test_uniforms_are_uniform():
    # 4096 requests x 8 nodes: mean 1/2, variance 1/12, KS distance small
    u = np.concatenate([uniforms_for(5, 0, b, 8)[0] for b in range(4096)])
    n = u.size
    assert abs(u.mean() - 0.5) < 4 * np.sqrt(1 / 12 / n)
    s = np.sort(u)
    ks = np.max(np.abs(s - (np.arange(1, n + 1) / n)))
    assert ks < 1.95 / np.sqrt(n)   # ~0.1% level
