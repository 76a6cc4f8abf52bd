"""Pins of the oracle's Philox4x64-10 and of the ISD uniforms (CPU only)."""
import math

import numpy as np
import pytest

from oracle import philox


def _numpy_block(ctr, key):
    # numpy.random.Philox increments the 256-bit counter before each block, so
    # its first block for counter c is Philox(c + 1).
    c = list(ctr)
    # subtract one with borrow across the four words
    for i in range(4):
        if c[i] > 0:
            c[i] -= 1
            break
        c[i] = (1 << 64) - 1
    g = np.random.Philox(counter=np.array(c, dtype=np.uint64),
                         key=np.array(list(key), dtype=np.uint64))
    return [int(x) for x in g.random_raw(4)]


@pytest.mark.parametrize("seed", range(6))
def test_philox_matches_numpy(seed):
    rng = np.random.default_rng(1000 + seed)
    for _ in range(25):
        ctr = [int(x) for x in rng.integers(0, 2**64, size=4, dtype=np.uint64)]
        ctr[0] = max(ctr[0], 1)   # keep the numpy borrow in word 0
        key = [int(x) for x in rng.integers(0, 2**64, size=2, dtype=np.uint64)]
        ours = [int(w) for w in philox.philox4x64_10(tuple(ctr), tuple(key))]
        assert ours == _numpy_block(ctr, key)


def test_philox_matches_numpy_small_counters():
    for step in range(1, 4):
        for c in range(3):
            ctr = (step, c, 1, 0)
            key = (0, 0)
            ours = [int(w) for w in philox.philox4x64_10(ctr, key)]
            assert ours == _numpy_block(ctr, key)


def test_philox_vectorised_equals_scalar():
    ctrs = np.arange(1, 40, dtype=np.uint64)
    vec = philox.philox4x64_10((ctrs, np.uint64(7), np.uint64(2), np.uint64(3)), (11, 13))
    for i, c in enumerate(ctrs):
        one = philox.philox4x64_10((int(c), 7, 2, 3), (11, 13))
        assert [int(w[i]) for w in vec] == [int(w) for w in one]


def test_weyl_constants_from_their_definitions():
    # W0 = floor(2^64 / golden ratio) = floor(2^64 (sqrt(5) - 1) / 2)
    s5 = math.isqrt(5 << 128)
    assert philox.PHILOX_W0 == (s5 - (1 << 64)) // 2
    # W1 = floor(2^64 (sqrt(3) - 1))
    assert philox.PHILOX_W1 == math.isqrt(3 << 128) - (1 << 64)


def test_uniform24_exact_and_in_range():
    words = np.array([0, (1 << 40) - 1, 1 << 40, (1 << 64) - 1], dtype=np.uint64)
    u = philox.uniform24(words)
    assert u[0] == 0.0 and u[1] == 0.0
    assert u[2] == 2.0 ** -24
    assert u[3] == 1.0 - 2.0 ** -24
    assert np.all(u < 1.0)
    # exactly representable in float32
    assert np.all(u.astype(np.float32).astype(np.float64) == u)


def test_draws_uniform_chi_square():
    req = np.arange(20000)
    u = philox.accept_uniforms(seed=0, step=5, requests=req, n_drafts=7).reshape(-1)
    counts, _ = np.histogram(u, bins=64, range=(0.0, 1.0))
    expected = u.size / 64
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    # chi-square with 63 dof: the 0.999 quantile is about 103.4
    assert chi2 < 103.4


def test_draws_differ_across_purposes_and_steps():
    req = np.arange(64)
    a = philox.accept_uniforms(0, 1, req, 3)
    b = philox.accept_uniforms(0, 2, req, 3)
    s = philox.sample_uniform(0, 1, req)
    r = philox.residual_uniform(0, 1, req)
    p = philox.propose_uniforms(0, 1, req, 3)
    allv = np.concatenate([a.ravel(), b.ravel(), s, r, p.ravel()])
    assert np.unique(allv).size == allv.size


def test_draw_layout_word_and_block():
    # u for draft i uses word (i-1) % 4 of block (i-1) // 4
    u = philox.accept_uniforms(seed=3, step=9, requests=np.array([5]), n_drafts=7)[0]
    blk0 = philox.philox4x64_10((9, 5, philox.PURPOSE_ACCEPT, 0), (3, 0))
    blk1 = philox.philox4x64_10((9, 5, philox.PURPOSE_ACCEPT, 1), (3, 0))
    words = [int(w) for w in blk0] + [int(w) for w in blk1]
    assert np.array_equal(u, philox.uniform24(np.array(words[:7], dtype=np.uint64)))
