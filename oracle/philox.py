"""Philox4x64-10, written from its published definition, and the ISD uniforms.

Test infrastructure (see ``oracle/__init__``): not for the product path.

Philox is the counter-based generator of J. K. Salmon, M. A. Moraes,
R. O. Dror and D. E. Shaw, "Parallel random numbers: as easy as 1, 2, 3"
(SC'11).  One call maps a 256-bit counter (four 64-bit words) and a 128-bit key
(two words) to four 64-bit words by ten rounds.  Each round multiplies words 0
and 2 by fixed odd constants, keeps both halves of the 128-bit products, and
permutes / xors them with the other two words and the round key.  Between rounds
the key is bumped by two Weyl constants.

The pages are silent on the random-number source of the accept rule (they only
state the rule: [IDLM] "Inference & ISD", [GN] "Inference & ISD").  A
counter-based generator makes every draw a pure function of
(seed, step, request, purpose, index), so a CPU and a GPU implementation can be
compared draw by draw.

Pins (tests/test_oracle_philox.py): the 4x64 instantiation is checked word for
word against ``numpy.random.Philox`` (a library implementation of the same
generator); the two Weyl constants are re-derived from the golden ratio and
sqrt(3); the uniform map is checked for range and uniformity.
"""

import numpy as np

MASK64 = (1 << 64) - 1

# Round multipliers for the 4x64 variant (from the SC'11 paper's table).
PHILOX_M0 = 0xD2E7470EE14C6C93
PHILOX_M1 = 0xCA5A826395121157
# Weyl key increments: frac(golden ratio) and sqrt(3) - 1, scaled by 2**64.
PHILOX_W0 = 0x9E3779B97F4A7C15
PHILOX_W1 = 0xBB67AE8584CAA73B

ROUNDS = 10

# Purposes of a draw: the third counter word.
PURPOSE_ACCEPT = 0   # u_i compared against min(1, p/q) for draft i
PURPOSE_SAMPLE = 1   # word 0: bonus / fresh token draw; word 1: residual draw
PURPOSE_PROPOSE = 2  # SAMPLE-mode proposals, one word per MASK row

_M32 = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def _mulhilo(a, m):
    """(hi, lo) 64-bit halves of the 128-bit product a*m, a: uint64 array."""
    a = np.asarray(a, dtype=np.uint64)
    m_lo = np.uint64(m & 0xFFFFFFFF)
    m_hi = np.uint64(m >> 32)
    a_lo = a & _M32
    a_hi = a >> _S32
    ll = a_lo * m_lo
    lh = a_lo * m_hi
    hl = a_hi * m_lo
    hh = a_hi * m_hi
    mid = (ll >> _S32) + (lh & _M32) + (hl & _M32)
    hi = hh + (lh >> _S32) + (hl >> _S32) + (mid >> _S32)
    lo = (mid << _S32) | (ll & _M32)
    return hi, lo


def philox4x64_10(ctr, key):
    """Philox4x64 with ten rounds.

    ctr: four counter words, each an int or a uint64 array (broadcast together).
    key: two key words (ints or arrays).
    Returns a tuple of four uint64 arrays.
    """
    with np.errstate(over="ignore"):
        c0, c1, c2, c3 = (np.asarray(np.uint64(x) if isinstance(x, int) else x,
                                     dtype=np.uint64) for x in ctr)
        k0, k1 = (np.asarray(np.uint64(x) if isinstance(x, int) else x,
                             dtype=np.uint64) for x in key)
        c0, c1, c2, c3 = np.broadcast_arrays(c0, c1, c2, c3)
        for r in range(ROUNDS):
            if r > 0:
                k0 = k0 + np.uint64(PHILOX_W0)
                k1 = k1 + np.uint64(PHILOX_W1)
            hi0, lo0 = _mulhilo(c0, PHILOX_M0)
            hi1, lo1 = _mulhilo(c2, PHILOX_M1)
            c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
    return c0, c1, c2, c3


def uniform24(word):
    """Top 24 bits of a 64-bit word as a float in [0, 1): exact in float32."""
    w = np.asarray(word, dtype=np.uint64)
    return (w >> np.uint64(40)).astype(np.float64) * (2.0 ** -24)


def draw(seed, step, request, purpose, index):
    """Uniform number ``index`` of one purpose, for a request at a step.

    Word ``index % 4`` of Philox(ctr = (step, request, purpose, index // 4),
    key = (seed, 0)).  ``request`` and ``index`` may be arrays.
    """
    request = np.asarray(request, dtype=np.uint64)
    index = np.asarray(index, dtype=np.int64)
    block = (index // 4).astype(np.uint64)
    words = philox4x64_10((np.uint64(step), request, np.uint64(purpose), block),
                          (np.uint64(seed), np.uint64(0)))
    stacked = np.stack(np.broadcast_arrays(*words), axis=0)
    lane = np.broadcast_to(index % 4, stacked.shape[1:])
    picked = np.take_along_axis(stacked, lane[None, ...].astype(np.int64), axis=0)[0]
    return uniform24(picked)


def accept_uniforms(seed, step, requests, n_drafts):
    """u[c, i-1] for draft i = 1..n_drafts of each request: shape [C, n_drafts]."""
    req = np.asarray(requests, dtype=np.uint64)[:, None]
    idx = np.arange(n_drafts, dtype=np.int64)[None, :]
    return draw(seed, step, req, PURPOSE_ACCEPT, idx)


def sample_uniform(seed, step, requests):
    """Draw for the bonus token (all drafts accepted) or the fresh token."""
    return draw(seed, step, np.asarray(requests, dtype=np.uint64), PURPOSE_SAMPLE, 0)


def residual_uniform(seed, step, requests):
    """Draw for the resample from the residual at the first rejection."""
    return draw(seed, step, np.asarray(requests, dtype=np.uint64), PURPOSE_SAMPLE, 1)


def propose_uniforms(seed, step, requests, n_mask):
    """Draws for SAMPLE-mode proposals of MASK rows 1..n_mask: [C, n_mask]."""
    req = np.asarray(requests, dtype=np.uint64)[:, None]
    idx = np.arange(n_mask, dtype=np.int64)[None, :]
    return draw(seed, step, req, PURPOSE_PROPOSE, idx)
