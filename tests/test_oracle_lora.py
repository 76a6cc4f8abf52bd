"""Pins of the oracle's gated LoRA (CPU only)."""
import numpy as np

from oracle.isd import gated_lora


def _case(seed=0, M=21, K=48, N=40, r=8):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((M, K)), rng.standard_normal((N, K)) * 0.1,
            rng.standard_normal((r, K)) * 0.1, rng.standard_normal((N, r)) * 0.1,
            (np.arange(M) % 7 >= 4).astype(np.uint8))


def test_ungated_rows_equal_the_base_projection_bitwise():
    x, w, a, b, g = _case()
    y = gated_lora(x, w, a, b, g, 1.0)
    base = x @ w.T
    assert np.array_equal(y[g == 0], base[g == 0])


def test_gated_rows_equal_the_merged_weight():
    x, w, a, b, g = _case(seed=1)
    s = 0.5
    y = gated_lora(x, w, a, b, g, s)
    merged = x @ (w + s * b @ a).T        # other association order
    np.testing.assert_allclose(y[g == 1], merged[g == 1], rtol=1e-12, atol=1e-12)
    assert not np.allclose(y[g == 1], (x @ w.T)[g == 1])
