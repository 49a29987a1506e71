"""CPU checks of the tolerance helpers the GPU parity tests use: the fp32
half-ulp against numpy's own spacing, and the per-element condition factor
reducing to the constant one for exponents below 64 in magnitude."""
import numpy as np

from tests import parity


def test_half_ulp32_is_half_of_numpy_spacing():
    a = np.array([1.0, 1.5, 63.99, 64.0, 100.0, 127.9, 128.0, 1e-3, -70.0, 2.0 ** -126])
    want = np.spacing(a.astype(np.float32)).astype(np.float64) / 2
    np.testing.assert_array_equal(parity.half_ulp32(np.abs(a)), np.abs(want))


def test_elementwise_kappa_reduces_to_the_constant_for_small_exponents():
    g = np.random.default_rng(1)
    x = g.normal(0, 2, (4, 50))
    lse = parity.row_lse(x, 0.0)
    assert np.all(np.abs((x - lse[:, None]) * parity.LOG2E) < 40)
    np.testing.assert_array_equal(parity.kappa_elementwise(x, lse, 0.0), parity.kappa(0.0))
    k30 = parity.kappa_elementwise(x, parity.row_lse(x, 30.0), 30.0)
    np.testing.assert_array_equal(k30, parity.kappa(30.0))


def test_elementwise_kappa_grows_with_the_exponent():
    x = np.array([[0.0, -30.0, -100.0, -140.0]])
    lse = parity.row_lse(x, 0.0)
    k = parity.kappa_elementwise(x, lse, 0.0)[0]
    # biased exponents 24 and -19: the constant covers them
    assert k[0] == parity.kappa(0.0) and k[1] == parity.kappa(0.0)
    # biased exponents -120 and -178: half an ulp (2^-18, 2^-17) times ln 2, and
    # the rounding of log2 e times the exponent
    assert k[2] >= parity.LN2 * 2.0 ** -18 + 100 * parity.LOG2E * 1.3e-8 * parity.LN2
    assert k[3] >= parity.LN2 * 2.0 ** -17 > parity.kappa(0.0)
    assert k[3] > k[2] > k[1]
