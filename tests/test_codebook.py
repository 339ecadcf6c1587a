"""The library's Lloyd-Max codebook (host code of libtq.so, no device needed) against the
oracle's, two unrelated constructions of the same tables.

The library solves for the thresholds of the positive half line by damped Newton steps
from the companding start, with closed-form cell means; the oracle alternates Lloyd
steps from an even grid over [-3, 3] and then takes Newton steps on the centroids of the
whole line, with Simpson-rule cell integrals ("How I built VeloxQuant-MLX", Stage 2, both).
Agreement of the fp32 centroids (and so of the fp64 midpoints the encoder compares with)
is then evidence about both.  The codebook is also checked on its own here: the
fixed-point conditions by adaptive quadrature, and Max's classical values."""
import math

import numpy as np
import pytest
from scipy import integrate
from scipy.stats import norm as gauss

import oracle


@pytest.fixture(scope="module")
def tq():
    import quantized_kv_cache_10_gb300 as m
    return m


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
def test_library_codebook_equals_oracle(tq, bits):
    lib = tq.tq_codebook_gaussian(bits)
    _, c32, mid = oracle.lloyd_max(bits)[:3]
    np.testing.assert_array_equal(lib["centroids"], c32)
    np.testing.assert_array_equal(lib["midpoints"], mid)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_library_codebook_fixed_point(tq, bits):
    """Each fp32 centroid is the RN of its cell's conditional mean, the cells bounded by
    the midpoints: checked by adaptive quadrature up to the fp32 rounding."""
    c = tq.tq_codebook_gaussian(bits)["centroids"].astype(np.float64)
    n = 1 << bits
    assert np.all(np.diff(c) > 0)
    np.testing.assert_array_equal(c, -c[::-1])
    bnd = np.concatenate([[-np.inf], (c[:-1] + c[1:]) / 2, [np.inf]])
    for i in range(n):
        a, b = bnd[i], bnd[i + 1]
        m0 = integrate.quad(gauss.pdf, a, b, epsabs=1e-16, epsrel=1e-13)[0]
        m1 = integrate.quad(lambda x: x * gauss.pdf(x), a, b, epsabs=1e-16, epsrel=1e-13)[0]
        # the fp32 rounding of c moves the bounds by ~2^-24 |c|, the mean by less
        assert abs(c[i] - m1 / m0) <= 2.0 ** -22 * max(1.0, abs(c[i])), (bits, i, c[i], m1 / m0)


def test_library_codebook_classical_values(tq):
    # Max (1960): positive levels of the N(0,1) quantiser with 2 and 4 levels, and sqrt(2/pi) at 1 bit
    assert abs(float(tq.tq_codebook_gaussian(1)["centroids"][1]) - math.sqrt(2 / math.pi)) < 1e-7
    c2 = tq.tq_codebook_gaussian(2)["centroids"]
    assert abs(c2[2] - 0.4528) < 1e-4 and abs(c2[3] - 1.510) < 1e-3


def test_library_codebook_argument_checks(tq):
    for bits in (0, 9, -1):
        with pytest.raises(tq.TQError):
            tq.tq_codebook_gaussian(bits)
