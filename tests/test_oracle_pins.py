"""The CPU oracle against its pins (no GPU). See ``oracle_pins.py``."""
import numpy as np
import pytest

from oracle import oracle as O

import oracle_pins


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    pin()


@pytest.fixture(scope="module")
def long_double_lib():
    return O.load(precision="long double")


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda f: f.__name__)
def test_oracle_pin_long_double(pin, long_double_lib, monkeypatch):
    """Every pin holds for the long-double build of the same source too."""
    monkeypatch.setattr(O, "_lib", long_double_lib)
    pin()


def test_long_double_second_order_at_small_eps():
    """At eps = 1e-6 the O(eps^2) divergence of nearly identical rows lies
    below what double keeps of the O(eps) terms that cancel (the double build
    is off by about 1e-3 relative there); the long-double build meets the
    second-order closed form to 1e-5 (its O(eps) remainder is about 1e-6)."""
    rng = np.random.default_rng(28)
    s = rng.normal(0, 2, (4, 4096))
    t = s + 1e-6 * rng.normal(0, 1, (4, 4096))
    for beta in (0.3, 0.5, 0.8):
        got = O.jsd(s, t, beta, grad=False, precision="long double")[0]
        ref = oracle_pins.jsd_second_order(s, t, beta)
        assert np.all(np.abs(got / ref - 1.0) <= 1e-5), (beta, got, ref)


def test_double_rounding_against_long_double():
    """The double oracle's own rounding at the Qwen vocabulary (151936), with a
    large common offset and masked tokens: loss, gradients and entropy agree
    with the long-double build to 1e-13 relative (measured: below 1e-15), far
    inside the 1e-5 tolerance the GPU kernels are held to."""
    rng = np.random.default_rng(29)
    v = 151936
    s = rng.normal(0, 4, (3, v)) + 1000.0
    t = s + rng.normal(0, 2, (3, v))
    s[0, :100] = -np.inf
    t[1, 50:60] = -np.inf
    for beta in (0.0, 0.5, 1.0):
        a = O.jsd(s, t, beta)
        b = O.jsd(s, t, beta, precision="long double")
        fin = np.isfinite(b[0])
        assert np.array_equal(fin, np.isfinite(a[0])), beta
        assert np.all(np.abs(a[0][fin] / b[0][fin] - 1.0) <= 1e-13), beta
        for k in (3, 4):
            assert np.max(np.abs(a[k] - b[k])) <= 1e-13 * np.max(np.abs(b[k])), (beta, k)
    a = O.entropy(s)
    b = O.entropy(s, precision="long double")
    assert np.all(np.abs(a[0] / b[0] - 1.0) <= 1e-13)
    assert np.max(np.abs(a[1] - b[1])) <= 1e-13 * np.max(np.abs(b[1]))
