"""The oracle against what the pages and mathematics fix (CPU only)."""
import numpy as np
import pytest

import oracle
from oracle import chunked_ref
from tests import pins


@pytest.mark.parametrize("pin", pins.SSD_PINS + pins.SS_PINS + pins.TRAP_PINS + pins.ROT_PINS
                         + pins.QUAT_PINS + pins.BWD_PINS + pins.TRAP_BWD_PINS,
                         ids=lambda f: f.__name__)
def test_pin_holds(pin):
    for name, err, tol in pin(0):
        assert err <= tol, f"{name}: error {err:.3e} > {tol:.1e}"


@pytest.mark.parametrize("name,code", sorted(oracle.MUTATIONS_SSD.items()))
def test_planted_ssd_mistake_is_caught(name, code):
    failed = [n for pin in pins.SSD_PINS for (n, err, tol) in pin(code) if not err <= tol]
    assert failed, f"planted mistake '{name}' passed every SSD pin"


@pytest.mark.parametrize("name,code", sorted(oracle.MUTATIONS_TRAP.items()))
def test_planted_trapezoidal_mistake_is_caught(name, code):
    failed = [n for pin in pins.TRAP_PINS for (n, err, tol) in pin(code) if not err <= tol]
    assert failed, f"planted mistake '{name}' passed every trapezoidal pin"


@pytest.mark.parametrize("name,code", sorted(oracle.MUTATIONS_ROT.items()))
def test_planted_rotation_variant_mistake_is_caught(name, code):
    failed = [n for pin in pins.ROT_PINS for (n, err, tol) in pin(code) if not err <= tol]
    assert failed, f"planted mistake '{name}' passed every rotation-variant pin"


@pytest.mark.parametrize("name,code", sorted(oracle.MUTATIONS_QUAT.items()))
def test_planted_quaternion_mistake_is_caught(name, code):
    failed = [n for pin in pins.QUAT_PINS for (n, err, tol) in pin(code) if not err <= tol]
    assert failed, f"planted mistake '{name}' passed every quaternion pin"


@pytest.mark.parametrize("name,code", sorted(oracle.MUTATIONS_BWD.items()))
def test_planted_backward_mistake_is_caught(name, code):
    failed = [n for pin in pins.BWD_PINS for (n, err, tol) in pin(code) if not err <= tol]
    assert failed, f"planted mistake '{name}' passed every backward pin"


@pytest.mark.parametrize("name,code", sorted(oracle.MUTATIONS_SS.items()))
def test_planted_selective_scan_mistake_is_caught(name, code):
    failed = [n for pin in pins.SS_PINS for (n, err, tol) in pin(code) if not err <= tol]
    assert failed, f"planted mistake '{name}' passed every selective-scan pin"


def test_segsum_definition():
    """segsum.rs page: out[i,j] = sum_{k=j+1..i} x_k for i >= j, -inf above the diagonal."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((2, 3, 11))
    s = chunked_ref.segsum(x)
    T = x.shape[-1]
    for i in range(T):
        for j in range(T):
            if i >= j:
                ref = x[..., j + 1:i + 1].sum(axis=-1)
                np.testing.assert_allclose(s[..., i, j], ref, rtol=0, atol=1e-12)
            else:
                assert np.all(np.isneginf(s[..., i, j]))
    assert np.all(np.diagonal(s, axis1=-2, axis2=-1) == 0.0)
    # exp(segsum) is the causal 1-semiseparable mask: L[i,k] = L[i,j] L[j,k] for k <= j <= i
    L = np.exp(s)
    for i in range(T):
        for j in range(i + 1):
            for k in range(j + 1):
                np.testing.assert_allclose(L[..., i, k], L[..., i, j] * L[..., j, k], rtol=1e-12)
    assert np.all(L[..., np.triu_indices(T, 1)[0], np.triu_indices(T, 1)[1]] == 0.0)


def test_segsum_constant_input():
    s = chunked_ref.segsum(np.full(6, -0.25))
    for i in range(6):
        for j in range(i + 1):
            assert s[i, j] == pytest.approx(-0.25 * (i - j), abs=1e-15)


def test_oracle_threading_is_bitwise_stable():
    x, dA, B, C, th, h0 = pins._problem(61, 3, 17, 2, 4, 2, 3, 4, theta=True, init=True)
    y1, f1 = oracle.ssd(x, dA, B, C, th, h0, nthreads=1)
    y4, f4 = oracle.ssd(x, dA, B, C, th, h0, nthreads=5)
    assert np.array_equal(y1, y4) and np.array_equal(f1, f4)


def test_oracle_empty_inputs():
    y, f = oracle.ssd(np.zeros((2, 0, 1, 3, 4)), np.zeros((2, 0, 3)), np.zeros((2, 0, 1, 1, 5)),
                      np.zeros((2, 0, 1, 1, 5)), init_state=np.ones((2, 3, 4, 5)))
    assert y.shape == (2, 0, 1, 3, 4) and np.all(f == 1.0)


@pytest.mark.parametrize("name,code", sorted(oracle.MUTATIONS_TRAP_BWD.items()))
def test_planted_trapezoidal_backward_mistake_is_caught(name, code):
    failed = [n for pin in pins.TRAP_BWD_PINS for (n, err, tol) in pin(code) if not err <= tol]
    assert failed, f"planted mistake '{name}' passed every trapezoidal backward pin"
