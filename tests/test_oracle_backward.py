"""Pins of the fp64 backward oracle (CPU): finite differences of the
independent C oracle's explicit forward, the value-shift invariant, and the
affinity of the output in the probe."""
import numpy as np
import pytest

import oracle
from oracle.backward import plx_backward


def _inputs(N, d, seed, rho_std=0.7):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((1, 1, N, d)) for _ in range(3))
    rho = rho_std * rng.standard_normal((1, 1, N, d))
    dout = rng.standard_normal((1, 1, N, d))
    return q, k, v, rho, dout


def _loss(q, k, v, rho, dout, scale):
    res = oracle.prefill("explicit", q, k, v, rho, scale)
    o = np.stack([res[(0, 0)][0]])
    return float(np.sum(o * dout[0]))


def test_backward_matches_finite_differences_of_the_c_oracle():
    N, d, scale = 7, 4, 0.6
    q, k, v, rho, dout = _inputs(N, d, 3)
    grads = plx_backward(q, k, v, rho, dout, scale)[:4]
    rng = np.random.default_rng(5)
    eps = 1e-6
    for which, g in enumerate(grads):
        for _ in range(6):
            i, c = int(rng.integers(N)), int(rng.integers(d))
            args = [a.copy() for a in (q, k, v, rho)]
            args[which][0, 0, i, c] += eps
            lp = _loss(*args, dout, scale)
            args[which][0, 0, i, c] -= 2 * eps
            lm = _loss(*args, dout, scale)
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - g[0, 0, i, c]) <= 1e-6 * max(1.0, abs(fd)), (which, i, c, fd, g[0, 0, i, c])


def test_backward_value_shift_invariant():
    # v_j + a for every j shifts every o_i by a, so sum_j dL/dv_j = sum_i dO_i
    q, k, v, rho, dout = _inputs(12, 6, 4)
    dv = plx_backward(q, k, v, rho, dout, 0.4)[2]
    assert np.allclose(dv[0, 0].sum(0), dout[0, 0].sum(0), atol=1e-12)


def test_backward_affine_in_probe():
    # o is affine in rho: dL/drho does not depend on rho; dq, dk, dv are affine in it
    q, k, v, r1, dout = _inputs(10, 5, 6)
    r2 = np.random.default_rng(7).standard_normal(r1.shape)
    g0 = plx_backward(q, k, v, 0 * r1, dout, 0.5)
    g1 = plx_backward(q, k, v, r1, dout, 0.5)
    g2 = plx_backward(q, k, v, r2, dout, 0.5)
    g12 = plx_backward(q, k, v, r1 + r2, dout, 0.5)
    assert np.allclose(g1[3], g2[3], atol=1e-12) and np.allclose(g0[3], g1[3], atol=1e-12)
    for n in range(3):
        assert np.allclose(g12[n] - g0[n], (g1[n] - g0[n]) + (g2[n] - g0[n]), atol=1e-10)


@pytest.mark.parametrize("shape,rho_std", [((1, 2, 37, 8), 0.4), ((2, 1, 20, 5), 1.0), ((1, 1, 1, 4), 0.3)])
def test_closed_form_matches_autograd(shape, rho_std):
    """The hand-derived closed form (dense fp64, for long sequences) against
    autograd of the explicit-covariance forward: every term and sign of the
    derivation is checked."""
    from oracle.backward import plx_backward, plx_backward_closed
    B, H, N, d = shape
    rng = np.random.default_rng(N * d)
    q, k, v, dout = (rng.standard_normal(shape) for _ in range(4))
    rho = rho_std * rng.standard_normal(shape)
    ref = plx_backward(q, k, v, rho, dout, 0.6)[:4]
    got = plx_backward_closed(q, k, v, rho, dout, 0.6)
    for (b, h), grads in got.items():
        for name, g, r in zip(("dq", "dk", "dv", "drho"), grads, ref):
            assert np.allclose(g, r[b, h], rtol=1e-10, atol=1e-12), f"{name} {shape} ({b}, {h})"
