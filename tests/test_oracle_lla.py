"""Pins of the fp64 LLA oracle (oracle/lla.py), on the CPU.

Local linear attention ("Parallax: Parameterized Local Linear Attention for
Language Modeling", zhichai.net section 1.2; gist.science "Enunciato del
Problema") fits v locally as a linear function of the key; its solved probe
rho* = (Sigma_KK + lambda I)^{-1} mu, mu = kbar - q, fed to Parallax's output
formula (zhichai.net section 1.3) is the fit's intercept at the query.

Pins, each fixed independently of the oracle's code:
- numpy's lstsq on the ridge-augmented weighted regression;
- exact recovery of linear data v = a + M k;
- the softmax limit at large lambda (scipy softmax);
- the independent C oracle's explicit Parallax form fed the solved probe;
- conjugate gradients after d steps equal the direct solve;
- affinity in v: shifting every value by a shifts o by a.

Planted mistakes each fail one of them: a flipped mu, an uncentred key
moment, the ridge on the wrong side, an unweighted moment, a CG sign slip, a
transposed value-key covariance, an output without its vbar term."""
import types

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from oracle import lla


def _inputs(rng, B, H, N, d, key_scale=1.0):
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d)) * key_scale
    v = rng.standard_normal((B, H, N, d))
    return q, k, v


def pin_ridge_least_squares(mod):
    """o_i is the intercept b of min sum_j w_ij |v_j - b - W (k_j - q_i)|^2 + lambda |W|_F^2,
    solved by numpy's lstsq on the weighted design with sqrt(lambda) I rows for W."""
    rng = np.random.default_rng(31)
    B, H, N, d = 1, 2, 9, 3
    q, k, v = _inputs(rng, B, H, N, d)
    scale, lam = 0.7, 0.3
    res = mod.lla_direct(q, k, v, scale, lam)
    for (b, h), (o, rho, rows) in res.items():
        for n, i in enumerate(rows):
            K, V = k[b, h, : i + 1], v[b, h, : i + 1]
            w = softmax(scale * K @ q[b, h, i])
            X = np.hstack([np.ones((i + 1, 1)), K - q[b, h, i]]) * np.sqrt(w)[:, None]
            Y = V * np.sqrt(w)[:, None]
            ridge = np.hstack([np.zeros((d, 1)), np.sqrt(lam) * np.eye(d)])
            coef, *_ = np.linalg.lstsq(np.vstack([X, ridge]), np.vstack([Y, np.zeros((d, d))]), rcond=None)
            np.testing.assert_allclose(o[n], coef[0], rtol=1e-9, atol=1e-9)


def pin_linear_data(mod):
    """v_j = a + M k_j exactly: at lambda = 0 with a full-rank prefix the fit is
    exact, so o_i = a + M q_i."""
    rng = np.random.default_rng(32)
    N, d = 14, 3
    q = rng.standard_normal((1, 1, N, d))
    k = rng.standard_normal((1, 1, N, d))
    a = rng.standard_normal(d)
    M = rng.standard_normal((d, d))
    v = a + k @ M.T
    rows = np.arange(d + 2, N)
    o, rho, _ = mod.lla_direct(q, k, v, 0.5, 0.0, rows=rows)[(0, 0)]
    np.testing.assert_allclose(o, a + q[0, 0, rows] @ M.T, rtol=1e-9, atol=1e-9)


def pin_softmax_limit(mod):
    """lambda -> infinity sends rho* to 0 and o to softmax attention."""
    rng = np.random.default_rng(33)
    q, k, v = _inputs(rng, 1, 1, 7, 4)
    o, rho, rows = mod.lla_direct(q, k, v, 0.8, 1e9)[(0, 0)]
    for n, i in enumerate(rows):
        w = softmax(0.8 * k[0, 0, : i + 1] @ q[0, 0, i])
        np.testing.assert_allclose(o[n], w @ v[0, 0, : i + 1], rtol=0, atol=1e-7)
        assert float(np.max(np.abs(rho[n]))) < 1e-7


def pin_parallax_with_solved_probe(mod):
    """Parallax's output formula, evaluated by the independent C oracle (explicit
    covariance form), with rho = the solved probe gives o."""
    rng = np.random.default_rng(34)
    q, k, v = _inputs(rng, 1, 2, 11, 4, key_scale=1.5)
    scale, lam = 0.6, 0.05
    for (b, h), (o, rho, rows) in mod.lla_direct(q, k, v, scale, lam).items():
        for n, i in enumerate(rows):
            out, _ = oracle.query("explicit", q[b, h, i], rho[n], k[b, h, : i + 1], v[b, h, : i + 1], scale)
            np.testing.assert_allclose(o[n], out, rtol=1e-9, atol=1e-9)


def pin_cg_reaches_the_solve(mod):
    """In exact arithmetic CG solves a d x d SPD system in at most d steps."""
    rng = np.random.default_rng(35)
    q, k, v = _inputs(rng, 1, 1, 10, 4)
    scale, lam = 0.5, 0.2
    direct = mod.lla_direct(q, k, v, scale, lam)[(0, 0)]
    cg = mod.lla_cg(q, k, v, scale, lam, max_iters=4)[(0, 0)]
    np.testing.assert_allclose(cg[1], direct[1], rtol=1e-8, atol=1e-8)
    np.testing.assert_allclose(cg[0], direct[0], rtol=1e-8, atol=1e-8)
    assert int(cg[3].max()) <= 4


def pin_value_shift(mod):
    """The fit's intercept is affine in the values: v_j + a gives o + a, and
    rho* (a function of q and k only) does not change."""
    rng = np.random.default_rng(37)
    q, k, v = _inputs(rng, 1, 1, 9, 3)
    a = rng.standard_normal(3)
    o1, r1, _ = mod.lla_direct(q, k, v, 0.7, 0.2)[(0, 0)]
    o2, r2, _ = mod.lla_direct(q, k, v + a, 0.7, 0.2)[(0, 0)]
    np.testing.assert_allclose(o2, o1 + a, rtol=1e-10, atol=1e-10)
    np.testing.assert_allclose(r2, r1, rtol=1e-12, atol=1e-12)


PINS = [pin_ridge_least_squares, pin_linear_data, pin_softmax_limit, pin_parallax_with_solved_probe,
        pin_cg_reaches_the_solve, pin_value_shift]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(lla)


def test_cg_tolerance_stops_rows_early():
    """With a tolerance the CG oracle stops each row once its residual is small
    enough, and the result is still close to the solve."""
    rng = np.random.default_rng(36)
    q, k, v = _inputs(rng, 1, 1, 40, 8)
    direct = lla.lla_direct(q, k, v, 0.35, 0.1)[(0, 0)]
    o, rho, rows, steps = lla.lla_cg(q, k, v, 0.35, 0.1, max_iters=100, tol=1e-6)[(0, 0)]
    assert int(steps.max()) <= 8 and int(steps.min()) >= 1
    np.testing.assert_allclose(o, direct[0], rtol=1e-5, atol=1e-5)


MUTANTS = {
    "mu_sign_flipped": ("mu = kbar - q[i]", "mu = q[i] - kbar"),
    "uncentred_key_moment": ("S = (kc * w[:, None]).T @ kc + lam * np.eye(d)",
                             "S = (k[: i + 1] * w[:, None]).T @ k[: i + 1] + lam * np.eye(d)"),
    "ridge_subtracted": ("+ lam * np.eye(d)      # S_i", "- lam * np.eye(d)      # S_i"),
    "unweighted_key_moment": ("S = (kc * w[:, None]).T @ kc", "S = kc.T @ kc / len(w)"),
    "cg_residual_sign": ("r = r - alpha * Ap", "r = r + alpha * Ap"),
    "value_covariance_transposed": ("C = (vc * w[:, None]).T @ kc", "C = (kc * w[:, None]).T @ vc"),
    "output_drops_vbar": ("o[n] = vbar - C @ rho[n]", "o[n] = -(C @ rho[n])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(lla.__file__).read()
    assert src.count(old) == 1, f"mutant anchor for {name} not unique"
    mod = types.ModuleType(f"lla_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    caught = 0
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, np.linalg.LinAlgError):
            caught += 1
    assert caught >= 1, f"mutant {name} passed every pin"
