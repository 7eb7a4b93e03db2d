"""fp64 Local Linear Attention (LLA) with the solved probe -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU legs
may import this module.  It shares no code with the CUDA library.

"Parallax: Parameterized Local Linear Attention for Language Modeling"
describes LLA as the method Parallax replaces (zhichai.net section 1.2;
gist.science, "Enunciato del Problema"): where softmax attention fits a
constant to the values near the query, LLA fits a linear function of the key,
b + W (k - q), and each token's optimal probe solves a linear system,
rho_i* = Sigma_i^{-1} mu_i, by conjugate gradients with a ridge lambda that
trades stability against falling back to softmax.  Parallax's output formula
(zhichai.net section 1.3) then gives the attention output with that probe.

Written out per query i of one head (causal prefix j <= i):

    w_ij   = softmax_j(scale q_i . k_j)
    kbar_i = sum_j w_ij k_j,      vbar_i = sum_j w_ij v_j
    S_i    = sum_j w_ij (k_j - kbar_i)(k_j - kbar_i)^T              (d x d)
    C_i    = sum_j w_ij (v_j - vbar_i)(k_j - kbar_i)^T              (d x d)
    mu_i   = kbar_i - q_i
    rho_i* = (S_i + lambda I)^{-1} mu_i
    o_i    = vbar_i - C_i rho_i*

The pages leave mu and the ridge's placement open.  The reading taken here is
the weighted least-squares one: o_i is the intercept at k = q_i of the ridge
fit of v on (k - q_i) with weights w_ij, ridge lambda on the slope only.
Solving its normal equations gives exactly the lines above.

``lla_direct`` solves each system with numpy's dense solver (the plain
definition).  ``lla_cg`` runs textbook conjugate gradients from rho = 0 on
the same system.  It follows the CUDA path's iteration rule: stop a row once
r.r <= tol^2 mu.mu, or after max_iters steps.  With it, iteration-limited
results can be compared step for step.

Pins (tests/test_oracle_lla.py):
- the ridge least-squares fit solved by numpy's lstsq;
- exact recovery of linear data v = a + M k;
- the softmax limit at large lambda;
- Parallax's output with the solved probe, computed by the independent C
  oracle;
- CG after d steps equals the direct solve.
"""
from __future__ import annotations

import numpy as np


def _row_stats(q, k, v, scale, i):
    """Weights, means and centred keys/values of query i's causal prefix (fp64)."""
    s = scale * (k[: i + 1] @ q[i])
    w = np.exp(s - s.max())
    w /= w.sum()
    kbar = w @ k[: i + 1]
    vbar = w @ v[: i + 1]
    kc = k[: i + 1] - kbar
    vc = v[: i + 1] - vbar
    return w, kbar, vbar, kc, vc


def _systems(q, k, v, scale, lam, i):
    w, kbar, vbar, kc, vc = _row_stats(q, k, v, scale, i)
    d = q.shape[1]
    S = (kc * w[:, None]).T @ kc + lam * np.eye(d)      # S_i + lambda I
    C = (vc * w[:, None]).T @ kc                        # C_i (d_v x d_k)
    mu = kbar - q[i]
    return S, C, mu, vbar


def _heads(q, heads):
    B, H = q.shape[:2]
    return [(b, h) for b in range(B) for h in range(H)] if heads is None else list(heads)


def lla_direct(q, k, v, scale: float, lam: float, heads=None, rows=None):
    """{(b, h): (o [R, d], rho [R, d], rows)} with rho = (S + lambda I)^{-1} mu
    from a dense solve, for the given rows (default: all) of the given heads."""
    q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
    N = q.shape[2]
    out = {}
    for (b, h) in _heads(q, heads):
        rr = np.arange(N) if rows is None else np.asarray(rows)
        o = np.zeros((len(rr), q.shape[3]))
        rho = np.zeros_like(o)
        for n, i in enumerate(rr):
            S, C, mu, vbar = _systems(q[b, h], k[b, h], v[b, h], scale, lam, int(i))
            rho[n] = np.linalg.solve(S, mu)
            o[n] = vbar - C @ rho[n]
        out[(b, h)] = (o, rho, rr)
    return out


def lla_cg(q, k, v, scale: float, lam: float, max_iters: int, tol: float = 0.0, heads=None, rows=None):
    """As lla_direct, with rho from conjugate gradients started at 0.  Each
    step: Ap = (S + lambda I) p; alpha = rs / p.Ap; rho += alpha p;
    r -= alpha Ap; rs' = r.r; p = r + (rs' / rs) p.  A row stops before a step
    once rs <= tol^2 mu.mu (or when p.Ap <= 0).  Returns
    {(b, h): (o, rho, rows, steps taken per row)}."""
    q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
    N = q.shape[2]
    out = {}
    for (b, h) in _heads(q, heads):
        rr = np.arange(N) if rows is None else np.asarray(rows)
        o = np.zeros((len(rr), q.shape[3]))
        rho = np.zeros_like(o)
        steps = np.zeros(len(rr), np.int64)
        for n, i in enumerate(rr):
            S, C, mu, vbar = _systems(q[b, h], k[b, h], v[b, h], scale, lam, int(i))
            x = np.zeros_like(mu)
            r = mu.copy()
            p = r.copy()
            rs = rs0 = float(r @ r)
            for _ in range(max_iters):
                if rs <= tol * tol * rs0:
                    break
                Ap = S @ p
                pAp = float(p @ Ap)
                if not pAp > 0.0:
                    break
                alpha = rs / pAp
                x = x + alpha * p
                r = r - alpha * Ap
                rs_new = float(r @ r)
                p = r + (rs_new / rs) * p
                rs = rs_new
                steps[n] += 1
            rho[n] = x
            o[n] = vbar - C @ x
        out[(b, h)] = (o, rho, rr, steps)
    return out
