"""Checks that pin the fp64 oracle to facts fixed independently of it.

Each ``pin_*`` function takes an oracle object (``oracle.OracleLib`` or any
object with the same ``query`` / ``prefill_head`` methods) and raises
AssertionError when the oracle disagrees with the fact.  The facts come from
"Parallax: Parameterized Local Linear Attention for Language Modeling"
(arXiv:2605.29157) as summarised on the pages, and from mathematics:

* zhichai.net section 2.1 (the attention family) and gist.science
  "Significato e Affermazioni" (W_R = 0 gives back the Transformer):
  a zero probe is softmax attention; uniform weights with no intercept are a
  linear-attention form (pinned for the centred PLX forms and for the
  no-intercept form itself).
* zhichai.net section 1.2 and gist.science "Enunciato del Problema": local
  linear attention is the intercept of a locally weighted linear regression
  of v on k around the query; the solved probe rho* makes PLX equal to it.
* closed forms for one and two keys, invariances, library routines (scipy
  softmax / logsumexp, numpy least squares, numpy weighted covariance) and a
  40-digit brute force with mpmath.

None of these re-types the oracle's own code path.
"""
from __future__ import annotations

import numpy as np
from scipy.special import logsumexp, softmax, expit

PLX_FORMS = ("explicit", "stream")


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol, what):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol * scale, f"{what}: max abs err {err:.3e} > {tol:.1e} * {scale:.3g}"


# ---------------------------------------------------------------- softmax part
def pin_sa_closed_forms(o):
    """Softmax attention against closed forms and scipy."""
    rng = _rng(11)
    d = 5
    q = rng.standard_normal(d)
    K = rng.standard_normal((2, d))
    V = rng.standard_normal((2, d))
    scale = 0.7
    # one key: the output is v_0 and the lse is the single scaled score
    out, lse = o.query("sa", q, None, K[:1], V[:1], scale)
    _close(out, V[0], 1e-15, "sa n=1 out")
    _close(lse, scale * q @ K[0], 1e-14, "sa n=1 lse")
    # two keys: weight of key 1 is the logistic of the score difference
    s = scale * K @ q
    p = expit(s[1] - s[0])
    out, lse = o.query("sa", q, None, K, V, scale)
    _close(out, (1 - p) * V[0] + p * V[1], 1e-14, "sa n=2 out")
    _close(lse, np.logaddexp(s[0], s[1]), 1e-14, "sa n=2 lse")
    # zero scale: uniform weights, plain mean, lse = ln n
    n = 9
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    out, lse = o.query("sa", q, None, K, V, 0.0)
    _close(out, V.mean(axis=0), 1e-14, "sa uniform out")
    _close(lse, np.log(n), 1e-14, "sa uniform lse")
    # random case against scipy's softmax / logsumexp
    n, d = 57, 16
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    scale = 1 / np.sqrt(d)
    out, lse = o.query("sa", q, None, K, V, scale)
    _close(out, softmax(scale * K @ q) @ V, 1e-13, "sa vs scipy softmax")
    _close(lse, logsumexp(scale * K @ q), 1e-13, "sa lse vs scipy logsumexp")


def pin_rho_zero_is_sa(o):
    """A zero probe reduces PLX to softmax attention (W_R = 0 is the
    Transformer)."""
    rng = _rng(12)
    for n, d in ((1, 4), (3, 4), (40, 16), (130, 64)):
        q = rng.standard_normal(d)
        K = rng.standard_normal((n, d))
        V = rng.standard_normal((n, d))
        ref = softmax(K @ q / np.sqrt(d)) @ V
        for form in PLX_FORMS:
            out, lse = o.query(form, q, np.zeros(d), K, V, 1 / np.sqrt(d))
            _close(out, ref, 1e-13, f"{form} rho=0 vs softmax attention (n={n})")
            _close(lse, logsumexp(K @ q / np.sqrt(d)), 1e-13, f"{form} rho=0 lse")


# ------------------------------------------------------------- covariance part
def pin_plx_closed_forms(o):
    """One key: the covariance vanishes, o = v_0.  Two keys with logistic
    weight p: Sigma_KV = p(1-p)(v_1-v_0)(k_1-k_0)^T."""
    rng = _rng(13)
    d = 6
    q, rho = rng.standard_normal(d), rng.standard_normal(d)
    K = rng.standard_normal((2, d))
    V = rng.standard_normal((2, d))
    scale = 0.45
    s = scale * K @ q
    p = expit(s[1] - s[0])
    vbar = (1 - p) * V[0] + p * V[1]
    expect = vbar - p * (1 - p) * (V[1] - V[0]) * ((K[1] - K[0]) @ rho)
    for form in PLX_FORMS:
        out, _ = o.query(form, q, rho, K[:1], V[:1], scale)
        _close(out, V[0], 1e-15, f"{form} n=1")
        out, lse = o.query(form, q, rho, K, V, scale)
        _close(out, expect, 1e-14, f"{form} n=2 closed form")
        _close(lse, np.logaddexp(s[0], s[1]), 1e-14, f"{form} n=2 lse")


def pin_local_linear_regression(o):
    """With the solved probe rho* = Sigma_KK^{-1} (kbar - q), PLX equals the
    intercept b of the weighted least-squares fit
        min_{b, W} sum_j w_j || v_j - b - W (k_j - q) ||^2,
    the local linear estimator at q.  This fixes the minus sign, the
    orientation (d_v x d_k) and the normalisation of Sigma_KV."""
    rng = _rng(14)
    for trial in range(4):
        d, n = 4, 32
        q = rng.standard_normal(d)
        K = rng.standard_normal((n, d)) * rng.uniform(0.5, 2.0, size=d)
        V = rng.standard_normal((n, d)) + K @ rng.standard_normal((d, d))
        scale = 0.6
        w = softmax(scale * K @ q)
        kbar = w @ K
        sigma_kk = np.cov(K.T, aweights=w, bias=True)
        rho_star = np.linalg.solve(sigma_kk, kbar - q)
        X = np.hstack([np.ones((n, 1)), K - q])
        sw = np.sqrt(w)[:, None]
        coef, *_ = np.linalg.lstsq(X * sw, V * sw, rcond=None)
        intercept = coef[0]
        for form in PLX_FORMS:
            out, _ = o.query(form, q, rho_star, K, V, scale)
            _close(out, intercept, 1e-10, f"{form} vs weighted least squares (trial {trial})")


def pin_uniform_weights_linear_attention(o):
    """Zero scale (bandwidth h -> inf) gives uniform causal weights 1/n over
    the prefix, and then
        o_i = (m_i/n)(1 + z_i.rho_i/n) - S_i rho_i / n,
    with prefix sums S_i = sum v_j k_j^T, z_i = sum k_j, m_i = sum v_j.
    With centred data (keys and values in +/- pairs) at even n the intercept
    vanishes and o_i = -S_i rho_i / n: linear attention with probe -rho."""
    rng = _rng(15)
    N, d = 24, 5
    Q = rng.standard_normal((N, d))
    R = rng.standard_normal((N, d))
    K = rng.standard_normal((N, d))
    V = rng.standard_normal((N, d))
    S = np.cumsum(V[:, :, None] * K[:, None, :], axis=0)
    z = np.cumsum(K, axis=0)
    m = np.cumsum(V, axis=0)
    n = np.arange(1, N + 1)[:, None]
    expect = (m / n) * (1 + np.sum(z * R, axis=1, keepdims=True) / n) \
        - np.einsum("iab,ib->ia", S, R) / n
    for form in PLX_FORMS:
        out, lse = o.prefill_head(form, Q, K, V, R, 0.0)
        _close(out, expect, 1e-12, f"{form} uniform weights vs prefix sums")
        _close(lse, np.log(n[:, 0]), 1e-13, f"{form} uniform lse")
    # centred: pairs (k, v), (-k, -v)
    half = rng.standard_normal((N // 2, d))
    Kc = np.repeat(half, 2, axis=0) * np.tile([1.0, -1.0], N // 2)[:, None]
    halfv = rng.standard_normal((N // 2, d))
    Vc = np.repeat(halfv, 2, axis=0) * np.tile([1.0, -1.0], N // 2)[:, None]
    Sc = np.cumsum(Vc[:, :, None] * Kc[:, None, :], axis=0)
    even = np.arange(1, N, 2)            # rows with an even prefix length
    lin = -np.einsum("iab,ib->ia", Sc[even], R[even]) / (even + 1)[:, None]
    for form in PLX_FORMS:
        out, _ = o.prefill_head(form, Q, Kc, Vc, R, 0.0, rows=even)
        _close(out, lin, 1e-12, f"{form} centred uniform = linear attention with -rho")


def pin_invariants(o):
    """Linearity in rho; a common shift of the values shifts the output; a
    constant value gives that constant; a common shift of the keys leaves the
    output unchanged and moves lse by scale * q.a."""
    rng = _rng(16)
    n, d = 33, 8
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    r1, r2 = rng.standard_normal(d), rng.standard_normal(d)
    scale = 0.5
    for form in PLX_FORMS:
        o0, l0 = o.query(form, q, np.zeros(d), K, V, scale)
        o1, _ = o.query(form, q, r1, K, V, scale)
        o2, _ = o.query(form, q, r2, K, V, scale)
        o12, _ = o.query(form, q, r1 + r2, K, V, scale)
        _close(o12 - o0, (o1 - o0) + (o2 - o0), 1e-12, f"{form} linear in rho")
        o3, _ = o.query(form, q, 2.5 * r1, K, V, scale)
        _close(o3 - o0, 2.5 * (o1 - o0), 1e-12, f"{form} homogeneous in rho")
        a = rng.standard_normal(d)
        ov, _ = o.query(form, q, r1, K, V + a, scale)
        _close(ov, o1 + a, 1e-12, f"{form} value shift")
        c = rng.standard_normal(d)
        oc, _ = o.query(form, q, r1, K, np.tile(c, (n, 1)), scale)
        _close(oc, c, 1e-12, f"{form} constant value")
        ok, lk = o.query(form, q, r1, K + a, V, scale)
        _close(ok, o1, 1e-12, f"{form} key shift")
        _close(lk, l0 + scale * q @ a, 1e-12, f"{form} key shift lse")


def pin_brute_force(o):
    """40-digit mpmath evaluation of the definition on tiny inputs."""
    import mpmath as mp
    mp.mp.dps = 40
    rng = _rng(17)
    for n, d in ((1, 1), (2, 3), (5, 2), (8, 4), (7, 4)):
        q, rho = rng.standard_normal(d), rng.standard_normal(d)
        K = rng.standard_normal((n, d))
        V = rng.standard_normal((n, d))
        scale = float(rng.uniform(0.2, 1.5))
        Km = [[mp.mpf(float(x)) for x in row] for row in K]
        Vm = [[mp.mpf(float(x)) for x in row] for row in V]
        qm = [mp.mpf(float(x)) for x in q]
        rm = [mp.mpf(float(x)) for x in rho]
        s = [mp.mpf(scale) * mp.fsum(qm[t] * Km[j][t] for t in range(d)) for j in range(n)]
        e = [mp.e ** sj for sj in s]
        tot = mp.fsum(e)
        w = [ej / tot for ej in e]
        vbar = [mp.fsum(w[j] * Vm[j][a] for j in range(n)) for a in range(d)]
        kbar = [mp.fsum(w[j] * Km[j][b] for j in range(n)) for b in range(d)]
        sig = [[mp.fsum(w[j] * (Vm[j][a] - vbar[a]) * (Km[j][b] - kbar[b]) for j in range(n))
                for b in range(d)] for a in range(d)]
        expect = [float(vbar[a] - mp.fsum(sig[a][b] * rm[b] for b in range(d))) for a in range(d)]
        lse = float(mp.log(tot))
        for form in PLX_FORMS:
            out, l = o.query(form, q, rho, K, V, scale)
            _close(out, expect, 1e-13, f"{form} brute force n={n} d={d}")
            _close(l, lse, 1e-13, f"{form} brute force lse")
        out, _ = o.query("sa", q, None, K, V, scale)
        _close(out, [float(x) for x in vbar], 1e-13, "sa brute force")


def pin_causal_prefix(o):
    """Causal prefill: row i attends to keys 0..i, the diagonal included."""
    rng = _rng(18)
    N, d = 19, 4
    Q, R = rng.standard_normal((N, d)), rng.standard_normal((N, d))
    K, V = rng.standard_normal((N, d)), rng.standard_normal((N, d))
    for form in ("sa",) + PLX_FORMS:
        out, lse = o.prefill_head(form, Q, K, V, R, 0.8)
        _close(out[0], V[0], 1e-15, f"{form} row 0 is v_0")
        for i in (0, 1, 7, N - 1):
            ref, lref = o.query(form, Q[i], R[i], K[: i + 1], V[: i + 1], 0.8)
            _close(out[i], ref, 1e-15, f"{form} row {i}")
        # the scores of row i: its lse equals scipy's over keys 0..i
        for i in (0, 5, N - 1):
            _close(lse[i], logsumexp(0.8 * K[: i + 1] @ Q[i]), 1e-13, f"{form} lse row {i}")


def pin_forms_agree(o):
    """The explicit d x d covariance form and the streaming identity agree
    (two different computations of the same quantity)."""
    rng = _rng(19)
    for n, d in ((3, 2), (64, 16), (300, 64), (257, 128)):
        q, rho = rng.standard_normal(d), 0.3 * rng.standard_normal(d)
        K = rng.standard_normal((n, d))
        V = rng.standard_normal((n, d))
        oe, le = o.query("explicit", q, rho, K, V, 1 / np.sqrt(d))
        os_, ls = o.query("stream", q, rho, K, V, 1 / np.sqrt(d))
        _close(os_, oe, 1e-10, f"explicit vs stream n={n} d={d}")
        _close(ls, le, 1e-13, "lse explicit vs stream")


def pin_empty(o):
    """No keys: o = 0, lse = -inf."""
    d = 4
    for form in ("sa",) + PLX_FORMS:
        out, lse = o.query(form, np.ones(d), np.ones(d), np.zeros((0, d)), np.zeros((0, d)), 1.0)
        assert np.all(out == 0) and lse == -np.inf, f"{form} empty"


def pin_no_intercept(o):
    """The family's no-intercept member (zhichai.net section 2.1: without the
    affine term the covariance loses its centring, vbar = kbar = 0).
    * Uniform weights (scale = 0): o_i = -S_i rho_i / n with the prefix sums
      S_i = sum_j v_j k_j^T, linear attention with probe -rho.
    * Against the centred form: Sigma_KV = M - vbar kbar^T for the raw moment
      M = sum w v k^T, so o_PLX - o_noint = (1 + rho.kbar) o_SA, with the
      weights, kbar and o_SA from scipy's softmax.
    * One key: o = -(rho.k_0) v_0."""
    rng = _rng(29)
    N, d = 20, 6
    Q = rng.standard_normal((N, d))
    R = rng.standard_normal((N, d))
    K = rng.standard_normal((N, d))
    V = rng.standard_normal((N, d))
    n = np.arange(1, N + 1)[:, None]
    S = np.cumsum(V[:, :, None] * K[:, None, :], axis=0)
    out, lse = o.prefill_head("noint", Q, K, V, R, 0.0)
    _close(out, -np.einsum("iab,ib->ia", S, R) / n, 1e-12, "noint uniform = linear attention with -rho")
    _close(lse, np.log(n[:, 0]), 1e-13, "noint uniform lse")
    scale = 0.45
    plx, _ = o.prefill_head("explicit", Q, K, V, R, scale)
    noint, lse = o.prefill_head("noint", Q, K, V, R, scale)
    for i in range(N):
        w = softmax(scale * K[: i + 1] @ Q[i])
        kbar = w @ K[: i + 1]
        osa = w @ V[: i + 1]
        _close(plx[i] - noint[i], (1.0 + R[i] @ kbar) * osa, 1e-12, f"noint vs centred row {i}")
        _close(lse[i], logsumexp(scale * K[: i + 1] @ Q[i]), 1e-13, f"noint lse row {i}")
    out, _ = o.query("noint", Q[0], R[0], K[:1], V[:1], scale)
    _close(out, -(R[0] @ K[0]) * V[0], 1e-14, "noint one key")


ALL_PINS = [pin_sa_closed_forms, pin_rho_zero_is_sa, pin_plx_closed_forms,
            pin_local_linear_regression, pin_uniform_weights_linear_attention,
            pin_invariants, pin_brute_force, pin_causal_prefix, pin_forms_agree,
            pin_empty, pin_no_intercept]
