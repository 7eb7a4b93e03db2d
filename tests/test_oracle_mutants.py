"""Each plausible mistake planted in a copy of the oracle (compiled on the
CPU) must fail at least one pin.  Shows the pins constrain every step:
softmax scale, normalisation, lse, causal prefix, centring, orientation,
sign, the streaming identity, and the no-intercept form."""
import os
import tempfile

import pytest

import oracle
from oracle import build
import pins

MUTANTS = {
    "sign_of_correction": ("out[a] = vbar[a] - corr;", "out[a] = vbar[a] + corr;"),
    "transposed_sigma": ("corr += row[b] * rho[b];", "corr += sigma[(size_t)b * d + a] * rho[b];"),
    "second_moment_not_covariance": (
        "double dv = w[j] * (vj[a] - vbar[a]);\n            double *row = sigma + (size_t)a * d;\n            for (int b = 0; b < d; ++b)\n                row[b] += dv * (kj[b] - kbar[b]);",
        "double dv = w[j] * vj[a];\n            double *row = sigma + (size_t)a * d;\n            for (int b = 0; b < d; ++b)\n                row[b] += dv * kj[b];"),
    "key_key_covariance": ("double dv = w[j] * (vj[a] - vbar[a]);", "double dv = w[j] * (kj[a] - kbar[a]);"),
    "stream_drops_c": ("out[t] = (1.0 + c) * vbar[t] - u[t];", "out[t] = vbar[t] - u[t];"),
    "stream_sign_c": ("out[t] = (1.0 + c) * vbar[t] - u[t];", "out[t] = (1.0 - c) * vbar[t] - u[t];"),
    "stream_probe_uses_query": ("r += rho[t] * kj[t];", "r += q[t] * kj[t];"),
    "stream_scaled_probe": ("r += rho[t] * kj[t];", "r += scale * rho[t] * kj[t];"),
    "unscaled_scores": ("w[j] = scale * dot;", "w[j] = dot;"),
    "lse_drops_max": ("return m + log(l);", "return log(l);"),
    "unnormalised_weights": ("w[j] /= l;", "w[j] /= 1.0;"),
    "causal_excludes_diagonal": ("K, V, i + 1, d, scale", "K, V, i, d, scale"),
    "bessel_correction": ("row[b] += dv * (kj[b] - kbar[b]);",
                          "row[b] += dv * (kj[b] - kbar[b]) * ((double)n / (double)(n > 1 ? n - 1 : 1));"),
    "noint_sign": ("out[a] = -acc;", "out[a] = acc;"),
    "noint_transposed_moment": ("acc += row[b] * rho[b];", "acc += mom[(size_t)b * d + a] * rho[b];"),
    "noint_unweighted_moment": ("double wv = w[j] * vj[a];", "double wv = vj[a];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(build.SRC).read()
    assert old in src, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "mut.c")
        so = os.path.join(tmp, "libmut.so")
        open(c, "w").write(mutated)
        build.build(src=c, out=so)
        mut = oracle.OracleLib(so)
        failures = []
        for pin in pins.ALL_PINS:
            try:
                pin(mut)
            except AssertionError as e:
                failures.append((pin.__name__, str(e)[:80]))
        assert failures, f"mutant {name} passed every pin"
