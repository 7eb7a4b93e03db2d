"""The fp64 oracle against what the pages and mathematics fix (CPU only)."""
import pytest

import oracle
import pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.default())


def test_prefill_driver_matches_per_row_queries():
    """The threaded [B,H,N,d] driver returns the same rows as single queries."""
    import numpy as np
    import plx_inputs
    x = plx_inputs.prefill(1, 2, 40, 8, seed=5, dtype="f32")
    res = oracle.prefill("stream", x.q, x.k, x.v, x.rho, x.scale, threads=3)
    for (b, h), (out, lse, rows) in res.items():
        assert list(rows) == list(range(40))
        for i in (0, 13, 39):
            ref, lref = oracle.query("stream", x.q[b, h, i], x.rho[b, h, i],
                                     x.k[b, h, : i + 1], x.v[b, h, : i + 1], x.scale)
            assert np.array_equal(out[i], ref) and lse[i] == lref


def test_decode_equals_prefill_last_row():
    """Decode at length L is prefill row L-1 on the same data."""
    import numpy as np
    import plx_inputs
    x = plx_inputs.prefill(2, 2, 33, 8, seed=6, dtype="f32")
    L = np.array([33, 17], np.int32)
    q = np.stack([x.q[b, :, L[b] - 1] for b in range(2)])
    r = np.stack([x.rho[b, :, L[b] - 1] for b in range(2)])
    dec = oracle.decode("explicit", q, r, x.k, x.v, L, x.scale)
    for b in range(2):
        for h in range(2):
            out, lse = oracle.query("explicit", x.q[b, h, L[b] - 1], x.rho[b, h, L[b] - 1],
                                    x.k[b, h, : L[b]], x.v[b, h, : L[b]], x.scale)
            assert np.array_equal(dec[(b, h)][0], out) and dec[(b, h)][1] == lse


def test_decode_clamps_and_empty():
    import numpy as np
    import plx_inputs
    x = plx_inputs.decode(2, 1, 8, 16, seed=7, seqlens=np.array([0, 99]))
    dec = oracle.decode("stream", x.q, x.rho, x.k_cache, x.v_cache, x.seqlens, x.scale)
    assert np.all(dec[(0, 0)][0] == 0) and dec[(0, 0)][1] == -np.inf
    full, lse = oracle.query("stream", x.q[1, 0], x.rho[1, 0], x.k_cache[1, 0], x.v_cache[1, 0],
                             x.scale)
    assert np.array_equal(dec[(1, 0)][0], full)


def test_worked_examples():
    """Hand-derived exact answers (tests/golden/worked_examples.json)."""
    import json
    import os
    import numpy as np
    path = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
    for case in json.load(open(path))["cases"]:
        for form in ("explicit", "stream"):
            out, lse = oracle.query(form, case["q"], case["rho"], np.array(case["k"], float),
                                    np.array(case["v"], float), case["scale"])
            assert np.allclose(out, case["out"], rtol=0, atol=1e-14), (case["name"], form, out)
            assert abs(lse - case["lse"]) < 1e-14, (case["name"], form, lse)
