"""Pins of the fp64 probe-projection oracle (oracle/projection.py), on the CPU.

rho = W_R x ("Parallax: Parameterized Local Linear Attention for Language
Modeling", zhichai.net section 1.3), split into heads like the attention's
q, k, v.  Pinned by a scalar brute force on tiny inputs, the identity and
one-hot projections (whose results are slices of x), and linearity; each
plausible mistake planted in a copy of the oracle fails at least one pin."""
import types

import numpy as np
import pytest

from oracle import projection


def brute_force(x, w_r, H):
    """rho[b][h][n][j] = sum_k W_R[h d + j][k] x[b][n][k], one scalar at a time."""
    B, N, Dx = x.shape
    d = w_r.shape[0] // H
    out = np.zeros((B, H, N, d))
    for b in range(B):
        for h in range(H):
            for n in range(N):
                for j in range(d):
                    s = 0.0
                    for k in range(Dx):
                        s += float(w_r[h * d + j, k]) * float(x[b, n, k])
                    out[b, h, n, j] = s
    return out


def pin_brute_force(fn):
    rng = np.random.default_rng(5)
    for (B, N, H, d, Dx) in [(2, 3, 2, 2, 5), (1, 4, 3, 3, 2), (2, 1, 1, 4, 7)]:
        x = rng.standard_normal((B, N, Dx))
        w = rng.standard_normal((H * d, Dx))
        np.testing.assert_allclose(fn(x, w, H), brute_force(x, w, H), rtol=1e-12, atol=1e-12)


def pin_identity(fn):
    """W_R = I (Dx = H d): rho is x split into heads, rho[b, h, n, j] = x[b, n, h d + j]."""
    rng = np.random.default_rng(6)
    B, N, H, d = 2, 5, 3, 4
    x = rng.standard_normal((B, N, H * d))
    rho = fn(x, np.eye(H * d), H)
    for h in range(H):
        np.testing.assert_array_equal(rho[:, h], x[:, :, h * d:(h + 1) * d])


def pin_one_hot(fn):
    """Row h d + j of W_R picks input column perm[h d + j]: the result is that column."""
    rng = np.random.default_rng(7)
    B, N, H, d, Dx = 2, 3, 2, 3, 9
    perm = rng.permutation(Dx)[:H * d]
    w = np.zeros((H * d, Dx))
    w[np.arange(H * d), perm] = 1.0
    x = rng.standard_normal((B, N, Dx))
    rho = fn(x, w, H)
    for h in range(H):
        for j in range(d):
            np.testing.assert_array_equal(rho[:, h, :, j], x[:, :, perm[h * d + j]])


def pin_linear(fn):
    rng = np.random.default_rng(8)
    B, N, H, d, Dx = 2, 4, 2, 3, 6
    x1, x2 = rng.standard_normal((2, B, N, Dx))
    w = rng.standard_normal((H * d, Dx))
    np.testing.assert_allclose(fn(2.5 * x1 + x2, w, H), 2.5 * fn(x1, w, H) + fn(x2, w, H), rtol=1e-12, atol=1e-12)


PINS = [pin_brute_force, pin_identity, pin_one_hot, pin_linear]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(projection.probe_projection)


def test_rows_helper_matches_full():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, 7, 5))
    w = rng.standard_normal((6, 5))
    full = projection.probe_projection(x, w, 3)
    rows = [0, 3, 6]
    np.testing.assert_array_equal(projection.probe_projection_rows(x, w, 3, 1, rows), full[1][:, rows])


MUTANTS = {
    "head_and_dim_interleaved": ("y.reshape(B, N, heads, d).transpose(0, 2, 1, 3)",
                                 "y.reshape(B, N, d, heads).transpose(0, 3, 1, 2)"),
    "token_major_memory_read_as_head_major": ("y.reshape(B, N, heads, d).transpose(0, 2, 1, 3)",
                                              "y.reshape(B, heads, N, d)"),
    "weights_reinterpreted_not_transposed": ("@ w_r.T", "@ w_r.reshape(Dx, Hd)"),
    "tokens_of_batches_mixed": ("x.reshape(B * N, Dx) @ w_r.T",
                                "x.transpose(1, 0, 2).reshape(B * N, Dx) @ w_r.T"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    old, new = MUTANTS[name]
    src = open(projection.__file__).read()
    assert src.count(old) == 1, f"mutant anchor for {name} not unique"
    mod = types.ModuleType(f"projection_{name}")
    exec(compile(src.replace(old, new), f"<mutant {name}>", "exec"), mod.__dict__)
    caught = 0
    for pin in PINS:
        try:
            pin(mod.probe_projection)
        except (AssertionError, ValueError):
            caught += 1
    assert caught >= 1, f"mutant {name} passed every pin"
