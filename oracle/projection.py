"""fp64 probe projection rho = W_R x -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU legs
may import this module.  It shares no code with the CUDA library.

"Parallax: Parameterized Local Linear Attention for Language Modeling"
(zhichai.net section 1.3) draws each token's probe from the layer input by a
learned linear map, rho_i = W_R x_i; the attention then splits the result into
heads like q, k and v.  Written out per output element:

    rho[b, h, n, j] = sum_k W_R[h d + j, k] x[b, n, k]

with W_R of shape [H d, Dx] (head h owns rows h d .. h d + d - 1) and x of
shape [B, N, Dx].  The sum is one numpy matrix product in float64 (a library
primitive); the head split is a reshape and a transpose.

Pins (tests/test_oracle_projection.py): a pure-Python triple loop on tiny
inputs, the identity projection (W_R = I gives the head split of x itself),
a one-hot W_R that picks single input columns, and linearity in x.
"""
from __future__ import annotations

import numpy as np


def probe_projection(x, w_r, heads: int) -> np.ndarray:
    """rho [B, H, N, d] (float64) from x [B, N, Dx] and W_R [H d, Dx]."""
    x = np.asarray(x, dtype=np.float64)
    w_r = np.asarray(w_r, dtype=np.float64)
    B, N, Dx = x.shape
    Hd, Dw = w_r.shape
    if Dw != Dx or Hd % heads != 0:
        raise ValueError("W_R must be [H d, Dx] with Dx the width of x")
    d = Hd // heads
    y = x.reshape(B * N, Dx) @ w_r.T                      # [B N, H d]: y[t, h d + j]
    return np.ascontiguousarray(y.reshape(B, N, heads, d).transpose(0, 2, 1, 3))


def probe_projection_rows(x, w_r, heads: int, b: int, rows) -> np.ndarray:
    """rho[b, :, rows, :] (float64, shape [H, len(rows), d]) for a few tokens
    of batch b: the same product restricted to those tokens."""
    xs = np.asarray(x[b, rows], dtype=np.float64)[None]    # [1, R, Dx]
    return probe_projection(xs, w_r, heads)[0]
