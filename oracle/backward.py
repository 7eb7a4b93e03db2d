"""fp64 gradients of causal PLX attention -- TEST INFRASTRUCTURE.

Only the test suite may import this module.  It shares no code with the CUDA
library.

The forward is the explicit form of "Parallax: Parameterized Local Linear
Attention for Language Modeling" (zhichai.net section 1.3; gist.science
"Meccanismo Principale"): for each query i,
    w_i = softmax_{j <= i}(scale q_i . k_j),  vbar_i = sum_j w_ij v_j,
    kbar_i = sum_j w_ij k_j,
    Sigma_i = sum_j w_ij (v_j - vbar_i)(k_j - kbar_i)^T   (d x d, built explicitly),
    o_i = vbar_i - Sigma_i rho_i.
It is written in torch double-precision tensor operations on the CPU, and
torch's reverse-mode automatic differentiation (a library routine) gives the
gradients of L = sum_i dO_i . o_i with respect to q, k, v and rho.  The pages
do not derive a backward pass; this is the plain definition differentiated.

Pins (tests/test_oracle_backward.py): central finite differences of the
independent C oracle's explicit forward, the value-shift invariant
sum_j dL/dv_j = sum_i dO_i, and the affinity of o in rho (dL/drho does not
depend on rho; the other gradients are affine in it).

``plx_backward_closed`` is a second, independent route for long sequences,
where the explicit form's [N, N, d] intermediates do not fit: the gradients
written out in closed form (the forward differentiated by hand, on dense
N x N fp64 matrices with numpy), pinned against ``plx_backward``.
"""
from __future__ import annotations

import numpy as np


def _forward_head(q, k, v, rho, scale):
    import torch
    N = q.shape[0]
    s = scale * (q @ k.T)
    mask = torch.ones(N, N, dtype=torch.bool).tril()
    s = s.masked_fill(~mask, float("-inf"))
    w = torch.softmax(s, dim=1)                                  # w_ij, zero for j > i
    vbar = w @ v
    kbar = w @ k
    vc = v[None, :, :] - vbar[:, None, :]                        # v_j - vbar_i   [i, j, d]
    kc = k[None, :, :] - kbar[:, None, :]                        # k_j - kbar_i   [i, j, d]
    sigma = torch.einsum("ij,ija,ijb->iab", w, vc, kc)           # d_v x d_k per query
    return vbar - torch.einsum("iab,ib->ia", sigma, rho)


def plx_backward(q, k, v, rho, dout, scale):
    """Gradients of L = sum(dout * o) for every (b, h).  Arrays [B, H, N, d];
    returns (dq, dk, dv, drho) as float64 numpy arrays, and o."""
    import torch
    B, H, N, d = q.shape
    outs = [np.zeros((B, H, N, d)) for _ in range(4)]
    o_all = np.zeros((B, H, N, d))
    for b in range(B):
        for h in range(H):
            tq, tk, tv, tr = (torch.tensor(np.asarray(a[b, h], np.float64), requires_grad=True)
                              for a in (q, k, v, rho))
            o = _forward_head(tq, tk, tv, tr, float(scale))
            L = (o * torch.tensor(np.asarray(dout[b, h], np.float64))).sum()
            grads = torch.autograd.grad(L, (tq, tk, tv, tr))
            for n in range(4):
                outs[n][b, h] = grads[n].numpy()
            o_all[b, h] = o.detach().numpy()
    return (*outs, o_all)


def plx_backward_closed(q, k, v, rho, dout, scale, heads=None):
    """Gradients of L = sum(dout * o) in closed form, fp64 numpy, for the
    listed (b, h) heads (all by default).  With s = scale q k^T, w = the causal
    softmax of s, r = rho k^T, vbar = w v, c_i = sum_j w_ij r_ij,
    o = (1 + c) vbar - (w o r) v, G = dO v^T, a_i = dO_i . vbar_i and
    D_i = dO_i . o_i + c_i a_i:
        dL/ds = w o ((1 + c - r) o G + a r - D),   dL/dr = w o (a - G),
        dq = scale (dL/ds) k,  drho = (dL/dr) k,
        dk = scale (dL/ds)^T q + (dL/dr)^T rho,  dv = (w o (1 + c - r))^T dO.
    Returns {(b, h): (dq, dk, dv, drho)}."""
    B, H, N, d = q.shape
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    tril = np.tril(np.ones((N, N), dtype=bool))
    res = {}
    for b, h in heads:
        Q, K, V, R, dO = (np.asarray(a[b, h], np.float64) for a in (q, k, v, rho, dout))
        s = scale * (Q @ K.T)
        s = np.where(tril, s, -np.inf)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        r = R @ K.T
        vbar = w @ V
        c = np.sum(w * r, axis=1, keepdims=True)
        o = (1.0 + c) * vbar - (w * r) @ V
        G = dO @ V.T
        a = np.sum(dO * vbar, axis=1, keepdims=True)
        D = np.sum(dO * o, axis=1, keepdims=True) + c * a
        ds = w * ((1.0 + c - r) * G + a * r - D)
        dr = w * (a - G)
        dq = scale * (ds @ K)
        drho = dr @ K
        dk = scale * (ds.T @ Q) + dr.T @ R
        dv = (w * (1.0 + c - r)).T @ dO
        res[(b, h)] = (dq, dk, dv, drho)
    return res
