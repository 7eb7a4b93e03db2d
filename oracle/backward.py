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
