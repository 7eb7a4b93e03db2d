"""plx_lla_f32 (local linear attention, probe solved by fp32 conjugate
gradients on the GPU) against the fp64 LLA oracle (oracle/lla.py).

Three kinds of check:
- iteration-matched: tol = 0 and a few steps, so the GPU and the oracle's
  textbook CG take the same steps; o and rho must agree to fp32 accuracy;
- converged: a tight tolerance, against the oracle's dense solve;
- residual (any size): for every sampled row the GPU reports converged, the
  fp64 residual |(S + lambda I) rho_gpu - mu| of the oracle's own system is
  within the tolerance (plus fp32 slack), and |o_gpu - o_direct| stays within
  what that residual allows, |C| |r| / lambda_min(S + lambda I)."""
import numpy as np
import pytest

import plx_inputs
from oracle import lla
from parity import assert_f32

pytestmark = pytest.mark.gpu


def run_lla(x, lam, max_iters, tol, keep_weights=False):
    import torch
    import parameterized_local_linear_02_b300 as plx
    t = {n: torch.from_numpy(getattr(x, n)).to("cuda") for n in ("q", "k", "v")}
    out, rho, lse, steps = plx.plx_lla_f32(t["q"], t["k"], t["v"], lam=lam, max_iters=max_iters, tol=tol,
                                           scale=x.scale, keep_weights=keep_weights)
    torch.cuda.synchronize()
    assert plx.plx_last_device_error() == 0
    return out.cpu().numpy(), rho.cpu().numpy(), lse.cpu().numpy(), steps.cpu().numpy()


def inputs(B, H, N, d, seed):
    return plx_inputs.prefill(B, H, N, d, seed=seed, dtype="f32", rho="zero")


def tensor_steps(N, d):
    """With the weights kept, the CG steps after the first run on the tensor
    cores (split tf32) for d in {64, 128} and N % 4 == 0 (the weight rows are
    read by TMA, whose row stride must be a multiple of 16 bytes)."""
    return d in (64, 128) and N % 4 == 0


@pytest.mark.parametrize("shape,lam", [((1, 2, 70, 64), 0.1), ((2, 1, 129, 128), 0.05), ((1, 1, 1, 32), 0.1),
                                       ((1, 1, 40, 96), 0.5),
                                       # the block-GEMM step (d = 64, 128) on one partial tile
                                       ((1, 1, 1, 128), 0.1), ((2, 3, 5, 64), 0.2), ((1, 2, 64, 128), 0.1)])
@pytest.mark.parametrize("keep", [False, True])
def test_lla_iteration_matched(shape, lam, keep):
    """tol = 0, 3 steps.  Rows with a prefix of at least 9 keys take all 3
    steps in both precisions and must match the fp64 CG to fp32 accuracy.
    Rows with fewer keys have at most a few distinct eigenvalues, so CG has
    solved them exactly after 1 or 2 steps.  A further step then divides fp32
    rounding noise by lambda; in fp64 that noise is invisible.  That is the
    precision sensitivity of CG the pages warn about.  Those rows are checked
    against the direct solve, within the bound their residual allows.
    keep: the weights kept by the first step, the later steps on the tensor
    cores where tensor_steps(N, d)."""
    B, H, N, d = shape
    x = inputs(B, H, N, d, seed=N + d)
    iters = 3
    out, rho, _, steps = run_lla(x, lam, iters, 0.0, keep_weights=keep)
    ref = lla.lla_cg(x.q, x.k, x.v, x.scale, lam, max_iters=iters)
    for (b, h), (o_ref, rho_ref, rows, st) in ref.items():
        assert np.all(steps[b, h] <= iters) and np.all(steps[b, h][8:] == iters)
        if N > 8:
            assert_f32(out[b, h][8:], o_ref[8:], f"{shape} o", tol=2e-4)
            assert_f32(rho[b, h][8:], rho_ref[8:], f"{shape} rho", tol=1e-3)
    early = list(range(min(N, 8)))
    _residual_checks(x, out, rho, steps, lam, 0.0, iters, None, early)


EPS32 = 2.0 ** -24


def _residual_checks(x, out, rho, steps, lam, tol, max_iters, heads, rows):
    """Per row: the fp64 residual of the GPU's rho in the oracle's system, and
    |o_gpu - o_direct| against what that residual allows.  fp32 slack: CG's
    recursive residual drifts from the true one by about
    eps (|S| |rho| + sum_j w_j |k_j . rho| |k_j| + |mu|), per step and per
    accumulated key; the output pass cancels terms of size |rho| |k| |v|."""
    q, k, v = (np.asarray(a, np.float64) for a in (x.q, x.k, x.v))
    direct = lla.lla_direct(q, k, v, x.scale, lam, heads=heads, rows=rows)
    n_conv = 0
    for (b, h), (o_ref, rho_ref, rr) in direct.items():
        for n, i in enumerate(rr):
            i = int(i)
            K, V, qi = k[b, h, : i + 1], v[b, h, : i + 1], q[b, h, i]
            s = x.scale * K @ qi
            w = np.exp(s - s.max())
            w /= w.sum()
            kc, vc = K - w @ K, V - w @ V
            S = (kc * w[:, None]).T @ kc + lam * np.eye(q.shape[-1])
            C = (vc * w[:, None]).T @ kc
            mu = w @ K - qi
            rg = rho[b, h, i]
            res = float(np.linalg.norm(S @ rg - mu))
            grow = 64 * EPS32 * (np.sqrt(i + 1.0) + 1.0)
            s_norm = float(np.linalg.norm(S, 2))
            # the kernels form Sigma p as sum_j w_j ((k_j . p) - (kbar . p)) k_j: the
            # scalar difference cancels terms of size |k_j . p|, so rounding enters
            # at that scale, not at |Sigma p|
            kbar = w @ K
            cancel = float(w @ ((np.abs(K @ rg) + abs(kbar @ rg)) * np.linalg.norm(K, axis=1)))
            if steps[b, h, i] < max_iters:
                n_conv += 1
                lim = tol * np.linalg.norm(mu) + grow * (s_norm * np.linalg.norm(rg) + cancel + np.linalg.norm(mu))
                assert res <= lim, f"row ({b},{h},{i}): residual {res:.3e} > {lim:.3e}"
            lmin = float(np.linalg.eigvalsh(S)[0])
            kmax = float(np.max(np.linalg.norm(K, axis=1)))
            vmax = float(np.max(np.linalg.norm(V, axis=1)))
            bound = np.linalg.norm(C, 2) * res / lmin + grow * (1.0 + np.linalg.norm(rg) * kmax) * vmax
            err = float(np.linalg.norm(out[b, h, i] - o_ref[n]))
            assert err <= bound, f"row ({b},{h},{i}): |o - o*| {err:.3e} > {bound:.3e}"
    return n_conv


@pytest.mark.parametrize("shape,lam", [((1, 2, 70, 64), 0.1), ((2, 1, 129, 128), 0.05), ((1, 1, 40, 32), 0.02),
                                       ((2, 1, 132, 128), 0.05), ((1, 2, 200, 64), 0.1)])
@pytest.mark.parametrize("keep", [False, True])
def test_lla_converged_matches_direct_solve(shape, lam, keep):
    B, H, N, d = shape
    x = inputs(B, H, N, d, seed=3 * N + d)
    tol, iters = 1e-5, 4 * d
    out, rho, _, steps = run_lla(x, lam, iters, tol, keep_weights=keep)
    n_conv = _residual_checks(x, out, rho, steps, lam, tol, iters, None, None)
    assert n_conv == B * H * N, f"only {n_conv} of {B * H * N} rows converged"
    ref = lla.lla_direct(x.q, x.k, x.v, x.scale, lam)
    for (b, h), (o_ref, rho_ref, rows) in ref.items():
        assert_f32(out[b, h], o_ref, f"{shape} o vs direct solve", tol=1e-3)


@pytest.mark.parametrize("shape,lam", [((1, 2, 200, 64), 1.0), ((1, 1, 160, 128), 0.5)])
@pytest.mark.parametrize("keep", [False, True])
def test_lla_well_conditioned_matches_direct_solve_at_fp32_tolerance(shape, lam, keep):
    """With a ridge that keeps (Sigma_KK + lambda I) well conditioned (lambda
    of the order of the key variance), the converged fp32 CG output meets the
    fp32 path's tolerance, 1e-4 of the RMS, against the dense fp64 solve (with
    keep, the steps after the first on the tensor cores in split tf32)."""
    B, H, N, d = shape
    x = inputs(B, H, N, d, seed=5 * N + d)
    tol, iters = 1e-6, 4 * d
    out, rho, _, steps = run_lla(x, lam, iters, tol, keep_weights=keep)
    ref = lla.lla_direct(x.q, x.k, x.v, x.scale, lam)
    for (b, h), (o_ref, rho_ref, rows) in ref.items():
        mx, mn = assert_f32(out[b, h], o_ref, f"{shape} lambda {lam} o vs direct solve", tol=1e-4)
        print(f"well-conditioned LLA {shape} lambda {lam}: max {mx:.2e} mean {mn:.2e}")


def test_lla_full_size_sampled_rows():
    """The bench's LLA workload in the launch configuration the bench times:
    B=4, H=16, N=2048, d=128 fp32, lambda = 0.1, at most 48 steps, tol 1e-4
    (rows near prefix length d need the most, about 36 in fp64), the softmax
    weights kept across the steps and the steps after the first on the tensor
    cores.  Sampled rows of three heads checked by their fp64 residuals and
    against the direct solve, for that path and for the fp32 path that
    recomputes the weights in every step; lse is the same kernel's in both."""
    B, H, N, d = 4, 16, 2048, 128
    x = inputs(B, H, N, d, seed=41)
    lam, tol, iters = 0.1, 1e-4, 48
    rows = [0, 1, 2, 63, 127, 128, 129, 500, 1023, 2047]
    heads = [(0, 0), (1, 9), (3, 15)]
    lses = []
    for keep in (True, False):
        out, rho, lse, steps = run_lla(x, lam, iters, tol, keep_weights=keep)
        lses.append(lse)
        n_conv = _residual_checks(x, out, rho, steps, lam, tol, iters, heads, rows)
        assert n_conv == len(rows) * len(heads), f"{n_conv} of {len(rows) * len(heads)} sampled rows converged"
        assert int(steps.max()) < iters
        print(f"keep {keep}: steps max {int(steps.max())}, mean {float(steps.mean()):.2f}; sampled rows converged {n_conv}")
    assert np.array_equal(lses[0], lses[1])


def test_lla_large_lambda_is_softmax_attention():
    """lambda large: rho* ~ mu / lambda -> 0 and o -> softmax attention (the
    oracle's textbook softmax form), to O(1 / lambda)."""
    import oracle
    x = inputs(1, 2, 100, 64, seed=7)
    out, rho, lse, _ = run_lla(x, 1e6, 4, 0.0)
    for (b, h), (o_ref, lse_ref, rows) in oracle.prefill("sa", x.q, x.k, x.v, np.zeros_like(x.q), x.scale).items():
        assert_f32(out[b, h][rows], o_ref, f"LLA at lambda 1e6 vs softmax attention ({b}, {h})", tol=1e-4)
        assert float(np.max(np.abs(lse[b, h][rows] - lse_ref))) <= 1e-5


@pytest.mark.parametrize("shape,tol", [((2, 3, 200, 64), 1e-4), ((1, 2, 130, 128), 0.0), ((3, 1, 70, 128), 1e-3),
                                       ((1, 1, 1, 64), 0.0), ((1, 2, 132, 128), 0.0), ((2, 2, 260, 128), 1e-4),
                                       ((1, 1, 4, 128), 0.0),
                                       # every row stops before its first step: no weights are stored
                                       ((1, 2, 90, 128), 2.0), ((1, 2, 92, 128), 2.0)])
def test_lla_kept_weights(shape, tol):
    """With a workspace of plx_lla_kept_weights_workspace_size the CG steps
    read the softmax weights the first step stored instead of recomputing them.
    - N % 4 != 0: the block step reads them (the same values in the same
      operations), so out, rho, lse and the step counts are the recomputing
      path's, bit for bit (rows that stop early included: tol > 0);
    - N % 4 == 0 (d = 64, 128): the steps after the first run on the tensor
      cores in split tf32.  lse (the same kernel) is equal bit for bit, and
      every row passes the oracle's residual checks (converged rows within
      tol, every output within what its fp64 residual allows)."""
    import parameterized_local_linear_02_b300 as plx
    B, H, N, d = shape
    assert plx.plx_lla_kept_weights_workspace_size(B, H, N, d) == (
        plx.plx_lla_workspace_size(B, H, N, d) + ((B * H * N * N * 4 + 255) // 256) * 256)
    x = inputs(B, H, N, d, seed=50 + N)
    iters = 12
    a = run_lla(x, 0.1, iters, tol, keep_weights=True)
    b = run_lla(x, 0.1, iters, tol)
    if not tensor_steps(N, d) or tol >= 2.0:
        for got, ref, name in zip(a, b, ("out", "rho", "lse", "steps")):
            assert np.array_equal(got, ref), name
        return
    out, rho, lse, steps = a
    assert np.array_equal(lse, b[2])
    assert np.all(steps <= iters)
    _residual_checks(x, out, rho, steps, 0.1, tol, iters, None, None)
