"""Error metric and tolerances for GPU-vs-oracle parity.

Errors are |gpu - oracle| element by element, divided by the RMS of the
oracle output over the compared elements.  Tolerances: bf16 inputs with fp32
accumulation, max <= 2e-2 and mean <= 2e-3; the fp32 path, max and mean
<= 1e-4.  lse (natural log) is compared in absolute terms: 1e-3 for the bf16
tensor-core path, 1e-5 for fp32 arithmetic."""
import numpy as np

BF16_MAX, BF16_MEAN = 2e-2, 2e-3
F32_TOL = 1e-4
LSE_BF16, LSE_F32 = 1e-3, 1e-5


def rel_errors(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "non-finite GPU output"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    d = np.abs(got - ref)
    return float(d.max()) / rms, float(d.mean()) / rms


def assert_bf16(got, ref, what=""):
    mx, mn = rel_errors(got, ref)
    assert mx <= BF16_MAX and mn <= BF16_MEAN, f"{what}: max {mx:.2e} mean {mn:.2e} (rel. to RMS)"
    return mx, mn


def assert_bf16_output(got, ref, what=""):
    """bf16 tolerance plus the rounding of the output itself to bf16 (unit
    roundoff 2^-8 of each element's magnitude), for results stored as bf16."""
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2)))
    mx, mn = rel_errors(got, ref)
    tmax = BF16_MAX + 2.0 ** -8 * float(np.max(np.abs(ref))) / rms
    tmean = BF16_MEAN + 2.0 ** -8 * float(np.mean(np.abs(ref))) / rms
    assert mx <= tmax and mn <= tmean, f"{what}: max {mx:.2e} (tol {tmax:.2e}) mean {mn:.2e} (tol {tmean:.2e})"
    return mx, mn


def assert_f32(got, ref, what="", tol=F32_TOL):
    mx, mn = rel_errors(got, ref)
    assert mx <= tol and mn <= tol, f"{what}: max {mx:.2e} mean {mn:.2e} (rel. to RMS)"
    return mx, mn


def assert_lse(got, ref, tol, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):          # -inf - -inf where both rows are empty
        err = np.where(both_inf, 0.0, np.abs(got - ref))
    assert float(err.max()) <= tol, f"{what}: lse max abs err {float(err.max()):.2e}"


SENTINEL = -768.0      # exact in fp32, bf16 and fp16; no kernel output here takes it


def canary(shape, dtype, guard=1024):
    """A device tensor of ``shape`` filled with NaN (so an element the kernel
    does not write shows up in the comparison), inside a buffer whose
    ``guard`` elements before and after hold SENTINEL.  Returns
    ``(tensor, intact)``; ``intact()`` is True while no write has left the
    tensor.  Integer dtypes (workspaces) are filled with 0xFF bytes instead of
    NaN."""
    import torch
    n = int(np.prod(shape))
    if dtype.is_floating_point:
        buf = torch.full((n + 2 * guard,), float("nan"), dtype=dtype, device="cuda")
        sent = torch.tensor(SENTINEL, dtype=dtype, device="cuda")
    else:
        buf = torch.full((n + 2 * guard,), 0xFF, dtype=dtype, device="cuda")
        sent = torch.tensor(0x5A, dtype=dtype, device="cuda")
    buf[:guard] = sent
    buf[guard + n:] = sent
    view = buf[guard:guard + n].view(shape)

    def intact():
        return bool(torch.all(buf[:guard] == sent)) and bool(torch.all(buf[guard + n:] == sent))
    return view, intact
