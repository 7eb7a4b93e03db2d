"""Seeded synthetic inputs for the PLX attention hot path.

This module is shared by the fp64 oracle's tests and by the CUDA path's tests
and benchmark.  It draws random numbers and rounds them to the storage type;
it holds none of the attention arithmetic.

Workload recipes (shapes and distributions follow the workloads of
"Parallax: Parameterized Local Linear Attention for Language Modeling",
arXiv:2605.29157, as summarised by gist.science, "Meccanismo Principale"):

* ``prefill``: q, k, v ~ N(0, 1) in layout [B, H, N, d] (d contiguous).
  The probe rho is one of
    - ``"normal"``: rho ~ N(0, rho_std^2) per token per head;
    - ``"proj"``: rho = W_R x with x ~ N(0, 1) of width ``x_width`` per token
      and W_R ~ N(0, 1/x_width) of shape [H*d, x_width] (the learned probe
      projection of the layer input, drawn at random);
    - ``"zero"``: rho = 0 (plain softmax attention).
  Keys are either ``"normal"`` or ``"planted"``: per (b, h), 64 centres
  kappa_c ~ N(0, I_d), every position j draws z_j ~ U{0..63} and
  k_j = kappa_{z_j} + 0.05 * eps_j, so the softmax weights are peaked and the
  covariance branch is non-trivial.
* ``decode``: q, rho [B, H, d]; k_cache, v_cache [B, H, S_cap, d]; q, k, v ~
  N(0, 1), rho ~ N(0, rho_std^2); seqlens either all S_cap (``"full"``) or
  drawn uniformly from [ctx/2, ctx] (``"ragged"``).

Host generation uses numpy's PCG64 stream seeded by ``seed`` and draws the
tensors in a fixed order.  Large decode caches can instead be drawn on a CUDA
device with torch's seeded Philox generator (``decode_device``); the oracle
then reads slices copied back to the host.

bf16 inputs are rounded once, round-to-nearest-even, and the oracle receives
exactly the rounded values (widened), so input quantisation is never counted
as kernel error.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "bf16_round", "bf16_bits_to_f32", "PrefillInputs", "DecodeInputs",
    "prefill", "decode", "decode_device", "ragged_seqlens", "CONFIGS",
    "ProbeInputs", "probe",
]


def bf16_round(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Round to bf16 (round-to-nearest-even via fp32).

    Returns ``(bits, values)``: the uint16 bit patterns and the rounded values
    widened back to float32 (exact)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    bits = ((u + bias) >> np.uint32(16)).astype(np.uint16)
    return bits, bf16_bits_to_f32(bits)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class PrefillInputs:
    B: int
    H: int
    N: int
    d: int
    dtype: str                     # "bf16" or "f32": storage type on the device
    scale: float
    q: np.ndarray                  # float32 values [B,H,N,d] (bf16-exact if dtype == "bf16")
    k: np.ndarray
    v: np.ndarray
    rho: np.ndarray
    bits: dict = field(default_factory=dict)   # uint16 bf16 patterns when dtype == "bf16"

    def device_tensors(self, device="cuda"):
        """torch tensors on ``device`` in the storage dtype, [B,H,N,d] contiguous."""
        import torch
        out = {}
        for name in ("q", "k", "v", "rho"):
            if self.dtype == "bf16":
                t = torch.from_numpy(self.bits[name].view(np.int16)).view(torch.bfloat16)
            else:
                t = torch.from_numpy(getattr(self, name))
            out[name] = t.to(device).contiguous()
        return out


@dataclass
class DecodeInputs:
    B: int
    H: int
    d: int
    S_cap: int
    scale: float
    q: np.ndarray          # float32 [B,H,d] (bf16-exact)
    rho: np.ndarray
    k_cache: np.ndarray    # float32 [B,H,S_cap,d] (bf16-exact)
    v_cache: np.ndarray
    seqlens: np.ndarray    # int32 [B]
    bits: dict = field(default_factory=dict)

    def device_tensors(self, device="cuda"):
        import torch
        out = {}
        for name in ("q", "rho", "k_cache", "v_cache"):
            t = torch.from_numpy(self.bits[name].view(np.int16)).view(torch.bfloat16)
            out[name] = t.to(device).contiguous()
        out["seqlens"] = torch.from_numpy(self.seqlens.astype(np.int32)).to(device)
        return out


def _normal(rng, shape, std=1.0):
    x = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def _store(x: np.ndarray, dtype: str):
    if dtype == "bf16":
        return bf16_round(x)
    if dtype == "f32":
        return None, np.ascontiguousarray(x, dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def prefill(B: int, H: int, N: int, d: int, *, seed: int, dtype: str = "bf16",
            rho: str = "normal", rho_std: float = 0.1, keys: str = "normal",
            x_width: int = 1024, scale: float | None = None,
            n_centres: int = 64, key_noise: float = 0.05) -> PrefillInputs:
    """Seeded prefill inputs, layout [B, H, N, d]."""
    rng = np.random.default_rng(seed)
    shape = (B, H, N, d)
    q = _normal(rng, shape)
    if keys == "normal":
        k = _normal(rng, shape)
    elif keys == "planted":
        centres = _normal(rng, (B, H, n_centres, d))
        z = rng.integers(0, n_centres, size=(B, H, N))
        k = np.take_along_axis(centres, z[..., None].repeat(d, axis=-1), axis=2)
        k = k + _normal(rng, shape, key_noise)
    else:
        raise ValueError(f"unknown keys {keys!r}")
    v = _normal(rng, shape)
    if rho == "normal":
        r = _normal(rng, shape, rho_std)
    elif rho == "proj":
        x = rng.standard_normal((B, N, x_width))                      # fp64
        w_r = rng.standard_normal((H * d, x_width)) / math.sqrt(x_width)
        r = (x @ w_r.T).reshape(B, N, H, d).transpose(0, 2, 1, 3)
        r = np.ascontiguousarray(r, dtype=np.float32)
    elif rho == "zero":
        r = np.zeros(shape, np.float32)
    else:
        raise ValueError(f"unknown rho {rho!r}")
    bits = {}
    vals = {}
    for name, arr in (("q", q), ("k", k), ("v", v), ("rho", r)):
        b, val = _store(arr, dtype)
        if b is not None:
            bits[name] = b
        vals[name] = val
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return PrefillInputs(B, H, N, d, dtype, float(scale), vals["q"], vals["k"],
                         vals["v"], vals["rho"], bits)


def ragged_seqlens(rng, B: int, ctx: int) -> np.ndarray:
    """Per-sequence lengths drawn uniformly from [ctx/2, ctx] (inclusive)."""
    return rng.integers(ctx // 2, ctx + 1, size=B).astype(np.int32)


def decode(B: int, H: int, d: int, S_cap: int, *, seed: int,
           seqlens: str | np.ndarray = "full", rho_std: float = 0.1,
           scale: float | None = None) -> DecodeInputs:
    """Seeded one-token decode inputs (host, bf16-rounded)."""
    rng = np.random.default_rng(seed)
    q = _normal(rng, (B, H, d))
    r = _normal(rng, (B, H, d), rho_std)
    kc = _normal(rng, (B, H, S_cap, d))
    vc = _normal(rng, (B, H, S_cap, d))
    if isinstance(seqlens, str):
        if seqlens == "full":
            sl = np.full(B, S_cap, np.int32)
        elif seqlens == "ragged":
            sl = ragged_seqlens(rng, B, S_cap)
        else:
            raise ValueError(f"unknown seqlens {seqlens!r}")
    else:
        sl = np.asarray(seqlens, np.int32)
    bits, vals = {}, {}
    for name, arr in (("q", q), ("rho", r), ("k_cache", kc), ("v_cache", vc)):
        bits[name], vals[name] = bf16_round(arr)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    return DecodeInputs(B, H, d, S_cap, float(scale), vals["q"], vals["rho"],
                        vals["k_cache"], vals["v_cache"], sl, bits)


def decode_device(B: int, H: int, d: int, S_cap: int, *, seed: int,
                  seqlens: str | np.ndarray = "full", rho_std: float = 0.1,
                  device="cuda"):
    """Seeded decode inputs drawn directly on a CUDA device (for caches too
    large to draw on the host quickly).  Uses torch's seeded Philox generator;
    every tensor is drawn in fp32 and rounded once to bf16 (RNE).

    Returns a dict of device tensors: q, rho [B,H,d] bf16; k_cache, v_cache
    [B,H,S_cap,d] bf16; seqlens int32 [B]."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = {}
    out["q"] = torch.randn((B, H, d), generator=g, device=device).to(torch.bfloat16)
    out["rho"] = (torch.randn((B, H, d), generator=g, device=device) * rho_std).to(torch.bfloat16)
    for name in ("k_cache", "v_cache"):
        t = torch.empty((B, H, S_cap, d), dtype=torch.bfloat16, device=device)
        # draw per (b) slab to bound the fp32 temporary
        for b in range(B):
            t[b].copy_(torch.randn((H, S_cap, d), generator=g, device=device))
        out[name] = t
    if isinstance(seqlens, str):
        if seqlens == "full":
            sl = np.full(B, S_cap, np.int32)
        elif seqlens == "ragged":
            sl = ragged_seqlens(np.random.default_rng(seed), B, S_cap)
        else:
            raise ValueError(f"unknown seqlens {seqlens!r}")
    else:
        sl = np.asarray(seqlens, np.int32)
    out["seqlens_host"] = sl
    out["seqlens"] = torch.from_numpy(sl).to(device)
    return out


@dataclass
class ProbeInputs:
    """Inputs of the probe projection: hidden states x [B, N, Dx] and the
    probe weights W_R [H * d, Dx], both bf16-exact float32 values."""
    B: int
    N: int
    H: int
    d: int
    Dx: int
    x: np.ndarray
    w_r: np.ndarray
    bits: dict = field(default_factory=dict)

    def device_tensors(self, device="cuda"):
        import torch
        return {name: torch.from_numpy(self.bits[name].view(np.int16)).view(torch.bfloat16).to(device).contiguous()
                for name in ("x", "w_r")}


def probe(B: int, N: int, H: int, d: int, Dx: int, *, seed: int, x_std: float = 1.0) -> ProbeInputs:
    """Seeded probe-projection inputs: x ~ N(0, x_std^2) of shape [B, N, Dx]
    and W_R ~ N(0, 1/Dx) of shape [H * d, Dx], each rounded once to bf16.
    Only the draws; the product is the oracle's."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, (B, N, Dx), x_std)
    w = _normal(rng, (H * d, Dx), 1.0 / math.sqrt(Dx))
    bits, vals = {}, {}
    for name, arr in (("x", x), ("w_r", w)):
        bits[name], vals[name] = bf16_round(arr)
    return ProbeInputs(B, N, H, d, Dx, vals["x"], vals["w_r"], bits)


# The five workloads of the benchmark/parity plan (sizes by what they are).
CONFIGS = {
    "tiny_f32": dict(kind="prefill", B=1, H=2, N=128, d=64, dtype="f32",
                     rho="normal", rho_std=0.1, keys="normal", seed=0),
    "prefill_b4_h16_n2048_d128": dict(kind="prefill", B=4, H=16, N=2048, d=128,
                                      dtype="bf16", rho="proj", keys="normal", seed=1),
    "prefill_b2_h16_n8192_d128_planted": dict(kind="prefill", B=2, H=16, N=8192, d=128,
                                              dtype="bf16", rho="normal", rho_std=0.1,
                                              keys="planted", seed=2),
    "decode_b64_h16_ctx4096_d128": dict(kind="decode", B=64, H=16, d=128, S_cap=4096,
                                        seqlens="full", rho_std=0.1, seed=3),
    "decode_sweep": dict(kind="decode_sweep", batches=(1, 8, 64, 256),
                         contexts=(2048, 8192, 32768, 131072), H=16, d=128,
                         seqlens="ragged", rho_std=0.1, seed=4),
}
