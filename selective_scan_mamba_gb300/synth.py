"""Seeded synthetic inputs, shaped like the layers the pages benchmark.

This module is the one piece shared by the CUDA path and the float64 oracle.  It
holds none of the scan's arithmetic: it only draws numbers (numpy
``default_rng(seed)``, drawn in the library's argument order) and rounds them to
the storage type the kernels read (bfloat16 with round-to-nearest-even, or
float32), so that both sides see bit-identical values.

Recipe (one seed per workload, 0 unless stated):
  * x, B, C, z, D ~ N(0, 1); the raw time step delta ~ s * N(0, 1) with s = 0.5
    ("drawn as in the tiny fp32 case") or s = 1 (130m-shaped layer);
  * delta bias b = inv_softplus(u), u = exp(U(ln 1e-3, ln 1e-1)), so that
    softplus(b) = u exactly in real arithmetic;
  * Mamba-1 A[d, n] = -(n + 1); Mamba-2 A_h = -U(1, 16);
  * decode state ~ N(0, 0.1^2) in float32.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F32 = "f32"
BF16 = "bf16"


def bf16_bits(a) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even); return the
    16-bit patterns as uint16.  Inputs are finite."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    # finite inputs stay below 0xFF800000, so the sum cannot wrap in 32 bits
    r = (u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_values(bits: np.ndarray) -> np.ndarray:
    """float32 values of bfloat16 bit patterns (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def to_storage(a, dtype: str) -> np.ndarray:
    """float32 values exactly representable in the storage type ``dtype``."""
    a = np.asarray(a, dtype=np.float32)
    if dtype == BF16:
        return bf16_values(bf16_bits(a)).reshape(a.shape)
    if dtype == F32:
        return a.copy()
    raise ValueError(f"unknown storage dtype {dtype!r}")


def inv_softplus(u):
    """The b with log(1 + e^b) = u (float64), written as u + log(-expm1(-u))."""
    u = np.asarray(u, dtype=np.float64)
    return u + np.log(-np.expm1(-u))


def _bias(rng, n):
    u = np.exp(rng.uniform(math.log(1e-3), math.log(1e-1), size=n))
    return inv_softplus(u).astype(np.float32)


@dataclass
class Inputs:
    """Arrays in the library's layouts.  ``arrays`` maps argument names to float32
    numpy arrays whose values are exact in the storage type given by ``dtypes``
    (absent optional arguments are simply missing)."""
    kind: str
    dims: dict
    arrays: dict = field(default_factory=dict)
    dtypes: dict = field(default_factory=dict)

    def f64(self, name):
        a = self.arrays.get(name)
        return None if a is None else a.astype(np.float64)


def mamba1(batch, dim, dstate, seqlen, *, dtype=BF16, delta_scale=0.5, with_z=False,
           with_D=True, ngroups=1, with_h0=False, seed=0) -> Inputs:
    """Mamba-1 scan inputs.  x, delta, z: [batch, dim, L]; B, C: [batch, G, N, L];
    A: [dim, N]; D, delta_bias: [dim]; h0: [batch, dim, N]."""
    rng = np.random.default_rng(seed)
    inp = Inputs("mamba1", dict(batch=batch, dim=dim, dstate=dstate, seqlen=seqlen,
                                ngroups=ngroups))
    a = inp.arrays
    a["x"] = to_storage(rng.standard_normal((batch, dim, seqlen), np.float32), dtype)
    a["delta"] = to_storage(delta_scale * rng.standard_normal((batch, dim, seqlen), np.float32),
                            dtype)
    a["delta_bias"] = _bias(rng, dim)
    a["A"] = np.tile(-np.arange(1, dstate + 1, dtype=np.float32), (dim, 1))
    a["B"] = to_storage(rng.standard_normal((batch, ngroups, dstate, seqlen), np.float32), dtype)
    a["C"] = to_storage(rng.standard_normal((batch, ngroups, dstate, seqlen), np.float32), dtype)
    if with_D:
        a["D"] = rng.standard_normal(dim).astype(np.float32)
    if with_z:
        a["z"] = to_storage(rng.standard_normal((batch, dim, seqlen), np.float32), dtype)
    if with_h0:
        a["h0"] = rng.standard_normal((batch, dim, dstate)).astype(np.float32)
    for k in ("x", "delta", "B", "C", "z"):
        if k in a:
            inp.dtypes[k] = dtype
    for k in ("delta_bias", "A", "D", "h0"):
        if k in a:
            inp.dtypes[k] = F32
    return inp


def ssd(batch, seqlen, nheads, headdim, dstate, ngroups=1, *, dtype=BF16, delta_scale=0.5,
        with_z=False, with_D=True, with_h0=False, seed=0) -> Inputs:
    """Mamba-2 SSD inputs.  x, z: [batch, L, H, P]; dt: [batch, L, H];
    B, C: [batch, L, G, N]; A, D, dt_bias: [H]; h0: [batch, H, P, N]."""
    rng = np.random.default_rng(seed)
    inp = Inputs("ssd", dict(batch=batch, seqlen=seqlen, nheads=nheads, headdim=headdim,
                             dstate=dstate, ngroups=ngroups))
    a = inp.arrays
    a["x"] = to_storage(rng.standard_normal((batch, seqlen, nheads, headdim), np.float32), dtype)
    a["dt"] = to_storage(delta_scale * rng.standard_normal((batch, seqlen, nheads), np.float32),
                         dtype)
    a["dt_bias"] = _bias(rng, nheads)
    a["A"] = (-rng.uniform(1.0, 16.0, size=nheads)).astype(np.float32)
    a["B"] = to_storage(rng.standard_normal((batch, seqlen, ngroups, dstate), np.float32), dtype)
    a["C"] = to_storage(rng.standard_normal((batch, seqlen, ngroups, dstate), np.float32), dtype)
    if with_D:
        a["D"] = rng.standard_normal(nheads).astype(np.float32)
    if with_z:
        a["z"] = to_storage(rng.standard_normal((batch, seqlen, nheads, headdim), np.float32),
                            dtype)
    if with_h0:
        a["h0"] = rng.standard_normal((batch, nheads, headdim, dstate)).astype(np.float32)
    for k in ("x", "dt", "B", "C", "z"):
        if k in a:
            inp.dtypes[k] = dtype
    for k in ("dt_bias", "A", "D", "h0"):
        if k in a:
            inp.dtypes[k] = F32
    return inp


def step_params(nheads, dstate, *, a_per_state=False, with_D=True, seed=0) -> Inputs:
    """Per-layer decode parameters: A ([H] or [H, N]), D and dt_bias ([H]) and the
    initial state scale.  Per-step tensors come from :func:`step_tokens`."""
    rng = np.random.default_rng(seed)
    inp = Inputs("step_params", dict(nheads=nheads, dstate=dstate, a_per_state=a_per_state))
    a = inp.arrays
    a["dt_bias"] = _bias(rng, nheads)
    if a_per_state:
        a["A"] = np.tile(-np.arange(1, dstate + 1, dtype=np.float32), (nheads, 1))
    else:
        a["A"] = (-rng.uniform(1.0, 16.0, size=nheads)).astype(np.float32)
    if with_D:
        a["D"] = rng.standard_normal(nheads).astype(np.float32)
    for k in a:
        inp.dtypes[k] = F32
    return inp


def step_state(batch, nheads, headdim, dstate, *, scale=0.1, seed=0) -> np.ndarray:
    """Initial decode state [batch, H, P, N] ~ N(0, scale^2), float32."""
    rng = np.random.default_rng((seed, 1))
    return (scale * rng.standard_normal((batch, nheads, headdim, dstate))).astype(np.float32)


def step_tokens(batch, nheads, headdim, dstate, ngroups=1, *, step=0, dtype=BF16,
                delta_scale=0.5, with_z=True, seed=0) -> Inputs:
    """Inputs of decode step ``step``: x, z [batch, H, P]; dt [batch, H];
    B, C [batch, G, N].  Each step has its own stream (seed, 2, step)."""
    rng = np.random.default_rng((seed, 2, step))
    inp = Inputs("step_tokens", dict(batch=batch, nheads=nheads, headdim=headdim, dstate=dstate,
                                     ngroups=ngroups, step=step))
    a = inp.arrays
    a["x"] = to_storage(rng.standard_normal((batch, nheads, headdim), np.float32), dtype)
    a["dt"] = to_storage(delta_scale * rng.standard_normal((batch, nheads), np.float32), dtype)
    a["B"] = to_storage(rng.standard_normal((batch, ngroups, dstate), np.float32), dtype)
    a["C"] = to_storage(rng.standard_normal((batch, ngroups, dstate), np.float32), dtype)
    if with_z:
        a["z"] = to_storage(rng.standard_normal((batch, nheads, headdim), np.float32), dtype)
    for k in a:
        inp.dtypes[k] = dtype
    return inp


# The five workloads (shapes of Mamba-130m/790m and Mamba2-130m/780m layers).
WORKLOADS = {
    "m1_tiny_f32": dict(kind="mamba1", batch=1, dim=64, dstate=16, seqlen=256, dtype=F32,
                        delta_scale=0.5, with_z=False),
    "m1_130m_layer": dict(kind="mamba1", batch=8, dim=1536, dstate=16, seqlen=2048, dtype=BF16,
                          delta_scale=1.0, with_z=True),
    "m1_790m_long": dict(kind="mamba1", batch=1, dim=3072, dstate=16,
                         seqlens=(1024, 4096, 16384, 32768), dtype=BF16, delta_scale=0.5,
                         with_z=False),
    "ssd_130m": dict(kind="ssd", batch=4, seqlen=4096, nheads=24, headdim=64, dstate=128,
                     ngroups=1, chunks=(64, 256), dtype=BF16, delta_scale=0.5, with_z=False),
    "step_780m": dict(kind="step", batch=64, nheads=48, headdim=64, dstate=128, ngroups=1,
                      steps=1024, dtype=BF16, delta_scale=0.5, with_z=True, state_scale=0.1),
}
