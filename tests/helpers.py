"""Shared test helpers: move seeded synthetic inputs to the GPU, and the parity metric."""
import numpy as np

from selective_scan_mamba_gb300 import synth


def to_device(inp, names=None):
    """CUDA torch tensors holding exactly the values in ``inp`` (bf16 bit-exact)."""
    import torch
    out = {}
    for k, v in inp.arrays.items():
        if names is not None and k not in names:
            continue
        if inp.dtypes[k] == synth.BF16:
            bits = synth.bf16_bits(v).view(np.int16)
            out[k] = torch.from_numpy(bits.copy()).cuda().view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda()
    return out


def to_numpy(t):
    import torch
    return t.detach().to(torch.float32).cpu().numpy().astype(np.float64)


def max_rel_err(got, ref):
    """max |got - ref| / max |ref| over the tensor."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(got))) if got.size else 0.0
    return float(np.max(np.abs(got - ref)) / scale)


def bf16_half_ulp(ref):
    """Half a bfloat16 ulp at |ref| (the rounding error a bfloat16 store may add)."""
    a = np.abs(np.asarray(ref, np.float64))
    e = np.floor(np.log2(np.maximum(a, 1e-38)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


# Tolerances: float32 inputs 1e-5 and bfloat16 inputs 2e-3, both relative to max|ref|
# over the tensor; a bfloat16 OUTPUT may in addition be off by the half-ulp of its own
# rounding (see check()).
TOL_F32 = 1e-5
TOL_BF16 = 2e-3


def check(got, ref, tol, out_bf16=False, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    if ref.size == 0:
        return
    assert np.all(np.isfinite(ref)), f"{what}: reference has non-finite values"
    assert np.all(np.isfinite(got)), f"{what}: {int((~np.isfinite(got)).sum())} non-finite outputs"
    scale = np.max(np.abs(ref))
    allowed = tol * scale + (bf16_half_ulp(ref) if out_bf16 else 0.0)
    err = np.abs(got - ref)
    bad = err > allowed
    if np.any(bad):
        i = np.unravel_index(np.argmax(err - allowed), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} outside tolerance; worst at {i}: got "
            f"{got[i]!r} ref {ref[i]!r} (tol {tol} * max|ref| {scale:.4g}); "
            f"max rel err {max_rel_err(got, ref):.3g}")
