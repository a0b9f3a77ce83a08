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


def _as_f64(a, device):
    """float64 torch tensor on ``device`` (no copy for a float64 numpy array on the CPU)."""
    import torch
    if isinstance(a, torch.Tensor):
        return a.detach().to(device=device, dtype=torch.float64)
    return torch.from_numpy(np.ascontiguousarray(a, np.float64)).to(device)


def check(got, ref, tol, out_bf16=False, what=""):
    """Element-by-element parity: every |got - ref| <= tol * max|ref| (plus half a
    bfloat16 ulp of ref for a bfloat16 output).  ``got`` and ``ref`` are numpy arrays or
    torch tensors; the comparison runs in float64 on got's device (the GPU when got is a
    CUDA tensor), so whole tensors of 10^8 elements check in well under a second."""
    import torch
    dev = got.device if isinstance(got, torch.Tensor) else "cpu"
    g = _as_f64(got, dev)
    r = _as_f64(ref, dev)
    assert tuple(g.shape) == tuple(r.shape), f"{what}: shape {tuple(g.shape)} vs {tuple(r.shape)}"
    if r.numel() == 0:
        return
    assert bool(torch.isfinite(r).all()), f"{what}: reference has non-finite values"
    nonfinite = int((~torch.isfinite(g)).sum())
    assert nonfinite == 0, f"{what}: {nonfinite} non-finite outputs"
    scale = float(r.abs().max())
    err = (g - r).abs_()
    if out_bf16:
        # half a bfloat16 ulp of |ref|: 2^(floor(log2|ref|) - 8); frexp gives |ref| = m 2^e
        # with m in [0.5, 1), so floor(log2|ref|) = e - 1
        _, e = torch.frexp(r.abs().clamp_min(1e-38))
        allowed = torch.ldexp(torch.ones_like(r), (e - 9).to(r.dtype)).add_(tol * scale)
        excess = err - allowed
    else:
        excess = err - tol * scale
    worst = float(excess.max())
    if worst > 0:
        bad = int((excess > 0).sum())
        i = np.unravel_index(int(excess.argmax()), tuple(r.shape))
        gi, ri = float(g[i]), float(r[i])
        raise AssertionError(
            f"{what}: {bad} of {r.numel()} outside tolerance; worst at {i}: got {gi!r} ref "
            f"{ri!r} (tol {tol} * max|ref| {scale:.4g}); max rel err "
            f"{float(err.max()) / scale if scale else float(err.max()):.3g}")


def rel_err(got, ref):
    """max |got - ref| / max |ref| in float64 on got's device (for reports)."""
    import torch
    dev = got.device if isinstance(got, torch.Tensor) else "cpu"
    g = _as_f64(got, dev)
    r = _as_f64(ref, dev)
    scale = float(r.abs().max()) if r.numel() else 0.0
    e = float((g - r).abs().max()) if r.numel() else 0.0
    return e / scale if scale else e
