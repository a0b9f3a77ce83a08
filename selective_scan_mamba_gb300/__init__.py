"""selective_scan_mamba_gb300 -- GB300-native selective state-space scans.

A thin Python binding over libssmscan's C ABI (include/ssmscan.h).  The functions keep
the C names:

  * ssm_scan_fwd, ssm_scan_bwd          -- Mamba-1 selective scan (diagonal A per channel)
                                           and its gradients
  * ssd_chunk_scan_fwd, ssd_scan_bwd    -- Mamba-2 chunked SSD scan (scalar A per head)
                                           and its gradients
  * ssm_state_update, ssm_state_update_tokens
                                        -- decode: one token or T tokens, in place on the
                                           state
  * ssm_mamba3_scan_fwd                 -- Mamba-3 complex-diagonal scan
  * ssm_s4d_scan_fwd, ssm_s4d_conv_fwd, ssm_s4d_kernel
                                        -- S4D recurrent form, FFT convolution form and
                                           convolution kernel

Each takes CUDA torch tensors of the current device in the library's layouts, checks
them, fills the C parameter struct and calls the library on the current torch stream
(or the one given).  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback, and a missing GPU or library raises.
"""
from __future__ import annotations

import ctypes

from . import _lib
from ._lib import SsmError  # noqa: F401

__all__ = [
    "ssm_scan_fwd", "ssm_scan_workspace_size", "ssm_scan_bwd", "ssm_scan_bwd_workspace_size",
    "ssd_chunk_scan_fwd", "ssd_chunk_scan_workspace_size", "ssd_scan_bwd",
    "ssd_scan_bwd_workspace_size", "ssm_state_update", "ssm_state_update_tokens",
    "ssm_mamba3_scan_fwd", "ssm_s4d_scan_fwd", "ssm_s4d_conv_fwd", "ssm_s4d_conv_workspace_size",
    "ssm_s4d_kernel", "wait_timeouts",
    "device_status", "SsmError", "lib",
]


def wait_timeouts() -> int:
    """Bounded device-side waits that gave up since the previous call (0 in correct
    operation); synchronises with the device and clears the count."""
    return int(_lib.load().ssm_wait_timeouts())


def device_status() -> None:
    """Waits for the current device and raises SsmError (status SSM_ERR_TIMEOUT) if a
    bounded device-side wait gave up since the previous check, which means the outputs
    of the calls in between are not valid, or SSM_ERR_CUDA if the device reports an
    error.  Clears the record."""
    _lib.check(_lib.load().ssm_device_status())


def lib():
    """The loaded shared library (ctypes.CDLL)."""
    return _lib.load()


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return _lib.SSM_BF16
    if t.dtype == torch.float32:
        return _lib.SSM_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


def _out_dtype(code):
    torch = _torch()
    return torch.bfloat16 if code == _lib.SSM_BF16 else torch.float32


def _ptr(t, name, shape=None, dtype=None):
    if t is None:
        return None
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the call runs on the current device "
                         f"cuda:{torch.cuda.current_device()}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _disc(disc):
    if disc in ("exp_euler", _lib.SSM_DISC_EXP_EULER, None):
        return _lib.SSM_DISC_EXP_EULER
    if disc in ("zoh", _lib.SSM_DISC_ZOH):
        return _lib.SSM_DISC_ZOH
    raise ValueError(f"unknown discretisation {disc!r}")


def _stream(stream):
    torch = _torch()
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if stream.device.index != torch.cuda.current_device():
        raise ValueError(f"stream is on {stream.device}, but the call runs on the current "
                         f"device cuda:{torch.cuda.current_device()}")
    return ctypes.c_void_p(stream.cuda_stream)


def _scan_params(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, h_final, disc):
    torch = _torch()
    batch, dim, L = x.shape
    if B.dim() == 3:
        B = B.unsqueeze(1)
        C = C.unsqueeze(1)
    G, N = B.shape[1], B.shape[2]
    f32 = torch.float32
    p = _lib.ScanParams()
    p.batch, p.dim, p.dstate, p.seqlen, p.ngroups = batch, dim, N, L, G
    p.in_dtype = _dtype_code(x)
    p.out_dtype = _dtype_code(y)
    p.x = _ptr(x, "x")
    p.delta = _ptr(delta, "delta", (batch, dim, L), x.dtype)
    p.delta_bias = _ptr(delta_bias, "delta_bias", (dim,), f32)
    p.delta_softplus = int(bool(delta_softplus))
    p.A = _ptr(A, "A", (dim, N), f32)
    p.B = _ptr(B, "B", (batch, G, N, L), x.dtype)
    p.C = _ptr(C, "C", (batch, G, N, L), x.dtype)
    p.D_skip = _ptr(D, "D", (dim,), f32)
    p.z = _ptr(z, "z", (batch, dim, L), x.dtype)
    p.h0 = _ptr(h0, "h0", (batch, dim, N), f32)
    p.y = _ptr(y, "y", (batch, dim, L))
    p.h_final = _ptr(h_final, "h_final", (batch, dim, N), f32)
    p.disc = _disc(disc)
    return p


_KERNELS = {"auto": _lib.SSM_SCAN_KERNEL_AUTO, "tmem": _lib.SSM_SCAN_KERNEL_TMEM,
            "tma": _lib.SSM_SCAN_KERNEL_TMA, "tiled": _lib.SSM_SCAN_KERNEL_TILED,
            "generic": _lib.SSM_SCAN_KERNEL_GENERIC}


def scan_opts(kernel="auto", threads_per_channel=0, max_segments=0, wait_limit=0,
              fault_test=0):
    """The C options struct of ssm_scan_fwd_ex (see include/ssmscan.h)."""
    o = _lib.ScanOpts()
    if kernel not in _KERNELS:
        raise ValueError(f"unknown kernel {kernel!r} ({', '.join(_KERNELS)})")
    o.kernel = _KERNELS[kernel]
    o.threads_per_channel = int(threads_per_channel)
    o.max_segments = int(max_segments)
    o.wait_limit = int(wait_limit)
    o.fault_test = int(fault_test)
    return o


def ssm_scan_workspace_size(x, B, out_dtype=None, disc="exp_euler", **opts) -> int:
    """Scratch bytes ssm_scan_fwd needs for these shapes, dtypes and options (y defaults
    to x's dtype); the options are those of :func:`scan_opts`."""
    p = _lib.ScanParams()
    p.batch, p.dim, p.seqlen = x.shape
    p.dstate = B.shape[-2]
    p.ngroups = 1 if B.dim() == 3 else B.shape[1]
    p.in_dtype = _dtype_code(x)
    p.out_dtype = _dtype_code(x) if out_dtype is None else _dtype_code(
        _torch().empty(0, dtype=out_dtype))
    p.disc = _disc(disc)
    o = scan_opts(**opts)
    return int(lib().ssm_scan_workspace_size(ctypes.byref(p), ctypes.byref(o)))


def ssm_scan_fwd(x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                 h0=None, *, y=None, h_final=None, out_dtype=None, return_final_state=False,
                 disc="exp_euler", workspace=None, stream=None, **opts):
    """Mamba-1 selective scan.

    x, delta, z: [batch, dim, L] (bfloat16 or float32); B, C: [batch, G, N, L] or
    [batch, N, L]; A: [dim, N] float32; D, delta_bias: [dim] float32; h0: [batch, dim, N]
    float32.  Returns y [batch, dim, L] (dtype ``out_dtype``, default x's), and the final
    state [batch, dim, N] float32 when ``return_final_state``.

    Runs ssm_scan_fwd_ex with the options of :func:`scan_opts` given as keywords (kernel,
    threads_per_channel, max_segments, ...; all automatic by default).  When the plan
    splits a long sequence in time it needs scratch: ``workspace`` (a uint8 CUDA tensor of
    at least ssm_scan_workspace_size bytes) or, if None, a tensor allocated here.
    """
    torch = _torch()
    if y is None:
        y = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
    if return_final_state and h_final is None:
        h_final = torch.empty((x.shape[0], x.shape[1], A.shape[1]), dtype=torch.float32,
                              device=x.device)
    p = _scan_params(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, y, h_final, disc)
    o = scan_opts(**opts)
    need = int(lib().ssm_scan_workspace_size(ctypes.byref(p), ctypes.byref(o)))
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
        ws_ptr, ws_bytes = _ptr(workspace, "workspace"), workspace.numel()
    _lib.check(lib().ssm_scan_fwd_ex(ctypes.byref(p), ctypes.byref(o), ws_ptr, ws_bytes,
                                     _stream(stream)))
    return (y, h_final) if return_final_state else y


def ssm_scan_bwd(x, delta, A, B, C, dy, D=None, z=None, delta_bias=None, delta_softplus=True,
                 h0=None, dh_final=None, *, return_dh0=True, workspace=None, stream=None):
    """Backward of ssm_scan_fwd (exponential-Euler, dstate 16, 32 or 64).

    Same inputs as the forward plus dy [batch, dim, L] (bfloat16 or float32) and the
    optional dh_final [batch, dim, N] float32.  Returns a dict of float32 gradients of
    sum(dy * y) + sum(dh_final * h_final): dx, ddelta [batch, dim, L], dA [dim, N],
    dB, dC [batch, G, N, L], and dD, dz, ddelta_bias for the inputs given, dh0
    [batch, dim, N] when ``return_dh0``.
    """
    torch = _torch()
    if B.dim() == 3:
        B = B.unsqueeze(1)
        C = C.unsqueeze(1)
    batch, dim, L = x.shape
    G, N = B.shape[1], B.shape[2]
    f32, dev = torch.float32, x.device
    p = _lib.ScanBwdParams()
    # the forward parameters; y is ignored by the backward, dy fixes its dtype
    p.fwd = _scan_params(x, delta, A, B, C, D, z, delta_bias, delta_softplus, h0, dy, None,
                         "exp_euler")
    out = {"dx": torch.empty((batch, dim, L), dtype=f32, device=dev),
           "ddelta": torch.empty((batch, dim, L), dtype=f32, device=dev),
           "dA": torch.empty((dim, N), dtype=f32, device=dev),
           "dB": torch.empty((batch, G, N, L), dtype=f32, device=dev),
           "dC": torch.empty((batch, G, N, L), dtype=f32, device=dev)}
    if D is not None:
        out["dD"] = torch.empty((dim,), dtype=f32, device=dev)
    if z is not None:
        out["dz"] = torch.empty((batch, dim, L), dtype=f32, device=dev)
    if delta_bias is not None:
        out["ddelta_bias"] = torch.empty((dim,), dtype=f32, device=dev)
    if return_dh0:
        out["dh0"] = torch.empty((batch, dim, N), dtype=f32, device=dev)
    p.dy = _ptr(dy, "dy", (batch, dim, L))
    p.dh_final = _ptr(dh_final, "dh_final", (batch, dim, N), f32)
    for name, field in (("dx", "dx"), ("ddelta", "ddelta"), ("dz", "dz"), ("dA", "dA"),
                        ("dB", "dB"), ("dC", "dC"), ("dD", "dD_skip"),
                        ("ddelta_bias", "ddelta_bias"), ("dh0", "dh0")):
        setattr(p, field, _ptr(out.get(name), name))
    need = int(lib().ssm_scan_bwd_workspace_size(ctypes.byref(p)))
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    _lib.check(lib().ssm_scan_bwd(ctypes.byref(p), ws_ptr, ws_bytes, _stream(stream)))
    return out


def ssm_scan_bwd_workspace_size(x, B, dy_dtype=None) -> int:
    """Scratch bytes ssm_scan_bwd needs for these shapes (0 if unsupported)."""
    p = _lib.ScanBwdParams()
    if B.dim() == 3:
        B = B.unsqueeze(1)
    p.fwd.batch, p.fwd.dim, p.fwd.seqlen = x.shape
    p.fwd.ngroups, p.fwd.dstate = B.shape[1], B.shape[2]
    p.fwd.in_dtype = _dtype_code(x)
    p.fwd.out_dtype = (_lib.SSM_F32 if dy_dtype is not None and dy_dtype == _torch().float32
                       else _lib.SSM_BF16)
    p.fwd.disc = 0
    return int(lib().ssm_scan_bwd_workspace_size(ctypes.byref(p)))


def ssm_mamba3_scan_fwd(x, delta, A_re, A_im, lam, B, C, D=None, z=None, delta_bias=None,
                        delta_softplus=True, h0=None, *, y=None, h_final=None, out_dtype=None,
                        return_final_state=False, workspace=None, stream=None):
    """Mamba-3 scan: complex diagonal A = A_re + i A_im, exponential-trapezoidal rule.

    x, delta, lam, z: [batch, dim, L] (bfloat16 or float32); B, C: [batch, G, N, L];
    A_re, A_im: [dim, N] float32; D, delta_bias: [dim] float32; h0: [batch, dim, N, 2]
    float32 (re, im).  Returns y and, when ``return_final_state``, h_final [batch, dim,
    N, 2] float32.
    """
    torch = _torch()
    if B.dim() == 3:
        B = B.unsqueeze(1)
        C = C.unsqueeze(1)
    batch, dim, L = x.shape
    G, N = B.shape[1], B.shape[2]
    f32 = torch.float32
    if y is None:
        y = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
    if return_final_state and h_final is None:
        h_final = torch.empty((batch, dim, N, 2), dtype=f32, device=x.device)
    p = _lib.Mamba3Params()
    p.batch, p.dim, p.dstate, p.seqlen, p.ngroups = batch, dim, N, L, G
    p.in_dtype = _dtype_code(x)
    p.out_dtype = _dtype_code(y)
    p.x = _ptr(x, "x")
    p.delta = _ptr(delta, "delta", (batch, dim, L), x.dtype)
    p.delta_bias = _ptr(delta_bias, "delta_bias", (dim,), f32)
    p.delta_softplus = int(bool(delta_softplus))
    p.A_re = _ptr(A_re, "A_re", (dim, N), f32)
    p.A_im = _ptr(A_im, "A_im", (dim, N), f32)
    p.lam = _ptr(lam, "lam", (batch, dim, L), x.dtype)
    p.B = _ptr(B, "B", (batch, G, N, L), x.dtype)
    p.C = _ptr(C, "C", (batch, G, N, L), x.dtype)
    p.D_skip = _ptr(D, "D", (dim,), f32)
    p.z = _ptr(z, "z", (batch, dim, L), x.dtype)
    p.h0 = _ptr(h0, "h0", (batch, dim, N, 2), f32)
    p.y = _ptr(y, "y", (batch, dim, L))
    p.h_final = _ptr(h_final, "h_final", (batch, dim, N, 2), f32)
    need = int(lib().ssm_mamba3_scan_workspace_size(ctypes.byref(p)))
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    _lib.check(lib().ssm_mamba3_scan_fwd(ctypes.byref(p), ws_ptr, ws_bytes, _stream(stream)))
    return (y, h_final) if return_final_state else y


def _complex_pairs(t, name, shape):
    """float32 [..., 2] (re, im) view of a complex64 tensor, or a float32 [..., 2] tensor"""
    torch = _torch()
    if t is None:
        return None
    if t.is_complex():
        t = torch.view_as_real(t.to(torch.complex64)).contiguous()
    _ptr(t, name, tuple(shape) + (2,), torch.float32)
    return t


def _s4d_params(log_dt, A, B, C, D=None):
    torch = _torch()
    dim = log_dt.shape[0]
    A_ = _complex_pairs(A, "A", (dim, A.shape[1]))
    N = A_.shape[1]
    p = _lib.S4dParams()
    p.dim, p.dstate = dim, N
    keep = [A_, _complex_pairs(B, "B", (dim, N)), _complex_pairs(C, "C", (dim, N))]
    p.log_dt = _ptr(log_dt, "log_dt", (dim,), torch.float32)
    p.A, p.B, p.C = (_ptr(k, n) for k, n in zip(keep, ("A", "B", "C")))
    p.D_skip = _ptr(D, "D", (dim,), torch.float32)
    return p, keep


def ssm_s4d_scan_fwd(u, log_dt, A, B, C, D=None, h0=None, *, y=None, h_final=None,
                     out_dtype=None, return_final_state=False, workspace=None, stream=None):
    """S4D recurrent form (exact ZOH, Delta = exp(log_dt)).

    u: [batch, dim, L] (bfloat16 or float32); log_dt: [dim] float32; A, B, C: [dim, N]
    complex64 or [dim, N, 2] float32; D: [dim]; h0: [batch, dim, N] complex64 or
    [batch, dim, N, 2] float32.  Returns y [batch, dim, L] and, when
    ``return_final_state``, h_final [batch, dim, N, 2] float32.
    """
    torch = _torch()
    batch, dim, L = u.shape
    p, keep = _s4d_params(log_dt, A, B, C, D)
    N = p.dstate
    if y is None:
        y = torch.empty(u.shape, dtype=out_dtype or u.dtype, device=u.device)
    if return_final_state and h_final is None:
        h_final = torch.empty((batch, dim, N, 2), dtype=torch.float32, device=u.device)
    h0_ = _complex_pairs(h0, "h0", (batch, dim, N))
    p.batch, p.seqlen = batch, L
    p.in_dtype = _dtype_code(u)
    p.out_dtype = _dtype_code(y)
    p.u = _ptr(u, "u")
    p.h0 = _ptr(h0_, "h0")
    p.y = _ptr(y, "y", (batch, dim, L))
    p.h_final = _ptr(h_final, "h_final", (batch, dim, N, 2), torch.float32)
    need = int(lib().ssm_s4d_scan_workspace_size(ctypes.byref(p)))
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=u.device)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    _lib.check(lib().ssm_s4d_scan_fwd(ctypes.byref(p), ws_ptr, ws_bytes, _stream(stream)))
    del keep, h0_
    return (y, h_final) if return_final_state else y


def ssm_s4d_conv_fwd(u, log_dt, A, B, C, D=None, *, y=None, out_dtype=None, workspace=None,
                     stream=None):
    """S4D convolution form by FFT on the GPU: y = K * u + D u from a zero state (L <= 8192).

    Same arguments as :func:`ssm_s4d_scan_fwd` without a state.  ``workspace``: a uint8
    CUDA tensor of at least ssm_s4d_conv_workspace_size bytes (allocated here if None).
    Returns y [batch, dim, L]."""
    torch = _torch()
    batch, dim, L = u.shape
    p, keep = _s4d_params(log_dt, A, B, C, D)
    if y is None:
        y = torch.empty(u.shape, dtype=out_dtype or u.dtype, device=u.device)
    p.batch, p.seqlen = batch, L
    p.in_dtype = _dtype_code(u)
    p.out_dtype = _dtype_code(y)
    p.u = _ptr(u, "u")
    p.y = _ptr(y, "y", (batch, dim, L))
    need = int(lib().ssm_s4d_conv_workspace_size(ctypes.byref(p)))
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=u.device)
        ws_ptr, ws_bytes = _ptr(workspace, "workspace"), workspace.numel()
    _lib.check(lib().ssm_s4d_conv_fwd(ctypes.byref(p), ws_ptr, ws_bytes, _stream(stream)))
    del keep
    return y


def ssm_s4d_conv_workspace_size(u, log_dt, A, B, C) -> int:
    """Scratch bytes ssm_s4d_conv_fwd needs for u's shape (0 if unsupported)."""
    p, keep = _s4d_params(log_dt, A, B, C)
    p.batch, _, p.seqlen = u.shape
    p.in_dtype = p.out_dtype = _dtype_code(u)
    n = int(lib().ssm_s4d_conv_workspace_size(ctypes.byref(p)))
    del keep
    return n


def ssm_s4d_kernel(log_dt, A, B, C, kernel_len, *, out=None, stream=None):
    """S4D convolution kernel K [dim, kernel_len] float32: K_l = Re sum_n C Bbar Abar^l."""
    torch = _torch()
    p, keep = _s4d_params(log_dt, A, B, C)
    if out is None:
        out = torch.empty((p.dim, int(kernel_len)), dtype=torch.float32, device=log_dt.device)
    _lib.check(lib().ssm_s4d_kernel(ctypes.byref(p), _ptr(out, "K", (p.dim, int(kernel_len)),
                                                         torch.float32), int(kernel_len),
                                    _stream(stream)))
    del keep
    return out


def _ssd_params(x, dt, A, B, C, chunk_size, D, z, dt_bias, dt_softplus, h0, y, h_final, disc):
    torch = _torch()
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    f32 = torch.float32
    p = _lib.SsdParams()
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups = batch, L, H, P, N, G
    p.chunk_size = int(chunk_size)
    p.in_dtype = _dtype_code(x)
    p.out_dtype = _dtype_code(y)
    p.x = _ptr(x, "x")
    p.dt = _ptr(dt, "dt", (batch, L, H), x.dtype)
    p.dt_bias = _ptr(dt_bias, "dt_bias", (H,), f32)
    p.dt_softplus = int(bool(dt_softplus))
    p.A = _ptr(A, "A", (H,), f32)
    p.B = _ptr(B, "B", (batch, L, G, N), x.dtype)
    p.C = _ptr(C, "C", (batch, L, G, N), x.dtype)
    p.D_skip = _ptr(D, "D", (H,), f32)
    p.z = _ptr(z, "z", (batch, L, H, P), x.dtype)
    p.h0 = _ptr(h0, "h0", (batch, H, P, N), f32)
    p.y = _ptr(y, "y", (batch, L, H, P))
    p.h_final = _ptr(h_final, "h_final", (batch, H, P, N), f32)
    p.disc = _disc(disc)
    return p


def ssd_scan_bwd(x, dt, A, B, C, dy, D=None, z=None, dt_bias=None, dt_softplus=True, h0=None,
                 dh_final=None, *, return_dh0=True, workspace=None, stream=None):
    """Backward of the SSD scan (exponential-Euler, dstate 16, 32, 64 or 128; in chunked
    form for (dstate, headdim) in {(128, 64), (64, 64), (128, 32), (64, 32)} when dy has
    x's dtype, else as the tied recurrence).

    Same inputs as ssd_chunk_scan_fwd plus dy [batch, L, H, P] and the optional dh_final
    [batch, H, P, N] float32.  Returns a dict of float32 gradients: dx [batch, L, H, P],
    ddt [batch, L, H], dA [H], dB, dC [batch, L, G, N], and dD, dz, ddt_bias for the
    inputs given, dh0 [batch, H, P, N] when ``return_dh0``.
    """
    torch = _torch()
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    f32, dev = torch.float32, x.device
    p = _lib.SsdBwdParams()
    # forward parameters; chunk size, y and h_final are ignored by the backward
    p.fwd = _ssd_params(x, dt, A, B, C, 64, D, z, dt_bias, dt_softplus, h0, dy, None, "exp_euler")
    out = {"dx": torch.empty((batch, L, H, P), dtype=f32, device=dev),
           "ddt": torch.empty((batch, L, H), dtype=f32, device=dev),
           "dA": torch.empty((H,), dtype=f32, device=dev),
           "dB": torch.empty((batch, L, G, N), dtype=f32, device=dev),
           "dC": torch.empty((batch, L, G, N), dtype=f32, device=dev)}
    if D is not None:
        out["dD"] = torch.empty((H,), dtype=f32, device=dev)
    if z is not None:
        out["dz"] = torch.empty((batch, L, H, P), dtype=f32, device=dev)
    if dt_bias is not None:
        out["ddt_bias"] = torch.empty((H,), dtype=f32, device=dev)
    if return_dh0:
        out["dh0"] = torch.empty((batch, H, P, N), dtype=f32, device=dev)
    p.dy = _ptr(dy, "dy", (batch, L, H, P))
    p.dh_final = _ptr(dh_final, "dh_final", (batch, H, P, N), f32)
    for name, field in (("dx", "dx"), ("ddt", "ddt"), ("dz", "dz"), ("dA", "dA"), ("dB", "dB"),
                        ("dC", "dC"), ("dD", "dD_skip"), ("ddt_bias", "ddt_bias"), ("dh0", "dh0")):
        setattr(p, field, _ptr(out.get(name), name))
    need = int(lib().ssd_scan_bwd_workspace_size(ctypes.byref(p)))
    ws_ptr, ws_bytes = None, 0
    if need:
        if workspace is None:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel()
    _lib.check(lib().ssd_scan_bwd(ctypes.byref(p), ws_ptr, ws_bytes, _stream(stream)))
    return out


def ssd_scan_bwd_workspace_size(x, B, dy_dtype=None) -> int:
    """Scratch bytes ssd_scan_bwd needs for these shapes (0 if unsupported); dy_dtype
    defaults to x's dtype."""
    p = _lib.SsdBwdParams()
    p.fwd.batch, p.fwd.seqlen, p.fwd.nheads, p.fwd.headdim = x.shape
    p.fwd.ngroups, p.fwd.dstate = B.shape[2], B.shape[3]
    p.fwd.chunk_size = 64
    p.fwd.in_dtype = _dtype_code(x)
    if dy_dtype is None:
        p.fwd.out_dtype = p.fwd.in_dtype
    else:
        p.fwd.out_dtype = _lib.SSM_F32 if dy_dtype == _torch().float32 else _lib.SSM_BF16
    return int(lib().ssd_scan_bwd_workspace_size(ctypes.byref(p)))


def ssd_chunk_scan_workspace_size(x, B, chunk_size) -> int:
    """Scratch bytes ssd_chunk_scan_fwd needs for these shapes and chunk size."""
    p = _lib.SsdParams()
    p.batch, p.seqlen, p.nheads, p.headdim = x.shape
    p.ngroups, p.dstate = B.shape[2], B.shape[3]
    p.chunk_size = int(chunk_size)
    p.in_dtype = _lib.SSM_BF16
    p.out_dtype = _lib.SSM_BF16
    return int(lib().ssd_chunk_scan_workspace_size(ctypes.byref(p)))


def ssd_chunk_scan_fwd(x, dt, A, B, C, chunk_size=64, D=None, z=None, dt_bias=None,
                       dt_softplus=True, h0=None, *, y=None, h_final=None, out_dtype=None,
                       return_final_state=False, disc="exp_euler", workspace=None, stream=None):
    """Mamba-2 chunked SSD scan.

    x, z: [batch, L, H, P]; dt: [batch, L, H]; B, C: [batch, L, G, N] (bfloat16 or
    float32); A, D, dt_bias: [H] float32; h0: [batch, H, P, N] float32.  Returns y
    [batch, L, H, P] and, when ``return_final_state``, the final state.
    """
    torch = _torch()
    if y is None:
        y = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
    if return_final_state and h_final is None:
        h_final = torch.empty((x.shape[0], x.shape[2], x.shape[3], B.shape[3]),
                              dtype=torch.float32, device=x.device)
    p = _ssd_params(x, dt, A, B, C, chunk_size, D, z, dt_bias, dt_softplus, h0, y, h_final, disc)
    need = int(lib().ssd_chunk_scan_workspace_size(ctypes.byref(p)))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    _lib.check(lib().ssd_chunk_scan_fwd(ctypes.byref(p), workspace.data_ptr(), workspace.numel(),
                                        _stream(stream)))
    return (y, h_final) if return_final_state else y


def ssm_state_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=True, *,
                     y=None, out_dtype=None, disc="exp_euler", stream=None):
    """One decode step, updating ``state`` [batch, H, P, N] float32 in place.

    x, z: [batch, H, P]; dt: [batch, H]; B, C: [batch, G, N]; A: [H] (Mamba-2 form) or
    [H, N] (Mamba-1 form); D, dt_bias: [H].  Returns y [batch, H, P].
    """
    torch = _torch()
    batch, H, P, N = state.shape
    G = B.shape[1]
    if y is None:
        y = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
    f32 = torch.float32
    p = _lib.StepParams()
    p.batch, p.nheads, p.headdim, p.dstate, p.ngroups = batch, H, P, N, G
    p.a_per_state = 1 if A.dim() == 2 else 0
    p.in_dtype = _dtype_code(x)
    p.out_dtype = _dtype_code(y)
    p.state = _ptr(state, "state", (batch, H, P, N), f32)
    p.x = _ptr(x, "x", (batch, H, P))
    p.dt = _ptr(dt, "dt", (batch, H), x.dtype)
    p.dt_bias = _ptr(dt_bias, "dt_bias", (H,), f32)
    p.dt_softplus = int(bool(dt_softplus))
    p.A = _ptr(A, "A", (H, N) if A.dim() == 2 else (H,), f32)
    p.B = _ptr(B, "B", (batch, G, N), x.dtype)
    p.C = _ptr(C, "C", (batch, G, N), x.dtype)
    p.D_skip = _ptr(D, "D", (H,), f32)
    p.z = _ptr(z, "z", (batch, H, P), x.dtype)
    p.y = _ptr(y, "y", (batch, H, P))
    p.disc = _disc(disc)
    _lib.check(lib().ssm_state_update(ctypes.byref(p), _stream(stream)))
    return y


def ssm_state_update_tokens(state, x, dt, A, B, C, D=None, z=None, dt_bias=None,
                            dt_softplus=True, *, y=None, out_dtype=None, disc="exp_euler",
                            stream=None):
    """T consecutive decode steps in one call, updating ``state`` [batch, H, P, N] float32
    in place (read and written once).

    Token-major inputs: x, z: [T, batch, H, P]; dt: [T, batch, H]; B, C: [T, batch, G, N];
    A: [H] or [H, N]; D, dt_bias: [H].  Returns y [T, batch, H, P] (output after each
    token).
    """
    torch = _torch()
    batch, H, P, N = state.shape
    T = x.shape[0]
    G = B.shape[2]
    if y is None:
        y = torch.empty(x.shape, dtype=out_dtype or x.dtype, device=x.device)
    f32 = torch.float32
    p = _lib.StepParams()
    p.batch, p.nheads, p.headdim, p.dstate, p.ngroups = batch, H, P, N, G
    p.a_per_state = 1 if A.dim() == 2 else 0
    p.in_dtype = _dtype_code(x)
    p.out_dtype = _dtype_code(y)
    p.state = _ptr(state, "state", (batch, H, P, N), f32)
    p.x = _ptr(x, "x", (T, batch, H, P))
    p.dt = _ptr(dt, "dt", (T, batch, H), x.dtype)
    p.dt_bias = _ptr(dt_bias, "dt_bias", (H,), f32)
    p.dt_softplus = int(bool(dt_softplus))
    p.A = _ptr(A, "A", (H, N) if A.dim() == 2 else (H,), f32)
    p.B = _ptr(B, "B", (T, batch, G, N), x.dtype)
    p.C = _ptr(C, "C", (T, batch, G, N), x.dtype)
    p.D_skip = _ptr(D, "D", (H,), f32)
    p.z = _ptr(z, "z", (T, batch, H, P), x.dtype)
    p.y = _ptr(y, "y", (T, batch, H, P))
    p.disc = _disc(disc)
    _lib.check(lib().ssm_state_update_tokens(ctypes.byref(p), int(T), _stream(stream)))
    return y
