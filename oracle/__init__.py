"""float64 CPU oracle for the selective state-space scan -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never uses it and
shares no code with it; the two meet only through the seeded input generator
(``selective_scan_mamba_gb300.synth``), which holds none of the method's
arithmetic.

The arithmetic lives in ``oracle.c`` (plain sequential loops in double
precision, each routine citing the passage it follows); this module compiles it
with the host C compiler on first use and calls it through ctypes.  Every array
argument is a float64 numpy array in the library's layout; ``None`` stands for an
optional input that is absent.

Parity pins: every routine is pinned by tests in ``tests/test_oracle_pins.py``
(closed forms, brute-force unrolled sums, chunked-versus-sequential agreement,
split continuation, degenerate cases, high-precision references for softplus and
phi1).  None is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

DISC_EXP_EULER = 0
DISC_ZOH = 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP, portable flags)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
                   "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _bind(path):
    lib = ctypes.CDLL(path)
    dp = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_softplus.restype = ctypes.c_double
    lib.oracle_softplus.argtypes = [ctypes.c_double]
    lib.oracle_phi1.restype = ctypes.c_double
    lib.oracle_phi1.argtypes = [ctypes.c_double]
    lib.oracle_s4d_kernel.restype = i
    lib.oracle_s4d_kernel.argtypes = [i, i, i] + [dp] * 5
    lib.oracle_s4d_recurrent.restype = i
    lib.oracle_s4d_recurrent.argtypes = [i, i, i, i] + [dp] * 9
    lib.oracle_mamba3_scan.restype = i
    lib.oracle_mamba3_scan.argtypes = [i, i, i, i, i] + [dp] * 3 + [i] + [dp] * 10
    lib.oracle_mamba1_scan_bwd.restype = i
    lib.oracle_mamba1_scan_bwd.argtypes = [i, i, i, i, i] + [dp] * 3 + [i] + [dp] * 17
    lib.oracle_mamba1_scan.restype = i
    lib.oracle_mamba1_scan.argtypes = [i, i, i, i, i, dp, dp, dp, i, dp, dp, dp, dp, dp, dp, i,
                                       dp, dp]
    lib.oracle_ssd_sequential.restype = i
    lib.oracle_ssd_sequential.argtypes = [i, i, i, i, i, i, dp, dp, dp, i, dp, dp, dp, dp, dp, dp,
                                          i, dp, dp]
    lib.oracle_ssd_chunked.restype = i
    lib.oracle_ssd_chunked.argtypes = [i, i, i, i, i, i, i, dp, dp, dp, i, dp, dp, dp, dp, dp, dp,
                                       i, dp, dp]
    lib.oracle_state_update.restype = i
    lib.oracle_state_update.argtypes = [i, i, i, i, i, i, dp, dp, dp, dp, i, dp, dp, dp, dp, dp,
                                        i, dp]
    lib.oracle_num_threads.restype = i
    lib.oracle_num_threads.argtypes = []
    lib.oracle_set_num_threads.restype = None
    lib.oracle_set_num_threads.argtypes = [i]
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(_LIB)
    return _lib


class use_library:
    """Context manager: route every call of this module to another build of the
    oracle (used by the test that plants mistakes in a copy of oracle.c)."""

    def __init__(self, path):
        self.path = path
        self.saved = None

    def __enter__(self):
        global _lib
        self.saved = _load()
        _lib = _bind(self.path)
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _f64(a, shape=None):
    """Contiguous float64 copy/view of an optional array, checked against shape."""
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and a.shape != tuple(shape):
        raise ValueError(f"oracle: expected shape {tuple(shape)}, got {a.shape}")
    return a


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def softplus(v: float) -> float:
    return _load().oracle_softplus(float(v))


def phi1(zv: float) -> float:
    return _load().oracle_phi1(float(zv))


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Threads the OpenMP loops over independent rows use (n < 1: all cores).  Timing
    only: every row is still computed sequentially by one thread, so results do not
    change."""
    _load().oracle_set_num_threads(int(n))


def mamba1_scan(x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=True,
                h0=None, disc=DISC_EXP_EULER, ngroups=None):
    """Mamba-1 selective scan.  x, delta, z: [batch, dim, L]; B, C: [batch, G, N, L];
    A: [dim, N].  Returns (y [batch, dim, L], h_final [batch, dim, N])."""
    x = _f64(x)
    batch, dim, L = x.shape
    A = _f64(A)
    N = A.shape[1]
    B = _f64(B)
    if B.ndim == 3:  # [batch, N, L] means one group
        B = B[:, None]
    G = B.shape[1] if ngroups is None else ngroups
    B = _f64(B, (batch, G, N, L))
    C = _f64(C if np.ndim(C) == 4 else np.asarray(C)[:, None], (batch, G, N, L))
    delta = _f64(delta, (batch, dim, L))
    A = _f64(A, (dim, N))
    D = _f64(D, (dim,))
    z = _f64(z, (batch, dim, L))
    delta_bias = _f64(delta_bias, (dim,))
    h0 = _f64(h0, (batch, dim, N))
    y = np.empty((batch, dim, L), np.float64)
    hf = np.empty((batch, dim, N), np.float64)
    rc = _load().oracle_mamba1_scan(batch, dim, N, L, G, _p(x), _p(delta), _p(delta_bias),
                                    int(bool(delta_softplus)), _p(A), _p(B), _p(C), _p(D), _p(z),
                                    _p(h0), int(disc), _p(y), _p(hf))
    if rc:
        raise ValueError("oracle_mamba1_scan: invalid arguments")
    return y, hf


def mamba1_scan_bwd(x, delta, A, B, C, dy, D=None, z=None, delta_bias=None,
                    delta_softplus=True, h0=None, dh_final=None):
    """Gradients of sum(dy * y) + sum(dh_final * h_final) for mamba1_scan
    (exponential-Euler).  Shapes as mamba1_scan with B, C [batch, G, N, L].  Returns a
    dict with dx, ddelta, dA, dB, dC and, for the inputs given, dD, dz, ddelta_bias,
    dh0 (dh0 always)."""
    x = _f64(x)
    batch, dim, L = x.shape
    A = _f64(A)
    N = A.shape[1]
    B = _f64(B)
    G = B.shape[1]
    B = _f64(B, (batch, G, N, L))
    C = _f64(C, (batch, G, N, L))
    delta = _f64(delta, (batch, dim, L))
    dy = _f64(dy, (batch, dim, L))
    D = _f64(D, (dim,))
    z = _f64(z, (batch, dim, L))
    delta_bias = _f64(delta_bias, (dim,))
    h0 = _f64(h0, (batch, dim, N))
    dh_final = _f64(dh_final, (batch, dim, N))
    out = {"dx": np.empty((batch, dim, L)), "ddelta": np.empty((batch, dim, L)),
           "dA": np.empty((dim, N)), "dB": np.empty((batch, G, N, L)),
           "dC": np.empty((batch, G, N, L)), "dh0": np.empty((batch, dim, N))}
    if D is not None:
        out["dD"] = np.empty(dim)
    if z is not None:
        out["dz"] = np.empty((batch, dim, L))
    if delta_bias is not None:
        out["ddelta_bias"] = np.empty(dim)
    rc = _load().oracle_mamba1_scan_bwd(
        batch, dim, N, L, G, _p(x), _p(delta), _p(delta_bias), int(bool(delta_softplus)), _p(A),
        _p(B), _p(C), _p(D), _p(z), _p(h0), _p(dy), _p(dh_final), _p(out["dx"]),
        _p(out["ddelta"]), _p(out["dA"]), _p(out["dB"]), _p(out["dC"]), _p(out.get("dD")),
        _p(out.get("dz")), _p(out.get("ddelta_bias")), _p(out["dh0"]))
    if rc:
        raise ValueError("oracle_mamba1_scan_bwd: invalid arguments")
    return out


def mamba3_scan(x, delta, A_re, A_im, lam, B, C, D=None, z=None, delta_bias=None,
                delta_softplus=True, h0=None):
    """Mamba-3 scan (complex diagonal A = A_re + i A_im, exponential-trapezoidal rule with
    weight lam [batch, dim, L]).  x, delta, z: [batch, dim, L]; B, C: [batch, G, N, L];
    A_re, A_im: [dim, N]; h0: [batch, dim, N] complex (or None).  Returns (y [batch, dim,
    L], h_final [batch, dim, N] complex128)."""
    x = _f64(x)
    batch, dim, L = x.shape
    A_re = _f64(A_re)
    N = A_re.shape[1]
    B = _f64(B)
    G = B.shape[1]
    B = _f64(B, (batch, G, N, L))
    C = _f64(C, (batch, G, N, L))
    delta = _f64(delta, (batch, dim, L))
    A_im = _f64(A_im, (dim, N))
    lam = _f64(lam, (batch, dim, L))
    D = _f64(D, (dim,))
    z = _f64(z, (batch, dim, L))
    delta_bias = _f64(delta_bias, (dim,))
    h0p = None
    if h0 is not None:
        h0c = np.asarray(h0, np.complex128).reshape(batch, dim, N)
        h0p = np.ascontiguousarray(np.stack([h0c.real, h0c.imag], axis=-1))
    y = np.empty((batch, dim, L), np.float64)
    hf = np.empty((batch, dim, N, 2), np.float64)
    rc = _load().oracle_mamba3_scan(batch, dim, N, L, G, _p(x), _p(delta), _p(delta_bias),
                                    int(bool(delta_softplus)), _p(A_re), _p(A_im), _p(lam),
                                    _p(B), _p(C), _p(D), _p(z), _p(h0p), _p(y), _p(hf))
    if rc:
        raise ValueError("oracle_mamba3_scan: invalid arguments")
    return y, hf[..., 0] + 1j * hf[..., 1]


def _pairs(a, shape):
    """complex array -> float64 (re, im) pairs of the given leading shape"""
    a = np.asarray(a, np.complex128).reshape(shape)
    return np.ascontiguousarray(np.stack([a.real, a.imag], axis=-1))


def s4d_kernel(log_dt, A, B, C, L):
    """S4D convolution kernel K [dim, L]: K_l = Re sum_n C Bbar Abar^l (exact ZOH).
    log_dt [dim]; A, B, C complex [dim, N]."""
    log_dt = _f64(log_dt)
    dim = log_dt.shape[0]
    N = np.asarray(A).shape[1]
    K = np.empty((dim, L), np.float64)
    rc = _load().oracle_s4d_kernel(dim, N, L, _p(log_dt), _p(_pairs(A, (dim, N))),
                                   _p(_pairs(B, (dim, N))), _p(_pairs(C, (dim, N))), _p(K))
    if rc:
        raise ValueError("oracle_s4d_kernel: invalid arguments")
    return K


def s4d_recurrent(u, log_dt, A, B, C, D=None, h0=None):
    """S4D recurrent form from h0 (complex [batch, dim, N], zeros when None).  u [batch,
    dim, L].  Returns (y [batch, dim, L], h_final complex [batch, dim, N])."""
    u = _f64(u)
    batch, dim, L = u.shape
    N = np.asarray(A).shape[1]
    y = np.empty((batch, dim, L), np.float64)
    hf = np.empty((batch, dim, N, 2), np.float64)
    rc = _load().oracle_s4d_recurrent(batch, dim, N, L, _p(u), _p(_f64(log_dt, (dim,))),
                                      _p(_pairs(A, (dim, N))), _p(_pairs(B, (dim, N))),
                                      _p(_pairs(C, (dim, N))), _p(_f64(D, (dim,))),
                                      _p(None if h0 is None else _pairs(h0, (batch, dim, N))),
                                      _p(y), _p(hf))
    if rc:
        raise ValueError("oracle_s4d_recurrent: invalid arguments")
    return y, hf[..., 0] + 1j * hf[..., 1]


def s4d_fft_conv(u, log_dt, A, B, C, D=None):
    """S4D convolution form: y = K * u (causal, by FFT of length 2L) + D u."""
    u = _f64(u)
    batch, dim, L = u.shape
    K = s4d_kernel(log_dt, A, B, C, L)
    n = 2 * L if L else 1
    y = np.fft.irfft(np.fft.rfft(u, n=n) * np.fft.rfft(K, n=n)[None], n=n)[..., :L]
    if D is not None:
        y = y + _f64(D, (dim,))[None, :, None] * u
    return y


def _ssd_args(x, dt, A, B, C, D, z, dt_bias, h0):
    x = _f64(x)
    batch, L, H, P = x.shape
    B = _f64(B)
    G, N = B.shape[2], B.shape[3]
    B = _f64(B, (batch, L, G, N))
    C = _f64(C, (batch, L, G, N))
    dt = _f64(dt, (batch, L, H))
    A = _f64(A, (H,))
    D = _f64(D, (H,))
    z = _f64(z, (batch, L, H, P))
    dt_bias = _f64(dt_bias, (H,))
    h0 = _f64(h0, (batch, H, P, N))
    return x, dt, A, B, C, D, z, dt_bias, h0, (batch, L, H, P, G, N)


def ssd_sequential(x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=True, h0=None,
                   disc=DISC_EXP_EULER):
    """Mamba-2 sequential scan.  x, z: [batch, L, H, P]; dt: [batch, L, H];
    B, C: [batch, L, G, N]; A, D, dt_bias: [H].  Returns (y, h_final [batch, H, P, N])."""
    x, dt, A, B, C, D, z, dt_bias, h0, (batch, L, H, P, G, N) = _ssd_args(
        x, dt, A, B, C, D, z, dt_bias, h0)
    y = np.empty((batch, L, H, P), np.float64)
    hf = np.empty((batch, H, P, N), np.float64)
    rc = _load().oracle_ssd_sequential(batch, L, H, P, N, G, _p(x), _p(dt), _p(dt_bias),
                                       int(bool(dt_softplus)), _p(A), _p(B), _p(C), _p(D), _p(z),
                                       _p(h0), int(disc), _p(y), _p(hf))
    if rc:
        raise ValueError("oracle_ssd_sequential: invalid arguments")
    return y, hf


def ssd_bwd(x, dt, A, B, C, dy, D=None, z=None, dt_bias=None, dt_softplus=True, h0=None,
            dh_final=None):
    """Gradients of sum(dy * y) + sum(dh_final * h_final) for ssd_sequential
    (exponential-Euler).  With a scalar A per head the Mamba-2 recurrence is the Mamba-1
    scan over the H*P channels of the heads, A tied across each head's channels and
    states and Delta shared by a head's P channels ("From S4 to Mamba-3", 03/System,
    mamba2_minimal.py), so its derivative is mamba1_scan_bwd on that view with the tied
    gradients summed.  Layouts as ssd_sequential; returns dx, ddt [batch, L, H], dA [H],
    dB, dC [batch, L, G, N], dh0 [batch, H, P, N] and dD, dz, ddt_bias for the inputs
    given."""
    x, dt, A, B, C, D, z, dt_bias, h0, (batch, L, H, P, G, N) = _ssd_args(
        x, dt, A, B, C, D, z, dt_bias, h0)
    dy = _f64(dy, (batch, L, H, P))
    dh_final = _f64(dh_final, (batch, H, P, N))

    def chan(a):  # [batch, L, H, P] -> [batch, H*P, L]
        return None if a is None else np.ascontiguousarray(a.reshape(batch, L, H * P).transpose(0, 2, 1))
    rep = lambda v: None if v is None else np.repeat(v, P)  # noqa: E731  [H] -> [H*P]
    g = mamba1_scan_bwd(
        chan(x), np.ascontiguousarray(np.repeat(dt, P, axis=2).transpose(0, 2, 1)),
        np.repeat(A[:, None], P * N).reshape(H * P, N),
        np.ascontiguousarray(B.transpose(0, 2, 3, 1)), np.ascontiguousarray(C.transpose(0, 2, 3, 1)),
        chan(dy), D=rep(D), z=chan(z), delta_bias=rep(dt_bias), delta_softplus=dt_softplus,
        h0=None if h0 is None else h0.reshape(batch, H * P, N),
        dh_final=None if dh_final is None else dh_final.reshape(batch, H * P, N))

    def back(a):  # [batch, H*P, L] -> [batch, L, H, P]
        return np.ascontiguousarray(a.transpose(0, 2, 1).reshape(batch, L, H, P))
    out = {"dx": back(g["dx"]),
           "ddt": g["ddelta"].reshape(batch, H, P, L).sum(axis=2).transpose(0, 2, 1).copy(),
           "dA": g["dA"].reshape(H, P * N).sum(axis=1),
           "dB": np.ascontiguousarray(g["dB"].transpose(0, 3, 1, 2)),
           "dC": np.ascontiguousarray(g["dC"].transpose(0, 3, 1, 2)),
           "dh0": g["dh0"].reshape(batch, H, P, N)}
    if D is not None:
        out["dD"] = g["dD"].reshape(H, P).sum(axis=1)
    if z is not None:
        out["dz"] = back(g["dz"])
    if dt_bias is not None:
        out["ddt_bias"] = g["ddelta_bias"].reshape(H, P).sum(axis=1)
    return out


def ssd_chunked(x, dt, A, B, C, chunk, D=None, z=None, dt_bias=None, dt_softplus=True, h0=None,
                disc=DISC_EXP_EULER):
    """Mamba-2 chunked SSD with chunk size ``chunk``; same layouts as ssd_sequential."""
    x, dt, A, B, C, D, z, dt_bias, h0, (batch, L, H, P, G, N) = _ssd_args(
        x, dt, A, B, C, D, z, dt_bias, h0)
    y = np.empty((batch, L, H, P), np.float64)
    hf = np.empty((batch, H, P, N), np.float64)
    rc = _load().oracle_ssd_chunked(batch, L, H, P, N, G, int(chunk), _p(x), _p(dt), _p(dt_bias),
                                    int(bool(dt_softplus)), _p(A), _p(B), _p(C), _p(D), _p(z),
                                    _p(h0), int(disc), _p(y), _p(hf))
    if rc:
        raise ValueError("oracle_ssd_chunked: invalid arguments")
    return y, hf


def state_update(state, x, dt, A, B, C, D=None, z=None, dt_bias=None, dt_softplus=True,
                 disc=DISC_EXP_EULER, inplace=False):
    """One decode step.  state: [batch, H, P, N] (a new array is returned and the input is
    not modified, unless ``inplace``: then ``state``, a C-contiguous float64 array, is
    advanced in place and returned); x, z: [batch, H, P]; dt: [batch, H]; B, C:
    [batch, G, N]; A: [H] or [H, N].  Returns (y [batch, H, P], new_state)."""
    if inplace:
        if not (isinstance(state, np.ndarray) and state.dtype == np.float64
                and state.flags.c_contiguous):
            raise ValueError("oracle: an in-place state must be a C-contiguous float64 array")
        st = state
    else:
        st = np.array(state, dtype=np.float64, copy=True, order="C")
    batch, H, P, N = st.shape
    B = _f64(B)
    G = B.shape[1]
    B = _f64(B, (batch, G, N))
    C = _f64(C, (batch, G, N))
    x = _f64(x, (batch, H, P))
    dt = _f64(dt, (batch, H))
    A = _f64(A)
    a_per_state = 1 if A.ndim == 2 else 0
    A = _f64(A, (H, N) if a_per_state else (H,))
    D = _f64(D, (H,))
    z = _f64(z, (batch, H, P))
    dt_bias = _f64(dt_bias, (H,))
    y = np.empty((batch, H, P), np.float64)
    rc = _load().oracle_state_update(batch, H, P, N, G, a_per_state, _p(st), _p(x), _p(dt),
                                     _p(dt_bias), int(bool(dt_softplus)), _p(A), _p(B), _p(C),
                                     _p(D), _p(z), int(disc), _p(y))
    if rc:
        raise ValueError("oracle_state_update: invalid arguments")
    return y, st
