"""GPU parity of S4D (ssm_s4d_scan_fwd, ssm_s4d_kernel) against the float64 oracle, whose
recurrent and FFT-convolution forms are pinned equal.

Tolerances: the kernel K is computed in double precision per element and rounded, so it
is held to 1e-6 of max|K|.  The recurrence runs in float32 with Abar rounded to float32;
its relative error grows with the memory length ~1/(Delta |Re A|) of the slowest state
(up to 2000 steps at Delta = 1e-3, Re A = -1/2), so float32 inputs are held to 1e-4 and
bfloat16 inputs to 2e-3 of max|y|."""
import numpy as np
import pytest

import selective_scan_mamba_gb300 as ssm
from selective_scan_mamba_gb300 import synth
from tests.helpers import TOL_BF16, check, to_numpy

pytestmark = pytest.mark.gpu
TOL_S4D_F32 = 1e-4


@pytest.fixture(autouse=True)
def _needs_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _params(dim, N, seed):
    """S4D-Lin: A_n = -1/2 + i pi n, log Delta uniform on [ln 1e-3, ln 1e-1], B = 1,
    C complex normal, D normal."""
    rng = np.random.default_rng(seed)
    A = np.broadcast_to(-0.5 + 1j * np.pi * np.arange(N), (dim, N)).astype(np.complex128)
    log_dt = rng.uniform(np.log(1e-3), np.log(1e-1), dim)
    B = np.ones((dim, N), np.complex128)
    C = rng.standard_normal((dim, N)) + 1j * rng.standard_normal((dim, N))
    D = rng.standard_normal(dim)
    return log_dt, A, B, C, D


def _dev_params(log_dt, A, B, C, D):
    import torch

    def pairs(a):
        return torch.from_numpy(np.ascontiguousarray(np.stack([a.real, a.imag], -1), np.float32)).cuda()
    return (torch.from_numpy(log_dt.astype(np.float32)).cuda(), pairs(A), pairs(B), pairs(C),
            torch.from_numpy(D.astype(np.float32)).cuda())


def _run(oracle, batch, dim, N, L, bf16, h0=True, seed=0):
    import torch
    log_dt, A, B, C, D = _params(dim, N, seed)
    # the device sees float32 parameters: the oracle reads the same rounded values
    log_dt, D = log_dt.astype(np.float32).astype(np.float64), D.astype(np.float32).astype(np.float64)
    C = C.astype(np.complex64).astype(np.complex128)
    A = A.astype(np.complex64).astype(np.complex128)
    rng = np.random.default_rng(seed + 1)
    u = rng.standard_normal((batch, dim, L)).astype(np.float32)
    if bf16:
        bits = synth.bf16_bits(u)
        u = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
        ut = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    else:
        ut = torch.from_numpy(u).cuda()
    h0c = (rng.standard_normal((batch, dim, N)) + 1j * rng.standard_normal((batch, dim, N))
           ).astype(np.complex64) if h0 else None
    dl, dA, dB, dC, dD = _dev_params(log_dt, A, B, C, D)
    y, hf = ssm.ssm_s4d_scan_fwd(ut, dl, dA, dB, dC, D=dD,
                                 h0=None if h0c is None else torch.from_numpy(h0c).cuda(),
                                 out_dtype=torch.float32, return_final_state=True)
    torch.cuda.synchronize()
    yr, hr = oracle.s4d_recurrent(u.astype(np.float64), log_dt, A, B, C, D=D,
                                  h0=None if h0c is None else h0c.astype(np.complex128))
    tol = TOL_BF16 if bf16 else TOL_S4D_F32
    check(to_numpy(y), yr, tol, what="y")
    hf = to_numpy(hf)
    check(np.stack([hf[..., 0], hf[..., 1]]), np.stack([hr.real, hr.imag]), tol, what="h_final")
    return u, (log_dt, A, B, C, D), to_numpy(y)


@pytest.mark.parametrize("N", [4, 16, 64])
def test_recurrent_fp32(oracle_mod, N):
    _run(oracle_mod, 2, 40 if N < 64 else 20, N, 300, False)


def test_recurrent_bf16_long(oracle_mod):
    _run(oracle_mod, 1, 64, 32, 1500, True, seed=3)


def test_recurrent_equals_fft_convolution(oracle_mod):
    """From a zero state the GPU recurrence equals the oracle's FFT convolution form."""
    u, (log_dt, A, B, C, D), y = _run(oracle_mod, 2, 16, 32, 257, False, h0=False, seed=5)
    yc = oracle_mod.s4d_fft_conv(u.astype(np.float64), log_dt, A, B, C, D=D)
    check(y, yc, TOL_S4D_F32, what="y vs FFT convolution")


@pytest.mark.parametrize("L", [1, 100, 4096])
def test_kernel(oracle_mod, L):
    import torch
    log_dt, A, B, C, D = _params(24, 32, 7)
    log_dt = log_dt.astype(np.float32).astype(np.float64)
    C = C.astype(np.complex64).astype(np.complex128)
    dl, dA, dB, dC, _ = _dev_params(log_dt, A, B, C, D)
    K = ssm.ssm_s4d_kernel(dl, dA, dB, dC, L)
    torch.cuda.synchronize()
    Kr = oracle_mod.s4d_kernel(log_dt, A.astype(np.complex64).astype(np.complex128), B, C, L)
    check(to_numpy(K), Kr, 1e-6, what="K")


def test_empty_sequence_copies_state():
    import torch
    log_dt, A, B, C, D = _params(8, 16, 1)
    dl, dA, dB, dC, dD = _dev_params(log_dt, A, B, C, D)
    h0 = torch.randn(2, 8, 16, 2, device="cuda")
    u = torch.empty((2, 8, 0), device="cuda")
    _, hf = ssm.ssm_s4d_scan_fwd(u, dl, dA, dB, dC, D=dD, h0=h0, return_final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(hf, h0)


@pytest.mark.parametrize("bf16", [False, True])
def test_time_split_long_sequence(oracle_mod, bf16):
    """Few channels and a long sequence: the plan cuts the sequence into segments (a
    states-only pass, then each segment from the carried state); h0 and h_final."""
    _run(oracle_mod, 1, 8, 16, 3000, bf16, seed=11)


def _conv(oracle, batch, dim, N, L, bf16, out_bf16=False, seed=0):
    """The FFT convolution form on the GPU against both float64 oracle forms (the FFT
    convolution and the recurrence from a zero state), which the oracle pins equal."""
    import torch
    log_dt, A, B, C, D = _params(dim, N, seed)
    log_dt, D = log_dt.astype(np.float32).astype(np.float64), D.astype(np.float32).astype(np.float64)
    C = C.astype(np.complex64).astype(np.complex128)
    A = A.astype(np.complex64).astype(np.complex128)
    rng = np.random.default_rng(seed + 1)
    u = rng.standard_normal((batch, dim, L)).astype(np.float32)
    if bf16:
        bits = synth.bf16_bits(u)
        u = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
        ut = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    else:
        ut = torch.from_numpy(u).cuda()
    dl, dA, dB, dC, dD = _dev_params(log_dt, A, B, C, D)
    y = ssm.ssm_s4d_conv_fwd(ut, dl, dA, dB, dC, D=dD,
                             out_dtype=torch.bfloat16 if out_bf16 else torch.float32)
    torch.cuda.synchronize()
    u64 = u.astype(np.float64)
    yc = oracle.s4d_fft_conv(u64, log_dt, A, B, C, D=D)
    yr, _ = oracle.s4d_recurrent(u64, log_dt, A, B, C, D=D)
    tol = TOL_BF16 if bf16 else TOL_S4D_F32
    check(y, yc, tol, out_bf16=out_bf16, what="y vs the oracle's FFT convolution")
    check(y, yr, tol, out_bf16=out_bf16, what="y vs the oracle's recurrence")


@pytest.mark.parametrize("bf16", [False, True])
def test_convolution_form_efficiency_sweep_shape(oracle_mod, bf16):
    """The pages' efficiency-sweep shape: batch 8, d_model 256, 32 complex states, L 4096."""
    _conv(oracle_mod, 8, 256, 32, 4096, bf16, out_bf16=bf16)


@pytest.mark.parametrize("batch,L,N", [(3, 1000, 16), (1, 1, 8), (2, 8192, 4), (5, 257, 64), (2, 200, 32),
                                       (1, 1500, 16), (2, 100, 8), (1, 2048, 32)])
def test_convolution_form_ragged_and_limits(oracle_mod, batch, L, N):
    """An odd batch (the last transform carries one row), lengths that are not powers of
    two, one step, the longest sequence the shared-memory transform takes (8192), and a
    length for every transform size N = 2^m (m = 1 and 8 run the kernel compiled for any
    size, m = 9 .. 14 the ones compiled for theirs)."""
    _conv(oracle_mod, batch, 6, N, L, False, seed=batch)


def test_convolution_form_refusals():
    import torch
    log_dt, A, B, C, D = _params(4, 8, 2)
    dl, dA, dB, dC, dD = _dev_params(log_dt, A, B, C, D)
    u = torch.randn(1, 4, 8193, device="cuda")
    assert ssm.ssm_s4d_conv_workspace_size(u, dl, dA, dB, dC) == 0
    with pytest.raises(ssm.SsmError) as err:
        ssm.ssm_s4d_conv_fwd(u, dl, dA, dB, dC, D=dD)
    assert err.value.status == 2 and "8192" in err.value.message
    # the convolution form carries no state
    from selective_scan_mamba_gb300 import _lib
    import ctypes
    p, keep = ssm._s4d_params(dl, dA, dB, dC, dD)
    u = torch.randn(1, 4, 64, device="cuda")
    y = torch.empty_like(u)
    h0 = torch.zeros(1, 4, 8, 2, device="cuda")
    p.batch, p.seqlen = 1, 64
    p.u, p.y, p.h0 = u.data_ptr(), y.data_ptr(), h0.data_ptr()
    assert _lib.load().ssm_s4d_conv_fwd(ctypes.byref(p), None, 0, None) == _lib.SSM_ERR_INVALID_ARG
    del keep


def test_convolution_form_empty_sequence():
    """L = 0: nothing to convolve; the call succeeds without scratch and writes nothing."""
    import torch
    log_dt, A, B, C, D = _params(4, 8, 3)
    dl, dA, dB, dC, dD = _dev_params(log_dt, A, B, C, D)
    u = torch.empty((2, 4, 0), device="cuda")
    assert ssm.ssm_s4d_conv_workspace_size(u, dl, dA, dB, dC) == 0
    y = ssm.ssm_s4d_conv_fwd(u, dl, dA, dB, dC, D=dD)
    torch.cuda.synchronize()
    assert y.shape == (2, 4, 0)
