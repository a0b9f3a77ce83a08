"""GPU parity of the Mamba-3 scan (ssm_mamba3_scan_fwd) against the float64 oracle.

Tolerances as the Mamba-1 scan: max |y_gpu - y_ref| <= 1e-5 max |y_ref| with float32
inputs, 2e-3 with bfloat16 inputs (plus the half-ulp of a bfloat16 output), the same for
the complex final state (compared on its real and imaginary parts)."""
import numpy as np
import pytest

import selective_scan_mamba_gb300 as ssm
from selective_scan_mamba_gb300 import synth
from tests.helpers import TOL_BF16, TOL_F32, check, to_device, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _needs_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _case(oracle, batch, dim, N, L, G, dtype, gated=True, h0=True, seed=0, theta=3.0,
          lam_one=False, out="f32"):
    import torch
    inp = synth.mamba1(batch, dim, N, L, dtype=dtype, delta_scale=0.8, with_z=gated,
                       ngroups=G, seed=seed)
    rng = np.random.default_rng(seed + 50)
    # the complex part and the trapezoid weight (lam stored at the input dtype)
    A_im = (theta * rng.standard_normal((dim, N))).astype(np.float32)
    lam = rng.uniform(0.0, 1.0, (batch, dim, L)).astype(np.float32)
    if lam_one:
        lam[:] = 1.0
    if dtype == synth.BF16:
        bits = synth.bf16_bits(lam)
        lam = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
        lam_t = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    else:
        lam_t = torch.from_numpy(lam).cuda()
    h0c = (rng.standard_normal((batch, dim, N, 2)).astype(np.float32) if h0 else None)
    t = to_device(inp)
    od = {"bf16": torch.bfloat16, "f32": torch.float32}[out]
    y, hf = ssm.ssm_mamba3_scan_fwd(t["x"], t["delta"], t["A"], torch.from_numpy(A_im).cuda(), lam_t,
                                    t["B"], t["C"], D=t["D"], z=t.get("z"),
                                    delta_bias=t["delta_bias"],
                                    h0=None if h0c is None else torch.from_numpy(h0c).cuda(),
                                    out_dtype=od, return_final_state=True)
    torch.cuda.synchronize()
    f = inp.f64
    yr, hr = oracle.mamba3_scan(f("x"), f("delta"), f("A"), A_im.astype(np.float64),
                                lam.astype(np.float64), f("B"), f("C"), D=f("D"),
                                z=f("z") if gated else None, delta_bias=f("delta_bias"),
                                h0=None if h0c is None else h0c[..., 0] + 1j * h0c[..., 1])
    tol = TOL_F32 if dtype == synth.F32 else TOL_BF16
    check(to_numpy(y), yr, tol, out_bf16=(out == "bf16"), what="y")
    hf = to_numpy(hf)
    check(np.stack([hf[..., 0], hf[..., 1]]), np.stack([hr.real, hr.imag]), tol, what="h_final")


@pytest.mark.parametrize("N", [4, 16, 64])
def test_bf16_gated_ragged(oracle_mod, N):
    """z, D, bias, complex h0; several CTAs per (batch, group); a ragged last chunk."""
    _case(oracle_mod, 2, 80 if N < 64 else 24, N, 100, 1, synth.BF16)


def test_fp32_groups_bf16_out(oracle_mod):
    _case(oracle_mod, 2, 64, 32, 77, 2, synth.F32, gated=False, h0=False, out="bf16")


def test_fp32_reduces_to_mamba1_scan(oracle_mod):
    """lambda = 1 and A_im = 0 on the GPU equals the GPU Mamba-1 scan (exp-Euler)."""
    import torch
    inp = synth.mamba1(2, 48, 16, 90, dtype=synth.F32, with_z=True, with_h0=True, seed=9)
    t = to_device(inp)
    y1, h1 = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                              delta_bias=t["delta_bias"], h0=t["h0"], out_dtype=torch.float32,
                              return_final_state=True)
    h0c = torch.stack([t["h0"], torch.zeros_like(t["h0"])], dim=-1).contiguous()
    y3, h3 = ssm.ssm_mamba3_scan_fwd(t["x"], t["delta"], t["A"], torch.zeros_like(t["A"]),
                                     torch.ones_like(t["x"]), t["B"], t["C"], D=t["D"], z=t["z"],
                                     delta_bias=t["delta_bias"], h0=h0c, out_dtype=torch.float32,
                                     return_final_state=True)
    torch.cuda.synchronize()
    check(to_numpy(y3), to_numpy(y1), TOL_F32, what="y")
    check(to_numpy(h3[..., 0]), to_numpy(h1), TOL_F32, what="h_final")
    assert float(h3[..., 1].abs().max()) == 0.0


def test_one_step_and_empty(oracle_mod):
    _case(oracle_mod, 1, 40, 8, 1, 1, synth.F32)
    import torch
    h0 = torch.randn(1, 8, 8, 2, device="cuda")
    x = torch.empty((1, 8, 0), device="cuda")
    A = torch.full((8, 8), -0.5, device="cuda")
    y, hf = ssm.ssm_mamba3_scan_fwd(x, x, A, A, x, torch.empty((1, 1, 8, 0), device="cuda"),
                                    torch.empty((1, 1, 8, 0), device="cuda"), h0=h0,
                                    return_final_state=True)
    torch.cuda.synchronize()
    assert torch.equal(hf, h0)


def test_130m_layer_shape(oracle_mod):
    """The 130m layer's channel count and dstate, 512 steps, every output compared."""
    _case(oracle_mod, 1, 1536, 16, 512, 1, synth.BF16, seed=4)


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_time_split_long_sequence(oracle_mod, out):
    """Few channels and a long sequence: the plan cuts the sequence into segments (a
    states-only pass, then each segment from the carried state), including the
    trapezoid's left-end term at every segment boundary; complex h0 and h_final."""
    _case(oracle_mod, 1, 16, 16, 2600, 1, synth.F32 if out == "f32" else synth.BF16, seed=13,
          out=out)
