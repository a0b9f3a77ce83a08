"""GPU parity of the SSD backward (ssd_scan_bwd) against the oracle's SSD backward (the
Mamba-1 backward with tied parameters, pinned by finite differences of the sequential
SSD routine).  Every gradient is float32: max |g - g_ref| <= 1e-4 max |g_ref|, as for
the Mamba-1 backward."""
import numpy as np
import pytest

import selective_scan_mamba_gb300 as ssm
from selective_scan_mamba_gb300 import synth
from tests.helpers import check, to_device, to_numpy

pytestmark = pytest.mark.gpu
TOL_GRAD = 1e-4


@pytest.fixture(autouse=True)
def _needs_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _run(oracle, batch, L, H, P, N, G, dtype, gated=True, h0=True, seed=0):
    import torch
    inp = synth.ssd(batch, L, H, P, N, G, dtype=dtype, with_z=gated, with_h0=h0, seed=seed)
    t = to_device(inp)
    rng = np.random.default_rng(seed + 7)
    dy = rng.standard_normal((batch, L, H, P)).astype(np.float32)
    if dtype == synth.BF16:
        bits = synth.bf16_bits(dy)
        dy = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
        dyt = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    else:
        dyt = torch.from_numpy(dy).cuda()
    dhf = rng.standard_normal((batch, H, P, N)).astype(np.float32)
    g = ssm.ssd_scan_bwd(t["x"], t["dt"], t["A"], t["B"], t["C"], dyt, D=t["D"], z=t.get("z"),
                         dt_bias=t["dt_bias"], h0=t.get("h0"), dh_final=torch.from_numpy(dhf).cuda())
    torch.cuda.synchronize()
    f = inp.f64
    ref = oracle.ssd_bwd(f("x"), f("dt"), f("A"), f("B"), f("C"), dy.astype(np.float64), D=f("D"),
                         z=f("z") if gated else None, dt_bias=f("dt_bias"),
                         h0=f("h0") if h0 else None, dh_final=dhf.astype(np.float64))
    for k, v in ref.items():
        check(to_numpy(g[k]), v, TOL_GRAD, what=k)


@pytest.mark.parametrize("N,P", [(32, 16), (128, 64)])
def test_bf16_gated_groups(oracle_mod, N, P):
    """z, D, dt_bias, h0, dh_final; two groups; several CTAs per (batch, group)."""
    _run(oracle_mod, 2, 70, 4, P, N, 2, synth.BF16)


def test_fp32_no_gate(oracle_mod):
    _run(oracle_mod, 1, 45, 3, 32, 64, 1, synth.F32, gated=False, h0=False)


def test_130m_heads_short_sequence(oracle_mod):
    """The 130m SSD's 24 heads x 64 and dstate 128 on 192 steps, every gradient compared."""
    _run(oracle_mod, 1, 192, 24, 64, 128, 1, synth.BF16, seed=2)


def test_long_sequence_checkpoint_blocks(oracle_mod):
    """1000 steps: 63 chunks in 8 checkpoint blocks of 8, the last one short; dstate 128
    with two heads sharing one group."""
    _run(oracle_mod, 1, 1000, 2, 16, 128, 1, synth.BF16, seed=4)


def test_chunked_form_ragged_groups(oracle_mod):
    """The chunked form (dstate 128, headdim 64): 1000 steps (15 full chunks and a ragged
    one), two groups of two heads, h0 and dh_final, the (batch, head) sequences spread
    over several slices of the workspace."""
    _run(oracle_mod, 2, 1000, 4, 64, 128, 2, synth.BF16, seed=5)


@pytest.mark.parametrize("N,P", [(64, 64), (128, 32), (64, 32)])
def test_chunked_form_fp32_gated(oracle_mod, N, P):
    """float32 inputs and dy through the chunked form, with the gate and a short tail."""
    _run(oracle_mod, 2, 300, 3, P, N, 1, synth.F32, seed=6)


def test_chunked_form_bf16_narrow_heads(oracle_mod):
    """bf16 through the chunked form with headdim 32 and dstate 64 (the narrowest tiles)."""
    _run(oracle_mod, 2, 200, 3, 32, 64, 1, synth.BF16, seed=8)


def test_chunked_form_single_step(oracle_mod):
    """One step: a chunk with 63 padded steps."""
    _run(oracle_mod, 1, 1, 2, 64, 64, 1, synth.BF16, seed=7)
