"""GPU parity of the Mamba-1 scan backward (ssm_scan_bwd) against the float64 oracle's
backward (itself pinned by finite differences).

Inputs and the output gradient dy come from the seeded generator (bf16 values exact on
both sides).  Every gradient is float32 and is compared with the oracle over the whole
tensor: max |g_gpu - g_ref| <= TOL_GRAD * max |g_ref|.  The GPU computes in float32 with
the same operations as the definition; the bound leaves room for float32 rounding in the
sums over time and over the channels of a group (dA, dbias, dB, dC).
"""
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


def _run(oracle, batch, dim, N, L, G, dtype, gated=True, skip=True, bias=True, h0=True,
         dhf=True, softplus=True, seed=0):
    import torch
    inp = synth.mamba1(batch, dim, N, L, dtype=dtype, delta_scale=0.8, with_z=gated,
                       with_h0=h0, ngroups=G, seed=seed)
    if not softplus:  # without softplus the step is delta + bias: keep it positive
        inp.arrays["delta"] = np.abs(inp.arrays["delta"]) * 0.1
        inp.arrays["delta_bias"] = np.full_like(inp.arrays["delta_bias"], 0.01)
    t = to_device(inp)
    rng = np.random.default_rng(seed + 100)
    dy64 = rng.standard_normal((batch, dim, L)).astype(np.float32)
    if dtype == synth.BF16:  # dy in bf16; the oracle reads the same rounded values
        bits = synth.bf16_bits(dy64)
        dy64 = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
        dy = torch.from_numpy(bits.view(np.int16).copy()).cuda().view(torch.bfloat16)
    else:
        dy = torch.from_numpy(dy64).cuda()
    dh_final = (rng.standard_normal((batch, dim, N)).astype(np.float32) if dhf else None)
    g = ssm.ssm_scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], dy,
                         D=t.get("D") if skip else None, z=t.get("z"),
                         delta_bias=t["delta_bias"] if bias else None, delta_softplus=softplus,
                         h0=t.get("h0"), dh_final=None if dh_final is None else torch.from_numpy(dh_final).cuda())
    torch.cuda.synchronize()
    f = inp.f64
    ref = oracle.mamba1_scan_bwd(f("x"), f("delta"), f("A"), f("B"), f("C"), dy64.astype(np.float64),
                                 D=f("D") if skip else None, z=f("z") if gated else None,
                                 delta_bias=f("delta_bias") if bias else None,
                                 delta_softplus=softplus, h0=f("h0") if h0 else None,
                                 dh_final=None if dh_final is None else dh_final.astype(np.float64))
    for k, v in ref.items():
        assert k in g, k
        check(to_numpy(g[k]), v, TOL_GRAD, what=k)
    return g, ref


@pytest.mark.parametrize("N", [16, 32, 64])
def test_bf16_all_inputs_ragged(oracle_mod, N):
    """z, D, bias, h0, dh_final; several CTAs per (batch, group); a ragged last chunk."""
    _run(oracle_mod, 2, 160 if N == 16 else 72, N, 100, 1, synth.BF16)


def test_fp32_groups_no_gate(oracle_mod):
    _run(oracle_mod, 2, 96, 16, 65, 2, synth.F32, gated=False, skip=False, bias=False,
         h0=False, dhf=False)


def test_fp32_no_softplus(oracle_mod):
    _run(oracle_mod, 1, 64, 32, 40, 1, synth.F32, softplus=False)


def test_one_step_and_empty(oracle_mod):
    _run(oracle_mod, 1, 70, 16, 1, 1, synth.BF16)
    g, ref = _run(oracle_mod, 1, 70, 16, 0, 1, synth.BF16)
    assert to_numpy(g["dA"]).max() == 0.0


def test_130m_layer_shape(oracle_mod):
    """The 130m layer's channel count and dstate on a shorter sequence (256 steps), the
    full backward compared element by element."""
    _run(oracle_mod, 1, 1536, 16, 256, 1, synth.BF16, seed=3)


@pytest.mark.parametrize("N", [16, 32])
def test_long_sequence_checkpoint_blocks(oracle_mod, N):
    """1500 steps, 94 chunks: with N = 16 a checkpoint per chunk; with N = 32 blocks of
    10 chunks (the last one short) rerun forwards from their checkpoints."""
    _run(oracle_mod, 2, 40, N, 1500, 1, synth.BF16, seed=5)
