"""GPU parity of the Mamba-2 chunked SSD scan (ssd_chunk_scan_fwd) against the float64
oracle's sequential scan (the reference the pages test the chunked form against).
Tolerances as in test_gpu_scan.py."""
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


def run_gpu(inp, chunk, out_dtype=None, disc="exp_euler", h0=True):
    import torch
    t = to_device(inp)
    od = {"bf16": torch.bfloat16, "f32": torch.float32}[out_dtype] if out_dtype else None
    y, hf = ssm.ssd_chunk_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], chunk, D=t.get("D"),
                                   z=t.get("z"), dt_bias=t["dt_bias"],
                                   h0=t.get("h0") if h0 else None, out_dtype=od,
                                   return_final_state=True, disc=disc)
    torch.cuda.synchronize()
    return to_numpy(y), to_numpy(hf)


def run_oracle(oracle, inp, disc=0, h0=True, heads=None):
    f = inp.f64
    args = dict(D=f("D"), z=f("z"), dt_bias=f("dt_bias"), h0=f("h0") if h0 else None, disc=disc)
    if heads is None:
        return oracle.ssd_sequential(f("x"), f("dt"), f("A"), f("B"), f("C"), **args)
    # sampled (b, h): run the oracle on one batch row and one head at a time
    H = f("x").shape[2]
    G = f("B").shape[2]
    ys, hs = [], []
    for b, h in heads:
        g = h // (H // G)
        sl = lambda a: None if a is None else a  # noqa: E731
        y, hf = oracle.ssd_sequential(
            f("x")[b:b + 1, :, h:h + 1], f("dt")[b:b + 1, :, h:h + 1], f("A")[h:h + 1],
            f("B")[b:b + 1, :, g:g + 1], f("C")[b:b + 1, :, g:g + 1],
            D=None if args["D"] is None else args["D"][h:h + 1],
            z=None if args["z"] is None else args["z"][b:b + 1, :, h:h + 1],
            dt_bias=args["dt_bias"][h:h + 1],
            h0=None if args["h0"] is None else args["h0"][b:b + 1, h:h + 1], disc=disc)
        ys.append(y[0, :, 0])
        hs.append(hf[0, 0])
    return np.stack(ys), np.stack(hs)


@pytest.mark.parametrize("chunk", [64, 128, 256])
@pytest.mark.parametrize("P,N", [(64, 128), (32, 64), (128, 64)])
def test_small_ragged(oracle_mod, chunk, P, N):
    """Several chunks and a ragged last chunk (L = 300), 2 groups, z, D, h0, bf16."""
    inp = synth.ssd(2, 300, 4, P, N, 2, dtype=synth.BF16, with_z=True, with_h0=True, seed=1)
    y, hf = run_gpu(inp, chunk)
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_BF16, out_bf16=True, what="y")
    check(hf, hr, TOL_BF16, what="h_final")


@pytest.mark.parametrize("chunk", [64, 256])
def test_fp32_inputs(oracle_mod, chunk):
    inp = synth.ssd(2, 200, 3, 64, 64, 1, dtype=synth.F32, with_z=True, with_h0=True, seed=2)
    y, hf = run_gpu(inp, chunk, out_dtype="f32")
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_F32, what="y")
    check(hf, hr, TOL_F32, what="h_final")


def test_zoh(oracle_mod):
    inp = synth.ssd(1, 130, 2, 64, 128, 1, dtype=synth.F32, with_z=False, seed=3)
    y, hf = run_gpu(inp, 64, out_dtype="f32", disc="zoh", h0=False)
    yr, hr = run_oracle(oracle_mod, inp, disc=1, h0=False)
    check(y, yr, TOL_F32, what="y")
    check(hf, hr, TOL_F32, what="h_final")


@pytest.mark.parametrize("L", [1, 63, 64, 65])
def test_short_sequences(oracle_mod, L):
    inp = synth.ssd(1, L, 2, 32, 64, 1, dtype=synth.BF16, with_z=True, with_h0=True, seed=4)
    y, hf = run_gpu(inp, 64, out_dtype="f32")
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_BF16, what="y")
    check(hf, hr, TOL_BF16, what="h_final")


def test_empty_sequence():
    inp = synth.ssd(1, 0, 2, 32, 64, 1, dtype=synth.BF16, with_h0=True, seed=5)
    y, hf = run_gpu(inp, 64)
    assert y.shape == (1, 0, 2, 32)
    assert np.array_equal(hf, inp.arrays["h0"].astype(np.float64))


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_ranges_cross_sequences(oracle_mod, out):
    """Enough (batch, head, chunk) units that the per-SM ranges hold several chunks, start
    and stop inside sequences and straddle sequence boundaries; ragged last chunk (4000 =
    62 x 64 + 32), gate, initial state, two groups."""
    inp = synth.ssd(2, 4000, 6, 64, 128, 2, dtype=synth.BF16, with_z=True, with_h0=True, seed=6)
    y, hf = run_gpu(inp, 64, out_dtype=out)
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_BF16, out_bf16=(out == "bf16"), what="y")
    check(hf, hr, TOL_BF16, what="h_final")


@pytest.mark.parametrize("batch,L,heads", [(1, 640, 3), (1, 12000, 1), (3, 2000, 5), (8, 1100, 4)],
                         ids=["fewer_cut_chunks_than_sms", "one_sequence", "mixed", "many_short_cuts"])
def test_cut_pieces(oracle_mod, batch, L, heads):
    """Range ends inside sequences in several arrangements, so that the cut chunks are dealt
    out in shares that split cuts across CTAs (pieces folded back in time order): fewer cut
    chunks than SMs (one chunk per range), one sequence cut at every range, and mixes of
    long and short cuts; initial state, gate, ragged last chunk."""
    inp = synth.ssd(batch, L, heads, 64, 128, 1, dtype=synth.BF16, with_z=True, with_h0=True, seed=7)
    y, hf = run_gpu(inp, 64, out_dtype="f32")
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_BF16, what="y")
    check(hf, hr, TOL_BF16, what="h_final")


_SSD_130M_REF = {}


def _ssd_130m_inputs_and_reference(oracle):
    """The 130m-shaped SSD inputs and their float64 sequential-scan reference (computed
    once and shared by the chunk sizes)."""
    if "inp" not in _SSD_130M_REF:
        cfg = synth.WORKLOADS["ssd_130m"]
        inp = synth.ssd(cfg["batch"], cfg["seqlen"], cfg["nheads"], cfg["headdim"], cfg["dstate"],
                        cfg["ngroups"], dtype=cfg["dtype"], delta_scale=cfg["delta_scale"],
                        with_z=False, seed=0)
        _SSD_130M_REF["inp"] = inp
        _SSD_130M_REF["ref"] = run_oracle(oracle, inp, h0=False)
    return _SSD_130M_REF["inp"], _SSD_130M_REF["ref"]


@pytest.mark.parametrize("chunk", [64, 256])
def test_130m_full_size(oracle_mod, chunk):
    """Mamba-2 SSD 130m-shaped: batch 4, 24 heads x headdim 64, d_state 128, ngroups 1,
    L 4096, in the benchmark's launch configuration.  Every element of y and h_final
    against the sequential oracle, with a float32 output at the bare 2e-3 max|ref| bound
    and with a bfloat16 output (plus half a bfloat16 ulp)."""
    import torch
    inp, (yr, hr) = _ssd_130m_inputs_and_reference(oracle_mod)
    t = to_device(inp)
    for od in (torch.float32, torch.bfloat16):
        y, hf = ssm.ssd_chunk_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], chunk, D=t["D"],
                                       dt_bias=t["dt_bias"], out_dtype=od, return_final_state=True)
        torch.cuda.synchronize()
        bf = od == torch.bfloat16
        tag = "bf16" if bf else "f32"
        check(y, yr, TOL_BF16, out_bf16=bf, what=f"y ({tag} out, chunk {chunk})")
        check(hf, hr, TOL_BF16, what=f"h_final ({tag} out, chunk {chunk})")
    if chunk == 256:
        _SSD_130M_REF.clear()


def test_zz_no_device_wait_gave_up():
    """Every bounded wait in the kernels above (copies, MMAs, warp hand-offs) completed:
    the library's timeout counter is still zero after this file's cases."""
    assert ssm.wait_timeouts() == 0
