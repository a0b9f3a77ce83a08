"""CUDA-graph capture of the multi-launch paths, replayed on new inputs, against the
float64 oracle.  The Mamba-1 scan with a time split (segment pass, then main pass) and
the tensor-core SSD (step sums, cut states, walk) each run as a chain of dependent
launches; a captured graph must replay that chain with the inputs copied into the
captured buffers, the workspace reused and the launch parameters (the SSD's cut plan)
unchanged."""
import numpy as np
import pytest

import selective_scan_mamba_gb300 as ssm
from selective_scan_mamba_gb300 import synth
from tests.helpers import TOL_BF16, check, to_device, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _needs_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _capture(fn):
    import torch
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up outside the capture (builds the library, caches tensor maps)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def _load(dst, src):
    for k, v in src.items():
        if k in dst:
            dst[k].copy_(v)


def test_scan_with_time_split_replays(oracle_mod):
    """256 channels of one batch row over 4096 steps: the plan splits the sequence into
    segments (a segment pass and a main pass)."""
    import torch
    sets = [synth.mamba1(1, 256, 16, 4096, dtype=synth.BF16, with_z=False, with_h0=True, seed=s)
            for s in (11, 12)]
    t = to_device(sets[0])
    x = t["x"]
    ws = torch.empty(max(1, ssm.ssm_scan_workspace_size(x, t["B"], out_dtype=torch.float32)),
                     dtype=torch.uint8, device="cuda")
    y = torch.empty(x.shape, dtype=torch.float32, device="cuda")
    hf = torch.empty((1, 256, 16), dtype=torch.float32, device="cuda")

    def call():
        ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                         delta_bias=t["delta_bias"], h0=t["h0"], y=y, h_final=hf,
                         workspace=ws)

    g = _capture(call)
    for inp in sets:
        _load(t, to_device(inp))
        g.replay()
        torch.cuda.synchronize()
        f = inp.f64
        yr, hr = oracle_mod.mamba1_scan(f("x"), f("delta"), f("A"), f("B"), f("C"), D=f("D"),
                                        delta_bias=f("delta_bias"), h0=f("h0"))
        check(to_numpy(y), yr, TOL_BF16, what="y")
        check(to_numpy(hf), hr, TOL_BF16, what="h_final")


def test_ssd_chain_replays(oracle_mod):
    """Tensor-core SSD with range ends inside sequences (cut pieces spread over CTAs)."""
    import torch
    sets = [synth.ssd(3, 2000, 5, 64, 128, 1, dtype=synth.BF16, with_z=True, with_h0=True,
                      seed=s) for s in (21, 22)]
    t = to_device(sets[0])
    ws = torch.empty(ssm.ssd_chunk_scan_workspace_size(t["x"], t["B"], 64), dtype=torch.uint8,
                     device="cuda")
    y = torch.empty(t["x"].shape, dtype=torch.float32, device="cuda")
    hf = torch.empty(t["h0"].shape, dtype=torch.float32, device="cuda")

    def call():
        ssm.ssd_chunk_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], 64, D=t["D"], z=t["z"],
                               dt_bias=t["dt_bias"], h0=t["h0"], y=y, h_final=hf, workspace=ws,
                               return_final_state=True)

    g = _capture(call)
    for inp in sets:
        _load(t, to_device(inp))
        g.replay()
        torch.cuda.synchronize()
        f = inp.f64
        yr, hr = oracle_mod.ssd_sequential(f("x"), f("dt"), f("A"), f("B"), f("C"), D=f("D"),
                                           z=f("z"), dt_bias=f("dt_bias"), h0=f("h0"))
        check(to_numpy(y), yr, TOL_BF16, what="y")
        check(to_numpy(hf), hr, TOL_BF16, what="h_final")
