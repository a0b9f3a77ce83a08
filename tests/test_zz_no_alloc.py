"""ssd_chunk_scan_fwd_noalloc: the chunked SSD scan for callers that cannot allocate
device memory (for example a plugin whose host framework owns every byte of device
memory, or a serving loop that may not allocate once running).  It keeps its scratch
in the library's own fixed device array instead of a caller workspace.

Checked here through the C ABI: two calls in a row match the regular entry point
(which gets a caller workspace) and the float64 oracle within the parity tolerance, on
the tensor-core and the CUDA-core paths, and a problem too big for the fixed array is
refused with a clear message.  The file name makes pytest
collect it last."""
import ctypes

import pytest

import selective_scan_mamba_gb300 as ssm
from selective_scan_mamba_gb300 import _lib, synth
from tests.helpers import TOL_BF16, TOL_F32, check, to_device


def _noalloc_fn():
    lib = _lib.load()
    fn = lib.ssd_chunk_scan_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(_lib.SsdParams), ctypes.c_void_p]
    cap = lib.ssd_noalloc_scratch_capacity
    cap.restype = ctypes.c_size_t
    cap.argtypes = []
    return lib, fn, int(cap())


def test_capacity_is_the_documented_32_mib():
    _, _, cap = _noalloc_fn()
    assert cap == 32 << 20


def test_oversized_problem_is_refused_on_the_host():
    """Refused before any GPU work: the size query alone decides."""
    lib, fn, cap = _noalloc_fn()
    p = _lib.SsdParams()
    # headdim 32 runs on the CUDA-core path, which keeps one fp32 state per chunk
    p.batch, p.seqlen, p.nheads, p.headdim, p.dstate, p.ngroups, p.chunk_size = \
        4, 65536, 24, 32, 128, 1, 64
    p.in_dtype = p.out_dtype = _lib.SSM_BF16
    fake = 0x7F0000000000
    for f in ("x", "dt", "A", "B", "C", "y"):
        setattr(p, f, fake)
    assert lib.ssd_chunk_scan_workspace_size(ctypes.byref(p)) > cap
    assert fn(ctypes.byref(p), None) == _lib.SSM_ERR_INVALID_ARG
    msg = lib.ssm_last_error().decode()
    assert "fixed" in msg and "scratch" in msg


# (P, N, in dtype): the tensor-core path (headdim 64, dstate 128, bf16) and the CUDA-core
# path (headdim 32; float32 inputs), which keeps its chunk decays at an offset inside the
# same scratch
NOALLOC_CASES = [(64, 128, synth.BF16, 64), (64, 128, synth.BF16, 256), (32, 64, synth.BF16, 64),
                 (64, 64, synth.F32, 128)]


@pytest.mark.gpu
@pytest.mark.parametrize("P,N,dtype,chunk", NOALLOC_CASES)
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(oracle_mod, P, N, dtype, chunk):
    """Two calls in a row through the C ABI: each matches the regular entry point (given a
    caller workspace) and the float64 sequential oracle, within the parity tolerance.
    Ragged length, two groups, gate, skip and initial state."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    lib, fn, cap = _noalloc_fn()
    inp = synth.ssd(2, 1000, 8, P, N, 2, dtype=dtype, with_z=True, with_h0=True, seed=21)
    t = to_device(inp)
    assert ssm.ssd_chunk_scan_workspace_size(t["x"], t["B"], chunk) <= cap
    y_ref, h_ref = ssm.ssd_chunk_scan_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], chunk,
                                          D=t["D"], z=t["z"], dt_bias=t["dt_bias"], h0=t["h0"],
                                          return_final_state=True)
    torch.cuda.synchronize()
    f = inp.f64
    y_or, h_or = oracle_mod.ssd_sequential(f("x"), f("dt"), f("A"), f("B"), f("C"), D=f("D"),
                                           z=f("z"), dt_bias=f("dt_bias"), h0=f("h0"))
    tol = TOL_BF16 if dtype == synth.BF16 else TOL_F32
    out_bf16 = dtype == synth.BF16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        y = torch.full_like(t["x"], float("nan"))
        hf = torch.full((2, 8, P, N), float("nan"), dtype=torch.float32, device="cuda")
        p = ssm._ssd_params(t["x"], t["dt"], t["A"], t["B"], t["C"], chunk, t["D"], t["z"],
                            t["dt_bias"], True, t["h0"], y, hf, "exp_euler")
        rc = fn(ctypes.byref(p), stream)
        assert rc == _lib.SSM_OK, lib.ssm_last_error().decode()
        torch.cuda.synchronize()
        check(y, y_ref, tol, out_bf16=out_bf16, what=f"y vs workspace entry point, call {call}")
        check(hf, h_ref, tol, what=f"h_final vs workspace entry point, call {call}")
        check(y, y_or, tol, out_bf16=out_bf16, what=f"y vs oracle, call {call}")
        check(hf, h_or, tol, what=f"h_final vs oracle, call {call}")
