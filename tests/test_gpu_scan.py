"""GPU parity of the Mamba-1 selective scan (ssm_scan_fwd) against the float64 oracle.

Inputs come from the seeded generator; the oracle reads the identical values.  The
tolerance is max|y_gpu - y_ref| <= 1e-5 max|y_ref| for float32 inputs and
2e-3 max|y_ref| for bfloat16 inputs with float32 state (the same for h_final); a
bfloat16 output may in addition differ by the half-ulp of its own rounding.
"""
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


def run_gpu(inp, out_dtype=None, disc="exp_euler", final=True, h0=True, softplus=True, **opts):
    import torch
    t = to_device(inp)
    od = {"bf16": torch.bfloat16, "f32": torch.float32}[out_dtype] if out_dtype else None
    y, hf = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t.get("D"),
                             z=t.get("z"), delta_bias=t["delta_bias"], delta_softplus=softplus,
                             h0=t.get("h0") if h0 else None, out_dtype=od,
                             return_final_state=True, disc=disc, **opts)
    torch.cuda.synchronize()
    return to_numpy(y), to_numpy(hf)


def run_oracle(oracle, inp, disc=0, h0=True, rows=None, softplus=True):
    f = inp.f64
    x, dl, z = f("x"), f("delta"), f("z")
    B, C, h0a = f("B"), f("C"), f("h0") if h0 else None
    A, D, bias = f("A"), f("D"), f("delta_bias")
    if rows is not None:  # a sample of (b, d) channels, run one at a time
        ys, hs = [], []
        for b, d in rows:
            y, h = oracle.mamba1_scan(x[b:b + 1, d:d + 1], dl[b:b + 1, d:d + 1], A[d:d + 1],
                                      B[b:b + 1, :1] if B.shape[1] == 1 else
                                      B[b:b + 1, d // (x.shape[1] // B.shape[1])][:, None],
                                      C[b:b + 1, :1] if C.shape[1] == 1 else
                                      C[b:b + 1, d // (x.shape[1] // C.shape[1])][:, None],
                                      D=None if D is None else D[d:d + 1],
                                      z=None if z is None else z[b:b + 1, d:d + 1],
                                      delta_bias=bias[d:d + 1], delta_softplus=softplus,
                                      h0=None if h0a is None else h0a[b:b + 1, d:d + 1], disc=disc)
            ys.append(y[0, 0])
            hs.append(h[0, 0])
        return np.stack(ys), np.stack(hs)
    return oracle.mamba1_scan(x, dl, A, B, C, D=D, z=z, delta_bias=bias, delta_softplus=softplus,
                              h0=h0a, disc=disc)


def test_tiny_fp32_config(oracle_mod):
    """Mamba-1 selective scan fwd, tiny, fp32: batch 1, d_inner 64, d_state 16, L 256."""
    inp = synth.mamba1(1, 64, 16, 256, dtype=synth.F32, delta_scale=0.5, with_z=False, seed=0)
    y, hf = run_gpu(inp, h0=False)
    yr, hr = run_oracle(oracle_mod, inp, h0=False)
    check(y, yr, TOL_F32, what="y")
    check(hf, hr, TOL_F32, what="h_final")


BF16_KERNELS = [("tmem", 4), ("tma", 2), ("tma", 4), ("tiled", 1), ("tiled", 2), ("tiled", 4)]


@pytest.mark.parametrize("kernel,tpc", BF16_KERNELS)
@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_bf16_kernels_multi_cta_ragged(oracle_mod, kernel, tpc, out):
    """Each bf16 kernel and threads-per-channel choice (named through ssm_scan_fwd_ex's
    options): several CTAs, CTAs spanning a batch boundary, a ragged last tile, z, D, h0."""
    inp = synth.mamba1(3, 200, 16, 136, dtype=synth.BF16, delta_scale=1.0, with_z=True,
                       with_h0=True, seed=1)
    y, hf = run_gpu(inp, out_dtype=out, kernel=kernel, threads_per_channel=tpc)
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_BF16, out_bf16=(out == "bf16"), what="y")
    check(hf, hr, TOL_BF16, what="h_final")


@pytest.mark.parametrize("path", ["tmem", "tma", "tiled"])
def test_bf16_softplus_extremes(oracle_mod, path):
    """delta + bias spread over about +-40: softplus in its linear range (v > 20), near 0
    and vanishing (v < -14, where the fast form may return 0), on each bf16 kernel."""
    inp = synth.mamba1(2, 96, 16, 200, dtype=synth.BF16, delta_scale=14.0, with_z=True,
                       with_h0=True, seed=11)
    y, hf = run_gpu(inp, out_dtype="f32", kernel=path)
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_BF16, what="y")
    check(hf, hr, TOL_BF16, what="h_final")


@pytest.mark.parametrize("tpc", [2, 4])
def test_fp32_tiled_with_gate_and_groups(oracle_mod, tpc):
    inp = synth.mamba1(2, 320, 16, 100, dtype=synth.F32, with_z=True, with_h0=True, ngroups=2,
                       seed=2)
    y, hf = run_gpu(inp, out_dtype="f32", kernel="tiled", threads_per_channel=tpc)
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_F32, what="y")
    check(hf, hr, TOL_F32, what="h_final")


@pytest.mark.parametrize("L,N,dtype,disc", [
    (33, 16, synth.BF16, "exp_euler"),   # row not a whole number of 16-byte chunks
    (31, 5, synth.F32, "exp_euler"),     # dstate outside the tiled set
    (64, 16, synth.F32, "zoh"),          # ZOH discretisation
    (17, 40, synth.BF16, "zoh"),
    (1, 16, synth.F32, "exp_euler"),
    (2, 3, synth.F32, "exp_euler"),
])
def test_generic_path(oracle_mod, L, N, dtype, disc):
    inp = synth.mamba1(2, 12, N, L, dtype=dtype, with_z=True, with_h0=True, seed=3)
    y, hf = run_gpu(inp, disc=disc)
    yr, hr = run_oracle(oracle_mod, inp, disc=1 if disc == "zoh" else 0)
    tol = TOL_F32 if dtype == synth.F32 else TOL_BF16
    check(y, yr, tol, out_bf16=(dtype == synth.BF16), what="y")
    check(hf, hr, tol, what="h_final")


def test_no_softplus_no_skip(oracle_mod):
    inp = synth.mamba1(2, 40, 16, 64, dtype=synth.F32, with_D=False, seed=4)
    # without softplus the step is delta + bias: keep it positive
    inp.arrays["delta"] = np.abs(inp.arrays["delta"]) * 0.1
    inp.arrays["delta_bias"] = np.full_like(inp.arrays["delta_bias"], 0.01)
    y, hf = run_gpu(inp, h0=False, softplus=False)
    yr, hr = run_oracle(oracle_mod, inp, h0=False, softplus=False)
    check(y, yr, TOL_F32, what="y")
    check(hf, hr, TOL_F32, what="h_final")


def test_empty_sequence_copies_state():
    import torch
    inp = synth.mamba1(2, 8, 16, 0, dtype=synth.BF16, with_h0=True, seed=5)
    y, hf = run_gpu(inp)
    assert y.shape == (2, 8, 0)
    assert np.array_equal(hf, inp.arrays["h0"].astype(np.float64))


def test_split_continuation_matches_full(oracle_mod):
    """scan(0:L) equals scan(0:k) followed by scan(k:L) from the carried state."""
    import torch
    inp = synth.mamba1(2, 64, 16, 256, dtype=synth.F32, with_z=True, with_h0=True, seed=6)
    t = to_device(inp)
    y, hf = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                             delta_bias=t["delta_bias"], h0=t["h0"], return_final_state=True)
    k = 96
    part = {n: t[n][..., :k].contiguous() for n in ("x", "delta", "z", "B", "C")}
    rest = {n: t[n][..., k:].contiguous() for n in ("x", "delta", "z", "B", "C")}
    y1, h1 = ssm.ssm_scan_fwd(part["x"], part["delta"], t["A"], part["B"], part["C"], D=t["D"],
                              z=part["z"], delta_bias=t["delta_bias"], h0=t["h0"],
                              return_final_state=True)
    y2, h2 = ssm.ssm_scan_fwd(rest["x"], rest["delta"], t["A"], rest["B"], rest["C"], D=t["D"],
                              z=rest["z"], delta_bias=t["delta_bias"], h0=h1,
                              return_final_state=True)
    torch.cuda.synchronize()
    yr, hr = run_oracle(oracle_mod, inp)
    check(to_numpy(torch.cat([y1, y2], dim=-1)), yr, TOL_F32, what="y split")
    check(to_numpy(h2), hr, TOL_F32, what="h split")


def _full_size(oracle, inp, what):
    """Runs the GPU scan twice on the same inputs, with a float32 output (checked at the
    bare arithmetic bound, 2e-3 max|ref|) and with a bfloat16 output (the same bound plus
    half a bfloat16 ulp of each reference value), and checks every element of y and of
    the final state against one float64 oracle run."""
    import torch
    t = to_device(inp)
    outs = {}
    for od in (torch.float32, torch.bfloat16):
        y, hf = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t.get("D"),
                                 z=t.get("z"), delta_bias=t["delta_bias"], out_dtype=od,
                                 return_final_state=True)
        outs[od] = (y, hf)
    torch.cuda.synchronize()
    yr, hr = run_oracle(oracle, inp, h0=False)
    for od, (y, hf) in outs.items():
        bf = od == torch.bfloat16
        check(y, yr, TOL_BF16, out_bf16=bf, what=f"{what} y ({'bf16' if bf else 'f32'} out)")
        check(hf, hr, TOL_BF16, what=f"{what} h_final ({'bf16' if bf else 'f32'} out)")


def test_130m_layer_full_size(oracle_mod):
    """Mamba-1 130m-shaped layer scan (batch 8, d_inner 1536, d_state 16, L 2048, bf16, z),
    in the launch configuration the benchmark times: every element of y and h_final."""
    cfg = synth.WORKLOADS["m1_130m_layer"]
    inp = synth.mamba1(cfg["batch"], cfg["dim"], cfg["dstate"], cfg["seqlen"], dtype=cfg["dtype"],
                       delta_scale=cfg["delta_scale"], with_z=cfg["with_z"], seed=0)
    _full_size(oracle_mod, inp, "130m layer")


@pytest.mark.parametrize("L", [1024, 4096, 16384, 32768])
def test_790m_long_context_full_size(oracle_mod, L):
    """Long-context sweep, Mamba-1 790m-shaped: batch 1, d_inner 3072, d_state 16, no z,
    h_final out; every element of y and h_final at each sweep length."""
    cfg = synth.WORKLOADS["m1_790m_long"]
    inp = synth.mamba1(cfg["batch"], cfg["dim"], cfg["dstate"], L, dtype=cfg["dtype"],
                       delta_scale=cfg["delta_scale"], with_z=False, seed=0)
    _full_size(oracle_mod, inp, f"790m L={L}")


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_time_split_many_segments(oracle_mod, out):
    """One batch row with few channels and a long sequence: the bf16 path splits the
    sequence into many time segments (a segment pass, then each segment starts from h0
    carried through the earlier ones).  Gate, initial state, non-uniform A, every channel
    checked, ragged length."""
    inp = synth.mamba1(1, 256, 16, 4096 - 64 + 16, dtype=synth.BF16, with_z=True,
                       with_h0=True, seed=11)
    inp.arrays["A"] = -np.exp(np.random.default_rng(12).uniform(-1.0, 2.5, (256, 16))
                              ).astype(np.float32)
    y, hf = run_gpu(inp, out_dtype=out)
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_BF16, out_bf16=(out == "bf16"), what="y")
    check(hf, hr, TOL_BF16, what="h_final")


def test_plain_entry_point_needs_no_scratch(oracle_mod):
    """ssm_scan_fwd(p, stream), called through the C ABI: one batch row with few channels
    and a long sequence, a shape that ssm_scan_fwd_ex splits in time through a workspace,
    runs in one pass without scratch and matches the oracle."""
    import ctypes
    import torch
    from selective_scan_mamba_gb300 import _lib
    inp = synth.mamba1(1, 256, 16, 4096, dtype=synth.BF16, with_z=True, with_h0=True, seed=13)
    t = to_device(inp)
    assert ssm.ssm_scan_workspace_size(t["x"], t["B"]) > 0  # the _ex plan would split
    y = torch.empty_like(t["x"])
    hf = torch.empty((1, 256, 16), dtype=torch.float32, device="cuda")
    p = ssm._scan_params(t["x"], t["delta"], t["A"], t["B"], t["C"], t["D"], t["z"],
                         t["delta_bias"], True, t["h0"], y, hf, "exp_euler")
    lib = _lib.load()
    rc = lib.ssm_scan_fwd(ctypes.byref(p), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _lib.SSM_OK, lib.ssm_last_error().decode()
    torch.cuda.synchronize()
    yr, hr = run_oracle(oracle_mod, inp)
    check(y, yr, TOL_BF16, out_bf16=True, what="y")
    check(hf, hr, TOL_BF16, what="h_final")


def test_same_buffers_with_another_shape(oracle_mod):
    """Tensor maps are cached by address, shape and box: the same allocations read as
    another (batch, dim, L) must not reuse a map of the first shape."""
    import torch
    first = synth.mamba1(2, 96, 16, 512, dtype=synth.BF16, delta_scale=0.8, with_z=True, with_h0=True,
                         seed=41)
    second = synth.mamba1(3, 40, 16, 768, dtype=synth.BF16, delta_scale=0.8, with_z=True, seed=42)
    pools = {}
    for inp in (first, second):
        t = to_device(inp)
        for k, v in t.items():
            flat = v.reshape(-1)
            if k not in pools or pools[k].numel() < flat.numel():
                pools[k] = torch.empty(max(flat.numel(), 4096), dtype=v.dtype, device="cuda")
    for inp in (first, second, first):
        t = {k: pools[k][:v.numel()].view(v.shape).copy_(v) for k, v in to_device(inp).items()}
        y, hf = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                                 delta_bias=t["delta_bias"], h0=t.get("h0"), out_dtype=torch.float32,
                                 return_final_state=True)
        torch.cuda.synchronize()
        yr, hr = run_oracle(oracle_mod, inp)
        check(to_numpy(y), yr, TOL_BF16, what="y")
        check(to_numpy(hf), hr, TOL_BF16, what="h_final")


def test_large_small_large_shared_memory(oracle_mod):
    """The TMEM kernel's shared memory grows with its channels per CTA: a large problem,
    a small one, then the large one again must each launch (the kernel's shared-memory
    limit is only ever raised) and match the oracle."""
    big = synth.mamba1(8, 1536, 16, 128, dtype=synth.BF16, delta_scale=0.8, with_z=True, seed=51)
    small = synth.mamba1(1, 256, 16, 128, dtype=synth.BF16, delta_scale=0.8, with_z=True, seed=52)
    for inp in (big, small, big):
        y, hf = run_gpu(inp, out_dtype="f32", h0=False, kernel="tmem")
        yr, hr = run_oracle(oracle_mod, inp, h0=False)
        check(y, yr, TOL_BF16, what="y")
        check(hf, hr, TOL_BF16, what="h_final")


def test_zz_no_device_wait_gave_up():
    """Every bounded wait in the kernels above completed (timeout counter still zero)."""
    assert ssm.wait_timeouts() == 0
