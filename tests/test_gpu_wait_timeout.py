"""A bounded device-side wait that runs out is reported, and the GPU stays usable.

The Mamba-1 TMEM kernel's testing hook (ssm_scan_opts.fault_test = 1) never issues the
input copy of the second 64-step tile, so nothing ever arrives on that tile's mbarrier.
Every wait for it polls wait_limit times and gives up; the block then stops issuing
copies and MMAs, lets the ones it issued before land, frees its tensor memory and
finishes.  The kernel neither faults nor hangs: the call returns SSM_OK (it is
asynchronous) and ssm_device_status() then reports SSM_ERR_TIMEOUT, once.  A normal call
afterwards runs correctly and the status is clean again.
"""
import ctypes

import pytest

import selective_scan_mamba_gb300 as ssm
from selective_scan_mamba_gb300 import _lib, synth
from tests.helpers import TOL_BF16, check, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _needs_gpu():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")


def _scan(t, y, **opts):
    return ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                            delta_bias=t["delta_bias"], y=y, **opts)


def test_wait_that_runs_out_is_reported_and_the_gpu_recovers(oracle_mod):
    import torch
    lib = _lib.load()
    assert lib.ssm_device_status() == _lib.SSM_OK, lib.ssm_last_error().decode()
    # four 64-step tiles, a few CTAs; the TMEM kernel in one pass (no time split)
    inp = synth.mamba1(2, 192, 16, 256, dtype=synth.BF16, with_z=True, seed=31)
    t = to_device(inp)
    y = torch.empty_like(t["x"])
    _scan(t, y, kernel="tmem", max_segments=1, wait_limit=1 << 12, fault_test=1)
    rc = lib.ssm_device_status()
    assert rc == _lib.SSM_ERR_TIMEOUT, (rc, lib.ssm_last_error().decode())
    msg = lib.ssm_last_error().decode()
    assert "TMEM kernel" in msg and "not valid" in msg
    # the record was cleared by reading it
    assert lib.ssm_device_status() == _lib.SSM_OK
    # the same call without the hook is correct, and nothing gives up
    _scan(t, y, kernel="tmem", max_segments=1)
    ssm.device_status()
    f = inp.f64
    yr, _ = oracle_mod.mamba1_scan(f("x"), f("delta"), f("A"), f("B"), f("C"), D=f("D"), z=f("z"),
                                   delta_bias=f("delta_bias"))
    check(y, yr, TOL_BF16, out_bf16=True, what="y after the timed-out call")


def test_binding_raises_on_a_timed_out_call():
    import torch
    inp = synth.mamba1(1, 64, 16, 192, dtype=synth.BF16, with_z=True, seed=32)
    t = to_device(inp)
    y = torch.empty_like(t["x"])
    _scan(t, y, kernel="tmem", max_segments=1, wait_limit=1 << 10, fault_test=1)
    with pytest.raises(ssm.SsmError) as err:
        ssm.device_status()
    assert err.value.status == _lib.SSM_ERR_TIMEOUT
    ssm.device_status()  # cleared


def test_fault_hook_refused_where_it_cannot_apply():
    """The hook needs the TMEM kernel and at least two tiles; otherwise the call is refused
    on the host and nothing runs."""
    inp = synth.mamba1(1, 64, 16, 64, dtype=synth.BF16, with_z=True, seed=33)
    t = to_device(inp)
    with pytest.raises(ssm.SsmError) as err:
        _scan(t, None, kernel="tmem", fault_test=1)
    assert err.value.status == _lib.SSM_ERR_UNSUPPORTED
    lib = _lib.load()
    p = ssm._scan_params(t["x"], t["delta"], t["A"], t["B"], t["C"], None, None, t["delta_bias"],
                         True, None, t["x"].new_empty(t["x"].shape), None, "exp_euler")
    o = ssm.scan_opts(kernel="generic", fault_test=1)
    assert lib.ssm_scan_fwd_ex(ctypes.byref(p), ctypes.byref(o), None, 0, None) == \
        _lib.SSM_ERR_UNSUPPORTED
