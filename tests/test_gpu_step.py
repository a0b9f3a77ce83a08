"""GPU parity of the decode step (ssm_state_update) against the float64 oracle, step by
step, and decode-equals-scan on the GPU.  Tolerances as in test_gpu_scan.py."""
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


def _steps(oracle, batch, H, P, N, G, nsteps, dtype, a_per_state=False, disc="exp_euler",
           with_z=True, rows=None, seed=0):
    import torch
    par = synth.step_params(H, N, a_per_state=a_per_state, seed=seed)
    tp = to_device(par)
    st0 = synth.step_state(batch, H, P, N, seed=seed)
    state = torch.from_numpy(st0).cuda()
    ref_state = st0.astype(np.float64)
    if rows is not None:
        ref_state = ref_state[rows]
    fp = par.f64
    tol = TOL_F32 if dtype == synth.F32 else TOL_BF16
    for k in range(nsteps):
        tok = synth.step_tokens(batch, H, P, N, G, step=k, dtype=dtype, with_z=with_z, seed=seed)
        tt = to_device(tok)
        y = ssm.ssm_state_update(state, tt["x"], tt["dt"], tp["A"], tt["B"], tt["C"], D=tp["D"],
                                 z=tt.get("z"), dt_bias=tp["dt_bias"], disc=disc,
                                 out_dtype=torch.float32)
        f = tok.f64
        sel = (lambda a: a) if rows is None else (lambda a: None if a is None else a[rows])
        yr, ref_state = oracle.state_update(ref_state, sel(f("x")), sel(f("dt")), fp("A"),
                                            sel(f("B")), sel(f("C")), D=fp("D"), z=sel(f("z")),
                                            dt_bias=fp("dt_bias"),
                                            disc=1 if disc == "zoh" else 0)
        torch.cuda.synchronize()
        if rows is None:
            yg, sg = to_numpy(y), to_numpy(state)
        else:
            idx = torch.tensor(rows, device=state.device)
            yg, sg = to_numpy(y[idx]), to_numpy(state[idx])
        check(yg, yr, tol, what=f"y step {k}")
        check(sg, ref_state, tol, what=f"state step {k}")


@pytest.mark.parametrize("N", [16, 32, 64, 128, 256, 24])
def test_mamba2_form(oracle_mod, N):
    _steps(oracle_mod, 3, 4, 8, N, 2, 6, synth.BF16)


def test_mamba2_form_fp32_zoh(oracle_mod):
    _steps(oracle_mod, 2, 4, 16, 64, 1, 5, synth.F32, disc="zoh")


def test_mamba1_form(oracle_mod):
    """Mamba-1 decode: heads are channels, headdim 1, A [channels, N]."""
    _steps(oracle_mod, 4, 48, 1, 16, 1, 8, synth.F32, a_per_state=True)


def test_decode_equals_scan_on_gpu():
    """Feeding the scan's inputs one step at a time through ssm_state_update reproduces
    ssm_scan_fwd's outputs and final state (step() equals the full forward)."""
    import torch
    batch, dim, N, L = 2, 64, 16, 40
    inp = synth.mamba1(batch, dim, N, L, dtype=synth.F32, with_z=True, with_h0=True, seed=7)
    t = to_device(inp)
    y, hf = ssm.ssm_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
                             delta_bias=t["delta_bias"], h0=t["h0"], return_final_state=True)
    state = t["h0"].clone().view(batch, dim, 1, N)
    ys = []
    for k in range(L):
        yk = ssm.ssm_state_update(state, t["x"][:, :, k:k + 1].contiguous(),
                                  t["delta"][:, :, k].contiguous(), t["A"],
                                  t["B"][:, :, :, k].contiguous(), t["C"][:, :, :, k].contiguous(),
                                  D=t["D"], z=t["z"][:, :, k:k + 1].contiguous(),
                                  dt_bias=t["delta_bias"])
        ys.append(yk)
    torch.cuda.synchronize()
    check(to_numpy(torch.cat(ys, dim=2)), to_numpy(y), TOL_F32, what="decode vs scan y")
    check(to_numpy(state.view(batch, dim, N)), to_numpy(hf), TOL_F32, what="decode vs scan h")


def test_780m_full_size_every_step(oracle_mod):
    """Decode state update, Mamba2-780m-shaped: batch 64, 48 heads x headdim 64, d_state
    128, 1024 consecutive steps on the GPU.  Two GPU states advance in lockstep from the
    same start, one writing y in float32 and one in bfloat16; after every step each y and
    each whole state is checked against the float64 oracle stepping the same inputs
    (float32 y at the bare 2e-3 max|ref| bound, bfloat16 y with half a bfloat16 ulp)."""
    import torch
    cfg = synth.WORKLOADS["step_780m"]
    batch, H, P, N, G = cfg["batch"], cfg["nheads"], cfg["headdim"], cfg["dstate"], cfg["ngroups"]
    par = synth.step_params(H, N, seed=0)
    tp = to_device(par)
    fp = par.f64
    st0 = synth.step_state(batch, H, P, N, seed=0)
    states = {od: torch.from_numpy(st0).cuda() for od in (torch.float32, torch.bfloat16)}
    ref_state = st0.astype(np.float64)
    for k in range(cfg["steps"]):
        tok = synth.step_tokens(batch, H, P, N, G, step=k, dtype=cfg["dtype"],
                                delta_scale=cfg["delta_scale"], with_z=cfg["with_z"], seed=0)
        tt = to_device(tok)
        ys = {od: ssm.ssm_state_update(st, tt["x"], tt["dt"], tp["A"], tt["B"], tt["C"],
                                       D=tp["D"], z=tt["z"], dt_bias=tp["dt_bias"], out_dtype=od)
              for od, st in states.items()}
        f = tok.f64
        yr, _ = oracle_mod.state_update(ref_state, f("x"), f("dt"), fp("A"), f("B"), f("C"),
                                        D=fp("D"), z=f("z"), dt_bias=fp("dt_bias"), inplace=True)
        torch.cuda.synchronize()
        ref_dev = torch.from_numpy(ref_state).cuda()
        for od in states:
            bf = od == torch.bfloat16
            tag = "bf16" if bf else "f32"
            check(ys[od], yr, TOL_BF16, out_bf16=bf, what=f"y step {k} ({tag} out)")
            check(states[od], ref_dev, TOL_BF16, what=f"state step {k} ({tag} out)")


def _tokens(oracle, batch, H, P, N, G, T, dtype, a_per_state=False, disc="exp_euler", seed=3,
            calls=2):
    """`calls` consecutive ssm_state_update_tokens calls of T tokens each (token-major
    stacks of step_tokens) against T oracle steps each."""
    import torch
    par = synth.step_params(H, N, a_per_state=a_per_state, seed=seed)
    tp = to_device(par)
    st0 = synth.step_state(batch, H, P, N, seed=seed)
    state = torch.from_numpy(st0).cuda()
    ref_state = st0.astype(np.float64)
    fp = par.f64
    tol = TOL_F32 if dtype == synth.F32 else TOL_BF16
    for call in range(calls):
        toks = [synth.step_tokens(batch, H, P, N, G, step=call * T + k, dtype=dtype, seed=seed)
                for k in range(T)]
        stack = {n: np.stack([tk.arrays[n] for tk in toks]) for n in ("x", "dt", "B", "C", "z")}
        if dtype == synth.BF16:  # exact bf16 values, as in tests.helpers.to_device
            dev = {n: torch.from_numpy(synth.bf16_bits(v).view(np.int16).copy()).cuda()
                   .view(torch.bfloat16) for n, v in stack.items()}
        else:
            dev = {n: torch.from_numpy(np.ascontiguousarray(v, np.float32)).cuda()
                   for n, v in stack.items()}
        y = ssm.ssm_state_update_tokens(state, dev["x"], dev["dt"], tp["A"], dev["B"], dev["C"],
                                        D=tp["D"], z=dev["z"], dt_bias=tp["dt_bias"], disc=disc,
                                        out_dtype=torch.float32)
        torch.cuda.synchronize()
        yg = to_numpy(y)
        for k, tk in enumerate(toks):
            f = tk.f64
            yr, ref_state = oracle.state_update(ref_state, f("x"), f("dt"), fp("A"), f("B"), f("C"),
                                                D=fp("D"), z=f("z"), dt_bias=fp("dt_bias"),
                                                disc=1 if disc == "zoh" else 0)
            check(yg[k], yr, tol, what=f"y call {call} token {k}")
        check(to_numpy(state), ref_state, tol, what=f"state after call {call}")


@pytest.mark.parametrize("T", [1, 4, 17])
@pytest.mark.parametrize("N", [128, 16, 24])
def test_tokens_mamba2_form(oracle_mod, T, N):
    """Multi-token decode: T tokens per call, state read and written once, equal to T
    single steps (vector path for N = 16 and 128, scalar path for N = 24)."""
    _tokens(oracle_mod, 3, 6, 16, N, 2, T, synth.BF16)


def test_tokens_fp32_zoh(oracle_mod):
    _tokens(oracle_mod, 2, 4, 8, 64, 1, 5, synth.F32, disc="zoh")


def test_tokens_mamba1_form_large_table(oracle_mod):
    """Mamba-1 form (headdim 1, A [channels, N]) with many tokens: the per-token table
    does not fit in shared memory and the step quantities are computed where used."""
    _tokens(oracle_mod, 2, 96, 1, 16, 1, 64, synth.F32, a_per_state=True, calls=1)


@pytest.mark.parametrize("N,P,T", [(256, 48, 40), (64, 64, 33), (128, 100, 9), (128, 64, 70),
                                   (256, 40, 12), (64, 24, 10)])
def test_tokens_register_kernel_shapes(oracle_mod, N, P, T):
    """The register-resident multi-token kernel (N in 64/128/256): heads that do not
    divide the CTA span (P = 40, 48, 100), CTAs whose rows cross a group, several staged
    token blocks (T > block) and a ragged last token group."""
    _tokens(oracle_mod, 2, 4, P, N, 2, T, synth.BF16, calls=1)


# A hybrid stack for the serving loop: (heads, headdim, dstate, groups, Mamba-1 form).  The
# Mamba-1 form has one channel per head (P = 1) and A per (channel, state).
MIXED_STACK = [
    (96, 1, 16, 1, True),
    (4, 16, 64, 2, False),
    (48, 1, 16, 1, True),
    (6, 8, 128, 1, False),
]


def test_mixed_stack_cuda_graph_serving_loop(oracle_mod):
    """A decode serving loop captured once as a CUDA graph: T tokens, each through a stack
    whose layers alternate the Mamba-1 form and the Mamba-2 form (scalar A per head, two
    groups in one layer).  The graph is replayed twice, every layer's state carried from
    one replay to the next; each y and each state is checked against the oracle stepping
    the same layers in the same order."""
    import torch
    batch, T = 4, 5
    layers = []
    for li, (H, P, N, G, m1) in enumerate(MIXED_STACK):
        par = synth.step_params(H, N, a_per_state=m1, seed=40 + li)
        st0 = synth.step_state(batch, H, P, N, seed=40 + li)
        toks = [synth.step_tokens(batch, H, P, N, G, step=k, seed=40 + li) for k in range(T)]
        layers.append(dict(
            par=par, tp=to_device(par), st0=st0, state=torch.from_numpy(st0).cuda(), toks=toks,
            tt=[to_device(tk) for tk in toks],
            ys=[torch.empty((batch, H, P), dtype=torch.float32, device="cuda") for _ in range(T)]))

    def loop(states):
        for k in range(T):
            for lay, st in zip(layers, states):
                tt, tp = lay["tt"][k], lay["tp"]
                ssm.ssm_state_update(st, tt["x"], tt["dt"], tp["A"], tt["B"], tt["C"], D=tp["D"],
                                     z=tt["z"], dt_bias=tp["dt_bias"], y=lay["ys"][k])

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        loop([lay["state"].clone() for lay in layers])  # first launches outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        loop([lay["state"] for lay in layers])
    ref = [lay["st0"].astype(np.float64) for lay in layers]
    for rep in range(2):
        graph.replay()
        torch.cuda.synchronize()
        for li, lay in enumerate(layers):
            fp = lay["par"].f64
            for k in range(T):
                f = lay["toks"][k].f64
                yr, ref[li] = oracle_mod.state_update(ref[li], f("x"), f("dt"), fp("A"), f("B"),
                                                      f("C"), D=fp("D"), z=f("z"),
                                                      dt_bias=fp("dt_bias"))
                check(to_numpy(lay["ys"][k]), yr, TOL_BF16, what=f"replay {rep} layer {li} token {k}")
            check(to_numpy(lay["state"]), ref[li], TOL_BF16, what=f"replay {rep} layer {li} state")


def test_mamba1_form_bf16_zoh_ragged(oracle_mod):
    """Mamba-1 decode in bf16 with ZOH and dstate 32; 3 x 37 rows do not fill the last
    warp's row slots."""
    _steps(oracle_mod, 3, 37, 1, 32, 1, 4, synth.BF16, a_per_state=True, disc="zoh")


@pytest.mark.parametrize("batch,H,G,dtype,disc,with_z", [
    (3, 37, 1, synth.BF16, "zoh", True),
    (2, 38, 2, synth.F32, "exp_euler", False),
    (64, 3072, 1, synth.BF16, "exp_euler", True),
], ids=["bf16_zoh_ragged", "fp32_two_groups_no_gate", "batch64_3072_channels"])
def test_mamba1_form_dstate16_row_kernel(oracle_mod, batch, H, G, dtype, disc, with_z):
    """Mamba-1 decode at dstate 16 (one row per (batch, channel), four lanes per row):
    rows that do not fill the last warp's slots, two groups of channels sharing B/C, no
    gate, and the hybrid stack's full layer (196,608 rows, several passes per warp)."""
    _steps(oracle_mod, batch, H, 1, 16, G, 3, dtype, a_per_state=True, disc=disc, with_z=with_z)
