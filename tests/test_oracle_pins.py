"""Pins for the float64 oracle, against facts that do not come from the oracle.

Each check ties the oracle to something fixed by the pages or by mathematics:
high-precision references (mpmath), brute-force unrolled sums written here
independently, closed forms, chunked-versus-sequential agreement, split
continuation, decode-versus-scan agreement and degenerate cases.  They are
chosen so that a dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one of them (see test_oracle_mutations.py,
which plants such mistakes in a copy of the oracle and checks they are caught).
"""
import math

import mpmath
import numpy as np
import pytest

from selective_scan_mamba_gb300 import synth

mpmath.mp.dps = 50


def rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / scale)


# ----------------------------------------------------------------------------------------
# P9: softplus and the inverse softplus used by the input recipe
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("v", [-745.0, -60.0, -20.0, -5.0, -1e-3, 0.0, 1e-8, 0.7, 3.0, 19.9,
                               20.1, 50.0, 700.0])
def test_softplus_matches_high_precision(oracle_mod, v):
    ref = float(mpmath.log1p(mpmath.exp(mpmath.mpf(v))))
    got = oracle_mod.softplus(v)
    assert abs(got - ref) <= 4e-16 * abs(ref) + 1e-320


def test_inverse_softplus_round_trip(oracle_mod):
    u = np.exp(np.linspace(math.log(1e-3), math.log(1e-1), 41))
    b = synth.inv_softplus(u)
    back = np.array([oracle_mod.softplus(v) for v in b])
    assert np.max(np.abs(back - u) / u) <= 1e-15


# ----------------------------------------------------------------------------------------
# P1: phi1(z) = (e^z - 1)/z with the Taylor switch at |z| < 1e-4
#     ("From S4 to Mamba-3", Likely questions Q01)
# ----------------------------------------------------------------------------------------
def _phi1_ref(zv):
    zv = mpmath.mpf(zv)
    return float(mpmath.expm1(zv) / zv) if zv != 0 else 1.0


def test_phi1_log_grid(oracle_mod):
    grid = np.concatenate([-np.logspace(-12, math.log10(50.0), 120),
                           np.logspace(-12, 0, 80)])
    worst = 0.0
    for zv in grid:
        ref = _phi1_ref(zv)
        worst = max(worst, abs(oracle_mod.phi1(zv) - ref) / abs(ref))
    # exp(z)-1 in double loses at most ~2^-53/|z| relative for |z| >= 1e-4,
    # and the Taylor cut adds at most |z|^3/24 below it.
    assert worst < 3e-12


def test_phi1_special_values(oracle_mod):
    assert oracle_mod.phi1(0.0) == 1.0
    lo = oracle_mod.phi1(np.nextafter(1e-4, 0.0))
    hi = oracle_mod.phi1(1e-4)
    assert abs(lo - hi) < 1e-11
    lo = oracle_mod.phi1(-np.nextafter(1e-4, 0.0))
    hi = oracle_mod.phi1(-1e-4)
    assert abs(lo - hi) < 1e-11


def test_zoh_steady_state(oracle_mod):
    """Constant input under ZOH has the fixed point h = -B x / A whatever the step
    size: started there, the state stays there; started at zero it approaches it
    as h_inf (1 - abar^t)."""
    L, N = 400, 3
    A = np.array([[-0.5, -2.0, -7.0]])
    Bv = np.array([0.3, -1.1, 2.0])
    h_inf = -Bv * 1.7 / A[0]
    for dval in (1e-6, 0.01, 0.3):
        x = np.full((1, 1, L), 1.7)
        delta = np.full((1, 1, L), dval)
        B = np.tile(Bv[None, None, :, None], (1, 1, 1, L))
        C = np.tile(np.eye(N)[None, None, :, :1], (1, 1, 1, L))  # y reads h[0]
        y, hf = oracle_mod.mamba1_scan(x, delta, A, B, C, delta_softplus=False,
                                       h0=h_inf[None, None], disc=oracle_mod.DISC_ZOH)
        assert rel_err(hf[0, 0], h_inf) < 1e-13
        assert np.max(np.abs(y[0, 0] - h_inf[0])) < 1e-13 * abs(h_inf[0])
        _, hf = oracle_mod.mamba1_scan(x, delta, A, B, C, delta_softplus=False,
                                       disc=oracle_mod.DISC_ZOH)
        expect = h_inf * (1.0 - np.exp(dval * A[0] * L))
        assert rel_err(hf[0, 0], expect) < 1e-11


# ----------------------------------------------------------------------------------------
# P2: brute-force unrolled sums on tiny inputs
# ----------------------------------------------------------------------------------------
def _brute_mamba1(x, raw, bias, A, B, C, D, z, h0, zoh, softplus=True):
    """y_t = sum_{s<=t} C_t (prod_{r=s+1..t} e^{D_r A}) w_s B_s x_s
             + C_t (prod_{r<=t} e^{D_r A}) h0 + D x_t, gated; h_L likewise."""
    batch, dim, L = x.shape
    G, N = B.shape[1], B.shape[2]
    per = dim // G
    y = np.zeros((batch, dim, L))
    hL = np.zeros((batch, dim, N))

    def sp(v):
        return math.log1p(math.exp(v)) if v < 30 else v + math.log1p(math.exp(-v))

    for b in range(batch):
        for d in range(dim):
            g = d // per
            dl = [(sp(raw[b, d, t] + bias[d]) if softplus else raw[b, d, t] + bias[d])
                  for t in range(L)]

            def decay(n, s0, t1):  # product of e^{dl_r A} for r in (s0, t1]
                p = 1.0
                for r in range(s0 + 1, t1 + 1):
                    p *= math.exp(dl[r] * A[d, n])
                return p

            def wgt(n, s):
                if not zoh:
                    return dl[s]
                zz = dl[s] * A[d, n]
                return dl[s] * (math.expm1(zz) / zz if zz != 0 else 1.0)

            for t in range(L):
                acc = 0.0
                for n in range(N):
                    for s in range(t + 1):
                        acc += C[b, g, n, t] * decay(n, s, t) * wgt(n, s) * B[b, g, n, s] * x[b, d, s]
                    acc += C[b, g, n, t] * decay(n, -1, t) * h0[b, d, n]
                acc += D[d] * x[b, d, t]
                if z is not None:
                    acc *= z[b, d, t] / (1.0 + math.exp(-z[b, d, t]))
                y[b, d, t] = acc
            for n in range(N):
                s_ = sum(decay(n, s, L - 1) * wgt(n, s) * B[b, g, n, s] * x[b, d, s] for s in range(L))
                hL[b, d, n] = s_ + decay(n, -1, L - 1) * h0[b, d, n]
    return y, hL


@pytest.mark.parametrize("zoh", [False, True])
@pytest.mark.parametrize("gated", [False, True])
def test_mamba1_brute_force(oracle_mod, zoh, gated):
    rng = np.random.default_rng(7)
    batch, dim, N, L, G = 2, 4, 3, 7, 2
    x = rng.standard_normal((batch, dim, L))
    raw = rng.standard_normal((batch, dim, L))
    bias = rng.standard_normal(dim) * 0.3
    A = -rng.uniform(0.2, 3.0, (dim, N))
    B = rng.standard_normal((batch, G, N, L))
    C = rng.standard_normal((batch, G, N, L))
    D = rng.standard_normal(dim)
    z = rng.standard_normal((batch, dim, L)) if gated else None
    h0 = rng.standard_normal((batch, dim, N))
    y, hf = oracle_mod.mamba1_scan(x, raw, A, B, C, D=D, z=z, delta_bias=bias, h0=h0,
                                   disc=oracle_mod.DISC_ZOH if zoh else oracle_mod.DISC_EXP_EULER)
    yb, hb = _brute_mamba1(x, raw, bias, A, B, C, D, z, h0, zoh)
    assert rel_err(y, yb) < 1e-13
    assert rel_err(hf, hb) < 1e-13


def _brute_ssd(x, raw, bias, A, B, C, D, z, h0, zoh=False):
    """y_t[p] = sum_{s<=t} sum_n C_t[n] e^{A sum_{r=s+1..t} D_r} w_s x_s[p] B_s[n]
               + sum_n C_t[n] e^{A sum_{r<=t} D_r} h0[p,n] + D x_t[p], gated."""
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    per = H // G
    y = np.zeros_like(x)
    for b in range(batch):
        for h in range(H):
            g = h // per
            dl = [math.log1p(math.exp(raw[b, t, h] + bias[h])) for t in range(L)]
            cs = np.concatenate([[0.0], np.cumsum(dl)])  # cs[k] = sum of first k steps
            for t in range(L):
                for p in range(P):
                    acc = 0.0
                    for s in range(t + 1):
                        w = dl[s]
                        if zoh:
                            zz = dl[s] * A[h]
                            w = dl[s] * math.expm1(zz) / zz
                        cb = sum(C[b, t, g, n] * B[b, s, g, n] for n in range(N))
                        acc += cb * math.exp(A[h] * (cs[t + 1] - cs[s + 1])) * w * x[b, s, h, p]
                    acc += math.exp(A[h] * cs[t + 1]) * sum(C[b, t, g, n] * h0[b, h, p, n]
                                                            for n in range(N))
                    acc += D[h] * x[b, t, h, p]
                    if z is not None:
                        acc *= z[b, t, h, p] / (1.0 + math.exp(-z[b, t, h, p]))
                    y[b, t, h, p] = acc
    return y


@pytest.mark.parametrize("zoh", [False, True])
def test_ssd_brute_force(oracle_mod, zoh):
    rng = np.random.default_rng(11)
    batch, L, H, P, N, G = 2, 6, 4, 3, 5, 2
    x = rng.standard_normal((batch, L, H, P))
    raw = rng.standard_normal((batch, L, H))
    bias = rng.standard_normal(H) * 0.3
    A = -rng.uniform(0.5, 4.0, H)
    B = rng.standard_normal((batch, L, G, N))
    C = rng.standard_normal((batch, L, G, N))
    D = rng.standard_normal(H)
    z = rng.standard_normal((batch, L, H, P))
    h0 = rng.standard_normal((batch, H, P, N))
    yb = _brute_ssd(x, raw, bias, A, B, C, D, z, h0, zoh)
    disc = oracle_mod.DISC_ZOH if zoh else oracle_mod.DISC_EXP_EULER
    ys, _ = oracle_mod.ssd_sequential(x, raw, A, B, C, D=D, z=z, dt_bias=bias, h0=h0, disc=disc)
    assert rel_err(ys, yb) < 1e-13
    for q in (1, 2, 4, 5, 6, 8):
        yc, _ = oracle_mod.ssd_chunked(x, raw, A, B, C, q, D=D, z=z, dt_bias=bias, h0=h0,
                                       disc=disc)
        assert rel_err(yc, yb) < 1e-13


# ----------------------------------------------------------------------------------------
# P3: geometric closed forms with constant Delta, B, C
# ----------------------------------------------------------------------------------------
def test_step_response_closed_form(oracle_mod):
    L, N = 300, 4
    Avals = np.array([-0.1, -1.0, -3.0, -9.0])
    dval, xval = 0.05, 0.8
    Bv = np.array([1.0, -0.5, 2.0, 0.25])
    Cv = np.array([0.3, 1.2, -0.7, 2.0])
    h0 = np.array([0.4, -1.0, 0.0, 3.0])
    x = np.full((1, 1, L), xval)
    delta = np.full((1, 1, L), dval)
    B = np.tile(Bv[None, None, :, None], (1, 1, 1, L))
    C = np.tile(Cv[None, None, :, None], (1, 1, 1, L))
    y, hf = oracle_mod.mamba1_scan(x, delta, Avals[None], B, C, D=np.array([0.6]),
                                   h0=h0[None, None], delta_softplus=False)
    abar = np.exp(dval * Avals)
    t = np.arange(1, L + 1)[:, None]
    h_t = dval * Bv * xval * (1 - abar ** t) / (1 - abar) + abar ** t * h0
    y_ref = h_t @ Cv + 0.6 * xval
    assert rel_err(y[0, 0], y_ref) < 1e-12
    assert rel_err(hf[0, 0], h_t[-1]) < 1e-12


def test_impulse_response_closed_form(oracle_mod):
    L, N = 200, 3
    Avals = np.array([-0.2, -1.5, -4.0])
    dval = 0.1
    Bv = np.array([1.0, 2.0, -1.0])
    Cv = np.array([0.5, -0.25, 3.0])
    x = np.zeros((1, 1, L))
    x[0, 0, 0] = 1.0
    delta = np.full((1, 1, L), dval)
    B = np.tile(Bv[None, None, :, None], (1, 1, 1, L))
    C = np.tile(Cv[None, None, :, None], (1, 1, 1, L))
    y, _ = oracle_mod.mamba1_scan(x, delta, Avals[None], B, C, delta_softplus=False)
    t = np.arange(L)[:, None]
    y_ref = (Cv * np.exp(dval * Avals) ** t * dval * Bv).sum(axis=1)
    assert rel_err(y[0, 0], y_ref) < 1e-12


# ----------------------------------------------------------------------------------------
# P4: chunked SSD equals the sequential scan, aligned and misaligned chunk sizes
#     ("From S4 to Mamba-3", 04/Approach and 09/Validation)
# ----------------------------------------------------------------------------------------
@pytest.mark.parametrize("L,Q", [(96, 32), (96, 64), (300, 64), (300, 256), (257, 1), (4059, 256),
                                 (0, 64)])
def test_ssd_chunked_equals_sequential(oracle_mod, L, Q):
    inp = synth.ssd(2, L, 4, 8, 16, 2, dtype=synth.F32, with_z=True, with_h0=True, seed=3)
    f = inp.f64
    ys, hs = oracle_mod.ssd_sequential(f("x"), f("dt"), f("A"), f("B"), f("C"), D=f("D"),
                                       z=f("z"), dt_bias=f("dt_bias"), h0=f("h0"))
    yc, hc = oracle_mod.ssd_chunked(f("x"), f("dt"), f("A"), f("B"), f("C"), Q, D=f("D"),
                                    z=f("z"), dt_bias=f("dt_bias"), h0=f("h0"))
    if L:
        assert rel_err(yc, ys) < 1e-12
    assert rel_err(hc, hs) < 1e-12


# ----------------------------------------------------------------------------------------
# P5: Mamba-2 is the special case of Mamba-1 with A, Delta shared across a head's channels
# ----------------------------------------------------------------------------------------
def test_ssd_is_mamba1_special_case(oracle_mod):
    batch, L, H, P, N = 2, 50, 3, 4, 6
    inp = synth.ssd(batch, L, H, P, N, 1, dtype=synth.F32, with_z=True, with_h0=True, seed=5)
    f = inp.f64
    ys, hs = oracle_mod.ssd_sequential(f("x"), f("dt"), f("A"), f("B"), f("C"), D=f("D"),
                                       z=f("z"), dt_bias=f("dt_bias"), h0=f("h0"))
    dim = H * P
    x1 = f("x").reshape(batch, L, dim).transpose(0, 2, 1)
    z1 = f("z").reshape(batch, L, dim).transpose(0, 2, 1)
    dt1 = np.repeat(f("dt"), P, axis=2).transpose(0, 2, 1)
    A1 = np.repeat(np.repeat(f("A")[:, None], P, axis=0), N, axis=1)
    B1 = f("B").transpose(0, 2, 3, 1)  # [batch, G=1, N, L]
    C1 = f("C").transpose(0, 2, 3, 1)
    D1 = np.repeat(f("D"), P)
    bias1 = np.repeat(f("dt_bias"), P)
    h01 = f("h0").reshape(batch, dim, N)
    y1, h1 = oracle_mod.mamba1_scan(x1, dt1, A1, B1, C1, D=D1, z=z1, delta_bias=bias1, h0=h01)
    assert rel_err(y1.transpose(0, 2, 1).reshape(batch, L, H, P), ys) < 1e-13
    assert rel_err(h1.reshape(batch, H, P, N), hs) < 1e-13


# ----------------------------------------------------------------------------------------
# P6: split continuation and decode-equals-scan ("From S4 to Mamba-3", 09/Validation:
#     step() equals a full forward)
# ----------------------------------------------------------------------------------------
def test_mamba1_split_continuation(oracle_mod):
    inp = synth.mamba1(2, 5, 4, 90, dtype=synth.F32, with_z=True, with_h0=True, ngroups=1, seed=9)
    f = inp.f64
    y, hf = oracle_mod.mamba1_scan(f("x"), f("delta"), f("A"), f("B"), f("C"), D=f("D"),
                                   z=f("z"), delta_bias=f("delta_bias"), h0=f("h0"))
    for k in (0, 1, 37, 89, 90):
        y1, h1 = oracle_mod.mamba1_scan(f("x")[..., :k], f("delta")[..., :k], f("A"),
                                        f("B")[..., :k], f("C")[..., :k], D=f("D"),
                                        z=f("z")[..., :k], delta_bias=f("delta_bias"), h0=f("h0"))
        y2, h2 = oracle_mod.mamba1_scan(f("x")[..., k:], f("delta")[..., k:], f("A"),
                                        f("B")[..., k:], f("C")[..., k:], D=f("D"),
                                        z=f("z")[..., k:], delta_bias=f("delta_bias"), h0=h1)
        assert rel_err(np.concatenate([y1, y2], axis=-1), y) < 1e-13
        assert rel_err(h2, hf) < 1e-13


def test_mamba1_decode_equals_scan(oracle_mod):
    batch, dim, N, L = 2, 6, 5, 40
    inp = synth.mamba1(batch, dim, N, L, dtype=synth.F32, with_z=True, with_h0=True, seed=13)
    f = inp.f64
    A = f("A") * np.linspace(0.3, 2.0, dim)[:, None]  # a general (non-structured) A
    y, hf = oracle_mod.mamba1_scan(f("x"), f("delta"), A, f("B"), f("C"), D=f("D"), z=f("z"),
                                   delta_bias=f("delta_bias"), h0=f("h0"))
    state = f("h0")[:, :, None, :]  # heads = channels, headdim 1
    for t in range(L):
        ys, state = oracle_mod.state_update(state, f("x")[:, :, t:t + 1], f("delta")[:, :, t], A,
                                            f("B")[:, :, :, t], f("C")[:, :, :, t], D=f("D"),
                                            z=f("z")[:, :, t:t + 1], dt_bias=f("delta_bias"))
        assert rel_err(ys[:, :, 0], y[:, :, t]) < 1e-13
    assert rel_err(state[:, :, 0, :], hf) < 1e-13


@pytest.mark.parametrize("zoh", [False, True])
def test_ssd_decode_equals_scan(oracle_mod, zoh):
    batch, L, H, P, N, G = 2, 30, 4, 3, 8, 2
    inp = synth.ssd(batch, L, H, P, N, G, dtype=synth.F32, with_z=True, with_h0=True, seed=17)
    f = inp.f64
    disc = oracle_mod.DISC_ZOH if zoh else oracle_mod.DISC_EXP_EULER
    y, hf = oracle_mod.ssd_sequential(f("x"), f("dt"), f("A"), f("B"), f("C"), D=f("D"),
                                      z=f("z"), dt_bias=f("dt_bias"), h0=f("h0"), disc=disc)
    state = f("h0")
    for t in range(L):
        ys, state = oracle_mod.state_update(state, f("x")[:, t], f("dt")[:, t], f("A"),
                                            f("B")[:, t], f("C")[:, t], D=f("D"), z=f("z")[:, t],
                                            dt_bias=f("dt_bias"), disc=disc)
        assert rel_err(ys, y[:, t]) < 1e-13
    assert rel_err(state, hf) < 1e-13


# ----------------------------------------------------------------------------------------
# P7: degenerate cases
# ----------------------------------------------------------------------------------------
def test_zero_step_keeps_state(oracle_mod):
    rng = np.random.default_rng(1)
    batch, dim, N, L = 1, 3, 4, 12
    x = rng.standard_normal((batch, dim, L))
    h0 = rng.standard_normal((batch, dim, N))
    B = rng.standard_normal((batch, 1, N, L))
    C = rng.standard_normal((batch, 1, N, L))
    D = rng.standard_normal(dim)
    A = -rng.uniform(0.5, 2, (dim, N))
    y, hf = oracle_mod.mamba1_scan(x, np.zeros_like(x), A, B, C, D=D, h0=h0,
                                   delta_softplus=False)
    expect = np.einsum("bnt,bdn->bdt", C[:, 0], h0) + D[None, :, None] * x
    assert rel_err(y, expect) < 1e-14
    assert np.array_equal(hf, h0)


def test_memoryless_limit(oracle_mod):
    rng = np.random.default_rng(2)
    batch, dim, N, L = 2, 3, 4, 15
    x = rng.standard_normal((batch, dim, L))
    raw = rng.standard_normal((batch, dim, L))
    B = rng.standard_normal((batch, 1, N, L))
    C = rng.standard_normal((batch, 1, N, L))
    D = rng.standard_normal(dim)
    A = np.full((dim, N), -1e300)  # exp(Delta*A) = 0: no memory
    y, _ = oracle_mod.mamba1_scan(x, raw, A, B, C, D=D, h0=rng.standard_normal((batch, dim, N)))
    dl = np.log1p(np.exp(raw))
    expect = dl * np.einsum("bnt,bnt->bt", C[:, 0], B[:, 0])[:, None, :] * x + D[None, :, None] * x
    assert rel_err(y, expect) < 1e-14


def test_zero_input_zero_output(oracle_mod):
    inp = synth.mamba1(2, 4, 3, 33, dtype=synth.F32, with_z=True, seed=4)
    f = inp.f64
    y, hf = oracle_mod.mamba1_scan(np.zeros_like(f("x")), f("delta"), f("A"), f("B"), f("C"),
                                   D=f("D"), z=f("z"), delta_bias=f("delta_bias"))
    assert not np.any(y) and not np.any(hf)


def test_linearity_in_input_and_state(oracle_mod):
    rng = np.random.default_rng(6)
    inp = synth.mamba1(2, 4, 3, 40, dtype=synth.F32, seed=8)
    f = inp.f64
    x2 = rng.standard_normal(f("x").shape)
    h1 = rng.standard_normal((2, 4, 3))
    h2 = rng.standard_normal((2, 4, 3))
    common = dict(D=f("D"), delta_bias=f("delta_bias"))
    ya, ha = oracle_mod.mamba1_scan(f("x"), f("delta"), f("A"), f("B"), f("C"), h0=h1, **common)
    yb, hb = oracle_mod.mamba1_scan(x2, f("delta"), f("A"), f("B"), f("C"), h0=h2, **common)
    yc, hc = oracle_mod.mamba1_scan(2.0 * f("x") - 3.0 * x2, f("delta"), f("A"), f("B"), f("C"),
                                    h0=2.0 * h1 - 3.0 * h2, **common)
    assert rel_err(yc, 2.0 * ya - 3.0 * yb) < 1e-13
    assert rel_err(hc, 2.0 * ha - 3.0 * hb) < 1e-13


def test_empty_sequence(oracle_mod):
    inp = synth.mamba1(1, 3, 2, 0, dtype=synth.F32, with_h0=True, seed=0)
    f = inp.f64
    y, hf = oracle_mod.mamba1_scan(f("x"), f("delta"), f("A"), f("B"), f("C"), D=f("D"),
                                   h0=f("h0"), delta_bias=f("delta_bias"))
    assert y.shape == (1, 3, 0)
    assert np.array_equal(hf, f("h0"))


# ----------------------------------------------------------------------------------------
# Stored fixture: the oracle's output on a tiny case (written by tests/golden/make_golden.py,
# which calls only the oracle); guards against unintended changes to its arithmetic.
# ----------------------------------------------------------------------------------------
def test_golden_fixture_unchanged(oracle_mod):
    import json
    import os
    from tests.golden import make_golden
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_tiny.json")
    with open(path) as fh:
        stored = json.load(fh)
    now = make_golden.compute(oracle_mod)
    for key, vals in stored["values"].items():
        assert rel_err(np.array(now[key]), np.array(vals)) < 1e-15, key


# ----------------------------------------------------------------------------------------
# Mamba-1 backward: the oracle's gradients against central finite differences of the
# (separately pinned) forward oracle, one random direction per input
# ----------------------------------------------------------------------------------------
def _bwd_inputs(seed, gated, skip, bias, h0, batch=2, dim=4, N=3, L=7, G=2):
    rng = np.random.default_rng(seed)
    inp = {
        "x": rng.standard_normal((batch, dim, L)),
        "delta": 0.7 * rng.standard_normal((batch, dim, L)),
        "A": -np.exp(0.5 * rng.standard_normal((dim, N))),
        "B": rng.standard_normal((batch, G, N, L)),
        "C": rng.standard_normal((batch, G, N, L)),
        "D": rng.standard_normal(dim) if skip else None,
        "z": rng.standard_normal((batch, dim, L)) if gated else None,
        "delta_bias": 0.3 * rng.standard_normal(dim) if bias else None,
        "h0": rng.standard_normal((batch, dim, N)) if h0 else None,
    }
    dy = rng.standard_normal((batch, dim, L))
    dhf = rng.standard_normal((batch, dim, N))
    return inp, dy, dhf


GRAD_OF = {"x": "dx", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
           "z": "dz", "delta_bias": "ddelta_bias", "h0": "dh0"}


@pytest.mark.parametrize("gated,skip,bias,h0,softplus", [
    (True, True, True, True, True), (False, False, False, False, True),
    (True, False, True, False, False), (False, True, False, True, False)])
def test_mamba1_bwd_finite_differences(oracle_mod, gated, skip, bias, h0, softplus):
    check_mamba1_bwd_fd(oracle_mod, gated, skip, bias, h0, softplus)


def check_mamba1_bwd_fd(oracle_mod, gated=True, skip=True, bias=True, h0=True, softplus=True):
    inp, dy, dhf = _bwd_inputs(5, gated, skip, bias, h0)
    if not softplus:  # keep Delta positive without softplus
        inp["delta"] = np.abs(inp["delta"]) + 0.05
        if inp["delta_bias"] is not None:
            inp["delta_bias"] = np.abs(inp["delta_bias"])

    def loss(args):
        y, hf = oracle_mod.mamba1_scan(**args, delta_softplus=softplus)
        return float((dy * y).sum() + (dhf * hf).sum())

    grads = oracle_mod.mamba1_scan_bwd(**inp, dy=dy, dh_final=dhf, delta_softplus=softplus)
    rng = np.random.default_rng(7)
    eps = 1e-6
    for name, val in inp.items():
        if val is None:
            assert GRAD_OF[name] not in grads or name == "h0"
            continue
        v = rng.standard_normal(val.shape)
        plus = dict(inp, **{name: val + eps * v})
        minus = dict(inp, **{name: val - eps * v})
        fd = (loss(plus) - loss(minus)) / (2 * eps)
        an = float((grads[GRAD_OF[name]] * v).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


def test_mamba1_bwd_empty_sequence(oracle_mod):
    """L = 0: h_final = h0, so dh0 = dh_final and every other gradient is empty or zero."""
    inp, _, dhf = _bwd_inputs(6, True, True, True, True, L=0)
    dy = np.zeros((2, 4, 0))
    g = oracle_mod.mamba1_scan_bwd(**inp, dy=dy, dh_final=dhf)
    assert np.array_equal(g["dh0"], dhf)
    assert np.all(g["dA"] == 0) and np.all(g["dD"] == 0) and np.all(g["ddelta_bias"] == 0)


def test_mamba1_bwd_one_step_closed_form(oracle_mod):
    """L = 1, one channel, one state, no gate: y = C (e^{Delta a} h0 + Delta B x) + D x with
    Delta = softplus(delta + bias); the derivatives written out by hand."""
    x, dl, a, Bv, Cv, Dv, bias, h0 = 0.8, -0.3, -1.1, 0.6, -0.9, 0.4, 0.2, 1.5
    v = dl + bias
    Dt = math.log1p(math.exp(v))
    sig = 1.0 / (1.0 + math.exp(-v))
    E = math.exp(Dt * a)
    inp = {"x": np.full((1, 1, 1), x), "delta": np.full((1, 1, 1), dl), "A": np.full((1, 1), a),
           "B": np.full((1, 1, 1, 1), Bv), "C": np.full((1, 1, 1, 1), Cv), "D": np.array([Dv]),
           "delta_bias": np.array([bias]), "h0": np.full((1, 1, 1), h0)}
    g = oracle_mod.mamba1_scan_bwd(**inp, dy=np.ones((1, 1, 1)))
    dDt = Cv * (Bv * x + h0 * E * a)
    want = {"dx": Cv * Dt * Bv + Dv, "ddelta": dDt * sig, "ddelta_bias": dDt * sig,
            "dA": Cv * h0 * E * Dt, "dB": Cv * Dt * x, "dC": E * h0 + Dt * Bv * x, "dD": x,
            "dh0": Cv * E}
    for k, w in want.items():
        assert abs(float(np.ravel(g[k])[0]) - w) <= 1e-14 * max(1.0, abs(w)), (k, g[k], w)


# ----------------------------------------------------------------------------------------
# Mamba-3 scan: reduction to exponential-Euler, an unrolled complex sum, a steady state
# and a pure rotation
# ----------------------------------------------------------------------------------------
def _m3_inputs(seed, batch=2, dim=3, N=4, L=9, G=1, gated=True):
    rng = np.random.default_rng(seed)
    return {
        "x": rng.standard_normal((batch, dim, L)),
        "delta": 0.6 * rng.standard_normal((batch, dim, L)),
        "A_re": -np.exp(0.5 * rng.standard_normal((dim, N))),
        "A_im": 2.0 * rng.standard_normal((dim, N)),
        "lam": rng.uniform(0.0, 1.0, (batch, dim, L)),
        "B": rng.standard_normal((batch, G, N, L)),
        "C": rng.standard_normal((batch, G, N, L)),
        "D": rng.standard_normal(dim),
        "z": rng.standard_normal((batch, dim, L)) if gated else None,
        "delta_bias": 0.2 * rng.standard_normal(dim),
        "h0": rng.standard_normal((batch, dim, N)) + 1j * rng.standard_normal((batch, dim, N)),
    }


def test_mamba3_reduces_to_exp_euler(oracle_mod):
    """The pages' reduction test (04/Approach): lambda = 1, theta = 0 is Mamba-1 with the
    exponential-Euler rule, states real."""
    inp = _m3_inputs(11, G=1)
    inp["lam"] = np.ones_like(inp["lam"])
    inp["A_im"] = np.zeros_like(inp["A_im"])
    inp["h0"] = inp["h0"].real.astype(np.complex128)
    y3, h3 = oracle_mod.mamba3_scan(**inp)
    y1, h1 = oracle_mod.mamba1_scan(inp["x"], inp["delta"], inp["A_re"], inp["B"], inp["C"],
                                    D=inp["D"], z=inp["z"], delta_bias=inp["delta_bias"],
                                    h0=inp["h0"].real)
    assert rel_err(y3, y1) < 1e-14
    assert rel_err(h3.real, h1) < 1e-14 and np.all(h3.imag == 0)


def _m3_unrolled(inp, softplus=True):
    """h_t = P(0..t) h0 + sum_s P(s+1..t) c_s with P the product of the complex decays and
    c_s = lambda_s Delta_s u_s + (1 - lambda_s) Delta_s Abar_s u_{s-1}: the recurrence
    summed out, written independently of the oracle."""
    x, dl, lam = inp["x"], inp["delta"], inp["lam"]
    batch, dim, L = x.shape
    N = inp["A_re"].shape[1]
    y = np.zeros((batch, dim, L))
    hf = np.zeros((batch, dim, N), np.complex128)
    for b in range(batch):
        for d in range(dim):
            A = inp["A_re"][d] + 1j * inp["A_im"][d]
            v = dl[b, d] + inp["delta_bias"][d]
            Dt = np.log1p(np.exp(v)) if softplus else v
            Ab = np.exp(Dt[:, None] * A[None, :])                      # [L, N]
            u = inp["B"][b, 0].T * x[b, d][:, None]                    # [L, N]
            c = (lam[b, d][:, None] * Dt[:, None] * u).astype(np.complex128)
            c[1:] += (1 - lam[b, d][1:, None]) * Dt[1:, None] * Ab[1:] * u[:-1]
            for t in range(L):
                h = np.prod(Ab[:t + 1], axis=0) * inp["h0"][b, d]
                for s_ in range(t + 1):
                    h = h + np.prod(Ab[s_ + 1:t + 1], axis=0) * c[s_]
                o = np.real(np.sum(inp["C"][b, 0, :, t] * h)) + inp["D"][d] * x[b, d, t]
                zt = inp["z"][b, d, t]
                y[b, d, t] = o * zt / (1 + np.exp(-zt))
                hf[b, d] = h
    return y, hf


def test_mamba3_unrolled_sum(oracle_mod):
    inp = _m3_inputs(12)
    y, hf = oracle_mod.mamba3_scan(**inp)
    yr, hr = _m3_unrolled(inp)
    assert rel_err(y, yr) < 1e-12
    assert np.max(np.abs(hf - hr)) < 1e-12 * np.max(np.abs(hr))


def test_mamba3_steady_state(oracle_mod):
    """Constant Delta, lambda, x and B from t = 1 on: the state converges to
    h* = Delta (lambda + (1 - lambda) Abar) B x / (1 - Abar)."""
    L, N = 400, 3
    Dt, lam_v, xv = 0.4, 0.3, 1.7
    A = np.array([-0.5 + 2.0j, -1.2 - 0.7j, -0.3 + 5.0j])
    Bv = np.array([0.8, -1.1, 0.4])
    inp = {"x": np.full((1, 1, L), xv), "delta": np.full((1, 1, L), Dt),
           "A_re": A.real[None], "A_im": A.imag[None], "lam": np.full((1, 1, L), lam_v),
           "B": np.broadcast_to(Bv[None, None, :, None], (1, 1, N, L)).copy(),
           "C": np.zeros((1, 1, N, L))}
    _, hf = oracle_mod.mamba3_scan(**inp, delta_softplus=False)
    Ab = np.exp(Dt * A)
    hstar = Dt * (lam_v + (1 - lam_v) * Ab) * Bv * xv / (1 - Ab)
    assert np.max(np.abs(hf[0, 0] - hstar)) < 1e-12 * np.max(np.abs(hstar))


def test_mamba3_pure_rotation(oracle_mod):
    """A_re = 0, lambda = 1, an impulse at t = 0: h_t = Delta_0 B_0 x_0 exp(i theta
    sum_{r=1..t} Delta_r), so Re(C h) traces a cosine of the accumulated phase."""
    L, theta = 12, 0.9
    rng = np.random.default_rng(3)
    dts = rng.uniform(0.1, 0.5, L)
    x = np.zeros((1, 1, L))
    x[0, 0, 0] = 1.3
    inp = {"x": x, "delta": dts[None, None], "A_re": np.zeros((1, 1)), "A_im": np.full((1, 1), theta),
           "lam": np.ones((1, 1, L)), "B": np.full((1, 1, 1, L), 0.7), "C": np.ones((1, 1, 1, L))}
    y, hf = oracle_mod.mamba3_scan(**inp, delta_softplus=False)
    phase = theta * np.concatenate([[0.0], np.cumsum(dts[1:])])
    want = dts[0] * 0.7 * 1.3 * np.cos(phase)
    assert np.max(np.abs(y[0, 0] - want)) < 1e-14
    assert abs(hf[0, 0, 0] - dts[0] * 0.7 * 1.3 * np.exp(1j * phase[-1])) < 1e-14


# ----------------------------------------------------------------------------------------
# S4D: convolution form equals recurrent form (the pages' test), ZOH against
# high-precision arithmetic, the continuous-time DC gain
# ----------------------------------------------------------------------------------------
def _s4d_params(seed, dim=3, N=4):
    rng = np.random.default_rng(seed)
    n = np.arange(N)
    A = np.broadcast_to(-0.5 + 1j * np.pi * n, (dim, N)).copy()          # S4D-Lin
    log_dt = rng.uniform(np.log(1e-3), np.log(1e-1), dim)
    B = np.ones((dim, N), np.complex128)
    C = rng.standard_normal((dim, N)) + 1j * rng.standard_normal((dim, N))
    D = rng.standard_normal(dim)
    return log_dt, A, B, C, D


@pytest.mark.parametrize("L", [1, 7, 64, 300])
def test_s4d_fft_conv_equals_recurrent(oracle_mod, L):
    log_dt, A, B, C, D = _s4d_params(21)
    u = np.random.default_rng(22).standard_normal((2, 3, L))
    yc = oracle_mod.s4d_fft_conv(u, log_dt, A, B, C, D=D)
    yr, _ = oracle_mod.s4d_recurrent(u, log_dt, A, B, C, D=D)
    assert rel_err(yc, yr) < 1e-12


@pytest.mark.parametrize("z", [1e-6 + 2e-6j, 3e-5 - 9e-5j, 1e-3 + 0.5j, -0.8 + 3.0j, -2.5 - 40.0j])
def test_s4d_zoh_against_high_precision(oracle_mod, z):
    """K_0 = Re(C Bbar) with N = 1, B = 1: C = 1 gives Re(Bbar), C = -i gives Im(Bbar);
    Bbar = Delta (e^z - 1)/z evaluated with 50 digits."""
    dt = 0.05
    A = np.array([[z / dt]])
    Bb = mpmath.mpf(dt) * (mpmath.exp(mpmath.mpc(z.real, z.imag)) - 1) / mpmath.mpc(z.real, z.imag)
    for Cv, want in ((1.0 + 0j, float(Bb.real)), (-1j, float(Bb.imag))):
        K = oracle_mod.s4d_kernel(np.array([np.log(dt)]), A, np.ones((1, 1)), np.array([[Cv]]), 1)
        # within the Taylor band the pages' polynomial is exact to O(z^3)
        tol = 1e-15 + (abs(z) ** 3 * dt if abs(z) < 1e-4 else 0.0)
        assert abs(K[0, 0] - want) <= tol * max(1.0, abs(want)) + 1e-18, (z, K[0, 0], want)


def test_s4d_dc_gain(oracle_mod):
    """A constant input settles at the continuous-time DC gain -C B / A, which ZOH
    reproduces exactly (real A, N = 1)."""
    a, dt = -0.7, 0.3
    L = 400
    y, _ = oracle_mod.s4d_recurrent(np.ones((1, 1, L)), np.array([np.log(dt)]), np.array([[a + 0j]]),
                                    np.array([[2.0 + 0j]]), np.array([[1.5 + 0j]]))
    assert abs(y[0, 0, -1] - (-1.5 * 2.0 / a)) < 1e-12


# ----------------------------------------------------------------------------------------
# SSD backward: finite differences of the sequential SSD oracle (a separate C routine)
# ----------------------------------------------------------------------------------------
SSD_GRAD_OF = {"x": "dx", "dt": "ddt", "A": "dA", "B": "dB", "C": "dC", "D": "dD", "z": "dz",
               "dt_bias": "ddt_bias", "h0": "dh0"}


@pytest.mark.parametrize("gated,softplus", [(True, True), (False, False)])
def test_ssd_bwd_finite_differences(oracle_mod, gated, softplus):
    rng = np.random.default_rng(31)
    batch, L, H, P, G, N = 2, 6, 4, 3, 2, 5
    inp = {"x": rng.standard_normal((batch, L, H, P)),
           "dt": (np.abs(rng.standard_normal((batch, L, H))) * 0.5 + 0.05) if not softplus
           else 0.7 * rng.standard_normal((batch, L, H)),
           "A": -np.exp(0.5 * rng.standard_normal(H)),
           "B": rng.standard_normal((batch, L, G, N)), "C": rng.standard_normal((batch, L, G, N)),
           "D": rng.standard_normal(H), "z": rng.standard_normal((batch, L, H, P)) if gated else None,
           "dt_bias": np.abs(0.3 * rng.standard_normal(H)), "h0": rng.standard_normal((batch, H, P, N))}
    dy = rng.standard_normal((batch, L, H, P))
    dhf = rng.standard_normal((batch, H, P, N))

    def loss(args):
        y, hf = oracle_mod.ssd_sequential(**args, dt_softplus=softplus)
        return float((dy * y).sum() + (dhf * hf).sum())

    grads = oracle_mod.ssd_bwd(**inp, dy=dy, dh_final=dhf, dt_softplus=softplus)
    eps = 1e-6
    for name, val in inp.items():
        if val is None:
            continue
        v = rng.standard_normal(val.shape)
        fd = (loss(dict(inp, **{name: val + eps * v})) - loss(dict(inp, **{name: val - eps * v}))) / (2 * eps)
        an = float((grads[SSD_GRAD_OF[name]] * v).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)
