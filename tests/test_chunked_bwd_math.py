"""The chunked form of the SSD backward, restated in float64 numpy from the formulas in the
header of csrc/ssd_bwd.cu, reproduces the oracle's SSD backward (the Mamba-1 backward
on the tied view): a CPU check of the derivation the GPU path is built on, with several
chunks, a ragged last chunk, two groups, the gate, h0 and dh_final ("From S4 to
Mamba-3", 03/System, mamba2_minimal.py; 04/Approach, "Chunked SSD")."""
import numpy as np
import pytest

from selective_scan_mamba_gb300 import synth


def _sigmoid(v):
    return 1.0 / (1.0 + np.exp(-v))


def chunked_bwd(x, dt_raw, A, B, C, dout, D, z, dt_bias, h0, dh_final, Q):
    """Every gradient of sum(dout * out) + sum(dh_final * h_final), chunk by chunk: chunk
    states chained forwards, the outputs' adjoint sums chained backwards, and the
    per-chunk products of the header's formulas.  States are held as [N, P]."""
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    hpg = H // G
    g_out = {"dx": np.zeros_like(x), "ddt": np.zeros((batch, L, H)), "dA": np.zeros(H),
             "dB": np.zeros_like(B), "dC": np.zeros_like(C), "dD": np.zeros(H),
             "dz": np.zeros_like(x), "ddt_bias": np.zeros(H), "dh0": np.zeros((batch, H, P, N))}
    chunks = [(s0, min(Q, L - s0)) for s0 in range(0, L, Q)]
    for b in range(batch):
        for h in range(H):
            g = h // hpg
            u = dt_raw[b, :, h] + dt_bias[h]
            dt = np.log1p(np.exp(u))
            a = dt * A[h]
            # forward: the state entering each chunk
            hp = h0[b, h].T.copy()
            ent, parts = [], []
            for s0, q in chunks:
                sl = slice(s0, s0 + q)
                cum = np.cumsum(a[sl])
                tot = cum[-1]
                F = np.exp(tot - cum) * dt[sl]
                ent.append(hp)
                parts.append((sl, cum, tot, F))
                hp = np.exp(tot) * hp + (B[b, sl, g] * F[:, None]).T @ x[b, sl, h]
            # outputs, the gate and the adjoint sums R_c
            dos, Rs = [], []
            for (sl, cum, tot, F), Hp in zip(parts, ent):
                xc, Bc, Cc = x[b, sl, h], B[b, sl, g], C[b, sl, g]
                E = np.tril(np.exp(cum[:, None] - cum[None, :]))
                CB = Cc @ Bc.T
                o = (CB * E * dt[sl][None, :]) @ xc + np.exp(cum)[:, None] * (Cc @ Hp) + D[h] * xc
                zc = z[b, sl, h]
                sg = _sigmoid(zc)
                do = dout[b, sl, h] * zc * sg
                g_out["dz"][b, sl, h] = dout[b, sl, h] * o * sg * (1.0 + zc * (1.0 - sg))
                dos.append(do)
                Rs.append((Cc * np.exp(cum)[:, None]).T @ do)
            # backwards: the adjoint of the state leaving each chunk
            Gc = dh_final[b, h].T.copy()
            adj = [None] * len(chunks)
            for c in range(len(chunks) - 1, -1, -1):
                adj[c] = Gc
                Gc = np.exp(parts[c][2]) * Gc + Rs[c]
            g_out["dh0"][b, h] = Gc.T
            # the chunk gradients
            for c, ((sl, cum, tot, F), Hp, Gl, do) in enumerate(zip(parts, ent, adj, dos)):
                xc, Bc, Cc, dtc = x[b, sl, h], B[b, sl, g], C[b, sl, g], dt[sl]
                E = np.tril(np.exp(cum[:, None] - cum[None, :]))
                CB = Cc @ Bc.T
                T = do @ xc.T
                V = CB * E * T
                Y = xc @ Gl.T                                  # Y[s][n] = G x_s
                U = np.exp(cum)[:, None] * (do @ Hp.T)          # e^{cum_t} h_p do_t
                g_out["dx"][b, sl, h] = D[h] * do + (CB * E * dtc[None, :]).T @ do + F[:, None] * (Bc @ Gl)
                g_out["dB"][b, sl, g] += (T * E * dtc[None, :]).T @ Cc + F[:, None] * Y
                g_out["dC"][b, sl, g] += (T * E * dtc[None, :]) @ Bc + U
                dF = np.sum(Bc * Y, axis=1)
                dw = V.sum(axis=0) + np.exp(tot - cum) * dF
                dcum = (V * dtc[None, :]).sum(axis=1) - dtc * V.sum(axis=0) + np.sum(Cc * U, axis=1) - F * dF
                dtot = np.sum(F * dF) + np.exp(tot) * np.sum(Gl * Hp)
                da = np.cumsum(dcum[::-1])[::-1] + dtot
                raw = (da * A[h] + dw) * _sigmoid(u[sl])
                g_out["ddt"][b, sl, h] = raw
                g_out["dA"][h] += np.sum(da * dtc)
                g_out["dD"][h] += np.sum(do * xc)
                g_out["ddt_bias"][h] += np.sum(raw)
    return g_out


@pytest.mark.parametrize("L,Q", [(37, 8), (64, 16), (5, 16)])
def test_chunked_derivation_matches_oracle_backward(oracle_mod, L, Q):
    inp = synth.ssd(2, L, 4, 6, 5, 2, dtype=synth.F32, with_z=True, with_h0=True, seed=11 + L)
    f = inp.f64
    rng = np.random.default_rng(L)
    dout = rng.standard_normal((2, L, 4, 6))
    dhf = rng.standard_normal((2, 4, 6, 5))
    got = chunked_bwd(f("x"), f("dt"), f("A"), f("B"), f("C"), dout, f("D"), f("z"), f("dt_bias"),
                      f("h0"), dhf, Q)
    ref = oracle_mod.ssd_bwd(f("x"), f("dt"), f("A"), f("B"), f("C"), dout, D=f("D"), z=f("z"),
                             dt_bias=f("dt_bias"), h0=f("h0"), dh_final=dhf)
    for k, v in ref.items():
        scale = max(1.0, float(np.max(np.abs(v))))
        assert np.max(np.abs(got[k] - v)) <= 1e-10 * scale, k
