"""Plants plausible mistakes in a COPY of the oracle (on the CPU) and checks that
the pins in test_oracle_pins.py catch every one of them.  The real oracle is
never modified."""
import os
import subprocess

import pytest

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, text in oracle.c, replacement): a dropped term, a wrong sign, a wrong
# index, a transposed operand, a wrong Taylor coefficient, and so on.
MUTATIONS = [
    ("drop_skip_term", "if (Dskip) acc += Dskip[d] * xt;", ""),
    ("gate_sign", "return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    ("y_before_update",
     "h[n] = exp(dt * a) * h[n] + input_weight(dt, a, disc) * B[bc] * xt;\n                    acc += C[bc] * h[n];",
     "acc += C[bc] * h[n];\n                    h[n] = exp(dt * a) * h[n] + input_weight(dt, a, disc) * B[bc] * xt;"),
    ("B_C_swapped", "* B[bc] * xt;", "* C[bc] * xt;"),
    ("taylor_coefficient", "return 1.0 + z / 2.0 + z * z / 6.0;", "return 1.0 + z / 2.0 + z * z / 2.0;"),
    ("softplus_sign", "return m + log1p(exp(-fabs(v)));", "return m - log1p(exp(-fabs(v)));"),
    ("bias_ignored", "double v = raw + (bias ? bias[idx] : 0.0);", "double v = raw;"),
    ("group_index", "int g = d / per_group;", "int g = d % ngroups;"),
    ("ssd_decay_sign", "acc += cb * exp(cum[i] - cum[j]) * w[j] * xs;",
     "acc += cb * exp(cum[j] - cum[i]) * w[j] * xs;"),
    ("ssd_carried_state_dropped", "acc += exp(cum[i]) * ch;", ""),
    ("ssd_chunk_state_decay", "double f = exp(cum[q - 1] - cum[j]) * w[j];",
     "double f = w[j];"),
    ("ssd_seq_B_index", "acc += Ct[n] * *hp;", "acc += Bt[n] * *hp;"),
    ("step_zoh_ignored", "hrow[n] = exp(d_t * a) * hrow[n] + input_weight(d_t, a, disc) * x[xi] * Bb[n];",
     "hrow[n] = exp(d_t * a) * hrow[n] + d_t * x[xi] * Bb[n];"),
    ("bwd_carry_decay_dropped", "g[n] = Gt * E;", "g[n] = Gt;"),
    ("bwd_dA_missing_delta", "dA[(size_t)d * N + n] += Gt * hprev * E * dt;",
     "dA[(size_t)d * N + n] += Gt * hprev * E;"),
    ("bwd_gate_derivative_sign", "(1.0 + zt * (1.0 - sg))", "(1.0 - zt * (1.0 - sg))"),
    ("bwd_dC_uses_prev_state", "dC[bc] += dout * hs[(tt + 1) * N + n];", "dC[bc] += dout * hs[tt * N + n];"),
    ("bwd_softplus_derivative", "ddt / (1.0 + exp(-v))", "ddt / (1.0 + exp(v))"),
    ("bwd_dD_ignores_gate", "if (dD) dD[d] += dout * xt;", "if (dD) dD[d] += dy[row + tt] * xt;"),
    ("bwd_dx_skip_term_dropped", "double dxt = Dskip ? dout * Dskip[d] : 0.0;", "double dxt = 0.0;"),
    ("bwd_ddelta_decay_term_dropped", "ddt += Gt * (B[bc] * xt + hprev * E * a);", "ddt += Gt * B[bc] * xt;"),
    ("m3_left_end_dropped", "double pr = hr[n] + (1.0 - lt) * dt * up;", "double pr = hr[n];"),
    ("m3_rotation_sign", "hi[n] = ar * pi + ai * pr;", "hi[n] = ar * pi - ai * pr;"),
    ("m3_left_end_current_input", "double up = t > 0 ? B[bc - 1] * xp : 0.0;", "double up = t > 0 ? B[bc] * xt : 0.0;"),
    ("m3_lambda_on_wrong_end", "hr[n] = ar * pr - ai * pi + lt * dt * cur;", "hr[n] = ar * pr - ai * pi + (1.0 - lt) * dt * cur;"),
    ("m3_angle_without_delta", "double ang = dt * A_im[(size_t)d * N + n];", "double ang = A_im[(size_t)d * N + n];"),
    ("m3_magnitude_sign", "double mag = exp(dt * A_re[(size_t)d * N + n]);", "double mag = exp(-dt * A_re[(size_t)d * N + n]);"),
    ("s4d_taylor_imag", "pi = zi / 2.0 + (2.0 * zr * zi) / 6.0;", "pi = zi / 2.0;"),
    ("s4d_expm1_term_dropped", "double nr = expm1(zr) * cos(zi) - 2.0 * s2 * s2;", "double nr = expm1(zr) * cos(zi);"),
    ("s4d_kernel_conjugate", "wi = wr * abi + wi * abr;", "wi = -wr * abi + wi * abr;"),
    ("s4d_phi1_division_conjugate", "pi = (ni * zr - nr * zi) / den;", "pi = (ni * zr + nr * zi) / den;"),
    ("s4d_in_place_complex_update",
     "double nr = abr * hr - abi * hi + bbr * u[row + t];\n"
     "                    hi = abr * hi + abi * hr + bbi * u[row + t];\n"
     "                    hr = nr;",
     "hr = abr * hr - abi * hi + bbr * u[row + t];\n"
     "                    hi = abr * hi + abi * hr + bbi * u[row + t];"),
    ("s4d_kernel_log_dt_as_dt", "double dt = exp(log_dt[d]);\n        for (size_t l = 0;",
     "double dt = log_dt[d];\n        for (size_t l = 0;"),
    ("s4d_output_imag_sign", "y[row + t] += C[k] * hr - C[k + 1] * hi;", "y[row + t] += C[k] * hr + C[k + 1] * hi;"),
    ("step_skip_dropped", "if (Dskip) acc += Dskip[hd] * x[xi];\n                if (z) acc *= silu(z[xi]);\n                y[xi] = acc;",
     "if (z) acc *= silu(z[xi]);\n                y[xi] = acc;"),
    ("zoh_phi1_of_A_not_DeltaA", "return delta * oracle_phi1(delta * a);", "return delta * oracle_phi1(a);"),
    ("phi1_taylor_branch_inverted", "if (fabs(z) < 1e-4) return", "if (fabs(z) > 1e-4) return"),
    ("ssd_causal_mask_drops_diagonal", "for (int j = 0; j <= i; ++j) {        /* decayed attention */",
     "for (int j = 0; j < i; ++j) {        /* decayed attention */"),
    ("ssd_exclusive_cumsum", "run += d_t * A[hd];\n                    cum[i] = run;",
     "cum[i] = run;\n                    run += d_t * A[hd];"),
    ("ssd_ragged_chunk_decay", "double chunk_decay = exp(cum[q - 1]);", "double chunk_decay = exp(cum[chunk - 1]);"),
    ("step_per_state_A_transposed", "double a = a_per_state ? A[(size_t)hd * dstate + n] : A[hd];",
     "double a = a_per_state ? A[(size_t)n * nheads + hd] : A[hd];"),
    ("step_y_before_update",
     "hrow[n] = exp(d_t * a) * hrow[n] + input_weight(d_t, a, disc) * x[xi] * Bb[n];\n"
     "                    acc += Cb[n] * hrow[n];",
     "acc += Cb[n] * hrow[n];\n"
     "                    hrow[n] = exp(d_t * a) * hrow[n] + input_weight(d_t, a, disc) * x[xi] * Bb[n];"),
]

PIN_CHECKS = [
    lambda o: pins.test_softplus_matches_high_precision(o, -5.0),
    lambda o: pins.test_softplus_matches_high_precision(o, 3.0),
    lambda o: pins.test_phi1_log_grid(o),
    lambda o: pins.test_zoh_steady_state(o),
    lambda o: pins.test_mamba1_brute_force(o, True, True),
    lambda o: pins.test_mamba1_brute_force(o, False, True),
    lambda o: pins.test_ssd_brute_force(o, True),
    lambda o: pins.test_ssd_brute_force(o, False),
    lambda o: pins.test_ssd_chunked_equals_sequential(o, 300, 64),
    lambda o: pins.test_step_response_closed_form(o),
    lambda o: pins.test_mamba1_decode_equals_scan(o),
    lambda o: pins.test_ssd_decode_equals_scan(o, False),
    lambda o: pins.test_ssd_decode_equals_scan(o, True),
    lambda o: pins.check_mamba1_bwd_fd(o),
    lambda o: pins.test_mamba3_reduces_to_exp_euler(o),
    lambda o: pins.test_mamba3_unrolled_sum(o),
    lambda o: pins.test_mamba3_steady_state(o),
    lambda o: pins.test_mamba3_pure_rotation(o),
    lambda o: pins.test_s4d_fft_conv_equals_recurrent(o, 64),
    lambda o: pins.test_s4d_zoh_against_high_precision(o, 1e-3 + 0.5j),
    lambda o: pins.test_s4d_zoh_against_high_precision(o, 3e-5 - 9e-5j),
    lambda o: pins.test_s4d_dc_gain(o),
    lambda o: pins.test_mamba1_bwd_one_step_closed_form(o),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, oracle_mod, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation {name} no longer applies"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    str(mutated), "-o", str(lib), "-lm"], check=True)
    caught = 0
    with oracle.use_library(str(lib)):
        for check in PIN_CHECKS:
            try:
                check(oracle)
            except AssertionError:
                caught += 1
    assert caught > 0, f"planted mistake {name!r} passed every pin"
