"""Each plausible mistake planted in a copy of the oracle fails at least one pin.

The mutants are textual edits of ``oracle/ss_oracle.c`` compiled into a
temporary library (CPU only).  A mutant that survives every pin would mean
the pins cannot tell that mistake from the right answer.
"""
import pytest

import oracle
import oracle_pins

MUTANTS = {
    "dropped_u_in_input_term": ("h[n] = a_bar * h[n] + b_bar * u;",
                                "h[n] = a_bar * h[n] + b_bar;"),
    "sign_of_A": ("exp(dt * (double)j->A[d * N + n])",
                  "exp(-dt * (double)j->A[d * N + n])"),
    "missing_dt_in_decay": ("exp(dt * (double)j->A[d * N + n])",
                            "exp((double)j->A[d * N + n])"),
    "missing_dt_in_input": ("const double b_bar = dt * load_elem(",
                            "const double b_bar = load_elem("),
    "A_transposed": ("j->A[d * N + n]", "j->A[n * dim + d]"),
    "dropped_D_skip": ("      y += Dd * u;\n", "\n"),
    "D_indexed_by_batch": ("const double Dd = j->D ? (double)j->D[d] : 0.0;",
                           "const double Dd = j->D ? (double)j->D[b] : 0.0;"),
    "gate_before_skip": ("      y += Dd * u;\n      if (j->z) y *= silu(load_elem(j->z, x_idx, j->dtype));\n",
                         "      if (j->z) y *= silu(load_elem(j->z, x_idx, j->dtype));\n      y += Dd * u;\n"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "softplus_dropped_log1p": ("return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));",
                               "return (x > 0.0 ? x : 0.0);"),
    "softplus_missing_abs": ("log1p(exp(-fabs(x)))", "log1p(exp(-x))"),
    "bias_ignored": ("load_elem(j->delta, x_idx, j->dtype) + bias;",
                     "load_elem(j->delta, x_idx, j->dtype);"),
    "B_layout_b_L_N": ("load_elem(j->B, (bc * N + n) * L + t, j->dtype)",
                       "load_elem(j->B, (bc * L + t) * N + n, j->dtype)"),
    "C_time_reversed": ("load_elem(j->C, (bc * N + n) * L + t, j->dtype)",
                        "load_elem(j->C, (bc * N + n) * L + (L - 1 - t), j->dtype)"),
    "per_channel_BC_row_of_batch": ("const int64_t bc = j->bc_per_channel ? row : b;",
                                    "const int64_t bc = b;"),
    "per_channel_BC_row_swapped": ("const int64_t bc = j->bc_per_channel ? row : b;",
                                   "const int64_t bc = j->bc_per_channel ? d * j->batch + b : b;"),
    "readout_before_update": (
        "        h[n] = a_bar * h[n] + b_bar * u;\n        y += load_elem(j->C, (bc * N + n) * L + t, j->dtype) * h[n];\n",
        "        y += load_elem(j->C, (bc * N + n) * L + t, j->dtype) * h[n];\n        h[n] = a_bar * h[n] + b_bar * u;\n"),
    "h0_ignored": ("h[n] = j->h0 ? j->h0[row * N + n] : 0.0;", "h[n] = 0.0;"),
    "channel_from_wrong_axis": ("const int64_t b = row / dim, d = row % dim;",
                                "const int64_t b = row % j->batch, d = row / j->batch;"),
    "bf16_widening_truncated": ("(uint32_t)((const uint16_t*)p)[i] << 16",
                                "((uint32_t)((const uint16_t*)p)[i] << 16) & 0xFFFF0000u & ~0x10000u"),
    "combine_swapped_factor": ("const double v = a2[i] * v1[i] + c2[i];",
                               "const double v = a1[i] * v1[i] + c2[i];"),
    "combine_product_wrong": ("const double a = a2[i] * a1[i];",
                              "const double a = a2[i] + a1[i] - 1.0;"),
    # the backward
    "bwd_carry_without_decay": ("        g[n] = an * gn;\n", "        g[n] = gn;\n"),
    "bwd_sigmoid_of_dt_not_x": ("ddt / (1.0 + exp(-xv[t]))", "ddt / (1.0 + exp(-dtv[t]))"),
    "bwd_dA_missing_dt": ("j->dA[d * N + n] += gn * dt * an * prev;",
                          "j->dA[d * N + n] += gn * an * prev;"),
    "bwd_silu_derivative_sign": ("s * (1.0 + zt * (1.0 - s))", "s * (1.0 - zt * (1.0 - s))"),
    "bwd_dC_from_previous_state": ("j->dC[(b * N + n) * L + t] += dyp * h[t * N + n];",
                                   "j->dC[(b * N + n) * L + t] += dyp * prev;"),
    "bwd_du_without_skip": ("double du = dyp * Dd, ddt = 0.0;", "double du = 0.0, ddt = 0.0;"),
    "bwd_dB_without_u": ("j->dB[(b * N + n) * L + t] += gn * dt * u;",
                         "j->dB[(b * N + n) * L + t] += gn * dt;"),
    "bwd_dlast_ignored": ("g[n] = j->dlast ? j->dlast[row * N + n] : 0.0;", "g[n] = 0.0;"),
    "bwd_dD_before_gate": ("      dD += dyp * u;\n", "      dD += dy * u;\n"),
    "bwd_dB_time_reversed": ("j->dB[(b * N + n) * L + t] += gn * dt * u;",
                             "j->dB[(b * N + n) * L + (L - 1 - t)] += gn * dt * u;"),
    # the Mamba-2 forward
    "ssd_group_by_modulo": ("const int64_t g = hd / (H / G);", "const int64_t g = hd % G;"),
    "ssd_decay_missing_dt": ("const double decay = exp(A * dt);", "const double decay = exp(A);"),
    "ssd_input_missing_dt": ("decay * h[p * N + n] + dt * load_elem(j->B, bcrow + n, j->dtype) * xp;",
                             "decay * h[p * N + n] + load_elem(j->B, bcrow + n, j->dtype) * xp;"),
    "ssd_readout_from_B": ("y += load_elem(j->C, bcrow + n, j->dtype) * h[p * N + n];",
                           "y += load_elem(j->B, bcrow + n, j->dtype) * h[p * N + n];"),
    "ssd_skip_dropped": ("j->y[xrow + p] = y + Dh * xp;", "j->y[xrow + p] = y;"),
    "ssd_bias_ignored": ("load_elem(j->dt, (b * L + t) * H + hd, j->dtype) + bias;",
                         "load_elem(j->dt, (b * L + t) * H + hd, j->dtype);"),
    "ssd_x_head_major": ("const int64_t xrow = ((b * L + t) * H + hd) * P;",
                         "const int64_t xrow = ((b * H + hd) * L + t) * P;"),
    "ssd_state_transposed": ("j->final_state[unit * P * N + i] = h[i];",
                             "j->final_state[unit * P * N + (i % N) * P + i / N] = h[i];"),
    "ssd_h0_ignored": ("h[i] = j->h0 ? j->h0[unit * P * N + i] : 0.0;", "h[i] = 0.0;"),
    "ssd_h0_transposed": ("h[i] = j->h0 ? j->h0[unit * P * N + i] : 0.0;",
                          "h[i] = j->h0 ? j->h0[unit * P * N + (i % N) * P + i / N] : 0.0;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = oracle.SOURCE.read_text()
    assert src.count(old) == 1, f"mutation {name} does not apply exactly once"
    mutant_src = tmp_path / "ss_oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.build(mutant_src, tmp_path / "libmutant.so", force=True)
    orc = oracle.Oracle(lib)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passes every pin"
