"""Plant plausible slips in copies of the oracle; the pins must catch each one.

Each mutation is a textual edit of oracle.c compiled into a temporary
library.  The real oracle is never modified.
"""
import os
import subprocess

import pytest

import oracle
import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTATIONS = {
    # one rounding of base + acc instead of two
    "single_rounding": ("orc_bf16_to_f64(bias)); /* second */", "acc); /* second */"),
    "sign_of_projection": ("acc += orc_bf16_to_f64(w[j])", "acc -= orc_bf16_to_f64(w[j])"),
    "operands_swapped": ("const uint16_t *w = W2 + v * r;", "const uint16_t *w = W1 + v * r;"),
    "tie_to_highest": ("if (score[v] > score[best])", "if (score[v] >= score[best])"),
    "step_index_ignored": ("bk = base + ((int64_t)b * gamma + k) * V;",
                           "bk = base + ((int64_t)b * gamma + 0) * V;"),
    "prev_not_advanced": ("            prev = best;\n", "            (void)best;\n"),
    "philox_multiplier": ("M0 = 0xD2511F53u", "M0 = 0xD2511F55u"),
    "philox_key_bump": ("k1 += W1;", "k1 += W0;"),
    "counter_layout": ("{(uint32_t)(v >> 2), (uint32_t)k, (uint32_t)b, 0u}",
                       "{(uint32_t)(v >> 2), (uint32_t)b, (uint32_t)k, 0u}"),
    "noise_word": ("return out[v & 3];", "return out[(v + 1) & 3];"),
    "uniform_bin_edge": ("2.0 * (double)(x >> 9) + 1.0", "2.0 * (double)(x >> 9)"),
    "gumbel_sign": ("return (float)(-log((double)e));", "return (float)(log((double)e));"),
    "temperature_multiplies": ("/ (double)T); /* fp32 quotient */",
                               "* (double)T); /* fp32 quotient */"),
    "ties_away_from_zero": ("(frac == 0.5 && fmod(n, 2.0) != 0.0)", "(frac == 0.5)"),
    "truncating_round": ("if (frac > 0.5 ||", "if (0 &&"),
    # group sampler
    "group_mass_dropped": ("const double s = m + log(S) - log(-log((double)U1));",
                           "const double s = m - log(-log((double)U1));"),
    "group_max_dropped": ("const double s = m + log(S) - log(-log((double)U1));",
                          "const double s = log(S) - log(-log((double)U1));"),
    "group_pick_uses_U1": ("    const double target = (double)U2 * S;\n    double run = 0.0;\n",
                           "    const double target = (double)U1 * S;\n    double run = 0.0;\n"),
    "group_counter_word": ("{(uint32_t)(j >> 1), (uint32_t)k, (uint32_t)b, 1u}",
                           "{(uint32_t)(j >> 1), (uint32_t)k, (uint32_t)b, 0u}"),
    # the group scores from z rounded to fp32: overflows at tiny T
    "group_z_in_fp32": ("            z[i] = orc_bf16_to_f64(logit[v0 + i]) / (double)T;",
                        "            z[i] = (double)(float)(orc_bf16_to_f64(logit[v0 + i]) / (double)T);"),
    # recurrent heads
    "cell_gate_swapped": ("val = (1.0 - z) * hp + z * xi;", "val = z * hp + (1.0 - z) * xi;"),
    "cell_gate_sign": ("1.0 / (1.0 + exp(-p));", "1.0 / (1.0 + exp(p));"),
    "cell_matrix_transposed": ("orc_row_dot(M + (int64_t)i * r, 1, hprev, r)",
                               "orc_row_dot(M + i, r, hprev, r)"),
    "cell_rnn_drops_input": ("val = tanh(p + xi);", "val = tanh(p);"),
    "cell_rnn_drops_recurrence": ("val = tanh(p + xi);", "val = tanh(xi);"),
    "cell_state_not_carried": ("memcpy(hbuf, hk, (size_t)r * sizeof *hk);",
                               "memset(hbuf, 0, (size_t)r * sizeof *hk);"),
    "cell_projects_input": ("* r : hbuf;\n", "* r : u;\n"),
    "cell_initial_state_is_input": ("const uint16_t *hprev = NULL;", "const uint16_t *hprev = u;"),
    "gru_update_gate_swapped": ("val = (1.0 - zg) * ng + zg * hp;",
                                "val = zg * ng + (1.0 - zg) * hp;"),
    "gru_reset_on_input": ("tanh(orc_bf16_to_f64(x[2 * r + i]) + rg * pg[2])",
                           "tanh(rg * (orc_bf16_to_f64(x[2 * r + i]) + pg[2]))"),
    "gru_gate_matrices_reversed": ("M + ((int64_t)g * r + i) * r, 1, hprev, r)",
                                   "M + ((int64_t)(2 - g) * r + i) * r, 1, hprev, r)"),
    "gru_tables_reversed": ("X + ((int64_t)g * V + prev) * r",
                            "X + ((int64_t)(2 - g) * V + prev) * r"),
}


@pytest.fixture(scope="module")
def philox_ref():
    pytest.importorskip("triton")
    return pins.philox_reference()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_mutation(name, tmp_path, philox_ref):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor for %s not found exactly once" % name
    path = tmp_path / "oracle_mut.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c11", "-fopenmp", "-o", str(lib),
                    str(path), "-lm"], check=True)
    O = oracle.Oracle(str(lib))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(O)
        except (AssertionError, oracle.OracleError) as e:
            caught.append((pin.__name__, str(e)[:120]))
            break
    assert caught, "no pin caught the planted mutation %r" % name
