"""Plant plausible mistakes in a copy of the oracle, on the CPU, and check that
the pins catch every one of them (each mutant must fail at least one pin)."""
import os

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssd_oracle.c")

# (name, original text, mutated text)
MUTANTS = [
    ("dropped_dt_in_update",
     "S[p * N + n] = decay * S[p * N + n] + dtv * Bt[n] * xt[p];",
     "S[p * N + n] = decay * S[p * N + n] + Bt[n] * xt[p];"),
    ("decay_sign_flipped", "exp(A[h] * dtv)", "exp(-A[h] * dtv)"),
    ("decay_on_new_term",
     "S[p * N + n] = decay * S[p * N + n] + dtv * Bt[n] * xt[p];",
     "S[p * N + n] = decay * (S[p * N + n] + dtv * Bt[n] * xt[p]);"),
    ("readout_uses_B", "acc += Ct[n] * S[p * N + n];", "acc += Bt[n] * S[p * N + n];"),
    ("readout_previous_state", "acc += Ct[n] * S[p * N + n];",
     "acc += Ct[n] * (S[p * N + n] - dtv * Bt[n] * xt[p]) / decay;"),
    ("dropped_D", "yt[p] = acc + Dh * xt[p];", "yt[p] = acc;"),
    ("group_index_modulo", "const int64_t g = h / heads_per_group;",
     "const int64_t g = h % G;"),
    ("checkpoint_off_by_one", "t % ckpt_every == 0", "(t + 1) % ckpt_every == 0"),
    ("cumsum_exclusive",
     "run += A[h] * dt[(b * seqlen + t) * nheads + h];\n"
     "                G[(b * nheads + h) * seqlen + t] = log2e * run;",
     "G[(b * nheads + h) * seqlen + t] = log2e * run;\n"
     "                run += A[h] * dt[(b * seqlen + t) * nheads + h];"),
    ("cumsum_natural_log", "= log2e * run;", "= run;"),
    ("cumsum_no_chunk_reset", "if (t % chunk == 0) run = 0.0;", "if (t == 0) run = 0.0;"),
    ("conv_shifted_window", "const int64_t ts = t - width + 1 + k;", "const int64_t ts = t - width + k;"),
    ("conv_reads_future", "const int64_t ts = t - width + 1 + k;", "const int64_t ts = t + k;"),
    ("conv_taps_reversed", "acc += weight[d * width + k] * xr[ts];",
     "acc += weight[d * width + (width - 1 - k)] * xr[ts];"),
    ("conv_dropped_bias", "double acc = bias ? bias[d] : 0.0;", "double acc = 0.0;"),
    ("conv_padding_drops_first", "if (ts >= 0) acc", "if (ts > 0) acc"),
    ("gdn_delta_sign", "vt[v] = ut[v] - acc;", "vt[v] = ut[v] + acc;"),
    ("gdn_gate_inverted", "const double gate = exp(g_last - g[(b * T + t) * H + hh]);",
     "const double gate = exp(g[(b * T + t) * H + hh] - g_last);"),
    ("gdn_no_state_decay", "double acc = S[kk * V + v] * decay;", "double acc = S[kk * V + v];"),
    ("gdn_g_last_first_token", "const double g_last = g[(b * T + t1 - 1) * H + hh];",
     "const double g_last = g[(b * T + t0) * H + hh];"),
    ("gdn_o_mask_drops_diagonal", "for (int64_t j = t0; j <= i; ++j) {", "for (int64_t j = t0; j < i; ++j) {"),
    ("gdn_o_inter_undecayed", "oi[v] = inter * exp(gi);", "oi[v] = inter;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    mutant = tmp_path / "mutant.c"
    mutant.write_text(text.replace(old, new, 1))
    lib = oracle.load(oracle.build(str(mutant), str(tmp_path / "libmutant.so")))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
