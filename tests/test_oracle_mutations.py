"""The pins are strong enough: each plausible mistake planted in a copy of the
C oracle (a dropped term, a wrong sign, index or layout, in the forward or in
its adjoint) fails at least one pin.

The mutants are compiled from a textual edit of oracle/gdn_ref.c into a
temporary directory; the committed oracle is never modified.
"""
import os

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "gdn_ref.c")

MUTANTS = {
    "pred_without_decay": ("pred[j] *= alpha;", "pred[j] *= 1.0;"),
    "correction_sign": ("(vt[j] - pred[j])", "(vt[j] + pred[j])"),
    "no_write_term": ("ai * Si[j] + bki * (vt[j] - pred[j])", "ai * Si[j]"),
    "beta_dropped": ("const double bki = b * kt[i];", "const double bki = kt[i];"),
    "decay_sign": ("gk ? 1.0 : exp(g[t * Hv + hv])", "gk ? 1.0 : exp(-g[t * Hv + hv])"),
    "no_scale": ("ot[j] *= scale;", "ot[j] *= 1.0;"),
    "gqa_modulo": ("h = hv / HG;", "h = hv % H;"),
    "initial_state_transposed": ("initial_state[((n * Hv + hv) * dv + j) * dk + i]",
                                 "initial_state[((n * Hv + hv) * dk + i) * dv + j]"),
    "final_state_transposed": ("final_state[((n * Hv + hv) * dv + j) * dk + i]",
                               "final_state[((n * Hv + hv) * dk + i) * dv + j]"),
    "read_uses_query_of_key": ("ot[j] += Si[j] * qi;", "ot[j] += Si[j] * kt[i];"),
    "decay_not_applied_to_state": ("Si[j] = ai * Si[j] +", "Si[j] = Si[j] +"),
    "channel_pred_without_decay": ("gk ? exp(gk[i]) * kt[i] : kt[i]", "kt[i]"),
    "channel_state_decay_first_channel": ("gk ? exp(gk[i]) : alpha", "gk ? exp(gk[0]) : alpha"),
    "channel_gate_stride": ("g + (t * Hv + hv) * dk", "g + (t * Hv + hv)"),
    "channel_gate_sign": ("const double ai = gk ? exp(gk[i])", "const double ai = gk ? exp(-gk[i])"),
    "l2norm_without_sqrt": ("1.0 / sqrt(ss + eps)", "1.0 / (ss + eps)"),
    "default_scale_wrong": ("scale = 1.0 / sqrt((double)dk); /* also catches NaN */",
                            "scale = 1.0 / (double)dk; /* also catches NaN */"),
    "sequence_start_ignored": ("t0 = cu_seqlens ? cu_seqlens[n] : 0", "t0 = 0"),
    # backward (adjoint) mistakes
    "bwd_no_read_gradient": ("dS[i * dv + j] += scale * qt[i] * dot[j];",
                             "dS[i * dv + j] += 0.0 * qt[i] * dot[j];"),
    "bwd_dq_from_old_state": ("acc += St[i * dv + j] * dot[j];", "acc += Sp[i * dv + j] * dot[j];"),
    "bwd_dk_without_prediction_term": ("dkt[i] -= acc;", "dkt[i] += 0.0 * acc;"),
    "bwd_dpred_sign": ("dD[i * dv + j] = dS[i * dv + j] - kt[i] * dvt[j];",
                       "dD[i * dv + j] = dS[i * dv + j] + kt[i] * dvt[j];"),
    "bwd_dg_without_alpha": ("dg[t * Hv + hv] = alpha * da;", "dg[t * Hv + hv] = da;"),
    "bwd_dbeta_dropped": ("dbeta[t * Hv + hv] = db;", "dbeta[t * Hv + hv] = 0.0;"),
    "bwd_state_gradient_not_decayed": ("dS[i] = alpha * dD[i];", "dS[i] = dD[i];"),
    "bwd_dv_without_beta": ("dvt[j] = b * acc;", "dvt[j] = acc;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    before, after = MUTANTS[name]
    with open(SRC) as f:
        text = f.read()
    assert text.count(before) == 1, f"mutation site for {name} not unique"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(before, after))
    lib = oracle.load_library(oracle.compile_library(str(src), str(tmp_path / "libm.so")))
    failed = []
    for pin in P.ALL_PINS + P.BACKWARD_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutant {name}"
