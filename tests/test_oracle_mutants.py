"""Planted mistakes in the oracle (on the CPU): each mutant of the oracle's C
source must fail at least one pin, so the pins would catch that mistake."""
import os

import pytest

import oracle as oracle_pkg
from tests import _pins

MUTANTS = {
    "residual_sign_flipped": ("w[j] = p[j] > q[j] ? p[j] - q[j] : 0.0;", "w[j] = q[j] > p[j] ? q[j] - p[j] : 0.0;"),
    "rejected_uniform_reused": ("y = so_sample(w, V, (double)in->u[k], &ctie, &out->residual_mass);",
                                "y = so_sample(w, V, (double)in->u[i], &ctie, &out->residual_mass);"),
    "target_row_off_by_one": ("const void* trow = (const char*)in->target + (size_t)i * rs;",
                              "const void* trow = (const char*)in->target + (size_t)(i + 1) * rs;"),
    "accept_inverted": ("acc = u < theta;", "acc = u > theta;"),
    "temperature_dropped": ("logp[j] = logit_at(row, dtype, j) / T - lse;", "logp[j] = logit_at(row, dtype, j) - lse;"),
    "tv_missing_half": ("out->tv[i] = 0.5 * s;", "out->tv[i] = s;"),
    "bonus_from_draft_row": ("""      tau = k;
      int ctie = 0;
      y = so_sample(p, V,""", """      tau = k;
      int ctie = 0;
      row_distribution((const char*)in->draft + (size_t)(k - 1) * rs, in->dtype, V, in->T, p, lp);
      y = so_sample(p, V,"""),
    "argmax_last_of_ties": ("if (z > m) { m = z; a = j; }", "if (z >= m) { m = z; a = j; }"),
    "cdf_not_strict": ("if (t < C) { y = j; break; }", "if (t <= C) { y = j; break; }"),
    "lse_missing_max": ("double lse = lmax + log(s);", "double lse = log(s);"),
    "entropy_in_bits": ("if (lp > -INFINITY) h -= exp(lp) * lp;", "if (lp > -INFINITY) h -= exp(lp) * lp / log(2.0);"),
    "entropy_sign_flipped": ("if (lp > -INFINITY) h -= exp(lp) * lp;", "if (lp > -INFINITY) h += exp(lp) * lp;"),
    "entropy_without_temperature": ("double lp = logit_at(row, dtype, j) / T - lse;",
                                    "double lp = logit_at(row, dtype, j) - lse;"),
    "grad_without_temperature": ("grad[j] = w * dl * (qj / T) * ((qj < pj ? 1.0 : 0.0) - beta);",
                                 "grad[j] = w * dl * qj * ((qj < pj ? 1.0 : 0.0) - beta);"),
    "grad_indicator_flipped": ("grad[j] = w * dl * (qj / T) * ((qj < pj ? 1.0 : 0.0) - beta);",
                               "grad[j] = w * dl * (qj / T) * ((qj > pj ? 1.0 : 0.0) - beta);"),
    "grad_beta_dropped": ("grad[j] = w * dl * (qj / T) * ((qj < pj ? 1.0 : 0.0) - beta);",
                          "grad[j] = w * dl * (qj / T) * (qj < pj ? 1.0 : 0.0);"),
    "tie_band_too_wide": ("#define SO_TIE_BAND 1e-6", "#define SO_TIE_BAND 1e-4"),
    "cdf_tie_below_boundary_missed": (
        "if (tie) *tie = fabs(t - C) < SO_TIE_BAND * S || fabs(t - Cprev) < SO_TIE_BAND * S;",
        "if (tie) *tie = fabs(t - C) < SO_TIE_BAND * S;"),
    "overlap_loss_log_missing": ("*loss = kind == 0 ? 1.0 - alpha : -log(alpha);", "*loss = kind == 0 ? 1.0 - alpha : -alpha;"),
    # batch drivers: row strides, the draft row's buffer, and the weight index
    "entropy_target_row_stride": ("so_entropy((const char*)J->target + (size_t)(b * (J->k + 1) + i) * rs",
                                  "so_entropy((const char*)J->target + (size_t)(b * J->k + i) * rs"),
    "entropy_draft_row_from_target": ("so_entropy((const char*)J->draft + (size_t)(b * J->k + (i - J->k - 1)) * rs",
                                      "so_entropy((const char*)J->target + (size_t)(b * J->k + (i - J->k - 1)) * rs"),
    "grad_target_row_stride": ("so_overlap_grad((const char*)J->target + (size_t)(b * (J->k + 1) + i) * rs",
                               "so_overlap_grad((const char*)J->target + (size_t)(b * J->k + i) * rs"),
    "grad_draft_row_stride": ("(const char*)J->draft + (size_t)(b * J->k + i) * rs, J->dtype",
                              "(const char*)J->draft + (size_t)(b * (J->k + 1) + i) * rs, J->dtype"),
    "grad_weight_per_chain": ("J->w ? (double)J->w[r] : 1.0", "J->w ? (double)J->w[b] : 1.0"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    src = open(oracle_pkg.SOURCE).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = src.replace(old, new)
    csrc = os.path.join(tmp_path, f"mutant_{name}.c")
    with open(csrc, "w") as f:
        f.write(mutated)
    so = oracle_pkg.compile_source(csrc, os.path.join(tmp_path, f"libmutant_{name}.so"))
    orc = oracle_pkg.Oracle(so)
    failures = []
    for pin in _pins.ALL_PINS:
        try:
            pin(orc)
        except AssertionError as e:
            failures.append(pin.__name__)
            break
        except Exception as e:   # a crash in the mutant also counts as detection
            failures.append(f"{pin.__name__}: {type(e).__name__}")
            break
    assert failures, f"mutant {name} passed every pin"
