"""The oracle's pins must catch plausible mistakes.

Each case copies ``oracle/oracle.c`` to a temporary directory, plants one
mistake by a textual replacement (a wrong operand order, a flipped sign, a
wrong index, a dropped term or a non-strict comparison), compiles the mutant
and runs the pins against it.  At least one pin must fail for every mutant.
The oracle source itself is never modified.
"""
import os

import numpy as np
import pytest
from scipy.special import logsumexp

import oracle
from tests import enum_cases

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "ratio_inverted": ("p / q;", "q / p;"),
    "residual_sign": ("double d = prob_of(zt[x], mt[a], Lt[a], T) - prob_of(zd[x], md[a], Ld[a], T);",
                      "double d = prob_of(zd[x], md[a], Ld[a], T) - prob_of(zt[x], mt[a], Lt[a], T);"),
    "sampling_uniform_column": ("(double)u[k], &stie", "(double)u[a], &stie"),
    "last_rejection_instead_of_first": ("a = i;\n                        decided = 1;", "a = i;"),
    "temperature_dropped": ("s += exp((z[x] - m) / T);", "s += exp(z[x] - m);"),
    "bonus_row_off_by_one": ("load_row(target, dtype, (size_t)b * (k + 1) + a, V, zt);",
                             "load_row(target, dtype, (size_t)b * (k + 1) + (a > 0 ? a - 1 : 0), V, zt);"),
    "p_uses_draft_normaliser": ("double p = prob_of(zt_x, mt[i], Lt[i], T);",
                                "double p = prob_of(zt_x, md[i], Ld[i], T);"),
    "non_strict_accept": ("if (!((double)u[i] < al))", "if (!((double)u[i] <= al))"),
    "non_strict_cdf": ("if (t < c) {", "if (t <= c) {"),
    "no_residual_clamp": ("w[x] = d > 0.0 ? d : 0.0;", "w[x] = d;"),
    # the near-tie diagnostics the parity tests rely on
    "sample_tie_in_cdf_units": ("double d0 = fabs(s - c_prev / S), d1 = fabs(s - c / S);",
                                "double d0 = fabs(t - c_prev), d1 = fabs(t - c);"),
    "sample_tie_one_boundary": ("*tie = d0 < d1 ? d0 : d1;", "*tie = d1;"),
    "accept_tie_over_every_test": (
        "                if (!decided) {\n                    double d = fabs((double)u[i] - al);\n"
        "                    if (d < atie) atie = d;",
        "                double d = fabs((double)u[i] - al);\n                if (d < atie) atie = d;\n"
        "                if (!decided) {"),
    "resid_mass_reports_the_point": ("            if (resid_mass) resid_mass[b] = S;\n            if (sample_tie)",
                                     "            if (resid_mass) resid_mass[b] = S * (double)u[k];\n"
                                     "            if (sample_tie)"),
    "window_band_in_cdf_units": ("double t_lo = (s - band) * S, t_hi = (s + band) * S",
                                 "double t_lo = s * S - band, t_hi = s * S + band"),
}


def _pins_pass(lib):
    """Run a compact version of the pins; return False at the first failure."""
    V, k = 4, 2
    for kb, T, seed in [(2, 1.0, 0), (1, 0.7, 1), (0, 1.6, 2), (2, 0.7, 5)]:
        batch, P = enum_cases.build(V=V, k=k, kb=kb, T=T, seed=seed)
        res = oracle.verify(batch["target"], batch["draft"], batch["tokens"],
                            batch["draft_len"], batch["uniforms"], T, lib=lib)
        if not (res["status"] == 0).all():
            return False
        if (res["out_tokens"] < 0).any() and (res["out_len"] == 0).any():
            return False
        got = enum_cases.joint_from_outputs(res["out_tokens"], res["out_len"], batch["weight"], P, V, k)
        if np.max(np.abs(got - enum_cases.target_joint(P, V, k))) > 1e-12:
            return False
    # the near-tie diagnostics against numpy, narrow and wide band
    from tests.test_oracle_diagnostics import check_linear
    for seed, band in ((3, 1e-5), (4, 0.02)):
        try:
            check_linear(lib, seed=seed, dtype="f32", T=1.0, band=band)
        except AssertionError:
            return False
    rng = np.random.default_rng(5)
    z = rng.normal(0, 3, 300).astype(np.float32)
    if abs(oracle.row_lse(z, 0.6, lib=lib) - logsumexp(z.astype(np.float64) / 0.6)) > 1e-10:
        return False
    # edge conventions: forbidden draft token at u = 0; s = 0 on a zero-weight token
    t = np.zeros((1, 2, 6), np.float32)
    t[0, 0, 2] = -np.inf
    r = oracle.verify(t, np.zeros((1, 1, 6), np.float32), np.array([[2]], np.int32),
                      np.array([1], np.int32), np.zeros((1, 2), np.float32), 1.0, lib=lib)
    if r["out_len"][0] != 1 or r["out_tokens"][0, 0] == 2:
        return False
    t = np.log(np.array([[[0.1, 0.4, 0.2, 0.2, 0.1], [0.2] * 5]], np.float32))
    d = np.log(np.array([[[0.5, 0.1, 0.2, 0.1, 0.1]]], np.float32))
    r = oracle.verify(t, d, np.array([[0]], np.int32), np.array([1], np.int32),
                      np.array([[0.9, 0.0]], np.float32), 1.0, lib=lib)
    if r["out_len"][0] != 1 or r["out_tokens"][0, 0] != 1:
        return False
    return True


def test_unmutated_oracle_passes_compact_pins():
    assert _pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = oracle.build(force=True, src=str(mpath), out=str(tmp_path / "libmutant.so"))
    lib = oracle.load(so)
    assert not _pins_pass(lib), f"mutant {name} survived the pins"
