"""Pins of the oracle's reward-weighted distillation loss (``oracle_kd``).

Each pin checks the oracle against something other than its own formula: a
library routine (scipy's relative entropy on independently computed
softmaxes), a closed form (a uniform draft), invariants (Gibbs, sum of the
gradient, the temperature identity), or the derivative of the oracle's own
loss by central differences.  Planted mistakes must be caught (bottom).
"""
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax
from scipy.stats import entropy

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def _rows(seed, n_seq=3, t_len=4, V=64, scale=2.0, noise=0.6):
    rng = np.random.default_rng(seed)
    t = (rng.normal(0, scale, (n_seq, t_len, V))).astype(np.float32)
    d = (t + rng.normal(0, noise, t.shape)).astype(np.float32)
    return t, d


def test_kl_matches_scipy_relative_entropy():
    t, d = _rows(0)
    for T in (1.0, 0.7, 1.9):
        r = oracle.kd(t, d, np.ones(t.shape[0]), T)
        for b in range(t.shape[0]):
            for j in range(t.shape[1]):
                p = softmax(t[b, j].astype(np.float64) / T)
                q = softmax(d[b, j].astype(np.float64) / T)
                assert abs(r["row_kl"][b, j] - entropy(p, q)) < 1e-12


def test_uniform_draft_closed_form():
    # KL(p || uniform) = log V - H(p)
    t, _ = _rows(1, V=37)
    d = np.zeros_like(t)
    r = oracle.kd(t, d, np.ones(t.shape[0]), 1.0)
    for b in range(t.shape[0]):
        for j in range(t.shape[1]):
            p = softmax(t[b, j].astype(np.float64))
            assert abs(r["row_kl"][b, j] - (np.log(37) - entropy(p))) < 1e-12


def test_identical_rows_give_zero_loss_and_gradient():
    t, _ = _rows(2)
    r = oracle.kd(t, t.copy(), np.full(t.shape[0], 3.0), 0.8)
    assert np.abs(r["row_kl"]).max() < 1e-14
    assert np.abs(r["grad"]).max() < 1e-15
    assert (r["status"] == 0).all()


def test_gibbs_inequality_and_gradient_sums_to_zero():
    t, d = _rows(3, V=200)
    r = oracle.kd(t, d, np.array([0.5, 1.0, 2.0]), 1.3)
    assert (r["row_kl"] > 0).all()
    assert np.abs(r["grad"].sum(axis=2)).max() < 1e-14


def test_gradient_is_the_derivative_of_the_loss():
    # central differences of the oracle's own loss in the draft logits; the
    # logits and the step are exact in fp32
    rng = np.random.default_rng(4)
    V, T = 12, 0.75
    t = (rng.integers(-128, 128, (1, 1, V)) / 64.0).astype(np.float32)
    d = (rng.integers(-128, 128, (1, 1, V)) / 64.0).astype(np.float32)
    w = np.array([1.7])
    g = oracle.kd(t, d, w, T)["grad"][0, 0]
    h = 1.0 / 512
    for x in range(V):
        dp, dm = d.copy(), d.copy()
        dp[0, 0, x] += h
        dm[0, 0, x] -= h
        fd = (oracle.kd(t, dp, w, T, grad=False)["loss"][0] - oracle.kd(t, dm, w, T, grad=False)["loss"][0]) / (2 * h)
        assert abs(fd - g[x]) < 1e-5 * max(1.0, abs(g[x])), (x, fd, g[x])


def test_loss_is_the_weighted_sum_of_the_rows():
    t, d = _rows(5)
    w = np.array([0.25, 4.0, 0.0])
    r = oracle.kd(t, d, w, 1.0)
    np.testing.assert_allclose(r["loss"], w * r["row_kl"].sum(axis=1), rtol=1e-15, atol=0)
    r2 = oracle.kd(t, d, 2 * w, 1.0)
    np.testing.assert_allclose(r2["loss"], 2 * r["loss"], rtol=1e-15)
    np.testing.assert_allclose(r2["grad"], 2 * r["grad"], rtol=1e-15)
    assert (r["grad"][2] == 0).all()          # zero weight, zero gradient


def test_temperature_identity():
    # KL at temperature T of z equals KL at T = 1 of z / T (T a power of two,
    # so z / T is exact in fp32)
    t, d = _rows(6)
    for T in (0.5, 2.0, 0.25):
        a = oracle.kd(t, d, np.ones(3), T)
        b = oracle.kd((t / T).astype(np.float32), (d / T).astype(np.float32), np.ones(3), 1.0)
        np.testing.assert_allclose(a["row_kl"], b["row_kl"], rtol=1e-12)
        np.testing.assert_allclose(a["grad"] * T, b["grad"], rtol=1e-9, atol=1e-15)


def test_masked_tokens():
    t, d = _rows(7, n_seq=1, t_len=2, V=16)
    t[0, 0, 3] = -np.inf          # p(3) = 0: the term is 0, KL stays finite
    d[0, 1, 5] = -np.inf          # q(5) = 0 < p(5): KL = +inf
    r = oracle.kd(t, d, np.ones(1), 1.0)
    p = softmax(t[0, 0].astype(np.float64))
    q = softmax(d[0, 0].astype(np.float64))
    assert abs(r["row_kl"][0, 0] - entropy(p, q)) < 1e-12
    assert r["row_kl"][0, 1] == np.inf
    assert (r["status"] == 0).all()


def test_invalid_rows_mark_only_their_rollout():
    t, d = _rows(8)
    t[1, 2, 7] = np.nan
    d[2, 0, :] = -np.inf
    r = oracle.kd(t, d, np.ones(3), 1.0)
    assert r["status"][1, 2] == oracle.STATUS_NONFINITE and r["status"][2, 0] == oracle.STATUS_NONFINITE
    assert np.isnan(r["loss"][1]) and np.isnan(r["loss"][2]) and np.isfinite(r["loss"][0])
    assert np.isnan(r["grad"][1, 2]).all() and np.isfinite(r["grad"][1, 1]).all()


def test_bf16_inputs_are_widened_exactly():
    t, d = _rows(9)
    tb, db = torch.from_numpy(t).to(torch.bfloat16), torch.from_numpy(d).to(torch.bfloat16)
    a = oracle.kd(tb, db, np.ones(3), 1.0)
    b = oracle.kd(tb.float().numpy(), db.float().numpy(), np.ones(3), 1.0)
    np.testing.assert_array_equal(a["row_kl"], b["row_kl"])
    np.testing.assert_array_equal(a["grad"], b["grad"])


# --- planted mistakes --------------------------------------------------------------

KD_MUTANTS = {
    "kl_direction_swapped": ("kl += p * (lp - lq);", "kl += p * (lq - lp);"),
    "kl_weighted_by_q": ("kl += p * (lp - lq);", "kl += q * (lp - lq);"),
    "gradient_sign": ("grad[(size_t)r * V + x] = w * (q - p) / T;", "grad[(size_t)r * V + x] = w * (p - q) / T;"),
    "gradient_temperature_dropped": ("grad[(size_t)r * V + x] = w * (q - p) / T;",
                                     "grad[(size_t)r * V + x] = w * (q - p);"),
    "draft_normaliser_from_target": ("const double lq = (zd[x] - md) / T - Ld;      /* log q(x) */",
                                     "const double lq = (zd[x] - mt) / T - Lt;      /* log q(x) */"),
    "weight_of_next_rollout": ("const double w = weights[r / t_len];", "const double w = weights[(r + 1) / t_len % n_seq];"),
    "loss_unweighted": ("loss[b] = weights[b] * s;", "loss[b] = s;"),
}


def _kd_pins_pass(lib):
    t, d = _rows(0, n_seq=2, t_len=2, V=24)
    w = np.array([0.5, 2.0])
    r = oracle.kd(t, d, w, 0.75, lib=lib)
    for b in range(2):
        for j in range(2):
            p = softmax(t[b, j].astype(np.float64) / 0.75)
            q = softmax(d[b, j].astype(np.float64) / 0.75)
            if abs(r["row_kl"][b, j] - entropy(p, q)) > 1e-12:
                return False
            if np.abs(r["grad"][b, j] - w[b] * (q - p) / 0.75).max() > 1e-12:
                return False
    if np.abs(r["loss"] - w * r["row_kl"].sum(axis=1)).max() > 1e-12:
        return False
    return True


def test_unmutated_kd_oracle_passes():
    assert _kd_pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(KD_MUTANTS))
def test_kd_mutant_is_caught(name, tmp_path):
    old, new = KD_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = oracle.build(force=True, src=str(mpath), out=str(tmp_path / "libmutant.so"))
    assert not _kd_pins_pass(oracle.load(so)), f"mutant {name} survived"
