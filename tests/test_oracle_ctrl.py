"""Pins of the oracle's draft-length controller (``oracle_ctrl_*``).

Each pin checks the oracle against something other than its own formulas:
the maximum-likelihood rate of the truncated geometric law found by a
numerical optimiser, the Beta-posterior mean (scipy), the expected emitted
length by exact enumeration of the law of the accepted count and by Monte
Carlo, numpy's linear interpolation, closed-form decisions (free
verification, compute-bound rounds, alpha = 0 and 1) and a small case worked
by hand.  Planted mistakes must be caught (bottom).
"""
import os

import numpy as np
import pytest
from scipy import optimize, stats

import oracle

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def law_of_accepted(alpha, n):
    """P(a = j), j = 0..n: the first rejection after j accepts (j < n), or all
    n drafts accepted."""
    return np.array([alpha ** j * (1 - alpha) for j in range(n)] + [alpha ** n])


def simulate_rounds(rng, alpha, k, rounds):
    """Accepted counts of `rounds` rounds of draft length k at per-draft
    acceptance alpha (independent Bernoulli tests, stop at the first failure)."""
    u = rng.random((rounds, k))
    ok = u < alpha
    return np.where(ok.all(axis=1), k, np.argmin(ok, axis=1))


def ctl(lib, n_slots=16, max_k=7, batch_sizes=(1,), table=None, **kw):
    table = np.ones((len(batch_sizes), max_k + 1)) if table is None else table
    return oracle.Controller(n_slots, max_k, batch_sizes, table, lib=lib, **kw)


# --- the acceptance estimate ---------------------------------------------------------

def pin_estimate_is_the_truncated_geometric_mle(lib):
    rng = np.random.default_rng(0)
    for alpha, k in ((0.3, 3), (0.75, 7), (0.9, 5)):
        a = simulate_rounds(rng, alpha, k, 40)
        c = ctl(lib, max_k=k, decay=1.0, prior_weight=0.0)
        for x in a:
            c.observe([0], [k], [x + 1])
        nll = lambda t: -sum(np.log(law_of_accepted(t, k)[x]) for x in a)
        mle = optimize.minimize_scalar(nll, bounds=(1e-9, 1 - 1e-9), method="bounded",
                                       options={"xatol": 1e-10}).x
        assert abs(c.alpha([0])[0] - mle) < 1e-6, (alpha, k, c.alpha([0])[0], mle)


def pin_estimate_is_the_beta_posterior_mean(lib):
    # w0 pseudo-tests at rate alpha0 = a Beta(alpha0 w0, (1 - alpha0) w0)
    # prior; with decay 1 the estimate is the posterior mean
    rng = np.random.default_rng(1)
    a = simulate_rounds(rng, 0.6, 4, 25)
    for alpha0, w0 in ((0.5, 2.0), (0.8, 10.0), (0.1, 0.5)):
        c = ctl(lib, max_k=4, decay=1.0, prior_alpha=alpha0, prior_weight=w0)
        for x in a:
            c.observe([3], [4], [x + 1])
        succ = a.sum()
        fail = (a < 4).sum()
        post = stats.beta(alpha0 * w0 + succ, (1 - alpha0) * w0 + fail).mean()
        assert abs(c.alpha([3])[0] - post) < 1e-14
        assert c.alpha([2])[0] == alpha0        # never observed: the prior


def pin_estimate_converges(lib):
    rng = np.random.default_rng(2)
    for alpha in (0.2, 0.55, 0.93):
        a = simulate_rounds(rng, alpha, 6, 20000)
        c = ctl(lib, max_k=6, decay=1.0, prior_weight=0.0)
        for x in a:
            c.observe([5], [6], [x + 1])
        tests = a.sum() + (a < 6).sum()
        assert abs(c.alpha([5])[0] - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / tests)


def pin_decay_is_exponential(lib):
    # the same observation m times: A = a (1 - d^m) / (1 - d), N likewise
    d, m, k, a = 0.8, 9, 5, 2
    c = ctl(lib, max_k=k, decay=d, prior_weight=0.0)
    for _ in range(m):
        c.observe([1], [k], [a + 1])
    g = (1 - d ** m) / (1 - d)
    assert abs(c.A[1] - a * g) < 1e-13 and abs(c.N[1] - (a + 1) * g) < 1e-13
    # a full acceptance has no rejection test: N grows by k only
    c2 = ctl(lib, max_k=k, decay=1.0, prior_weight=0.0)
    c2.observe([0], [k], [k + 1])
    assert c2.A[0] == k and c2.N[0] == k


def pin_row_status(lib):
    c = ctl(lib, n_slots=6, max_k=3, decay=1.0, prior_weight=0.0)
    st = c.observe([0, 1, 1, 7, -1, 2, 3, 4, 5], [3, 3, 3, 3, 3, 4, 3, 0, 2], [2, 1, 1, 1, 1, 1, 0, 1, 4])
    #                ok  dup dup out neg badk  out0 k=0 len>k+1
    assert list(st) == [0, 5, 5, 5, 5, 2, 1, 1, 2], st
    assert c.A[0] == 1 and c.N[0] == 2
    assert (c.A[1:] == 0).all() and (c.N[1:] == 0).all()


# --- expected tokens and round time -------------------------------------------------

def pin_expected_tokens_by_enumeration(lib):
    for alpha in (0.0, 0.13, 0.5, 0.77, 0.999, 1.0):
        for n in range(0, 12):
            exact = float(np.dot(np.arange(1, n + 2), law_of_accepted(alpha, n)))
            assert abs(lib.oracle_ctrl_expected_tokens(alpha, n) - exact) < 1e-13 * (n + 1)
    assert lib.oracle_ctrl_expected_tokens(1.0, 6) == 7.0
    assert lib.oracle_ctrl_expected_tokens(0.0, 6) == 1.0


def pin_expected_tokens_by_simulation(lib):
    rng = np.random.default_rng(3)
    alpha, n = 0.7, 5
    a = simulate_rounds(rng, alpha, n, 200000)
    mc = (a + 1).mean()
    sd = (a + 1).std() / np.sqrt(a.size)
    assert abs(lib.oracle_ctrl_expected_tokens(alpha, n) - mc) < 4 * sd


def pin_round_time_interpolates_linearly(lib):
    rng = np.random.default_rng(4)
    bs = np.array([1, 8, 32, 33, 256], np.int32)
    table = rng.uniform(0.5, 5.0, (bs.size, 4))
    c = ctl(lib, max_k=3, batch_sizes=bs, table=table)
    for B in (1, 2, 7, 8, 20, 32, 33, 100, 256, 1000, 0):
        for n in range(4):
            want = np.interp(B, bs, table[:, n])       # clamps outside, like the oracle
            assert abs(c.round_time(B, n) - want) < 1e-14 * want, (B, n)
    for j, B in enumerate(bs):                          # exactly the row at a profiled size
        assert [c.round_time(B, n) for n in range(4)] == list(table[j])


# --- the choice ---------------------------------------------------------------------

def pin_choice_closed_forms(lib):
    K = 7
    ids = np.arange(5, dtype=np.int32)
    # free verification: T(B, n) = T(B, 0): E_n grows with n, so max_k
    c = ctl(lib, max_k=K, table=np.full((1, K + 1), 2.0), prior_alpha=0.3)
    assert c.choose(ids)["choice"] == K
    # compute-bound rounds T = (n + 1) T0: E_n / (n + 1) < 1 for alpha < 1, so off
    c = ctl(lib, max_k=K, table=(np.arange(K + 1) + 1.0)[None], prior_alpha=0.95)
    r = c.choose(ids)
    assert r["choice"] == 0 and (r["next_len"] == 0).all()
    # alpha = 0: every E_n = 1 and T non-decreasing in n: off, even on ties
    c = ctl(lib, max_k=K, table=np.full((1, K + 1), 1.0), prior_alpha=0.0)
    assert c.choose(ids)["choice"] == 0
    # alpha = 1 with sub-linear time: (n + 1) / (1 + n/2) grows: max_k
    c = ctl(lib, max_k=K, table=(1.0 + 0.5 * np.arange(K + 1))[None], prior_alpha=1.0)
    assert c.choose(ids)["choice"] == K


def pin_choice_worked_case(lib):
    # alpha = 1/2: E_n = 1, 3/2, 7/4, 15/8; T = 1, 6/5, 3/2, 2 give rates
    # 1, 5/4, 7/6, 15/16: one draft
    c = ctl(lib, max_k=3, table=np.array([[1.0, 1.2, 1.5, 2.0]]), prior_alpha=0.5)
    r = c.choose(np.array([0], np.int32))
    assert r["choice"] == 1
    np.testing.assert_allclose(r["rates"], [1.0, 1.25, 7 / 6, 15 / 16], rtol=1e-15)
    # per-sequence mode, slots at 1/2 (one draft, as above) and 9/10: E =
    # 1, 1.9, 2.71, 3.439 gives rates 1, 1.583, 1.807, 1.7195: two drafts
    c = ctl(lib, max_k=3, table=np.array([[1.0, 1.2, 1.5, 2.0]]), mode=1, decay=1.0, prior_weight=0.0)
    c.observe([0, 1], [3, 3], [2, 4])           # slot 0: 1 of 2 tests; slot 1: 3 of 3
    c.A[1], c.N[1] = 9.0, 10.0                   # rate 9/10 for slot 1
    r = c.choose(np.array([0, 1], np.int32))
    assert list(r["next_len"]) == [1, 2] and r["choice"] == 2


def pin_choice_by_brute_force(lib):
    # batch mode against enumeration-based expectations and numpy's
    # interpolation, on random states and tables
    rng = np.random.default_rng(5)
    for trial in range(20):
        K = int(rng.integers(1, 9))
        bs = np.sort(rng.choice(np.arange(1, 600), size=3, replace=False)).astype(np.int32)
        base = rng.uniform(1.0, 3.0, (3, 1))
        table = base * (1.0 + rng.uniform(0.0, 0.6, (3, 1)) * np.arange(K + 1)[None])
        c = ctl(lib, n_slots=40, max_k=K, batch_sizes=bs, table=table, decay=1.0, prior_weight=1.0,
                prior_alpha=float(rng.uniform()))
        c.A[:] = rng.uniform(0, 20, 40)
        c.N[:] = c.A + rng.uniform(0, 20, 40)
        ids = rng.permutation(40)[: int(rng.integers(1, 40))].astype(np.int32)
        B = ids.size
        al = (c.A[ids] + c.prior_alpha * 1.0) / (c.N[ids] + 1.0)
        E = np.array([[np.dot(np.arange(1, n + 2), law_of_accepted(x, n)) for n in range(K + 1)] for x in al])
        T = np.array([np.interp(B, bs, table[:, n]) for n in range(K + 1)])
        rates = E.sum(axis=0) / T
        r = c.choose(ids)
        srt = np.sort(rates)
        if K == 0 or (srt[-1] - srt[-2]) / srt[-1] > 1e-9:
            assert r["choice"] == int(np.argmax(rates)), (trial, rates, r)
        np.testing.assert_allclose(r["rates"], rates, rtol=1e-12)
        c.mode = 1
        r1 = c.choose(ids)
        per = E / T[None]
        for b in range(B):
            s = np.sort(per[b])
            if (s[-1] - s[-2]) / s[-1] > 1e-9:
                assert r1["next_len"][b] == int(np.argmax(per[b]))


def pin_bad_ids_get_no_draft(lib):
    c = ctl(lib, n_slots=4, max_k=3, table=np.full((1, 4), 1.0), prior_alpha=0.9)
    r = c.choose(np.array([0, 9, -2, 3], np.int32))
    assert list(r["next_len"]) == [3, 0, 0, 3] and list(r["status"]) == [0, 5, 5, 0]


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__[4:] for p in PINS])
def test_controller_pin(pin):
    pin(oracle.load())


# --- planted mistakes --------------------------------------------------------------

CTRL_MUTANTS = {
    "tests_counted_as_drafted": ("N[id] = decay * N[id] + (double)(a + r);", "N[id] = decay * N[id] + (double)k;"),
    "rejection_not_counted": ("const int r = (a < k) ? 1 : 0;", "const int r = 0;"),
    "decay_missing_on_tests": ("N[id] = decay * N[id] + (double)(a + r);", "N[id] = N[id] + (double)(a + r);"),
    "prior_dropped": ("return (A + alpha0 * w0) / den;", "return A / den;"),
    "expected_tokens_from_one": ("for (int j = 0; j <= n; ++j)\n        e += pow",
                                 "for (int j = 1; j <= n; ++j)\n        e += pow"),
    "ties_to_longer_draft": ("if (R[n] > top) {", "if (R[n] >= top) {"),
    "interpolation_neighbours_swapped": (
        "const double t0 = table[(size_t)j * K1 + n], t1 = table[(size_t)(j + 1) * K1 + n];",
        "const double t1 = table[(size_t)j * K1 + n], t0 = table[(size_t)(j + 1) * K1 + n];"),
    "batch_rate_not_divided_by_time": ("R[n] = R[n] / T[n];", "R[n] = R[n] / T[0];"),
    "long_emitted_length_accepted": ("len < 0 || len > k + 1", "len < 0 || len > k + 2"),
    "repeated_id_kept": ("if (c != b && seq_ids[c] == id)", "if (c > b && seq_ids[c] == id)"),
}


def _ctrl_pins_pass(lib):
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            return False
    return True


def test_unmutated_controller_oracle_passes():
    assert _ctrl_pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(CTRL_MUTANTS))
def test_controller_mutant_is_caught(name, tmp_path):
    old, new = CTRL_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/present"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = oracle.build(force=True, src=str(mpath), out=str(tmp_path / "libmutant.so"))
    assert not _ctrl_pins_pass(oracle.load(so)), f"mutant {name} survived"
