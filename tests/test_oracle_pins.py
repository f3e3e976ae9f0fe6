"""Pins of the fp64 oracle to facts outside itself (no GPU needed).

Each test checks the oracle against something the pages or the mathematics
fix: exact enumeration of the output distribution, special cases that reduce
to a library routine, closed forms, and edge conventions.
"""
import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax
from scipy import stats

import oracle
from tests import enum_cases
from workloads import gumbel_argmax_tokens, philox_uniforms


# --- exact widening of the logits -----------------------------------------

def test_logit_widening_matches_torch():
    g = torch.Generator().manual_seed(11)
    x = torch.randn(257, generator=g) * 40
    x[3], x[7], x[9] = float("-inf"), 1e-40, -0.0
    xb = x.to(torch.bfloat16)
    np.testing.assert_array_equal(oracle.logit_values(xb), xb.float().double().numpy())
    np.testing.assert_array_equal(oracle.logit_values(x), x.double().numpy())


# --- log-sum-exp and softmax against scipy ---------------------------------

@pytest.mark.parametrize("T", [1.0, 0.6, 2.5, 1e-3])
def test_lse_and_probs_match_scipy(T):
    rng = np.random.default_rng(5)
    z = (rng.standard_t(3, 5000) * 2.5).astype(np.float32)
    z[[10, 20, 30]] = -np.inf
    ref = logsumexp(z.astype(np.float64) / T)
    assert abs(oracle.row_lse(z, T) - ref) <= 1e-12 * max(1.0, abs(ref))
    p = oracle.row_probs(z, T)
    np.testing.assert_allclose(p, softmax(z.astype(np.float64) / T), rtol=1e-12, atol=1e-300)
    assert p[10] == 0.0


# --- exhaustive enumeration: the output distribution is the target's -------

@pytest.mark.parametrize("kb", [0, 1, 2])
@pytest.mark.parametrize("T,seed", [(1.0, 0), (0.7, 1), (1.6, 2)])
def test_enumeration_reproduces_target_joint(kb, T, seed):
    V, k = 4, 2
    batch, P = enum_cases.build(V=V, k=k, kb=kb, T=T, seed=seed)
    res = oracle.verify(batch["target"], batch["draft"], batch["tokens"], batch["draft_len"],
                        batch["uniforms"], T)
    assert (res["status"] == 0).all()
    assert abs(batch["weight"].sum() - 1.0) < 1e-12
    got = enum_cases.joint_from_outputs(res["out_tokens"], res["out_len"], batch["weight"], P, V, k)
    want = enum_cases.target_joint(P, V, k)
    assert np.max(np.abs(got - want)) < 1e-12


def test_enumeration_acceptance_length_distribution():
    """With the same enumeration, P(a >= 1) must equal sum_x min(p0, q0)."""
    V, k = 4, 2
    batch, _ = enum_cases.build(V=V, k=k, kb=2, T=1.0, seed=3)
    res = oracle.verify(batch["target"], batch["draft"], batch["tokens"], batch["draft_len"],
                        batch["uniforms"], 1.0)
    p0 = softmax(batch["target"][0, 0].astype(np.float64))
    q0 = softmax(batch["draft"][0, 0].astype(np.float64))
    acc = batch["weight"][res["out_len"] >= 2].sum()
    assert abs(acc - np.minimum(p0, q0).sum()) < 1e-12


# --- q = p accepts every draft ----------------------------------------------

def test_identical_draft_accepts_all():
    rng = np.random.default_rng(9)
    B, k, V = 64, 5, 300
    t = (rng.normal(0, 3, (B, k + 1, V))).astype(np.float32)
    d = t[:, :k].copy()
    tok = rng.integers(0, V, (B, k)).astype(np.int32)
    kl = rng.integers(0, k + 1, B).astype(np.int32)
    u = philox_uniforms(B * (k + 1), seed=4).reshape(B, k + 1)
    res = oracle.verify(t, d, tok, kl, u, 0.9)
    np.testing.assert_array_equal(res["out_len"], kl + 1)
    for b in range(B):
        np.testing.assert_array_equal(res["out_tokens"][b, :kl[b]], tok[b, :kl[b]])
        np.testing.assert_array_equal(res["alpha"][b, :kl[b]], 1.0)


# --- T -> 0: accept iff the draft is the target's argmax --------------------

def _separated_rows(rng, n, V, gap=0.25):
    rows = np.empty((n, V), np.float32)
    for r in range(n):
        rows[r] = (rng.permutation(V) * gap - V * gap / 2).astype(np.float32)
    return rows


@pytest.mark.parametrize("T", [1e-3, 0.0])
def test_low_temperature_is_argmax(T):
    rng = np.random.default_rng(21)
    B, k, V = 200, 3, 64
    t = _separated_rows(rng, B * (k + 1), V).reshape(B, k + 1, V)
    d = _separated_rows(rng, B * k, V).reshape(B, k, V)
    # make the draft agree with the target's argmax on about half the rows
    agree = rng.random((B, k)) < 0.5
    d[agree] = t[:, :k][agree]
    tok = d.argmax(axis=2).astype(np.int32)          # x_i ~ q_i at T -> 0
    kl = np.full(B, k, np.int32)
    u = philox_uniforms(B * (k + 1), seed=6).reshape(B, k + 1)
    res = oracle.verify(t, d, tok, kl, u, T)
    amax = t.argmax(axis=2)
    for b in range(B):
        ok = tok[b] == amax[b, :k]
        a = k if ok.all() else int(np.argmin(ok))
        assert res["out_len"][b] == a + 1
        np.testing.assert_array_equal(res["out_tokens"][b, :a], tok[b, :a])
        assert res["out_tokens"][b, a] == amax[b, a]


def test_greedy_ties_take_lowest_id():
    V, k = 8, 1
    t = np.zeros((1, 2, V), np.float32)
    t[0, 0, [2, 5]] = 3.0
    t[0, 1, [1, 6]] = 4.0
    d = np.zeros((1, 1, V), np.float32)
    res = oracle.verify(t, d, np.array([[5]], np.int32), np.array([1], np.int32),
                        np.zeros((1, 2), np.float32), 0.0)
    assert res["out_len"][0] == 1 and res["out_tokens"][0, 0] == 2
    res = oracle.verify(t, d, np.array([[2]], np.int32), np.array([1], np.int32),
                        np.zeros((1, 2), np.float32), 0.0)
    assert res["out_len"][0] == 2 and list(res["out_tokens"][0]) == [2, 1]


# --- k_b = 0 is plain categorical sampling ----------------------------------

def test_no_draft_is_inverse_cdf_sampling():
    rng = np.random.default_rng(2)
    B, k, V = 500, 3, 50
    t = rng.normal(0, 2, (B, k + 1, V)).astype(np.float32)
    d = np.full((B, k, V), np.nan, np.float32)
    tok = np.full((B, k), -1, np.int32)
    kl = np.zeros(B, np.int32)
    u = philox_uniforms(B * (k + 1), seed=8).reshape(B, k + 1)
    res = oracle.verify(t, d, tok, kl, u, 1.3)
    assert (res["out_len"] == 1).all()
    for b in range(B):
        p = softmax(t[b, 0].astype(np.float64) / 1.3)
        c = np.cumsum(p)
        want = int(np.searchsorted(c, float(u[b, k]) * c[-1], side="right"))
        if res["sample_tie"][b] > 1e-12:
            assert res["out_tokens"][b, 0] == want


def test_no_draft_enumeration_is_exact():
    V = 4
    rng = np.random.default_rng(4)
    row = rng.normal(0, 1.5, V).astype(np.float32)
    p = softmax(row.astype(np.float64))
    cuts = np.cumsum(p)
    pieces = list(zip(np.concatenate([[0.0], cuts[:-1]]), cuts))
    mass = np.zeros(V)
    for lo, hi in pieces:
        u = np.array([[0, 0, np.float32(0.5 * (lo + hi))]], np.float32)
        res = oracle.verify(row.reshape(1, 1, V).repeat(3, 1), np.full((1, 2, V), np.nan, np.float32),
                            np.full((1, 2), -1, np.int32), np.zeros(1, np.int32), u, 1.0)
        mass[res["out_tokens"][0, 0]] += hi - lo
    np.testing.assert_allclose(mass, p, atol=1e-15)


# --- statistical closed forms ------------------------------------------------

def test_acceptance_rate_and_token_law_statistically():
    """Independent rows: P(accept draft 0) = sum min(p0, q0) = 1 - TV(p0, q0),
    E[a] = sum_j prod_{i<j} alpha_i, and the emitted token at positions 0
    and 1 follows p_0 and p_1 (chi-square)."""
    rng = np.random.default_rng(13)
    B, k, V, T = 200_000, 3, 8, 1.0
    base_t = rng.normal(0, 1.0, (k + 1, V)).astype(np.float32)
    base_d = (base_t[:k] + rng.normal(0, 0.8, (k, V))).astype(np.float32)
    t = np.broadcast_to(base_t, (B, k + 1, V)).copy()
    d = np.broadcast_to(base_d, (B, k, V)).copy()
    g = torch.Generator().manual_seed(3)
    tok = gumbel_argmax_tokens(torch.from_numpy(d.reshape(B * k, V)), T, g, chunk=1 << 16)
    tok = tok.numpy().reshape(B, k)
    kl = np.full(B, k, np.int32)
    u = philox_uniforms(B * (k + 1), seed=12).reshape(B, k + 1)
    res = oracle.verify(t, d, tok, kl, u, T)
    p = softmax(base_t.astype(np.float64) / T, axis=1)
    q = softmax(base_d.astype(np.float64) / T, axis=1)
    alpha = np.minimum(p[:k], q).sum(axis=1)
    assert np.allclose(alpha, 1 - 0.5 * np.abs(p[:k] - q).sum(axis=1))
    a = res["out_len"] - 1
    acc0 = (a >= 1).mean()
    assert abs(acc0 - alpha[0]) < 5 * np.sqrt(alpha[0] * (1 - alpha[0]) / B)
    ea = sum(np.prod(alpha[:j]) for j in range(1, k + 1))
    assert abs(a.mean() - ea) < 5 * a.std() / np.sqrt(B)
    for pos in (0, 1):
        sel = res["out_len"] > pos
        counts = np.bincount(res["out_tokens"][sel, pos], minlength=V)
        _, pval = stats.chisquare(counts, p[pos] * sel.sum())
        assert pval > 1e-4, (pos, pval)


# --- edge conventions ---------------------------------------------------------

def test_forbidden_draft_token_rejected_even_at_u_zero():
    """p(x) = 0 (target logit -inf) gives alpha = 0; u = 0 is not < 0."""
    V = 6
    t = np.zeros((1, 2, V), np.float32)
    t[0, 0, 2] = -np.inf
    d = np.zeros((1, 1, V), np.float32)
    res = oracle.verify(t, d, np.array([[2]], np.int32), np.array([1], np.int32),
                        np.zeros((1, 2), np.float32), 1.0)
    assert res["alpha"][0, 0] == 0.0 and res["out_len"][0] == 1
    assert res["out_tokens"][0, 0] != 2


def test_zero_draft_probability_accepts():
    """q(x) = 0 with p(x) > 0 gives r = +inf: always accepted."""
    V = 6
    t = np.zeros((1, 2, V), np.float32)
    d = np.zeros((1, 1, V), np.float32)
    d[0, 0, 4] = -np.inf
    u = np.array([[np.float32(1 - 2 ** -24), 0.5]], np.float32)
    res = oracle.verify(t, d, np.array([[4]], np.int32), np.array([1], np.int32), u, 1.0)
    assert res["alpha"][0, 0] == 1.0 and res["out_len"][0] == 2


def test_sampling_never_picks_zero_weight_token():
    """s = 0 must pick the first token with positive residual weight."""
    V = 5
    t = np.log(np.array([[[0.1, 0.4, 0.2, 0.2, 0.1], [0.2] * 5]], np.float32))
    d = np.log(np.array([[[0.5, 0.1, 0.2, 0.1, 0.1]]], np.float32))
    # draft token 0: p/q = 0.2 -> reject for u = 0.9; residual is zero on 0
    u = np.array([[0.9, 0.0]], np.float32)
    res = oracle.verify(t, d, np.array([[0]], np.int32), np.array([1], np.int32), u, 1.0)
    assert res["out_len"][0] == 1 and res["out_tokens"][0, 0] == 1


def test_status_codes_and_padding_not_read():
    rng = np.random.default_rng(1)
    B, k, V = 6, 2, 32
    t = rng.normal(size=(B, k + 1, V)).astype(np.float32)
    d = rng.normal(size=(B, k, V)).astype(np.float32)
    tok = rng.integers(0, V, (B, k)).astype(np.int32)
    kl = np.array([2, 3, 2, 2, 1, 0], np.int32)
    tok[2, 1] = V                    # bad token
    t[3, 1, 5] = np.nan              # NaN in a needed row
    t[4, 2] = np.nan                 # NaN only in padding (k_b = 1): fine
    d[4, 1] = np.nan
    t[5, 1:] = np.inf                # padding of a k_b = 0 sequence: fine
    u = philox_uniforms(B * (k + 1), seed=1).reshape(B, k + 1)
    res = oracle.verify(t, d, tok, kl, u, 1.0)
    assert list(res["status"] & 0xFF) == [0, oracle.STATUS_BAD_DRAFT_LEN, oracle.STATUS_BAD_TOKEN,
                                          oracle.STATUS_NONFINITE, 0, 0]
    for b in (1, 2, 3):
        assert res["out_len"][b] == 0 and (res["out_tokens"][b] == -1).all()
    t2 = t.copy()
    t2[0, 0] = -np.inf               # all -inf needed row
    assert oracle.verify(t2, d, tok, kl, u, 1.0)["status"][0] == oracle.STATUS_NONFINITE
    t3 = t.copy()
    t3[0, 1, 0] = np.inf
    assert oracle.verify(t3, d, tok, kl, u, 1.0)["status"][0] == oracle.STATUS_NONFINITE
    t4 = t.copy()
    t4[0, 1, :5] = -np.inf           # masked tokens are allowed
    assert oracle.verify(t4, d, tok, kl, u, 1.0)["status"][0] == 0


def test_bf16_and_f32_inputs_agree_on_identical_values():
    rng = np.random.default_rng(3)
    B, k, V = 16, 3, 200
    t = torch.from_numpy(rng.normal(0, 3, (B, k + 1, V)).astype(np.float32)).to(torch.bfloat16)
    d = (t[:, :k].float() + torch.from_numpy(rng.normal(0, 1, (B, k, V)).astype(np.float32))).to(torch.bfloat16)
    tok = torch.from_numpy(rng.integers(0, V, (B, k)).astype(np.int32))
    kl = torch.full((B,), k, dtype=torch.int32)
    u = philox_uniforms(B * (k + 1), seed=2).reshape(B, k + 1)
    r16 = oracle.verify(t, d, tok, kl, u, 0.8)
    r32 = oracle.verify(t.float(), d.float(), tok, kl, u, 0.8)
    np.testing.assert_array_equal(r16["out_tokens"], r32["out_tokens"])
    np.testing.assert_array_equal(r16["lse_t"], r32["lse_t"])
