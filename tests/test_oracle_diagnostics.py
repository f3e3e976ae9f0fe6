"""Pins of the oracle's near-tie diagnostics to an independent computation.

The parity tests use ``accept_tie``, ``sample_tie``, ``resid_mass`` and the
draw window ``sample_lo``/``sample_hi`` of the oracle to decide which
sequences are near-ties and which tokens are valid there.  Here each of them
is checked against ``tests/diag_reference.py`` (numpy and scipy, none of the
oracle's code) on batches with many rejections (residual masses well below
1, so a slip between C and C/S units shows), at a narrow and a wide band.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import diag_reference as ref_np
from workloads import philox_uniforms


def batch(seed, B=48, k=4, V=600, dtype="f32", sigma=1.5):
    rng = np.random.default_rng(seed)
    t = rng.normal(0, 2.0, (B, k + 1, V)).astype(np.float32)
    d = (t[:, :k] + rng.normal(0, sigma, (B, k, V))).astype(np.float32)
    kl = rng.integers(0, k + 1, B).astype(np.int32)
    tok = np.empty((B, k), np.int32)
    for b in range(B):
        for i in range(k):
            e = np.exp(d[b, i].astype(np.float64) - d[b, i].max())
            tok[b, i] = rng.choice(V, p=e / e.sum())
    u = philox_uniforms(B * (k + 1), seed=seed).reshape(B, k + 1)
    if dtype == "bf16":
        tb = torch.from_numpy(t).to(torch.bfloat16)
        db = torch.from_numpy(d).to(torch.bfloat16)
        return tb, db, tok, kl, u
    return t, d, tok, kl, u


def check_linear(lib, seed, dtype, T, band):
    t, d, tok, kl, u = batch(seed, dtype=dtype)
    got = oracle.verify(t, d, tok, kl, u, T, lib=lib, tie_band=band)
    want = ref_np.linear(t, d, tok, kl, u, T, band)
    assert (got["status"] == 0).all()
    # a draw that sits on a boundary to 1e-12 could go either way in two
    # summation orders; no such draw occurs in these batches
    assert (want["sample_tie"] > 1e-12).all()
    np.testing.assert_array_equal(got["out_len"], want["out_len"])
    np.testing.assert_array_equal(got["out_tokens"][np.arange(len(kl)), got["out_len"] - 1], want["y"])
    a, b = got["alpha"], want["alpha"]
    m = ~np.isnan(b)
    np.testing.assert_array_equal(np.isnan(a), np.isnan(b))
    np.testing.assert_allclose(a[m], b[m], rtol=1e-12, atol=0)
    np.testing.assert_allclose(got["accept_tie"], want["accept_tie"], rtol=0, atol=1e-12)
    np.testing.assert_allclose(got["resid_mass"], want["resid_mass"], rtol=1e-12, atol=0)
    np.testing.assert_allclose(got["sample_tie"], want["sample_tie"], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(got["sample_lo"], want["sample_lo"])
    np.testing.assert_array_equal(got["sample_hi"], want["sample_hi"])
    # the batches exercise what the checks are for: residual draws (S < 1),
    # later tests that did not run, and windows of more than one token
    assert (want["resid_mass"] < 0.9).sum() >= 10
    assert (want["sample_hi"] > want["sample_lo"]).any() or band < 1e-3
    return got, want


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [1.0, 0.6])
@pytest.mark.parametrize("band", [1e-5, 0.02])
def test_linear_diagnostics_match_numpy(dtype, T, band):
    check_linear(oracle.load(), seed=3 + int(T * 10), dtype=dtype, T=T, band=band)


def test_window_always_holds_the_drawn_token():
    got, _ = check_linear(oracle.load(), seed=11, dtype="f32", T=1.0, band=0.05)
    y = got["out_tokens"][np.arange(len(got["out_len"])), got["out_len"] - 1]
    assert ((got["sample_lo"] <= y) & (y <= got["sample_hi"])).all()


def test_greedy_window_is_the_argmax():
    t, d, tok, kl, u = batch(5, B=16)
    got = oracle.verify(t, d, tok, kl, u, 0.0)
    y = got["out_tokens"][np.arange(16), got["out_len"] - 1]
    np.testing.assert_array_equal(got["sample_lo"], y)
    np.testing.assert_array_equal(got["sample_hi"], y)


def test_accept_tie_counts_only_the_tests_that_ran():
    """Hand-made case: the second test never runs (the first rejects), so its
    |u - alpha| = 0 must not enter accept_tie."""
    p0 = np.array([0.1, 0.6, 0.3])
    q0 = np.array([0.5, 0.25, 0.25])
    t = np.log(np.stack([p0, p0, p0]))[None].astype(np.float32)
    d = np.log(np.stack([q0, q0]))[None].astype(np.float32)
    tok = np.array([[0, 1]], np.int32)
    al0 = np.float32(0.1) / np.float32(0.5)
    u = np.array([[0.9, 1.0 - 1e-7, 0.5]], np.float32)   # test 1 would sit at alpha = 1 exactly
    r = oracle.verify(t, d, tok, np.array([2], np.int32), u, 1.0)
    assert r["out_len"][0] == 1
    assert abs(r["accept_tie"][0] - abs(0.9 - al0)) < 1e-6


def test_tree_chain_diagnostics_equal_the_linear_ones():
    """A chain tree is the linear rule: its diagnostics must equal the
    linear oracle's (which the tests above pin to numpy)."""
    t, d, tok, kl, u = batch(7, B=32, k=3, V=400)
    B, k = 32, 3
    M = k + 1
    par = np.tile(np.arange(-1, M - 1, dtype=np.int32), (B, 1))
    ttok = np.zeros((B, M), np.int32)
    ttok[:, 1:] = tok
    dd = np.concatenate([d, np.full((B, 1, d.shape[2]), np.nan, np.float32)], axis=1)
    uu = np.empty((B, M), np.float32)
    uu[:, 0] = u[:, k]
    uu[:, 1:] = u[:, :k]
    for band in (1e-5, 0.02):
        lin = oracle.verify(t, d, tok, kl, u, 1.0, tie_band=band)
        tr = oracle.tree_verify(t, dd, par, ttok, kl + 1, uu, 1.0, tie_band=band)
        for key in ("accept_tie", "sample_tie", "resid_mass"):
            np.testing.assert_array_equal(tr[key], lin[key])
        for key in ("sample_lo", "sample_hi", "out_len"):
            np.testing.assert_array_equal(tr[key], lin[key])


@pytest.mark.parametrize("n_children", [1, 2, 3])
def test_tree_root_fan_diagnostics_match_numpy(n_children):
    """A root whose children are leaves, every child rejected (u near 1):
    the residual recursion, its mass and the draw window by numpy."""
    rng = np.random.default_rng(40 + n_children)
    V, M = 300, n_children + 1
    hits = 0
    for trial in range(20):
        t = rng.normal(0, 2.0, (1, M, V)).astype(np.float32)
        d = (t + rng.normal(0, 2.0, (1, M, V))).astype(np.float32)
        par = np.array([[-1] + [0] * n_children], np.int32)
        # tokens the drafter favours most over the target: rejected at u ~ 1
        fav = np.argsort(d[0, 0].astype(np.float64) - t[0, 0])[::-1][:n_children]
        tok = np.array([[0] + list(fav)], np.int32)
        u = np.array([[rng.random()] + [0.999999] * n_children], np.float32)
        for band in (1e-5, 0.03):
            r = oracle.tree_verify(t, d, par, tok, np.array([M], np.int32), u, 1.0, tie_band=band)
            j, atie, alphas, draw = ref_np.root_fan(t[0, 0], d[0, 0], tok[0, 1:], u[0, 1:], float(u[0, 0]), 1.0,
                                                    band)
            np.testing.assert_allclose(r["alpha"][0, 1:1 + len(alphas)], alphas, rtol=1e-12)
            assert abs(r["accept_tie"][0] - atie) < 1e-12
            if j >= 0:
                assert r["out_nodes"][0, 0] == j + 1
                continue
            hits += 1
            y, S, stie, lo, hi = draw
            assert r["out_len"][0] == 1 and r["out_tokens"][0, 0] == y
            assert abs(r["resid_mass"][0] - S) <= 1e-12 * S
            assert abs(r["sample_tie"][0] - stie) < 1e-12
            assert (r["sample_lo"][0], r["sample_hi"][0]) == (lo, hi)
    assert hits >= 10
