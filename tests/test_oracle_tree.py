"""Pins of the oracle's tree verification (``oracle_tree_verify``).

- Exhaustive enumeration: over every draft assignment of a tiny tree (each
  child an independent draw from the drafter at its parent) and every piece
  of the uniforms, the emitted tokens completed under the target table have
  exactly the target's joint law (the exactness the pages claim for
  rejection-sampling verification, here for branching drafts).
- A chain (one child per node) gives exactly what the linear oracle gives.
- Special cases: identical draft and target rows accept the first child,
  a root with no children samples categorically from p (numpy's search of
  the CDF), greedy follows the first argmax, a masked draft token (q = 0)
  with p > 0 is accepted, the structure and the rows the walk reads are
  checked.
Planted mistakes must be caught (bottom).
"""
import os

import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from tests import tree_cases as tc

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")


def pin_enumeration_is_lossless(lib):
    for shape in ("fan2", "fan3", "mixed", "binary2"):
        for T, seed in ((1.0, 1), (0.6, 2)):
            b, P = tc.build(shape, V=3, T=T, seed=seed, lib=lib)
            L = b["depth"] + 1
            assert abs(b["weight"].sum() - 1.0) < 1e-12
            got = tc.joint_from_outputs(b["out_tokens"], b["out_len"], b["weight"], P, 3, L)
            assert np.abs(got - tc.target_joint(P, 3, L)).max() < 1e-12, (shape, T)


def random_chain(rng, B, k, V, dtype=np.float32):
    t = rng.normal(0, 2.0, (B, k + 1, V)).astype(np.float32)
    d = (t[:, :k] + rng.normal(0, 0.8, (B, k, V))).astype(np.float32)
    tok = rng.integers(0, V, (B, k)).astype(np.int32)
    # make some drafts likely: the draft argmax
    m = rng.random((B, k)) < 0.6
    tok[m] = d.argmax(axis=2)[m]
    kb = rng.integers(0, k + 1, B).astype(np.int32)
    u = rng.random((B, k + 1)).astype(np.float32)
    return t, d, tok, kb, u


def chain_as_tree(t, d, tok, kb, u):
    B, k1, V = t.shape
    k = k1 - 1
    M = k + 1
    par = np.tile(np.arange(-1, M - 1, dtype=np.int32), (B, 1))
    tt = np.zeros((B, M), np.int32)
    tt[:, 1:] = tok
    dd = np.concatenate([d, np.zeros((B, 1, V), d.dtype)], axis=1)
    uu = np.zeros((B, M), np.float32)
    uu[:, 0] = u[:, k]
    uu[:, 1:] = u[:, :k]
    return t, dd, par, tt, (kb + 1).astype(np.int32), uu


def pin_chain_equals_linear(lib):
    rng = np.random.default_rng(3)
    for k, V, T, bf16 in ((3, 257, 1.0, False), (5, 64, 0.7, True), (2, 1000, 0.0, False), (4, 33, 1.3, True)):
        t, d, tok, kb, u = random_chain(rng, 40, k, V)
        if bf16:
            t = torch.from_numpy(t).to(torch.bfloat16)
            d = torch.from_numpy(d).to(torch.bfloat16)
        lin = oracle.verify(t, d, tok, kb, u, T, lib=lib)
        tt = t if not bf16 else t.float().numpy()
        dd_ = d if not bf16 else d.float().numpy()
        tree = oracle.tree_verify(*chain_as_tree(np.asarray(tt), np.asarray(dd_), tok, kb, u), T, lib=lib)
        np.testing.assert_array_equal(tree["out_len"], lin["out_len"])
        np.testing.assert_array_equal(tree["out_tokens"], lin["out_tokens"])
        np.testing.assert_array_equal(tree["status"], lin["status"])
        if T > 0:
            np.testing.assert_array_equal(tree["accept_tie"], lin["accept_tie"])
            np.testing.assert_array_equal(tree["sample_tie"], lin["sample_tie"])
        for b in range(40):
            n = tree["out_len"][b]
            assert list(tree["out_nodes"][b, :n - 1]) == list(range(1, n))


def fan(rng, V, t_children, T_same=False):
    M = t_children + 1
    t = rng.normal(0, 2.0, (1, M, V)).astype(np.float32)
    d = t.copy() if T_same else rng.normal(0, 2.0, (1, M, V)).astype(np.float32)
    par = np.array([[-1] + [0] * t_children], np.int32)
    tok = np.array([[0] + list(rng.integers(0, V, t_children))], np.int32)
    return t, d, par, tok, np.array([M], np.int32)


def pin_identical_rows_accept_the_first_child(lib):
    rng = np.random.default_rng(4)
    # binary tree of 7 nodes, q = p at every node: alpha = 1 at each first child
    par = np.array([[-1, 0, 0, 1, 1, 2, 2]], np.int32)
    t = rng.normal(0, 2.0, (1, 7, 50)).astype(np.float32)
    tok = np.array([[0, 5, 6, 7, 8, 9, 10]], np.int32)
    for _ in range(10):
        u = rng.random((1, 7)).astype(np.float32)
        r = oracle.tree_verify(t, t.copy(), par, tok, np.array([7], np.int32), u, 1.0, lib=lib)
        assert list(r["out_nodes"][0, :2]) == [1, 3] and r["out_len"][0] == 3
        assert r["alpha"][0, 1] == 1.0 and r["alpha"][0, 3] == 1.0


def pin_root_only_is_categorical_sampling(lib):
    rng = np.random.default_rng(5)
    V = 300
    for T in (1.0, 0.5, 2.0):
        t = rng.normal(0, 2.0, (64, 1, V)).astype(np.float32)
        u = rng.random((64, 1)).astype(np.float32)
        r = oracle.tree_verify(t, np.zeros_like(t), np.full((64, 1), -1, np.int32), np.zeros((64, 1), np.int32),
                               np.ones(64, np.int32), u, T, lib=lib)
        for b in range(64):
            c = np.cumsum(softmax(t[b, 0].astype(np.float64) / T))
            y = int(np.searchsorted(c / c[-1], float(u[b, 0]), side="right"))
            if r["sample_tie"][b] > 1e-9:
                assert r["out_tokens"][b, 0] == y and r["out_len"][b] == 1


def pin_greedy_follows_the_argmax(lib):
    rng = np.random.default_rng(6)
    V = 40
    par = np.array([[-1, 0, 0, 0, 1, 1, 3]], np.int32)
    for trial in range(30):
        t = rng.normal(0, 2.0, (1, 7, V)).astype(np.float32)
        tok = rng.integers(0, V, (1, 7)).astype(np.int32)
        # plant the argmax among the candidates now and then
        for node, kids in ((0, [1, 2, 3]), (1, [4, 5]), (3, [6])):
            if rng.random() < 0.7:
                tok[0, kids[int(rng.integers(len(kids)))]] = int(np.argmax(t[0, node]))
        r = oracle.tree_verify(t, np.zeros_like(t), par, tok, np.array([7], np.int32),
                               rng.random((1, 7)).astype(np.float32), 0.0, lib=lib)
        cur, path = 0, []
        while True:
            kids = [c for c in range(7) if par[0, c] == cur]
            hit = [c for c in kids if tok[0, c] == int(np.argmax(t[0, cur]))]
            if not hit:
                break
            cur = hit[0]
            path.append(cur)
        assert list(r["out_nodes"][0, :len(path)]) == path
        assert r["out_tokens"][0, len(path)] == int(np.argmax(t[0, cur])) and r["out_len"][0] == len(path) + 1


def pin_masked_draft_token_is_accepted(lib):
    rng = np.random.default_rng(7)
    t, d, par, tok, n = fan(rng, 20, 2)
    d[0, 0, tok[0, 1]] = -np.inf                       # q(x) = 0 < p(x): r = +inf
    u = np.array([[0.5, 0.999, 0.5]], np.float32)
    r = oracle.tree_verify(t, d, par, tok, n, u, 1.0, lib=lib)
    assert r["alpha"][0, 1] == 1.0 and list(r["out_nodes"][0, :1]) == [1]


def pin_structure_and_rows_are_checked(lib):
    rng = np.random.default_rng(8)
    V = 16
    t = rng.normal(0, 1.0, (6, 4, V)).astype(np.float32)
    d = rng.normal(0, 1.0, (6, 4, V)).astype(np.float32)
    par = np.tile(np.array([-1, 0, 0, 1], np.int32), (6, 1))
    tok = np.tile(np.array([0, 1, 2, 3], np.int32), (6, 1))
    n = np.full(6, 4, np.int32)
    par[0, 2] = 2                   # its own parent
    par[1, 3] = -1                  # no parent
    n[2] = 5                        # more nodes than the rows
    tok[3, 2] = V                   # token outside the vocabulary
    t[4, 0, 3] = np.nan             # the root row is always read
    d[5, 3, :] = np.nan             # node 3 has no children: its draft row is never read
    t[5, 2, :] = -np.inf            # node 2 is visited only if node 1 is rejected
    u = np.full((6, 4), 0.0, np.float32)     # u = 0 accepts every child with alpha > 0
    r = oracle.tree_verify(t, d, par, tok, n, u, 1.0, lib=lib)
    assert list(r["status"][:5]) == [2, 2, 2, 3, 4], r["status"]
    assert (r["out_len"][:5] == 0).all() and (r["out_tokens"][:5] == -1).all()
    assert r["status"][5] == 0 and r["out_len"][5] == 3


def pin_near_tie_diagnostics_of_a_rejected_fan(lib):
    """Root with three leaf children, each drafted where q exceeds p most and
    tested at u ~ 1 (all rejected): alpha, accept_tie, the final residual
    mass, sample_tie and the draw window against numpy's recursion."""
    from tests import diag_reference as ref_np
    rng = np.random.default_rng(44)
    V, M = 300, 4
    for _ in range(6):
        t = rng.normal(0, 2.0, (1, M, V)).astype(np.float32)
        d = (t + rng.normal(0, 2.0, (1, M, V))).astype(np.float32)
        fav = np.argsort(d[0, 0].astype(np.float64) - t[0, 0])[::-1][:3]
        par = np.array([[-1, 0, 0, 0]], np.int32)
        tok = np.array([[0] + list(fav)], np.int32)
        u = np.array([[rng.random(), 0.999999, 0.999999, 0.999999]], np.float32)
        for band in (1e-5, 0.03):
            r = oracle.tree_verify(t, d, par, tok, np.array([M], np.int32), u, 1.0, lib=lib, tie_band=band)
            j, atie, alphas, draw = ref_np.root_fan(t[0, 0], d[0, 0], tok[0, 1:], u[0, 1:], float(u[0, 0]), 1.0,
                                                    band)
            assert abs(r["accept_tie"][0] - atie) < 1e-12
            if j >= 0:
                continue
            y, S, stie, lo, hi = draw
            assert r["out_tokens"][0, 0] == y
            assert abs(r["resid_mass"][0] - S) <= 1e-12 * S
            assert abs(r["sample_tie"][0] - stie) < 1e-12
            assert (r["sample_lo"][0], r["sample_hi"][0]) == (lo, hi)


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__[4:] for p in PINS])
def test_tree_pin(pin):
    pin(oracle.load())


# --- planted mistakes --------------------------------------------------------------

TREE_MUTANTS = {
    "residual_not_carried": ("r[xx] = w[xx] / S;", "r[xx] = r[xx] + 0.0 * w[xx] / S;"),
    "residual_without_draft": ("const double v = r[xx] - q[xx];", "const double v = r[xx];"),
    "sampling_uniform_of_a_test": ("y = inverse_cdf(w, V, S, (double)u[0], &stie);",
                                   "y = inverse_cdf(w, V, S, (double)u[1 < M ? 1 : 0], &stie);"),
    "greedy_inverted": ("const int ok = (tok[c] == am);", "const int ok = (tok[c] != am);"),
    "parent_may_be_itself": ("if (par[j] < 0 || par[j] >= j)", "if (par[j] < 0 || par[j] > j)"),
    "masked_draft_rejected": ("(q[x] == 0.0) ? (r[x] > 0.0 ? INFINITY : 0.0)", "(q[x] == 0.0) ? 0.0"),
    "accepted_parent_token_emitted": ("                on[len] = next;\n                ot[len++] = tok[next];",
                                      "                on[len] = next;\n                ot[len++] = tok[cur];"),
    "accept_tie_of_rejections_only": ("                if (d < atie) atie = d;\n                if ((double)u[c] < al) {",
                                      "                if (d < atie && !((double)u[c] < al)) atie = d;\n"
                                      "                if ((double)u[c] < al) {"),
    "resid_mass_of_the_normalised_residual": (
        "                    final_w[(size_t)b * V + x] = w[x] / S;\n            if (resid_mass) resid_mass[b] = S;",
        "                    final_w[(size_t)b * V + x] = w[x] / S;\n            if (resid_mass) resid_mass[b] = 1.0;"),
    "bonus_from_the_draft": ("                    w[x] = r[x];\n                    S += w[x];",
                             "                    w[x] = prob_of(zd[x], 0.0, 0.0, 1.0);\n                    S += w[x];"),
}


def _tree_pins_pass(lib):
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            return False
    return True


def test_unmutated_tree_oracle_passes():
    assert _tree_pins_pass(oracle.load())


@pytest.mark.parametrize("name", sorted(TREE_MUTANTS))
def test_tree_mutant_is_caught(name, tmp_path):
    old, new = TREE_MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/present ({src.count(old)})"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(old, new))
    so = oracle.build(force=True, src=str(mpath), out=str(tmp_path / "libmutant.so"))
    assert not _tree_pins_pass(oracle.load(so)), f"mutant {name} survived"
