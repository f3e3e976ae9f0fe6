"""The tree input generator keeps the layout the tree entry point documents:
parents before children, tokens in the vocabulary, the rows the walk may
read finite, and every row it must never read (draft rows of nodes without
children, rows past a sequence's last node) NaN."""
import numpy as np
import torch

from workloads import get_tree_workload, make_tree_inputs, tree_parents


def test_full_tree_parents():
    assert tree_parents(()) == [-1]
    assert tree_parents((3,)) == [-1, 0, 0, 0]
    assert tree_parents((2, 2)) == [-1, 0, 0, 1, 1, 2, 2]
    par = tree_parents((4, 2, 3))
    assert len(par) == 1 + 4 + 8 + 24
    assert all(0 <= par[j] < j for j in range(1, len(par)))


def test_generated_trees_follow_the_layout():
    for name, over in (("tree", dict(B=5, V=700, dtype="f32")), ("tree_wide", dict(B=9, V=300, dtype="bf16"))):
        w = get_tree_workload(name, **over)
        inp = make_tree_inputs(w)
        B, M, V = inp["target"].shape
        par = inp["parents"].numpy()
        tok = inp["tokens"].numpy()
        nn = inp["n_nodes"].numpy()
        t = inp["target"].float().numpy()
        d = inp["draft"].float().numpy()
        u = inp["uniforms"].numpy()
        assert M == w.M and V == w.V
        assert ((u >= 0) & (u < 1)).all()
        for b in range(B):
            n = nn[b]
            assert 1 <= n <= M
            assert all(0 <= par[b, j] < j for j in range(1, M))
            assert ((tok[b, 1:] >= 0) & (tok[b, 1:] < V)).all()
            has_kids = {int(par[b, j]) for j in range(1, n)}
            for j in range(M):
                if j < n:
                    assert np.isfinite(t[b, j]).all()
                else:
                    assert np.isnan(t[b, j]).all()
                if j < n and j in has_kids:
                    assert np.isfinite(d[b, j]).all()
                else:
                    assert np.isnan(d[b, j]).all()
        if not w.ragged:
            assert (nn == M).all()


def test_children_are_draws_from_the_parent_draft():
    # every child's token has positive probability under its parent's draft
    # row, and the most likely tokens come up most often
    w = get_tree_workload("tree", B=40, V=64, dtype="f32", draft_sigma=0.5)
    inp = make_tree_inputs(w)
    d = inp["draft"].numpy()
    tok = inp["tokens"].numpy()
    par = inp["parents"].numpy()
    ranks = []
    for b in range(40):
        for j in range(1, w.M):
            row = d[b, par[b, j]].astype(np.float64)
            assert np.isfinite(row).all()
            ranks.append(int((row > row[tok[b, j]]).sum()))
    assert np.median(ranks) < 8          # draws concentrate on the top of q
