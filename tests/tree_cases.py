"""Exhaustive enumeration of tree verification on a tiny prefix-conditioned
"model" (the tree form of ``enum_cases``).

The draft tree has a fixed shape; every child's token is an independent draw
from the drafter's distribution at its parent (the reading under which the
multi-candidate rule is exact), so all V^(nodes-1) token assignments are
enumerated with their probability.  Each test uniform is split at the
acceptance probability the verifier used for that child, and the sampling
uniform at the CDF points of the weights the verifier drew from (both read
from the oracle's diagnostics: a wrong rule gives a wrong output law whatever
the split points).  The decision is evaluated once per piece, at its
midpoint, and weighted by the piece lengths times the drafts' probability.
Completing each emitted prefix under the target table must reproduce the
target's own joint law over depth + 1 tokens.
"""
from __future__ import annotations

import itertools

import numpy as np
from scipy.special import softmax

import oracle
from workloads import make_tables

SHAPES = {
    "fan2": [-1, 0, 0],                 # one node, two candidates
    "fan3": [-1, 0, 0, 0],              # three candidates
    "chain2": [-1, 0, 1],               # the linear case, k = 2
    "mixed": [-1, 0, 1, 0],             # first candidate has a child
    "binary2": [-1, 0, 0, 1, 1, 2],     # two levels, branching 2, 2, 1
}


def depths(parents):
    d = [0] * len(parents)
    for j in range(1, len(parents)):
        d[j] = d[parents[j]] + 1
    return d


def path_of(j, parents, toks):
    out = []
    while j > 0:
        out.append(toks[j])
        j = parents[j]
    return tuple(reversed(out))


def _pieces(points):
    """Pieces of [0, 1) between the points; pieces narrower than 1e-12 come
    only from rounding (a CDF that ends at 1 - 1e-16) and carry no weight."""
    pts = sorted(set(float(p) for p in points if 0.0 <= p <= 1.0) | {0.0, 1.0})
    return [(a, b) for a, b in zip(pts[:-1], pts[1:]) if b - a > 1e-12]


def _mid32(a, b):
    m = np.float32(0.5 * (a + b))
    if not (a < float(m) < b):
        raise AssertionError(f"piece [{a}, {b}) too narrow for a float32 midpoint")
    return m


def build(shape="binary2", V=3, T=1.0, seed=0, scale=1.5, lib=None):
    """Enumeration batch for one tree shape: target, draft [N,M,V] f32,
    parents, tokens [N,M] i32, n_nodes [N], uniforms [N,M] f32, weight,
    margin [N], plus the oracle's outputs for each case and the target table."""
    parents = SHAPES[shape]
    M = len(parents)
    D = max(depths(parents))
    rng = np.random.default_rng(seed)
    tabT = {p: r.astype(np.float32) for p, r in make_tables(rng, V, D + 1, scale).items()}
    tabD = {p: r.astype(np.float32) for p, r in make_tables(rng, V, D + 1, scale).items()}
    internal = {parents[j] for j in range(1, M)}

    def P(pre):
        return softmax(tabT[tuple(pre)].astype(np.float64) / T)

    def Q(pre):
        return softmax(tabD[tuple(pre)].astype(np.float64) / T)

    nan_row = np.full(V, np.nan, np.float32)
    par = np.asarray(parents, np.int32)
    cases = []
    for assign in itertools.product(range(V), repeat=M - 1):
        tk = [-1] + list(assign)
        qprob = 1.0
        for j in range(1, M):
            qprob *= Q(path_of(parents[j], parents, tk))[tk[j]]
        if qprob == 0.0:
            continue
        t_rows = np.stack([tabT[path_of(j, parents, tk)] for j in range(M)])
        d_rows = np.stack([tabD[path_of(j, parents, tk)] if j in internal else nan_row for j in range(M)])
        tok = np.asarray([0] + list(assign), np.int32)

        def run(u):
            return oracle.tree_verify(t_rows[None], d_rows[None], par[None], tok[None], np.array([M], np.int32),
                                      u[None], T, final_w=True, lib=lib)

        def explore(fixed):
            u = np.full(M, 0.5, np.float32)
            for c, (lo, hi) in fixed.items():
                u[c] = _mid32(lo, hi)
            r = run(u)
            tested = [c for c in range(1, M) if not np.isnan(r["alpha"][0, c])]
            unfixed = [c for c in tested if c not in fixed]
            if unfixed:
                c = min(unfixed)
                for piece in _pieces([r["alpha"][0, c]]):
                    explore({**fixed, c: piece})
                return
            weight = qprob
            margin = 1.0
            for c, (lo, hi) in fixed.items():
                weight *= hi - lo
                margin = min(margin, float(u[c]) - lo, hi - float(u[c]))
            for lo, hi in _pieces(np.cumsum(r["final_w"][0])[:-1]):
                uu = u.copy()
                uu[0] = _mid32(lo, hi)
                out = run(uu)
                cases.append({"target": t_rows, "draft": d_rows, "tokens": tok, "uniforms": uu,
                              "weight": weight * (hi - lo),
                              "margin": min(margin, float(uu[0]) - lo, hi - float(uu[0])),
                              "out_tokens": out["out_tokens"][0], "out_len": int(out["out_len"][0]),
                              "out_nodes": out["out_nodes"][0]})

        explore({})
    N = len(cases)
    batch = {
        "target": np.stack([c["target"] for c in cases]),
        "draft": np.stack([c["draft"] for c in cases]),
        "parents": np.tile(par, (N, 1)),
        "tokens": np.stack([c["tokens"] for c in cases]),
        "n_nodes": np.full(N, M, np.int32),
        "uniforms": np.stack([c["uniforms"] for c in cases]),
        "weight": np.asarray([c["weight"] for c in cases]),
        "margin": np.asarray([c["margin"] for c in cases]),
        "out_tokens": np.stack([c["out_tokens"] for c in cases]),
        "out_len": np.asarray([c["out_len"] for c in cases], np.int32),
        "out_nodes": np.stack([c["out_nodes"] for c in cases]),
        "T": T, "V": V, "M": M, "depth": D,
    }
    return batch, P


def joint_from_outputs(out_tokens, out_len, weight, P, V, L):
    """Complete each emitted prefix under the target table to L tokens and
    accumulate the weighted joint."""
    joint = np.zeros((V,) * L)
    for row, n, w in zip(out_tokens, out_len, weight):
        emitted = tuple(int(t) for t in row[:n])
        for tail in itertools.product(range(V), repeat=L - n):
            y = emitted + tail
            pr = w
            for j in range(n, L):
                pr *= P(y[:j])[y[j]]
            joint[y] += pr
    return joint


def target_joint(P, V, L):
    joint = np.zeros((V,) * L)
    for y in itertools.product(range(V), repeat=L):
        pr = 1.0
        for j in range(L):
            pr *= P(y[:j])[y[j]]
        joint[y] = pr
    return joint
