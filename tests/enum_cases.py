"""Exhaustive enumeration of speculative-sampling verification on a tiny,
prefix-conditioned "model".

Every random input of the verifier (the drafted tokens x_i ~ q_i(.|prefix),
the accept uniforms u_i and the sampling uniform s) is enumerated exactly:
the drafts over all V^k_b outcomes, each uniform over the pieces of [0,1)
on which the verifier's decision cannot change.  The decision is evaluated
once per piece, at its midpoint, and weighted by the piece's length times
the drafts' probability.  Completing the emitted prefix autoregressively
under the target table must then give exactly the target's own joint
distribution over the k+1 tokens: the exactness the pages claim for
rejection-sampling verification ("Accelerating RL Post-Training Rollouts via
System-Integrated Speculative Decoding", §2 core mechanism; "Online Draft
Co-Training ...", the analogy: the output distribution is the same as the
proof-reader writing alone).

The piece boundaries are computed here with scipy's softmax, independently
of the verifier under test; the decisions come from the verifier.  A superset
of the true boundaries is used for the sampling uniform (the CDF points of
every weight vector the verifier might sample from), so each piece lies
inside one decision region.
"""
from __future__ import annotations

import itertools

import numpy as np
from scipy.special import softmax

from workloads import make_tables


def _pieces(points):
    pts = sorted(set(float(p) for p in points if 0.0 <= p <= 1.0) | {0.0, 1.0})
    return [(a, b) for a, b in zip(pts[:-1], pts[1:]) if b > a]


def _mid32(a, b):
    m = np.float32(0.5 * (a + b))
    if not (a < float(m) < b):
        raise AssertionError(f"piece [{a}, {b}) too narrow for a float32 midpoint")
    return m


def build(V=4, k=2, kb=2, T=1.0, seed=0, scale=1.5):
    """Return the enumeration batch and the target table.

    Arrays (N cases): target [N,k+1,V] f32, draft [N,k,V] f32, tokens [N,k]
    i32, draft_len [N] i32, uniforms [N,k+1] f32, weight [N] f64, and
    ``margin`` [N]: the distance of each midpoint uniform to its piece's ends
    (how far the case is from any decision boundary).
    """
    rng = np.random.default_rng(seed)
    tabT = {p: r.astype(np.float32) for p, r in make_tables(rng, V, k + 1, scale).items()}
    tabD = {p: r.astype(np.float32) for p, r in make_tables(rng, V, max(k, 1), scale).items()}

    def P(pre):
        return softmax(tabT[tuple(pre)].astype(np.float64) / T)

    def Q(pre):
        return softmax(tabD[tuple(pre)].astype(np.float64) / T)

    tgt, drf, tok, kl, uni, wts, mrg = [], [], [], [], [], [], []
    nan_row = np.full(V, np.nan, np.float32)
    for xs in itertools.product(range(V), repeat=kb):
        qprob = 1.0
        for j in range(kb):
            qprob *= Q(xs[:j])[xs[j]]
        if qprob == 0.0:
            continue
        alphas = [min(1.0, P(xs[:j])[xs[j]] / Q(xs[:j])[xs[j]]) for j in range(kb)]
        u_pieces = [_pieces([a]) for a in alphas]
        s_points = []
        for a in range(kb + 1):
            w = np.maximum(0.0, P(xs[:a]) - Q(xs[:a])) if a < kb else P(xs[:kb])
            if w.sum() > 0:
                s_points.extend(np.cumsum(w) / w.sum())
        s_pieces = _pieces(s_points)
        t_rows = [tabT[xs[:j]] if j <= kb else nan_row for j in range(k + 1)]
        d_rows = [tabD[xs[:j]] if j < kb else nan_row for j in range(k)]
        for combo in itertools.product(*u_pieces, s_pieces):
            u = np.zeros(k + 1, np.float32)
            weight = qprob
            margin = 1.0
            for j, (lo, hi) in enumerate(combo[:-1]):
                u[j] = _mid32(lo, hi)
                weight *= hi - lo
                margin = min(margin, float(u[j]) - lo, hi - float(u[j]))
            lo, hi = combo[-1]
            u[k] = _mid32(lo, hi)
            weight *= hi - lo
            margin = min(margin, float(u[k]) - lo, hi - float(u[k]))
            tgt.append(np.stack(t_rows))
            drf.append(np.stack(d_rows) if k else np.zeros((0, V), np.float32))
            tok.append(list(xs) + [-1] * (k - kb))
            kl.append(kb)
            uni.append(u)
            wts.append(weight)
            mrg.append(margin)
    batch = {
        "target": np.ascontiguousarray(np.stack(tgt), dtype=np.float32),
        "draft": np.ascontiguousarray(np.stack(drf), dtype=np.float32),
        "tokens": np.asarray(tok, np.int32).reshape(len(tok), k),
        "draft_len": np.asarray(kl, np.int32),
        "uniforms": np.stack(uni).astype(np.float32),
        "weight": np.asarray(wts),
        "margin": np.asarray(mrg),
        "T": T, "k": k, "V": V,
    }
    return batch, P


def joint_from_outputs(out_tokens, out_len, weight, P, V, k):
    """Complete each emitted prefix under the target table and accumulate the
    weighted joint over all (k+1)-token strings."""
    joint = np.zeros((V,) * (k + 1))
    for row, n, w in zip(out_tokens, out_len, weight):
        emitted = tuple(int(t) for t in row[:n])
        for tail in itertools.product(range(V), repeat=k + 1 - n):
            y = emitted + tail
            pr = w
            for j in range(n, k + 1):
                pr *= P(y[:j])[y[j]]
            joint[y] += pr
    return joint


def target_joint(P, V, k):
    joint = np.zeros((V,) * (k + 1))
    for y in itertools.product(range(V), repeat=k + 1):
        pr = 1.0
        for j in range(k + 1):
            pr *= P(y[:j])[y[j]]
        joint[y] = pr
    return joint
