"""The oracle's per-sequence diagnostics restated with numpy and scipy.

The parity tests decide from these diagnostics which sequences are near-ties
(excluded from the exact comparison) and which tokens a draw at a near-tie
may validly give, so a slip in them would silently hide mismatches.  This
module recomputes them from their definitions with library routines
(``scipy.special.softmax``, ``numpy.cumsum``, ``numpy.searchsorted``), with
none of the oracle's code:

  accept_tie   min |u_i - alpha_i| over the acceptance tests that ran, i.e.
               up to and including the first rejection (1 if none ran);
  resid_mass   S, the mass of the weights of the final draw: max(0, p_a - q_a)
               after a rejection at a, p_{k_b} when every draft was accepted
               (p_a itself if the residual is exactly zero);
  sample_tie   the distance of the sampling uniform s to the two ends of the
               drawn token's interval [C(y-1)/S, C(y)/S] of the normalised CDF;
  sample_lo/hi the smallest and largest token with positive weight whose
               interval comes within `band` of s (a draw whose CDF is off by
               less than `band` can give any token between them).

The rule itself (accept iff u_i < min(1, p_i(x_i)/q_i(x_i)), first
rejection, inverse CDF in ascending token id) is the standard speculative
sampling rule read into "Accelerating RL Post-Training Rollouts via
System-Integrated Speculative Decoding", §2 core mechanism.
"""
from __future__ import annotations

import numpy as np
from scipy.special import softmax


def as_f64(x):
    """float32 array or uint16 bf16 bits (or a torch tensor) -> float64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


def draw_diagnostics(w, s, band):
    """(y, S, sample_tie, lo, hi) of the inverse-CDF draw over weights w."""
    C = np.cumsum(w)
    S = C[-1]
    y = int(np.searchsorted(C, s * S, side="right"))
    while y < len(w) and w[y] == 0.0:       # a zero-weight token is never the answer
        y += 1
    if y >= len(w):
        y = int(np.nonzero(w > 0)[0][-1])
    c_hi = C[y]
    c_lo = C[y - 1] if y > 0 else 0.0
    tie = min(abs(s - c_lo / S), abs(s - c_hi / S))
    C_prev = np.concatenate([[0.0], C[:-1]])
    ok = (w > 0) & (C >= (s - band) * S) & (C_prev <= (s + band) * S)
    idx = np.nonzero(ok)[0]
    return y, S, tie, int(idx[0]), int(idx[-1])


def linear(target, draft, tokens, draft_len, uniforms, T, band):
    """Outputs and diagnostics of every sequence of a batch (T > 0)."""
    t = as_f64(target)
    d = as_f64(draft)
    tok = np.asarray(tokens)
    kl = np.asarray(draft_len)
    u = np.asarray(uniforms, dtype=np.float64)
    B, k1, V = t.shape
    k = k1 - 1
    out = {name: np.full(B, np.nan) for name in ("accept_tie", "resid_mass", "sample_tie")}
    out["alpha"] = np.full((B, max(k, 1)), np.nan)
    out["out_len"] = np.zeros(B, np.int64)
    out["y"] = np.full(B, -1)
    out["sample_lo"] = np.full(B, -1)
    out["sample_hi"] = np.full(B, -1)
    for b in range(B):
        kb = int(kl[b])
        p = [softmax(t[b, i] / T) for i in range(kb + 1)]
        q = [softmax(d[b, i] / T) for i in range(kb)]
        a, atie = kb, 1.0
        for i in range(kb):
            x = int(tok[b, i])
            r = np.inf if (q[i][x] == 0 and p[i][x] > 0) else (0.0 if q[i][x] == 0 else p[i][x] / q[i][x])
            al = min(1.0, r)
            out["alpha"][b, i] = al
            if a == kb:
                atie = min(atie, abs(u[b, i] - al))
                if not u[b, i] < al:
                    a = i
        w = np.maximum(p[a] - q[a], 0.0) if a < kb else p[kb].copy()
        if w.sum() == 0.0:
            w = p[a].copy()
        y, S, stie, lo, hi = draw_diagnostics(w, u[b, k], band)
        out["accept_tie"][b] = atie
        out["resid_mass"][b] = S
        out["sample_tie"][b] = stie
        out["sample_lo"][b], out["sample_hi"][b] = lo, hi
        out["out_len"][b] = a + 1
        out["y"][b] = y
    out["alpha"] = out["alpha"][:, :k]
    return out


def root_fan(target_row, draft_row, child_tokens, child_uniforms, s, T, band):
    """Tree verification at a root whose children are all leaves: the
    children are tested in order against the residual r (r = p at first,
    r <- max(0, r - q)/S after each rejection); an accepted child ends the
    walk at that child, whose bonus draw needs its own row, so only the
    all-rejected outcome is returned in full.  Returns (accepted child index
    or -1, accept_tie, alphas, and for -1: y, S, sample_tie, lo, hi)."""
    p = softmax(as_f64(target_row) / T)
    q = softmax(as_f64(draft_row) / T)
    r = p.copy()
    atie, alphas = 1.0, []
    S = 1.0
    w = r
    for j, (x, uc) in enumerate(zip(child_tokens, child_uniforms)):
        ratio = np.inf if (q[x] == 0 and r[x] > 0) else (0.0 if q[x] == 0 else r[x] / q[x])
        al = min(1.0, ratio)
        alphas.append(al)
        atie = min(atie, abs(uc - al))
        if uc < al:
            return j, atie, alphas, None
        w = np.maximum(r - q, 0.0)
        if w.sum() == 0.0:
            w = r.copy()
        S = w.sum()
        r = w / S
    return -1, atie, alphas, draw_diagnostics(w, s, band)
