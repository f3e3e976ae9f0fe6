"""Comparison of the CUDA path with the fp64 oracle on the same inputs.

Tolerances:
  * accepted lengths and emitted token ids: identical, except where the
    oracle reports a near-tie: an executed accept test with
    |u_i - min(1, r_i)| < NEAR_TIE, or a sampling uniform within NEAR_TIE
    (in units of C/S) of a CDF boundary of the drawn token.  Near-ties are
    counted; for an accept-test near-tie the whole sequence is excluded, for
    a sampling near-tie only the drawn token.
  * min(1, p/q): relative 1e-5 (values >= 1e-30).
  * log-sum-exp: 1e-5 * max(1, |lse|) (an fp32 number near 400 has an ulp of
    3e-5, so an absolute 1e-5 is not representable there).
  * the draw's mass S: 1e-5 * S + 1e-6.  For a residual draw S = sum max(0,
    p - q) is a difference of probabilities; each fp32 p(x), q(x) carries a
    relative error of about 3e-7 (ex2.approx plus the rounding of its
    argument), so |dS| <= 3e-7 * (sum p + sum q) = 6e-7 whatever S is, and a
    purely relative bound cannot hold as S -> 0.

``compare_diagnostics`` returns, per quantity, the largest error divided by
its tolerance: every value must be below 1.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

NEAR_TIE = 1e-5
RTOL = 1e-5


def run_gpu(verifier, inp, stream=None):
    out_tokens, out_len = verifier.verify(inp["target"], inp["draft"], inp["tokens"], inp["draft_len"],
                                          inp["uniforms"], inp["T"], stream=stream)
    torch.cuda.synchronize()
    return out_tokens.cpu().numpy(), out_len.cpu().numpy()


def run_oracle(inp, idx=None, nthreads=0):
    """Run the oracle on all sequences or on the subset ``idx``."""
    sel = (lambda t: t) if idx is None else (lambda t: t[idx])
    return oracle.verify(sel(inp["target"]).cpu(), sel(inp["draft"]).cpu(), sel(inp["tokens"]).cpu(),
                         sel(inp["draft_len"]).cpu(), sel(inp["uniforms"]).cpu(), inp["T"],
                         nthreads=nthreads)


def compare(gpu_tokens, gpu_len, ref, draft_len):
    """Return a dict of counts; ``mismatch`` must be 0."""
    B = gpu_len.shape[0]
    res = {"sequences": B, "mismatch": 0, "accept_ties": 0, "sample_ties": 0, "errors": 0,
           "bad": []}
    for b in range(B):
        st = int(ref["status"][b]) & 0xFF
        if st != 0:
            res["errors"] += 1
            if gpu_len[b] != 0 or not (gpu_tokens[b] == -1).all():
                res["mismatch"] += 1
                res["bad"].append((b, "error sequence emitted"))
            continue
        if ref["accept_tie"][b] < NEAR_TIE:
            res["accept_ties"] += 1
            continue
        n = int(ref["out_len"][b])
        if gpu_len[b] != n:
            res["mismatch"] += 1
            res["bad"].append((b, f"len {gpu_len[b]} != {n}"))
            continue
        if not np.array_equal(gpu_tokens[b, :n - 1], ref["out_tokens"][b, :n - 1]):
            res["mismatch"] += 1
            res["bad"].append((b, "accepted prefix"))
            continue
        if not (gpu_tokens[b, n:] == -1).all():
            res["mismatch"] += 1
            res["bad"].append((b, "padding"))
            continue
        if ref["sample_tie"][b] < NEAR_TIE:
            res["sample_ties"] += 1
            if not (0 <= gpu_tokens[b, n - 1]):
                res["mismatch"] += 1
                res["bad"].append((b, "invalid drawn token"))
            continue
        if gpu_tokens[b, n - 1] != ref["out_tokens"][b, n - 1]:
            res["mismatch"] += 1
            res["bad"].append((b, f"drawn {gpu_tokens[b, n - 1]} != {ref['out_tokens'][b, n - 1]}"))
    return res


MASS_ABS = 1e-6


def compare_diagnostics(dbg, ref, draft_len, out_len, skipped_ok=False):
    """Largest error / tolerance of LSE, alpha and the drawn mass.  With
    ``skipped_ok`` (early exit) rows after a rejection may hold NaN: they were
    not read."""
    kb = np.asarray(draft_len)
    B, k1 = ref["lse_t"].shape
    k = k1 - 1
    lse_t = dbg["lse_t"].cpu().numpy()
    lse_d = dbg["lse_d"].cpu().numpy()
    alpha = dbg["alpha"].cpu().numpy()
    mass = dbg["mass"].cpu().numpy()
    worst = {"lse": 0.0, "alpha": 0.0, "mass": 0.0}
    for b in range(B):
        if int(ref["status"][b]) & 0xFF:
            continue
        a_ref = int(ref["out_len"][b]) - 1
        skip = lambda i, v: skipped_ok and i > a_ref and np.isnan(v)
        for i in range(kb[b] + 1):
            r = ref["lse_t"][b, i]
            if skip(i, lse_t[b, i]):
                continue
            worst["lse"] = max(worst["lse"], abs(lse_t[b, i] - r) / (RTOL * max(1.0, abs(r))))
        for i in range(kb[b]):
            r = ref["lse_d"][b, i]
            if skip(i, lse_d[b, i]):
                continue
            worst["lse"] = max(worst["lse"], abs(lse_d[b, i] - r) / (RTOL * max(1.0, abs(r))))
            ra = ref["alpha"][b, i]
            if ra >= 1e-30:
                worst["alpha"] = max(worst["alpha"], abs(alpha[b, i] - ra) / (RTOL * ra))
        a = int(ref["out_len"][b]) - 1
        if ref["accept_tie"][b] >= NEAR_TIE and out_len[b] == a + 1 and np.isfinite(mass[b, a]):
            rm = ref["resid_mass"][b]
            worst["mass"] = max(worst["mass"], abs(mass[b, a] - rm) / (RTOL * rm + MASS_ABS))
    return worst


def check_invariants(gpu_tokens, gpu_len, draft_len, tokens, V):
    """Properties that hold at any size (every sequence, no oracle)."""
    kb = np.asarray(draft_len)
    tok = np.asarray(tokens)
    for b in range(gpu_len.shape[0]):
        n = int(gpu_len[b])
        assert 1 <= n <= kb[b] + 1, (b, n, kb[b])
        assert np.array_equal(gpu_tokens[b, :n - 1], tok[b, :n - 1]), b
        assert 0 <= gpu_tokens[b, n - 1] < V, b
        assert (gpu_tokens[b, n:] == -1).all(), b
