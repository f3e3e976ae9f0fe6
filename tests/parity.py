"""Comparison of the CUDA path with the fp64 oracle on the same inputs.

Tolerances:
  * accepted lengths and emitted token ids: identical, except where the
    oracle reports a near-tie: an executed accept test with
    |u_i - min(1, r_i)| < NEAR_TIE, or a sampling uniform within NEAR_TIE
    (in units of C/S) of a CDF boundary of the drawn token.  Near-ties are
    counted.  For an accept-test near-tie the whole sequence is excluded;
    for a sampling near-tie the accepted prefix must still match and the
    drawn token must lie in the oracle's window of valid draws (the tokens
    whose CDF interval comes within NEAR_TIE of the uniform).
  * min(1, p/q): relative 1e-5 (values >= 1e-30).
  * log-sum-exp: 1e-5 * max(1, |lse|) (an fp32 number near 400 has an ulp of
    3e-5, so an absolute 1e-5 is not representable there).
  * the draw's mass S (residual max(0, p - q) or the bonus row's 1):
    relative 1e-5.

Alongside, every comparison also counts the sequences that differ from the
oracle outside a tighter band, TIGHT_TIE = 1e-7, as a measure of how close
the fp32 kernel comes to the fp64 decisions.

``compare_diagnostics`` returns, per quantity, the largest error divided by
its tolerance: every value must be below 1.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

NEAR_TIE = 1e-5
TIGHT_TIE = 1e-7
RTOL = 1e-5


CANARY = -0x5A5A5A5B    # guard word written around every output buffer
GUARD = 64               # guard words on each side (256 bytes: the outputs stay aligned)


def guarded(n, device, dtype=torch.int32):
    """An n-element output inside a buffer with GUARD canary words on each
    side: (buffer, view)."""
    buf = torch.full((n + 2 * GUARD,), CANARY, dtype=dtype, device=device)
    return buf, buf[GUARD:GUARD + n]


def assert_guards(*bufs):
    """Nothing was written outside the outputs (a stand-in for a memory
    checker: a stray write next to an output shows here)."""
    for buf in bufs:
        g = torch.cat([buf[:GUARD], buf[-GUARD:]]).cpu()
        assert bool((g == CANARY).all()), "an output's guard words were overwritten"


def run_gpu(verifier, inp, stream=None):
    B, k1 = inp["target"].shape[:2]
    dev = inp["target"].device
    bt, out_tokens = guarded(B * k1, dev)
    bl, out_len = guarded(B, dev)
    verifier.verify(inp["target"], inp["draft"], inp["tokens"], inp["draft_len"], inp["uniforms"], inp["T"],
                    out_tokens=out_tokens.view(B, k1), out_len=out_len, stream=stream)
    torch.cuda.synchronize()
    assert_guards(bt, bl)
    return out_tokens.view(B, k1).cpu().numpy(), out_len.cpu().numpy()


def run_oracle(inp, idx=None, nthreads=0):
    """Run the oracle on all sequences or on the subset ``idx``."""
    sel = (lambda t: t) if idx is None else (lambda t: t[idx])
    return oracle.verify(sel(inp["target"]).cpu(), sel(inp["draft"]).cpu(), sel(inp["tokens"]).cpu(),
                         sel(inp["draft_len"]).cpu(), sel(inp["uniforms"]).cpu(), inp["T"],
                         nthreads=nthreads, tie_band=NEAR_TIE)


def compare(gpu_tokens, gpu_len, ref, draft_len):
    """Return a dict of counts; ``mismatch`` must be 0.  ``tight_mismatch``
    counts the sequences that differ from the oracle although no test and
    no draw of theirs came within TIGHT_TIE of a boundary."""
    B = gpu_len.shape[0]
    res = {"sequences": B, "mismatch": 0, "accept_ties": 0, "sample_ties": 0, "errors": 0,
           "tight_accept_ties": 0, "tight_sample_ties": 0, "tight_mismatch": 0, "bad": []}
    for b in range(B):
        st = int(ref["status"][b]) & 0xFF
        if st != 0:
            res["errors"] += 1
            if gpu_len[b] != 0 or not (gpu_tokens[b] == -1).all():
                res["mismatch"] += 1
                res["bad"].append((b, "error sequence emitted"))
            continue
        n = int(ref["out_len"][b])
        same = gpu_len[b] == n and np.array_equal(gpu_tokens[b], ref["out_tokens"][b])
        a_tie, s_tie = ref["accept_tie"][b], ref["sample_tie"][b]
        res["tight_accept_ties"] += int(a_tie < TIGHT_TIE)
        res["tight_sample_ties"] += int(a_tie >= TIGHT_TIE and s_tie < TIGHT_TIE)
        if not same and a_tie >= TIGHT_TIE and s_tie >= TIGHT_TIE:
            res["tight_mismatch"] += 1
        if a_tie < NEAR_TIE:
            res["accept_ties"] += 1
            continue
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
        y = int(gpu_tokens[b, n - 1])
        if s_tie < NEAR_TIE:
            res["sample_ties"] += 1
            lo, hi = int(ref["sample_lo"][b]), int(ref["sample_hi"][b])
            if not lo <= y <= hi:
                res["mismatch"] += 1
                res["bad"].append((b, f"drawn {y} outside the near-tie window [{lo}, {hi}]"))
            continue
        if y != ref["out_tokens"][b, n - 1]:
            res["mismatch"] += 1
            res["bad"].append((b, f"drawn {y} != {ref['out_tokens'][b, n - 1]}"))
    return res


def compare_diagnostics(dbg, ref, draft_len, out_len, skipped_ok=False):
    """Largest error / tolerance of LSE, alpha and the drawn mass.  With
    ``skipped_ok`` (early exit) rows after a rejection may hold NaN: they were
    not read."""
    kb = np.asarray(draft_len)
    B, k1 = ref["lse_t"].shape
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
        if ref["accept_tie"][b] >= NEAR_TIE and out_len[b] == a + 1:
            rm = ref["resid_mass"][b]
            if not np.isfinite(mass[b, a]):
                worst["mass"] = np.inf
            else:
                worst["mass"] = max(worst["mass"], abs(mass[b, a] - rm) / (RTOL * rm))
    return worst


def report(case, res, worst=None, **extra):
    """Print one case's near-tie counts and worst diagnostics, and append
    them as a JSON line to the file named by SV_PARITY_REPORT, if set."""
    import json
    import os
    line = {"case": case, **{k: v for k, v in res.items() if k != "bad"}, "near_tie_band": NEAR_TIE,
            "tight_band": TIGHT_TIE, **extra}
    if worst is not None:
        line["worst_over_tolerance"] = {k: float(v) for k, v in worst.items()}
    print("parity", json.dumps(line))
    path = os.environ.get("SV_PARITY_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(line) + "\n")
    return line


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
