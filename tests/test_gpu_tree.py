"""Parity of tree verification (``spec_verify_tree``, through the C ABI) with
the fp64 oracle.

The kernel sums each row in fp32 (ex2.approx) and takes each test in fp64
from those sums: p(x)/q(x) from its logarithm, (z^t - z^d) c minus the log2
ratio of the row sums, and after h rejections r(x)/q(x) = max(0, p/q - c_h)
/ P_h with c_h, P_h from the residual masses.  The residual weights are
formed as A e^t (1 - 2^delta), with no cancellation where p ~ c_h q, so the
masses carry the rows' fp32 error (~1e-7 relative) and the tests come within
1e-5 of the oracle's.  A sequence whose oracle walk came within 1e-5 of a
test threshold is a near-tie (excluded and counted); one whose draw came
within 1e-5 of a CDF boundary must still match on its accepted path and draw
a token inside the oracle's window of valid draws.  A draw from a diffuse
tail lands that close to a boundary whenever the drawn token's probability
is that small, so up to a quarter of the sequences (plus two) may be
near-ties.  Every other sequence must match the oracle exactly: tokens,
accepted nodes and lengths.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_71_gb300 as svp
from speculative_decoding_verification_71_gb300 import build as svbuild
from tests import tree_cases
from workloads import get_tree_workload, make_tree_inputs, get_workload, make_inputs

pytestmark = pytest.mark.gpu
DEV = "cuda"
ACCEPT_TIE = 1e-5
SAMPLE_TIE = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    svbuild.build()
    svp.load_library()


def run_gpu(inp, alpha=True):
    B, M, V = inp["target"].shape
    a = torch.empty(B, M, dtype=torch.float32, device=DEV) if alpha else None
    ot, on, ol, st = svp.verify_tree(inp["target"], inp["draft"], inp["parents"], inp["tokens"], inp["n_nodes"],
                                     inp["uniforms"], inp["T"], alpha=a)
    torch.cuda.synchronize()
    return ot.cpu().numpy(), on.cpu().numpy(), ol.cpu().numpy(), st.cpu().numpy(), (a.cpu().numpy() if alpha else None)


def run_ref(inp):
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    return oracle.tree_verify(cpu["target"], cpu["draft"], cpu["parents"], cpu["tokens"], cpu["n_nodes"],
                              cpu["uniforms"], cpu["T"], tie_band=SAMPLE_TIE)


def compare(g, ref, T):
    """Exact match outside near-ties; at a sampling near-tie the accepted
    path matches and the drawn token lies in the oracle's window.  Returns
    the number of near-tie sequences."""
    ot, on, ol, st, al = g
    B = len(ol)
    a_near = ref["accept_tie"] < ACCEPT_TIE if T > 0 else np.zeros(B, bool)
    s_near = (ref["sample_tie"] < SAMPLE_TIE) & ~a_near if T > 0 else np.zeros(B, bool)
    ok = ~(a_near | s_near)
    np.testing.assert_array_equal(st, ref["status"] & 0xff)
    np.testing.assert_array_equal(ol[ok], ref["out_len"][ok])
    np.testing.assert_array_equal(ot[ok], ref["out_tokens"][ok])
    np.testing.assert_array_equal(on[ok], ref["out_nodes"][ok])
    for b in np.nonzero(s_near)[0]:
        n = int(ref["out_len"][b])
        assert ol[b] == n, (b, ol[b], n)
        np.testing.assert_array_equal(on[b], ref["out_nodes"][b])
        np.testing.assert_array_equal(ot[b, :n - 1], ref["out_tokens"][b, :n - 1])
        assert ref["sample_lo"][b] <= ot[b, n - 1] <= ref["sample_hi"][b], (b, ot[b, n - 1])
    near = a_near | s_near
    if al is not None:
        ra = ref["alpha"]
        both = ok[:, None] & ~np.isnan(ra)
        assert np.array_equal(np.isnan(al[ok]), np.isnan(ra[ok]))
        err = np.abs(al[both] - ra[both])
        assert (err <= ACCEPT_TIE).all(), err.max()
    return int(near.sum())


CASES = [
    # workload, overrides
    ("tree", dict(B=24, V=1000, dtype="f32")),
    ("tree", dict(B=24, V=4099, dtype="f32", T=0.7)),          # unaligned rows: scalar loads
    ("tree", dict(B=16, V=32000, dtype="bf16")),
    ("tree_wide", dict(B=32, V=20000, dtype="bf16", T=1.3)),
    ("tree_wide", dict(B=16, V=1001, dtype="bf16")),            # unaligned bf16
    ("tree", dict(B=8, V=151936, dtype="bf16")),                # the full vocabulary
    ("tree", dict(B=8, V=65536, dtype="f32", draft_sigma=3.0)),  # a poor drafter: many rejections
    ("tree_wide", dict(B=24, V=5000, dtype="f32", T=0.0)),      # greedy
    ("tree", dict(B=16, V=3000, dtype="bf16", T=0.0, draft_sigma=0.1)),
    ("tree_wide", dict(B=400, V=4096, dtype="bf16")),           # more CTAs than fit at once: in waves
]


@pytest.mark.parametrize("name,over", CASES, ids=[f"{n}-{o}" for n, o in CASES])
def test_tree_matches_the_oracle(name, over):
    w = get_tree_workload(name, **over)
    inp = make_tree_inputs(w, device=DEV)
    g = run_gpu(inp)
    ref = run_ref(inp)
    ties = compare(g, ref, w.T)
    assert ties <= len(g[2]) // 4 + 2, ties
    assert (g[3] == 0).all()


@pytest.mark.parametrize("shape", ["fan2", "fan3", "mixed", "binary2"])
def test_enumeration_batch_decisions(shape):
    """The exhaustive-enumeration batch of the oracle pin: every case is far
    from its decision boundaries, so the kernel must decide each exactly."""
    batch, _ = tree_cases.build(shape, V=3, T=1.0, seed=1)
    far = batch["margin"] >= ACCEPT_TIE
    inp = {k: torch.from_numpy(np.ascontiguousarray(batch[k])).to(DEV)
           for k in ("target", "draft", "parents", "tokens", "n_nodes", "uniforms")}
    inp["T"] = 1.0
    ot, on, ol, st, _ = run_gpu(inp, alpha=False)
    assert (st == 0).all()
    np.testing.assert_array_equal(ol[far], batch["out_len"][far])
    np.testing.assert_array_equal(ot[far], batch["out_tokens"][far])
    np.testing.assert_array_equal(on[far], batch["out_nodes"][far])
    assert far.mean() > 0.9


def test_chain_tree_equals_linear_verification():
    """A chain of k_b + 1 nodes on the GPU gives what spec_verify gives on
    the GPU for the same inputs (two kernels, one rule)."""
    w = dataclasses.replace(get_workload("ragged"), B=64, k=4, V=20000)
    lin = make_inputs(w, device=DEV)
    B, k, V = 64, 4, 20000
    M = k + 1
    ver = svp.SpecVerifier(B, k, V, torch.bfloat16)
    lt, ll = ver.verify(lin["target"], lin["draft"], lin["tokens"], lin["draft_len"], lin["uniforms"], lin["T"])
    par = torch.arange(-1, M - 1, dtype=torch.int32, device=DEV).view(1, M).repeat(B, 1)
    tok = torch.zeros(B, M, dtype=torch.int32, device=DEV)
    tok[:, 1:] = lin["tokens"].clamp(min=0)
    draft = torch.cat([lin["draft"], torch.full((B, 1, V), float("nan"), dtype=torch.bfloat16, device=DEV)], dim=1)
    uni = torch.empty(B, M, dtype=torch.float32, device=DEV)
    uni[:, 0] = lin["uniforms"][:, k]
    uni[:, 1:] = lin["uniforms"][:, :k]
    inp = {"target": lin["target"], "draft": draft.contiguous(), "parents": par, "tokens": tok,
           "n_nodes": (lin["draft_len"] + 1).to(torch.int32), "uniforms": uni, "T": lin["T"]}
    ot, on, ol, st, _ = run_gpu(inp, alpha=False)
    ref = run_ref(inp)
    near = (ref["accept_tie"] < ACCEPT_TIE) | (ref["sample_tie"] < SAMPLE_TIE)
    lt, ll = lt.cpu().numpy(), ll.cpu().numpy()
    np.testing.assert_array_equal(ol[~near], ll[~near])
    np.testing.assert_array_equal(ot[~near], lt[~near])
    assert near.sum() <= 64 // 4 + 2


def test_errors_mark_only_their_sequence():
    w = get_tree_workload("tree", B=8, V=3000, dtype="f32")
    inp = make_tree_inputs(w, device=DEV)
    inp["parents"][0, 5] = 5                  # its own parent
    inp["n_nodes"][1] = 16                    # more nodes than M
    inp["tokens"][2, 3] = 3000                # outside the vocabulary
    inp["target"][3, 0, 17] = float("nan")    # the root row is always read
    inp["draft"][4, 0, :] = float("-inf")     # the root's draft row is all -inf
    inp["target"][5, 0, 9] = float("inf")
    g = run_gpu(inp)
    ref = run_ref(inp)
    assert list(g[3][:6]) == [svp.SV_ERR_BAD_DRAFT_LEN, svp.SV_ERR_BAD_DRAFT_LEN, svp.SV_ERR_BAD_TOKEN,
                              svp.SV_ERR_NONFINITE, svp.SV_ERR_NONFINITE, svp.SV_ERR_NONFINITE]
    assert (g[2][:6] == 0).all() and (g[0][:6] == -1).all() and (g[1][:6] == -1).all()
    compare(g, ref, w.T)


def test_root_only_and_repeated_calls():
    w = get_tree_workload("tree_wide", B=64, V=7000, dtype="bf16")
    inp = make_tree_inputs(w, device=DEV)
    inp["n_nodes"][:16] = 1                   # speculation off for these: plain sampling
    a = run_gpu(inp)
    compare(a, run_ref(inp), w.T)
    assert (a[2][:16] == 1).all()
    for _ in range(4):
        b = run_gpu(inp)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)


def test_back_to_back_calls_into_the_same_outputs():
    """Calls enqueued back to back on one stream with no host wait between
    them, into the same output buffers (each call's walk may start while the
    previous one runs; its outputs are written after the previous call is
    complete): the last call's outputs are the oracle's."""
    ws = [get_tree_workload("tree", B=24, V=20000, dtype="bf16", seed=31),
          get_tree_workload("tree", B=24, V=20000, dtype="bf16", seed=32, draft_sigma=3.0),
          get_tree_workload("tree", B=24, V=20000, dtype="bf16", seed=33, T=0.0)]
    inps = [make_tree_inputs(w, device=DEV) for w in ws]
    B, M = 24, inps[0]["target"].shape[1]
    assert all(i["target"].shape[1] == M for i in inps)
    stream = torch.cuda.Stream()
    ot = torch.empty(B, M, dtype=torch.int32, device=DEV)
    on = torch.empty(B, M, dtype=torch.int32, device=DEV)
    ol = torch.empty(B, dtype=torch.int32, device=DEV)
    st = torch.empty(B, dtype=torch.int32, device=DEV)
    al = torch.empty(B, M, dtype=torch.float32, device=DEV)
    for rep in range(4):
        for inp in inps:
            svp.verify_tree(inp["target"], inp["draft"], inp["parents"], inp["tokens"], inp["n_nodes"],
                            inp["uniforms"], inp["T"], out_tokens=ot, out_nodes=on, out_len=ol, status=st, alpha=al,
                            stream=stream)
    stream.synchronize()
    last = inps[-1]
    compare((ot.cpu().numpy(), on.cpu().numpy(), ol.cpu().numpy(), st.cpu().numpy(), al.cpu().numpy()),
            run_ref(last), last["T"])


def test_graph_capture():
    w = get_tree_workload("tree", B=16, V=8192, dtype="bf16")
    inp = make_tree_inputs(w, device=DEV)
    B, M, V = inp["target"].shape
    outs = [torch.empty(B, M, dtype=torch.int32, device=DEV) for _ in range(2)] + \
           [torch.empty(B, dtype=torch.int32, device=DEV) for _ in range(2)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        svp.verify_tree(inp["target"], inp["draft"], inp["parents"], inp["tokens"], inp["n_nodes"],
                        inp["uniforms"], inp["T"], *outs, stream=s)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            svp.verify_tree(inp["target"], inp["draft"], inp["parents"], inp["tokens"], inp["n_nodes"],
                            inp["uniforms"], inp["T"], *outs, stream=s)
        for o in outs:
            o.fill_(-7)
        g.replay()
        s.synchronize()
    ref = run_ref(inp)
    compare((outs[0].cpu().numpy(), outs[1].cpu().numpy(), outs[2].cpu().numpy(), outs[3].cpu().numpy(), None),
            ref, w.T)
