"""Parity of the draft-length controller (``spec_ctrl_*``, through the C ABI)
with the fp64 oracle, round after round.

Both sides compute in fp64 with one rounding per multiply and add, in the
same order, for the acceptance state, so the counts and the estimate alpha
agree exactly.  The expected tokens E_n = sum_j alpha^j are built by
repeated multiplication on the GPU and with pow() in the oracle, and the
batch sums run in another order, so a decision may differ only where the
oracle's best and second-best rates lie within 1e-12 of each other
(relative); such near-ties are counted and must be rare.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_71_gb300 as svp
from speculative_decoding_verification_71_gb300 import build as svbuild

pytestmark = pytest.mark.gpu
DEV = "cuda"
NEAR_TIE = 1e-12


@pytest.fixture(scope="module", autouse=True)
def _built():
    svbuild.build()
    svp.load_library()


def cost_table(rng, n_points, max_k, slope=(0.05, 0.6)):
    """Round times growing in n and in B (the memory- to compute-bound move)."""
    bs = np.sort(rng.choice(np.arange(1, 2048), size=n_points, replace=False)).astype(np.int32)
    t0 = np.linspace(1.0, 3.0, n_points)[:, None] * rng.uniform(0.9, 1.1, (n_points, 1))
    grow = np.linspace(slope[0], slope[1], n_points)[:, None]
    table = t0 * (1.0 + grow * np.arange(max_k + 1)[None] * rng.uniform(0.8, 1.2, (n_points, max_k + 1)))
    return bs, table


def pair(rng, n_slots, max_k, mode, decay, prior_alpha, prior_weight, n_points=4):
    bs, table = cost_table(rng, n_points, max_k)
    gpu = svp.DraftController(n_slots, max_k)
    gpu.set_cost(bs, table)
    gpu.set_params(decay, prior_alpha, prior_weight, mode)
    ref = oracle.Controller(n_slots, max_k, bs, table, decay=decay, prior_alpha=prior_alpha,
                            prior_weight=prior_weight, mode=mode)
    return gpu, ref


def simulate_out_len(rng, true_alpha, draft_len):
    """Emitted lengths of one verified round: accepted prefix + 1."""
    out = np.empty_like(draft_len)
    for b, (al, k) in enumerate(zip(true_alpha, draft_len)):
        a = 0
        while a < k and rng.random() < al:
            a += 1
        out[b] = a + 1
    return out


def t32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(DEV)


def check_choice(got_len, got_choice, ref, mode):
    r = ref
    if mode == svp.SV_CTRL_BATCH:
        if r["margin"][0] <= NEAR_TIE:
            return 1
        assert got_choice == r["choice"], (got_choice, r["choice"], r["rates"])
        np.testing.assert_array_equal(got_len, r["next_len"])
        return 0
    near = r["margin"] <= NEAR_TIE
    np.testing.assert_array_equal(got_len[~near], r["next_len"][~near])
    if not near.any():
        assert got_choice == r["choice"]
    return int(near.sum())


CASES = [
    # n_slots, max_k, mode, decay, prior_alpha, prior_weight, rounds
    (300, 7, svp.SV_CTRL_BATCH, 0.9, 0.5, 2.0, 12),
    (300, 7, svp.SV_CTRL_PER_SEQUENCE, 0.9, 0.5, 2.0, 12),
    (64, 3, svp.SV_CTRL_BATCH, 1.0, 0.7, 0.0, 20),
    (64, 3, svp.SV_CTRL_PER_SEQUENCE, 0.5, 0.2, 10.0, 20),
    (2048, 31, svp.SV_CTRL_PER_SEQUENCE, 0.95, 0.6, 1.0, 6),
    (2048, 31, svp.SV_CTRL_BATCH, 0.95, 0.6, 1.0, 6),
    (40, 0, svp.SV_CTRL_BATCH, 0.9, 0.5, 2.0, 3),           # speculation never possible
]


@pytest.mark.parametrize("n_slots,max_k,mode,decay,a0,w0,rounds", CASES,
                         ids=[f"s{c[0]}-k{c[1]}-m{c[2]}-d{c[3]}" for c in CASES])
def test_rounds_match_the_oracle(n_slots, max_k, mode, decay, a0, w0, rounds):
    rng = np.random.default_rng(n_slots * 31 + max_k + mode)
    gpu, ref = pair(rng, n_slots, max_k, mode, decay, a0, w0)
    true_alpha = rng.beta(4, 2, n_slots)
    true_alpha[: n_slots // 8] = 0.0                      # a drafter that never matches
    true_alpha[n_slots // 8: n_slots // 4] = 1.0          # ... and one that always does
    active = rng.permutation(n_slots)[: max(1, (n_slots * 7) // 8)]
    kb = rng.integers(0, max_k + 1, active.size)
    ties = decisions = 0
    for r in range(rounds):
        out = simulate_out_len(rng, true_alpha[active], kb)
        out[rng.random(active.size) < 0.05] = 0            # sequences the verifier flagged
        st_ref = ref.observe(active, kb, out)
        gpu.observe(t32(active), t32(kb), t32(out))
        assert set(np.unique(st_ref)) <= {oracle.CTRL_USED, oracle.CTRL_SKIPPED}
        # the estimate: exact
        np.testing.assert_array_equal(gpu.alpha(t32(active)).cpu().numpy(), ref.alpha(active))
        # the batch shrinks as sequences finish; the rest keep their slots
        active = active[rng.random(active.size) > 0.12]
        if active.size == 0:
            break
        nl, ch = gpu.choose(t32(active))
        rr = ref.choose(active)
        nl, ch = nl.cpu().numpy(), int(ch.item())
        ties += check_choice(nl, ch, rr, mode)
        decisions += 1 if mode == svp.SV_CTRL_BATCH else active.size
        kb = nl.astype(np.int64)
    assert gpu.status() == svp.SV_OK
    assert ties <= max(1, decisions // 100), (ties, decisions)
    all_ids = np.arange(n_slots)
    np.testing.assert_array_equal(gpu.alpha(t32(all_ids)).cpu().numpy(), ref.alpha(all_ids))


def test_batch_size_moves_the_toggle():
    # profiled: speculation pays at small batches, not at large ones
    K = 4
    bs = np.array([1, 64, 512], np.int32)
    table = np.array([[1.0, 1.02, 1.04, 1.06, 1.08],         # memory-bound: drafts are nearly free
                      [1.0, 1.30, 1.60, 1.90, 2.20],
                      [1.0, 1.90, 2.80, 3.70, 4.60]])        # compute-bound: each draft costs a step
    gpu = svp.DraftController(1024, K)
    gpu.set_cost(bs, table)
    gpu.set_params(1.0, 0.8, 4.0, svp.SV_CTRL_BATCH)
    ref = oracle.Controller(1024, K, bs, table, decay=1.0, prior_alpha=0.8, prior_weight=4.0)
    seen = []
    for B in (1, 8, 32, 64, 128, 300, 512, 1024):
        ids = np.arange(B)
        nl, ch = gpu.choose(t32(ids))
        rr = ref.choose(ids)
        assert int(ch.item()) == rr["choice"]
        assert (nl.cpu().numpy() == rr["choice"]).all()
        seen.append(rr["choice"])
    assert seen[0] == K and seen[-1] == 0                  # on at B = 1, off at B = 1024
    assert all(a >= b for a, b in zip(seen, seen[1:]))      # never back on as B grows


def test_errors_are_reported_and_rows_skipped():
    gpu = svp.DraftController(8, 3)
    gpu.set_cost([1], [[1.0, 1.1, 1.2, 1.3]])
    gpu.set_params(1.0, 0.5, 0.0, svp.SV_CTRL_BATCH)
    gpu.observe(t32([0, 1]), t32([3, 3]), t32([2, 4]))
    assert gpu.status() == svp.SV_OK
    before = gpu.alpha(t32(np.arange(8))).cpu().numpy()
    gpu.observe(t32([2, 2, 3]), t32([3, 3, 3]), t32([1, 1, 4]))          # slot 2 twice
    assert gpu.status() == svp.SV_ERR_INVALID_ARG
    after = gpu.alpha(t32(np.arange(8))).cpu().numpy()
    assert after[2] == before[2] == 0.5                   # not updated (still the prior)
    assert after[3] == 1.0                                # the valid row was used
    gpu.reset()
    assert gpu.status() == svp.SV_OK
    gpu.observe(t32([0, 1]), t32([3, 4]), t32([5, 1]))                   # len > k + 1, k > max_k
    assert gpu.status() == svp.SV_ERR_BAD_DRAFT_LEN
    gpu.reset()
    gpu.observe(t32([9]), t32([1]), t32([1]))                            # id outside the slots
    assert gpu.status() == svp.SV_ERR_INVALID_ARG
    gpu.reset()
    nl, ch = gpu.choose(t32([0, 11, 1]))
    assert nl.cpu().tolist()[1] == 0 and gpu.status() == svp.SV_ERR_INVALID_ARG
    a = gpu.alpha(t32([5, -1])).cpu().numpy()
    assert a[0] == 0.5 and np.isnan(a[1])
    # resetting some slots only
    gpu.reset()
    gpu.observe(t32([4, 5]), t32([3, 3]), t32([4, 4]))
    gpu.reset(t32([5]))
    a = gpu.alpha(t32([4, 5])).cpu().numpy()
    assert a[0] == 1.0 and a[1] == 0.5
    # host checks
    with pytest.raises(svp.SpecVerifyError):
        gpu.set_cost([4, 2], [[1.0] * 4, [1.0] * 4])
    with pytest.raises(svp.SpecVerifyError):
        gpu.set_cost([1], [[1.0, 0.0, 1.0, 1.0]])
    with pytest.raises(svp.SpecVerifyError):
        gpu.set_params(0.0, 0.5, 1.0)
    fresh = svp.DraftController(4, 2)
    with pytest.raises(svp.SpecVerifyError):
        fresh.choose(t32([0]))                            # no round-time table yet


def test_empty_batch_and_choice_only():
    gpu = svp.DraftController(4, 2)
    gpu.set_cost([1], [[1.0, 1.0, 1.0]])
    gpu.observe(t32([]), t32([]), t32([]))
    nl, ch = gpu.choose(t32([]))
    assert nl.numel() == 0 and int(ch.item()) == 0
    assert gpu.status() == svp.SV_OK


def test_a_decode_loop_in_one_cuda_graph():
    """verify -> observe -> choose, captured once and replayed: the same
    results as the eager loop, and the controller state equals the oracle
    controller fed with the same verified lengths."""
    from workloads import get_workload, make_inputs
    import dataclasses
    B, k, V = 48, 5, 6144
    w = dataclasses.replace(get_workload("ragged"), B=B, k=k, V=V)
    inp = make_inputs(w, device=DEV)
    ver = svp.SpecVerifier(B, k, V, inp["target"].dtype)
    bs = np.array([1, 32, 64], np.int32)
    table = np.array([[1.0 + 0.02 * n for n in range(k + 1)], [1.0 + 0.15 * n for n in range(k + 1)],
                      [1.0 + 0.5 * n for n in range(k + 1)]])
    ids = t32(np.arange(B))

    def make():
        c = svp.DraftController(B, k)
        c.set_cost(bs, table)
        c.set_params(0.8, 0.6, 2.0, svp.SV_CTRL_PER_SEQUENCE)
        return c

    def run(ctrl, rounds, graph):
        draft_len = inp["draft_len"].clone()
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=DEV)
        out_len = torch.empty(B, dtype=torch.int32, device=DEV)
        nxt = torch.empty(B, dtype=torch.int32, device=DEV)
        choice = torch.empty(1, dtype=torch.int32, device=DEV)
        s = torch.cuda.Stream()
        hist = []

        def step():
            ver.verify(inp["target"], inp["draft"], inp["tokens"], draft_len, inp["uniforms"], inp["T"],
                       out_tokens=out_tokens, out_len=out_len, stream=s)
            ctrl.observe(ids, draft_len, out_len, stream=s)
            ctrl.choose(ids, nxt, choice, stream=s)
            draft_len.copy_(nxt)

        with torch.cuda.stream(s):
            if graph:
                step()                                    # warm up outside the capture
                s.synchronize()
                ctrl.reset(stream=s)
                draft_len.copy_(inp["draft_len"])
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    step()
            for _ in range(rounds):
                before = draft_len.clone()
                if graph:
                    g.replay()
                else:
                    step()
                hist.append((before.clone(), out_len.clone(), out_tokens.clone()))
        s.synchronize()
        return hist

    eager_ctrl, graph_ctrl = make(), make()
    he = run(eager_ctrl, 6, graph=False)
    hg = run(graph_ctrl, 6, graph=True)
    for (k0, l0, t0), (k1, l1, t1) in zip(he, hg):
        assert torch.equal(k0, k1) and torch.equal(l0, l1) and torch.equal(t0, t1)
    ref = oracle.Controller(B, k, bs, table, decay=0.8, prior_alpha=0.6, prior_weight=2.0, mode=1)
    for kb, ol, _ in he:
        ref.observe(np.arange(B), kb.cpu().numpy(), ol.cpu().numpy())
    np.testing.assert_array_equal(graph_ctrl.alpha(ids).cpu().numpy(), ref.alpha(np.arange(B)))
    # the lengths actually changed: the controller is in the loop
    assert any(not torch.equal(he[0][0], h[0]) for h in he[1:])
    assert eager_ctrl.status() == svp.SV_OK and graph_ctrl.status() == svp.SV_OK
