"""Replica path on CPU: two gloo ranks each verify their shard of a batch
with the oracle; summed counters and concatenated outputs equal one run over
the whole batch (the path shards by sequence with no data exchange)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from speculative_decoding_verification_71_gb300.replicas import max_over_ranks, reduce_counts, shard


def test_shard_covers_the_batch_once():
    for B in (0, 1, 7, 256, 1023):
        for world in (1, 2, 3, 8):
            parts = [shard(B, r, world) for r in range(world)]
            assert parts[0][0] == 0 and parts[-1][1] == B
            for (a, b), (c, d) in zip(parts, parts[1:]):
                assert b == c
            sizes = [b - a for a, b in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard(4, 2, 2)


def _counts(res, kb):
    ok = (res["status"] & 0xFF) == 0
    a = res["out_len"] - 1
    return {"sequences": int(ok.sum()), "drafts_proposed": int(kb[ok].sum()),
            "drafts_accepted": int(a[ok].sum()), "emitted": int(res["out_len"][ok].sum()),
            "spec_off": int((kb[ok] == 0).sum()), "zero_residual": 0, "error_sequences": int((~ok).sum())}


def _inputs():
    from workloads import get_workload, make_inputs
    w = get_workload("ragged", B=24, V=2000)
    return make_inputs(w, device="cpu")


def _worker(rank, world, port, outq):
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    inp = _inputs()
    B = inp["target"].shape[0]
    s, e = shard(B, rank, world)
    res = oracle.verify(inp["target"][s:e], inp["draft"][s:e], inp["tokens"][s:e], inp["draft_len"][s:e],
                        inp["uniforms"][s:e], inp["T"])
    kb = inp["draft_len"][s:e].numpy()
    total = reduce_counts(_counts(res, kb))
    slowest = max_over_ranks(float(rank + 1))
    outq.put((rank, res["out_tokens"], res["out_len"], total, slowest))
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_match_one_process():
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted([q.get(timeout=120) for _ in range(2)], key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    inp = _inputs()
    ref = oracle.verify(inp["target"], inp["draft"], inp["tokens"], inp["draft_len"], inp["uniforms"], inp["T"])
    np.testing.assert_array_equal(np.concatenate([g[1] for g in got]), ref["out_tokens"])
    np.testing.assert_array_equal(np.concatenate([g[2] for g in got]), ref["out_len"])
    want = _counts(ref, inp["draft_len"].numpy())
    for k, v in want.items():
        assert got[0][3][k] == v and got[1][3][k] == v, k
    assert got[0][4] == got[1][4] == 2.0
