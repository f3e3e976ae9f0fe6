"""The allocation-free entry point gives the same outputs as the context-based
one.  spec_verify_noalloc serves callers that cannot call cudaMalloc (code
under an allocator it does not own, or that must not synchronise the device):
its workspace is a fixed array inside the library.  Two calls in a row, on
different inputs, check that the shared array carries nothing over."""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_verification_71_gb300 as svp
from speculative_decoding_verification_71_gb300 import build as svbuild
from workloads import get_workload, make_inputs

pytestmark = pytest.mark.gpu


def _noalloc_abi(inp, out_tokens, out_len):
    """Call the C entry point directly (through the C ABI, no wrapper)."""
    lib = svp.load_library()
    B, k1, V = inp["target"].shape
    dt = svp.SV_F32 if inp["target"].dtype == torch.float32 else svp.SV_BF16
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t is not None else None
    st = lib.spec_verify_noalloc(B, k1 - 1, V, dt, p(inp["target"]), p(inp["draft"]), p(inp["tokens"]),
                                 p(inp["draft_len"]), p(inp["uniforms"]), float(inp["T"]), p(out_tokens),
                                 p(out_len), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == svp.SV_OK, st
    torch.cuda.synchronize()


def test_noalloc_matches_context_entry_point_twice():
    svbuild.build()
    cases = [get_workload("ragged", B=48, k=3, V=20000, seed=31),
             get_workload("long_draft", B=20, k=7, V=12288, seed=32)]
    for w in cases:   # two calls in a row on the shared array
        inp = make_inputs(w, device="cuda")
        ver = svp.SpecVerifier(w.B, w.k, w.V, w.torch_dtype)
        ver.set_kernel(svp.SV_KERNEL_CLUSTER)   # the schedule this entry point runs: equal to the bit
        ref_t, ref_l = ver.verify(inp["target"], inp["draft"], inp["tokens"], inp["draft_len"],
                                  inp["uniforms"], inp["T"])
        out_t = torch.full_like(ref_t, 7)
        out_l = torch.full_like(ref_l, 7)
        _noalloc_abi(inp, out_t, out_l)
        np.testing.assert_array_equal(out_l.cpu().numpy(), ref_l.cpu().numpy())
        np.testing.assert_array_equal(out_t.cpu().numpy(), ref_t.cpu().numpy())


MORE_CASES = [
    ("ragged", dict(B=64, k=3, V=8192, T=0.0, seed=33)),          # greedy: no draft rows, no uniforms used
    ("tiny", dict()),                                              # fp32, the small workload
    ("tiny", dict(B=4096, k=3, V=256, seed=34)),                   # B (k + 1) = 16384: the array's capacity
]


def test_noalloc_greedy_fp32_and_full_capacity():
    """Greedy and fp32 instances, and a batch that fills the array, each twice
    in a row: equal to the context entry point (itself checked against the
    oracle) and to the oracle, and nothing written past the batch's rows."""
    import oracle
    svbuild.build()
    for name, over in MORE_CASES:
        w = get_workload(name, **over)
        inp = make_inputs(w, device="cuda")
        ver = svp.SpecVerifier(w.B, w.k, w.V, w.torch_dtype)
        ver.set_kernel(svp.SV_KERNEL_CLUSTER)   # the schedule this entry point runs: equal to the bit
        ref_t, ref_l = ver.verify(inp["target"], inp["draft"], inp["tokens"], inp["draft_len"],
                                  inp["uniforms"], inp["T"])
        ref = oracle.verify(inp["target"].cpu(), inp["draft"].cpu(), inp["tokens"].cpu(), inp["draft_len"].cpu(),
                            inp["uniforms"].cpu(), inp["T"])
        far = (ref["accept_tie"] >= 1e-5) & (ref["sample_tie"] >= 1e-5)
        for _ in range(2):
            # outputs inside larger buffers: the rows after the batch must keep their sentinel
            big_t = torch.full((w.B + 8, w.k + 1), -77, dtype=torch.int32, device="cuda")
            big_l = torch.full((w.B + 8,), -77, dtype=torch.int32, device="cuda")
            _noalloc_abi(inp, big_t[:w.B], big_l[:w.B])
            got_t, got_l = big_t[:w.B].cpu().numpy(), big_l[:w.B].cpu().numpy()
            np.testing.assert_array_equal(got_l, ref_l.cpu().numpy())
            np.testing.assert_array_equal(got_t, ref_t.cpu().numpy())
            np.testing.assert_array_equal(got_l[far], ref["out_len"][far])
            np.testing.assert_array_equal(got_t[far], ref["out_tokens"][far])
            assert bool((big_t[w.B:] == -77).all()) and bool((big_l[w.B:] == -77).all())


def test_noalloc_rejects_sizes_beyond_the_array():
    svbuild.build()
    lib = svp.load_library()
    P = None
    assert lib.spec_verify_noalloc(4097, 1, 100, svp.SV_BF16, P, P, P, P, P, 1.0, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_noalloc(4096, 7, 100, svp.SV_BF16, P, P, P, P, P, 1.0, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_noalloc(8, 32, 100, svp.SV_BF16, P, P, P, P, P, 1.0, P, P, P) == svp.SV_ERR_INVALID_ARG
