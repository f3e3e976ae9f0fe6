"""The C-ABI library builds, loads and exports every symbol the header
declares; host-side argument checks reject bad calls without touching a GPU."""
import ctypes
import os
import re

import pytest

import speculative_decoding_verification_71_gb300 as svp
from speculative_decoding_verification_71_gb300 import build as svbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    svbuild.build()
    return svp.load_library()


def declared_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b((?:sv|spec_verify|spec_kd|spec_ctrl)\w*)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(svp.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for code, name in enumerate(["SV_OK", "SV_ERR_INVALID_ARG", "SV_ERR_BAD_DRAFT_LEN",
                                 "SV_ERR_BAD_TOKEN", "SV_ERR_NONFINITE", "SV_ERR_TIMEOUT",
                                 "SV_ERR_CUDA", "SV_ERR_UNSUPPORTED"]):
        assert lib.sv_status_string(code).decode() == name


def test_null_context_is_rejected_on_the_host(lib):
    P = None
    assert lib.spec_verify(P, 1, 1, P, P, P, P, P, 1.0, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_compact(P, 1, 1, P, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_debug(P, 1, 1, P, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_stats(P, P, None) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_reset_stats(P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.sv_set_pipeline(P, 4, 2) == svp.SV_ERR_INVALID_ARG
    assert lib.sv_set_wait_limit_ns(P, 0) == svp.SV_ERR_INVALID_ARG
    assert lib.sv_get_config(P, None, None, None, None, None, None) == svp.SV_ERR_INVALID_ARG
    assert lib.sv_set_cluster(P, 2) == svp.SV_ERR_INVALID_ARG
    assert lib.sv_launch_shape(P, 4, None, None) == svp.SV_ERR_INVALID_ARG
    assert lib.sv_rows_shape(P, None, None, None) == svp.SV_ERR_INVALID_ARG
    d = ctypes.c_double()
    assert lib.sv_measure_ex2(0, ctypes.byref(d), None) == svp.SV_ERR_INVALID_ARG
    assert lib.sv_measure_ex2(16, None, None) == svp.SV_ERR_INVALID_ARG
    assert lib.sv_set_early_exit(P, 1) == svp.SV_ERR_INVALID_ARG
    # the distillation loss checks its sizes, temperature and pointers on the host
    assert lib.spec_kd_loss(0, 1, 10, 1, P, P, P, 1.0, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_kd_loss(1, 1, 10, 1, P, P, P, 1.0, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_kd_loss(1, 1, 10, 5, P, P, P, 1.0, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    one = ctypes.c_void_p(16)
    assert lib.spec_kd_loss(1, 1, 10, 1, one, one, one, 0.0, one, one, None, P) == svp.SV_ERR_INVALID_ARG
    assert lib.sv_destroy(P) == svp.SV_OK


def test_create_rejects_bad_sizes_before_any_cuda_call(lib):
    h = ctypes.c_void_p()
    for args in [(0, 3, 100, 1), (4, -1, 100, 1), (4, 3, 0, 1), (4, 3, 100, 7), (1 << 25, 7, 100, 1),
                 (4, 32, 100, 1), (4, 3, 1 << 20, 0)]:
        assert lib.sv_create(ctypes.byref(h), *args) == svp.SV_ERR_INVALID_ARG, args
    assert lib.sv_create(None, 4, 3, 100, 1) == svp.SV_ERR_INVALID_ARG


def test_binding_fails_loudly_without_the_library(tmp_path):
    with pytest.raises(RuntimeError, match="not found"):
        svp.load_library(str(tmp_path / "missing.so"))


def test_product_does_not_use_the_oracle():
    """The library and its binding never import, load or name the oracle."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_71_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h", ".cuh", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"import\s+oracle|from\s+oracle|liboracle|oracle\.c", text), f


def test_controller_host_checks(lib):
    P = None
    out = ctypes.c_void_p()
    assert lib.spec_ctrl_create(None, 4, 3) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_create(ctypes.byref(out), 0, 3) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_create(ctypes.byref(out), 4, 32) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_create(ctypes.byref(out), 4, -1) == svp.SV_ERR_INVALID_ARG
    assert not out.value
    assert lib.spec_ctrl_destroy(P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_set_cost(P, 1, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_set_params(P, 0.9, 0.5, 2.0, 0) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_reset(P, 0, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_observe(P, 1, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_choose(P, 1, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_alpha(P, 1, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_ctrl_status(P, P) == svp.SV_ERR_INVALID_ARG


def test_tree_host_checks(lib):
    P = None
    # sizes, dtype, temperature and pointers are checked before any launch
    assert lib.spec_verify_tree(1, 0, 10, 1, P, P, P, P, P, P, 1.0, P, P, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_tree(1, 65, 10, 1, P, P, P, P, P, P, 1.0, P, P, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_tree(1, 4, 0, 1, P, P, P, P, P, P, 1.0, P, P, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_tree(1, 4, 10, 7, P, P, P, P, P, P, 1.0, P, P, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_tree(1, 4, 10, 1, P, P, P, P, P, P, -1.0, P, P, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_tree(1, 4, 10, 1, P, P, P, P, P, P, 1.0, P, P, P, P, P, P) == svp.SV_ERR_INVALID_ARG
    assert lib.spec_verify_tree(0, 4, 10, 1, P, P, P, P, P, P, 1.0, P, P, P, P, P, P) == svp.SV_OK


def test_host_tensors_are_rejected_before_any_call(lib):
    # CPU tensors must never reach a kernel as device pointers
    import torch
    t = torch.zeros(2, 3, 8, dtype=torch.float32)
    i = torch.zeros(2, 3, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        svp.verify_tree(t, t, i, i, torch.ones(2, dtype=torch.int32), torch.zeros(2, 3), 1.0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        svp.kd_loss(t, t, torch.ones(2), 1.0)
    with pytest.raises(ValueError, match="CUDA tensor"):
        svp.spec_verify_noalloc(t, t[:, :2], i[:, :2], torch.ones(2, dtype=torch.int32), torch.zeros(2, 3), 1.0,
                                i, torch.zeros(2, dtype=torch.int32))
