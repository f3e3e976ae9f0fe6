"""Lossless speculative-sampling verification on GB300 (sm_103a).

A thin ctypes binding over ``libspecverify.so`` (C ABI in
``include/specverify.h``).  Every step of the verification runs in the
library's CUDA kernels; this module only marshals arguments: it checks
shapes and dtypes, passes device pointers and the current CUDA stream, and
allocates output tensors when the caller does not supply them.  There is no
CPU fallback: if the library is missing or cannot be loaded, the first call
raises.

The low-level functions carry the C names (``sv_create``, ``spec_verify``,
``spec_verify_compact``, ``spec_verify_debug``, ``spec_verify_stats``,
``spec_verify_reset_stats``, ``sv_destroy`` ...).  ``SpecVerifier`` wraps a
context for convenient use from PyTorch.
"""
from __future__ import annotations

import ctypes
import os

import torch

__all__ = [
    "SpecVerifier", "SpecVerifyError", "Stats", "load_library", "library_path",
    "SV_OK", "SV_ERR_INVALID_ARG", "SV_ERR_BAD_DRAFT_LEN", "SV_ERR_BAD_TOKEN",
    "SV_ERR_NONFINITE", "SV_ERR_TIMEOUT", "SV_ERR_CUDA", "SV_ERR_UNSUPPORTED",
    "SV_F32", "SV_BF16", "EXPORTED_SYMBOLS", "DraftController", "verify_tree", "SV_CTRL_BATCH", "SV_CTRL_PER_SEQUENCE",
    "measure_ex2",
]

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_BAD_DRAFT_LEN, SV_ERR_BAD_TOKEN = 0, 1, 2, 3
SV_ERR_NONFINITE, SV_ERR_TIMEOUT, SV_ERR_CUDA, SV_ERR_UNSUPPORTED = 4, 5, 6, 7
SV_F32, SV_BF16 = 0, 1
SV_CTRL_BATCH, SV_CTRL_PER_SEQUENCE = 0, 1
SV_KERNEL_AUTO, SV_KERNEL_CLUSTER, SV_KERNEL_PIECES = 0, 1, 2
SV_CTRL_MAX_POINTS = 12

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libspecverify.so")
_lib = None

EXPORTED_SYMBOLS = (
    "sv_status_string", "sv_last_cuda_error", "sv_create", "sv_destroy", "spec_verify",
    "spec_verify_compact", "spec_verify_debug", "spec_verify_stats", "spec_verify_reset_stats",
    "sv_set_pipeline", "sv_set_cluster", "sv_set_early_exit", "sv_set_diagnostics", "sv_get_config", "sv_launch_shape",
    "sv_set_wait_limit_ns", "sv_set_kernel", "sv_kernel_for", "sv_rows_shape", "sv_set_timeline", "sv_measure_ex2",
    "spec_verify_noalloc", "spec_kd_loss", "spec_kd_launch_shape",
    "spec_ctrl_create", "spec_ctrl_destroy", "spec_ctrl_set_cost", "spec_ctrl_set_params", "spec_ctrl_reset",
    "spec_ctrl_observe", "spec_ctrl_choose", "spec_ctrl_alpha", "spec_ctrl_status",
    "spec_verify_tree",
)


class Stats(ctypes.Structure):
    _fields_ = [
        ("mean_emitted", ctypes.c_double), ("mean_accepted", ctypes.c_double),
        ("accept_rate", ctypes.c_double), ("calls", ctypes.c_longlong),
        ("sequences", ctypes.c_longlong), ("drafts_proposed", ctypes.c_longlong),
        ("drafts_accepted", ctypes.c_longlong), ("emitted", ctypes.c_longlong),
        ("spec_off", ctypes.c_longlong), ("zero_residual", ctypes.c_longlong),
        ("error_sequences", ctypes.c_longlong), ("error_bits", ctypes.c_uint),
        ("rows_skipped", ctypes.c_longlong),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


class SpecVerifyError(RuntimeError):
    def __init__(self, status, where, detail=""):
        self.status = status
        name = _status_name(status)
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


def library_path() -> str:
    return _LIB_PATH


def load_library(path: str | None = None):
    """Load the C-ABI library (once).  Raises if it is absent: build it with
    ``speculative_decoding_verification_71_gb300.build.build()``."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libspecverify.so not found at {p}; build it first (build.build())")
    lib = ctypes.CDLL(p)
    c, P = ctypes, ctypes.c_void_p
    lib.sv_status_string.restype = c.c_char_p
    lib.sv_status_string.argtypes = [c.c_int]
    lib.sv_last_cuda_error.restype = c.c_char_p
    lib.sv_last_cuda_error.argtypes = [P]
    lib.sv_create.restype = c.c_int
    lib.sv_create.argtypes = [c.POINTER(P), c.c_int, c.c_int, c.c_int, c.c_int]
    lib.sv_destroy.restype = c.c_int
    lib.sv_destroy.argtypes = [P]
    lib.spec_verify.restype = c.c_int
    lib.spec_verify.argtypes = [P, c.c_int, c.c_int, P, P, P, P, P, c.c_float, P, P, P]
    lib.spec_verify_compact.restype = c.c_int
    lib.spec_verify_compact.argtypes = [P, c.c_int, c.c_int, P, P, P, P, P]
    lib.spec_verify_debug.restype = c.c_int
    lib.spec_verify_debug.argtypes = [P, c.c_int, c.c_int, P, P, P, P, P]
    lib.spec_verify_stats.restype = c.c_int
    lib.spec_verify_stats.argtypes = [P, P, c.POINTER(Stats)]
    lib.spec_verify_reset_stats.restype = c.c_int
    lib.spec_verify_reset_stats.argtypes = [P, P]
    lib.sv_set_pipeline.restype = c.c_int
    lib.sv_set_pipeline.argtypes = [P, c.c_int, c.c_int]
    lib.sv_set_early_exit.restype = c.c_int
    lib.sv_set_early_exit.argtypes = [P, c.c_int]
    lib.sv_set_diagnostics.restype = c.c_int
    lib.sv_set_diagnostics.argtypes = [P, c.c_int]
    lib.sv_set_cluster.restype = c.c_int
    lib.sv_set_cluster.argtypes = [P, c.c_int]
    lib.sv_set_kernel.restype = c.c_int
    lib.sv_set_kernel.argtypes = [P, c.c_int]
    lib.sv_set_timeline.restype = c.c_int
    lib.sv_set_timeline.argtypes = [P, P, c.c_int]
    lib.sv_kernel_for.restype = c.c_int
    lib.sv_kernel_for.argtypes = [P, c.c_int, c.POINTER(c.c_int)]
    lib.sv_get_config.restype = c.c_int
    lib.sv_get_config.argtypes = [P] + [c.POINTER(c.c_int)] * 6
    lib.spec_kd_loss.restype = c.c_int
    lib.spec_kd_loss.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int, P, P, P, c.c_float, P, P, P, P]
    lib.spec_kd_launch_shape.restype = c.c_int
    lib.spec_kd_launch_shape.argtypes = [c.c_int, c.c_int, c.c_int, c.POINTER(c.c_int), c.POINTER(c.c_int),
                                         c.POINTER(c.c_int)]
    lib.sv_launch_shape.restype = c.c_int
    lib.sv_launch_shape.argtypes = [P, c.c_int, c.POINTER(c.c_int), c.POINTER(c.c_int)]
    lib.sv_rows_shape.restype = c.c_int
    lib.sv_rows_shape.argtypes = [P, c.POINTER(c.c_int), c.POINTER(c.c_int), c.POINTER(c.c_int)]
    lib.sv_set_wait_limit_ns.restype = c.c_int
    lib.sv_set_wait_limit_ns.argtypes = [P, c.c_longlong]
    lib.sv_measure_ex2.restype = c.c_int
    lib.sv_measure_ex2.argtypes = [c.c_int, c.POINTER(c.c_double), c.POINTER(c.c_double)]
    lib.spec_ctrl_create.restype = c.c_int
    lib.spec_ctrl_create.argtypes = [c.POINTER(P), c.c_int, c.c_int]
    lib.spec_ctrl_destroy.restype = c.c_int
    lib.spec_ctrl_destroy.argtypes = [P]
    lib.spec_ctrl_set_cost.restype = c.c_int
    lib.spec_ctrl_set_cost.argtypes = [P, c.c_int, P, P]
    lib.spec_ctrl_set_params.restype = c.c_int
    lib.spec_ctrl_set_params.argtypes = [P, c.c_double, c.c_double, c.c_double, c.c_int]
    lib.spec_ctrl_reset.restype = c.c_int
    lib.spec_ctrl_reset.argtypes = [P, c.c_int, P, P]
    lib.spec_ctrl_observe.restype = c.c_int
    lib.spec_ctrl_observe.argtypes = [P, c.c_int, P, P, P, P]
    lib.spec_ctrl_choose.restype = c.c_int
    lib.spec_ctrl_choose.argtypes = [P, c.c_int, P, P, P, P]
    lib.spec_ctrl_alpha.restype = c.c_int
    lib.spec_ctrl_alpha.argtypes = [P, c.c_int, P, P, P]
    lib.spec_ctrl_status.restype = c.c_int
    lib.spec_ctrl_status.argtypes = [P, P]
    lib.spec_verify_tree.restype = c.c_int
    lib.spec_verify_tree.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int, P, P, P, P, P, P, c.c_float,
                                     P, P, P, P, P, P]
    lib.spec_verify_noalloc.restype = c.c_int
    lib.spec_verify_noalloc.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int, P, P, P, P, P, c.c_float, P, P, P]
    if path is None:
        _lib = lib
    return lib


def _status_name(status):
    names = ["SV_OK", "SV_ERR_INVALID_ARG", "SV_ERR_BAD_DRAFT_LEN", "SV_ERR_BAD_TOKEN",
             "SV_ERR_NONFINITE", "SV_ERR_TIMEOUT", "SV_ERR_CUDA", "SV_ERR_UNSUPPORTED"]
    return names[status] if 0 <= status < len(names) else f"status {status}"


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream_handle(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _check_dev(name, t, dtype, shape, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        # the kernels read device memory: a host pointer must never reach them
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class SpecVerifier:
    """A verification context: fixed workspace for up to ``max_B`` sequences
    of up to ``max_k`` drafts over vocabulary ``V`` in ``dtype``
    (torch.float32 or torch.bfloat16), on the current CUDA device."""

    def __init__(self, max_B: int, max_k: int, V: int, dtype=torch.bfloat16, device=None):
        self.lib = load_library()
        if dtype not in (torch.float32, torch.bfloat16):
            raise TypeError("dtype must be torch.float32 or torch.bfloat16")
        self.max_B, self.max_k, self.V, self.dtype = max_B, max_k, V, dtype
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else
                                   torch.device(device).index or 0)
        self._ctx = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            st = self.lib.sv_create(ctypes.byref(self._ctx), max_B, max_k, V,
                                    SV_F32 if dtype == torch.float32 else SV_BF16)
        if st != SV_OK:
            raise SpecVerifyError(st, "sv_create", self.lib.sv_last_cuda_error(None).decode())

    # -- lifetime -------------------------------------------------------
    def close(self):
        if self._ctx:
            self.lib.sv_destroy(self._ctx)
            self._ctx = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    @property
    def handle(self):
        return self._ctx

    def _raise(self, st, where):
        raise SpecVerifyError(st, where, self.lib.sv_last_cuda_error(self._ctx).decode())

    # -- the verification ------------------------------------------------
    def verify(self, target, draft, tokens, draft_len, uniforms, temperature,
               out_tokens=None, out_len=None, stream=None):
        """Enqueue one verification on ``stream`` (default: current stream).

        target [B,k+1,V], draft [B,k,V] (dtype of the context), tokens [B,k]
        int32, draft_len [B] int32, uniforms [B,k+1] float32.  Returns
        (out_tokens [B,k+1] int32, out_len [B] int32), allocated if not given.
        """
        B, k1, V = target.shape
        k = k1 - 1
        dev = target.device
        _check_dev("target", target, self.dtype, (B, k + 1, self.V), dev)
        if draft is not None:
            _check_dev("draft", draft, self.dtype, (B, k, self.V), dev)
        if tokens is not None:
            _check_dev("tokens", tokens, torch.int32, (B, k), dev)
        _check_dev("draft_len", draft_len, torch.int32, (B,), dev)
        if uniforms is not None:
            _check_dev("uniforms", uniforms, torch.float32, (B, k + 1), dev)
        if out_tokens is None:
            out_tokens = torch.empty(B, k + 1, dtype=torch.int32, device=dev)
        if out_len is None:
            out_len = torch.empty(B, dtype=torch.int32, device=dev)
        _check_dev("out_tokens", out_tokens, torch.int32, (B, k + 1), dev)
        _check_dev("out_len", out_len, torch.int32, (B,), dev)
        st = self.lib.spec_verify(self._ctx, B, k, _ptr(target), _ptr(draft), _ptr(tokens),
                                  _ptr(draft_len), _ptr(uniforms), float(temperature),
                                  _ptr(out_tokens), _ptr(out_len), _stream_handle(stream))
        if st != SV_OK:
            self._raise(st, "spec_verify")
        return out_tokens, out_len

    def compact(self, out_tokens, out_len, packed=None, offsets=None, stream=None):
        """Packed token list and exclusive-scan offsets of a verification's outputs."""
        B, k1 = out_tokens.shape
        dev = out_tokens.device
        if packed is None:
            packed = torch.empty(B * k1, dtype=torch.int32, device=dev)
        if offsets is None:
            offsets = torch.empty(B + 1, dtype=torch.int32, device=dev)
        st = self.lib.spec_verify_compact(self._ctx, B, k1 - 1, _ptr(out_tokens), _ptr(out_len),
                                          _ptr(packed), _ptr(offsets), _stream_handle(stream))
        if st != SV_OK:
            self._raise(st, "spec_verify_compact")
        return packed, offsets

    def debug(self, B, k, stream=None):
        """Per-row diagnostics of the last call (float64 device tensors); the
        call must have run with ``set_diagnostics(True)``."""
        dev = self.device
        lse_t = torch.empty(B, k + 1, dtype=torch.float64, device=dev)
        lse_d = torch.empty(B, max(k, 1), dtype=torch.float64, device=dev)
        alpha = torch.empty(B, max(k, 1), dtype=torch.float64, device=dev)
        mass = torch.empty(B, k + 1, dtype=torch.float64, device=dev)
        st = self.lib.spec_verify_debug(self._ctx, B, k, _ptr(lse_t), _ptr(lse_d), _ptr(alpha),
                                        _ptr(mass), _stream_handle(stream))
        if st != SV_OK:
            self._raise(st, "spec_verify_debug")
        return {"lse_t": lse_t, "lse_d": lse_d[:, :k], "alpha": alpha[:, :k], "mass": mass}

    def stats(self, stream=None):
        """Synchronise and read the counters.  Returns (status, dict)."""
        s = Stats()
        st = self.lib.spec_verify_stats(self._ctx, _stream_handle(stream), ctypes.byref(s))
        if st == SV_ERR_CUDA:
            self._raise(st, "spec_verify_stats")
        return st, s.as_dict()

    def reset_stats(self, stream=None):
        st = self.lib.spec_verify_reset_stats(self._ctx, _stream_handle(stream))
        if st != SV_OK:
            self._raise(st, "spec_verify_reset_stats")

    def set_pipeline(self, stages: int, ctas_per_sm: int = 0):
        """Staging slots (64 KB each) per CTA and CTAs per SM (0 = as many as
        fit); (0, 0) = automatic."""
        st = self.lib.sv_set_pipeline(self._ctx, int(stages), int(ctas_per_sm))
        if st != SV_OK:
            self._raise(st, "sv_set_pipeline")

    def set_wait_limit_ns(self, ns: int):
        st = self.lib.sv_set_wait_limit_ns(self._ctx, int(ns))
        if st != SV_OK:
            self._raise(st, "sv_set_wait_limit_ns")

    def set_cluster(self, cluster: int):
        """CTAs that share each sequence, one vocabulary slice each (1, 2, 4
        or 8); 0 = chosen per call from the batch size."""
        st = self.lib.sv_set_cluster(self._ctx, int(cluster))
        if st != SV_OK:
            self._raise(st, "sv_set_cluster")

    def set_kernel(self, kernel: int):
        """SV_KERNEL_AUTO (default), SV_KERNEL_CLUSTER or SV_KERNEL_PIECES."""
        st = self.lib.sv_set_kernel(self._ctx, int(kernel))
        if st != SV_OK:
            self._raise(st, "sv_set_kernel")

    def set_timeline(self, buf):
        """Per-CTA timestamps of the following calls into ``buf`` (a uint64
        CUDA tensor of at least (grid CTAs + 1) * 8 words, or int64), or
        None to stop.  The caller keeps ``buf`` alive while it is set."""
        ptr = buf.data_ptr() if buf is not None else None
        st = self.lib.sv_set_timeline(self._ctx, ptr, buf.numel() if buf is not None else 0)
        if st != SV_OK:
            self._raise(st, "sv_set_timeline")

    def kernel_for(self, B: int) -> int:
        """The kernel a call with batch B runs on 16-byte aligned rows."""
        kern = ctypes.c_int()
        st = self.lib.sv_kernel_for(self._ctx, int(B), ctypes.byref(kern))
        if st != SV_OK:
            self._raise(st, "sv_kernel_for")
        return kern.value

    def set_early_exit(self, on: bool):
        """Skip the rows of a sequence after its first rejection once it is
        decided (same outputs; fewer bytes read; diagnostics of skipped rows
        stay NaN)."""
        st = self.lib.sv_set_early_exit(self._ctx, 1 if on else 0)
        if st != SV_OK:
            self._raise(st, "sv_set_early_exit")

    def set_diagnostics(self, on: bool):
        """Record the per-row diagnostics that ``debug`` returns (off by
        default: the stores cost the verify call time)."""
        st = self.lib.sv_set_diagnostics(self._ctx, 1 if on else 0)
        if st != SV_OK:
            self._raise(st, "sv_set_diagnostics")

    def config(self):
        vals = [ctypes.c_int() for _ in range(6)]
        st = self.lib.sv_get_config(self._ctx, *[ctypes.byref(v) for v in vals])
        if st != SV_OK:
            self._raise(st, "sv_get_config")
        return dict(zip(("stages", "ctas_per_sm", "threads", "smem_bytes", "grid_ctas", "cluster"),
                        (v.value for v in vals)))

    def launch_shape(self, B: int):
        """(cluster size, CTAs in the grid) of a call with batch B."""
        cs, ctas = ctypes.c_int(), ctypes.c_int()
        st = self.lib.sv_launch_shape(self._ctx, int(B), ctypes.byref(cs), ctypes.byref(ctas))
        if st != SV_OK:
            self._raise(st, "sv_launch_shape")
        return cs.value, ctas.value

    def rows_shape(self):
        """(threads, shared-memory bytes, CTAs) of row streaming's streaming
        kernels, or None if this context cannot run row streaming."""
        vals = [ctypes.c_int() for _ in range(3)]
        st = self.lib.sv_rows_shape(self._ctx, *[ctypes.byref(v) for v in vals])
        if st == SV_ERR_UNSUPPORTED:
            return None
        if st != SV_OK:
            self._raise(st, "sv_rows_shape")
        return tuple(v.value for v in vals)


def spec_verify_noalloc(target, draft, tokens, draft_len, uniforms, temperature, out_tokens, out_len,
                        stream=None):
    """Verification without a context, for callers that may not allocate
    device memory: the library keeps the workspace in a fixed array of its
    own (limits: B <= 4096, k <= 31, B * (k+1) <= 16384).  The output buffers
    must be supplied.  Calls that may overlap on the GPU share that array and
    must be ordered on one stream.  Raises SpecVerifyError on a bad argument.
    """
    lib = load_library()
    B, k1, V = target.shape
    k = k1 - 1
    dev = target.device
    dtype = target.dtype
    if dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be float32 or bfloat16")
    _check_dev("target", target, dtype, (B, k + 1, V), dev)
    if draft is not None:
        _check_dev("draft", draft, dtype, (B, k, V), dev)
    if tokens is not None:
        _check_dev("tokens", tokens, torch.int32, (B, k), dev)
    _check_dev("draft_len", draft_len, torch.int32, (B,), dev)
    if uniforms is not None:
        _check_dev("uniforms", uniforms, torch.float32, (B, k + 1), dev)
    _check_dev("out_tokens", out_tokens, torch.int32, (B, k + 1), dev)
    _check_dev("out_len", out_len, torch.int32, (B,), dev)
    st = lib.spec_verify_noalloc(B, k, V, SV_F32 if dtype == torch.float32 else SV_BF16, _ptr(target),
                                 _ptr(draft), _ptr(tokens), _ptr(draft_len), _ptr(uniforms),
                                 float(temperature), _ptr(out_tokens), _ptr(out_len), _stream_handle(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_noalloc")
    return out_tokens, out_len


def kd_loss(target, draft, weights, temperature=1.0, grad=True, stream=None):
    """Reward-weighted distillation loss of the draft and its gradient in the
    draft logits (see ``spec_kd_loss`` in include/specverify.h).  target,
    draft: [n_seq, t_len, V] float32 or bfloat16 on the GPU; weights: [n_seq]
    float32 (w(r) per rollout).  Returns (row_kl [n_seq, t_len] float32,
    loss [n_seq] float32, grad [n_seq, t_len, V] in the logits' dtype or
    None)."""
    lib = load_library()
    n_seq, t_len, V = target.shape
    dtype = target.dtype
    if dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be float32 or bfloat16")
    dev = target.device
    _check_dev("target", target, dtype, (n_seq, t_len, V), dev)
    _check_dev("draft", draft, dtype, (n_seq, t_len, V), dev)
    _check_dev("weights", weights, torch.float32, (n_seq,), dev)
    row_kl = torch.empty((n_seq, t_len), dtype=torch.float32, device=dev)
    loss = torch.empty((n_seq,), dtype=torch.float32, device=dev)
    g = torch.empty((n_seq, t_len, V), dtype=dtype, device=dev) if grad else None
    st = lib.spec_kd_loss(n_seq, t_len, V, SV_BF16 if dtype == torch.bfloat16 else SV_F32,
                          target.data_ptr(), draft.data_ptr(), weights.data_ptr(), float(temperature),
                          row_kl.data_ptr(), loss.data_ptr(), g.data_ptr() if g is not None else None,
                          _stream_handle(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_kd_loss")
    return row_kl, loss, g


def measure_ex2(iters=4096):
    """(ex2 per SM per clock, ex2 per second) of the special-function unit on
    the current device (sv_measure_ex2)."""
    lib = load_library()
    per_clk, per_s = ctypes.c_double(), ctypes.c_double()
    st = lib.sv_measure_ex2(int(iters), ctypes.byref(per_clk), ctypes.byref(per_s))
    if st != SV_OK:
        raise SpecVerifyError(st, "sv_measure_ex2")
    return per_clk.value, per_s.value


def kd_launch_shape(V, dtype=torch.bfloat16, grad=True):
    """(CTAs per cluster, row buffers per CTA, grid CTAs) of ``kd_loss`` for
    rows of V logits."""
    lib = load_library()
    cs, nb, ctas = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    st = lib.spec_kd_launch_shape(int(V), SV_BF16 if dtype == torch.bfloat16 else SV_F32, int(bool(grad)),
                                  ctypes.byref(cs), ctypes.byref(nb), ctypes.byref(ctas))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_kd_launch_shape")
    return cs.value, nb.value, ctas.value


class DraftController:
    """Draft-length controller and speculation toggle (``spec_ctrl_*`` in
    include/specverify.h): per-slot acceptance state on the device, a
    profiled round-time table, and the choice of the next round's draft
    lengths.  ``n_slots`` sequence slots, draft lengths 0..``max_k``."""

    def __init__(self, n_slots: int, max_k: int, device=None):
        self.lib = load_library()
        self.n_slots, self.max_k = int(n_slots), int(max_k)
        self.device = torch.device("cuda", torch.cuda.current_device() if device is None else
                                   torch.device(device).index or 0)
        self._c = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            st = self.lib.spec_ctrl_create(ctypes.byref(self._c), self.n_slots, self.max_k)
        if st != SV_OK:
            raise SpecVerifyError(st, "spec_ctrl_create")

    def close(self):
        if self._c:
            self.lib.spec_ctrl_destroy(self._c)
            self._c = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _ok(self, st, where):
        if st != SV_OK:
            raise SpecVerifyError(st, where)

    def set_cost(self, batch_sizes, round_time):
        """batch_sizes [P] increasing; round_time [P, max_k + 1] (host)."""
        import numpy as np
        bs = np.ascontiguousarray(batch_sizes, dtype=np.int32).reshape(-1)
        t = np.ascontiguousarray(round_time, dtype=np.float64).reshape(bs.size, self.max_k + 1)
        self._ok(self.lib.spec_ctrl_set_cost(self._c, bs.size, bs.ctypes.data_as(ctypes.c_void_p),
                                             t.ctypes.data_as(ctypes.c_void_p)), "spec_ctrl_set_cost")

    def set_params(self, decay=0.9, prior_alpha=0.5, prior_weight=2.0, mode=SV_CTRL_BATCH):
        self._ok(self.lib.spec_ctrl_set_params(self._c, float(decay), float(prior_alpha), float(prior_weight),
                                               int(mode)), "spec_ctrl_set_params")

    def _ids(self, seq_ids):
        _check_dev("seq_ids", seq_ids, torch.int32, (seq_ids.numel(),), self.device)
        return seq_ids.numel()

    def reset(self, seq_ids=None, stream=None):
        n = 0 if seq_ids is None else self._ids(seq_ids)
        self._ok(self.lib.spec_ctrl_reset(self._c, n, _ptr(seq_ids), _stream_handle(stream)), "spec_ctrl_reset")

    def observe(self, seq_ids, draft_len, out_len, stream=None):
        B = self._ids(seq_ids)
        _check_dev("draft_len", draft_len, torch.int32, (B,), self.device)
        _check_dev("out_len", out_len, torch.int32, (B,), self.device)
        self._ok(self.lib.spec_ctrl_observe(self._c, B, _ptr(seq_ids), _ptr(draft_len), _ptr(out_len),
                                            _stream_handle(stream)), "spec_ctrl_observe")

    def choose(self, seq_ids, next_draft_len=None, choice=None, stream=None):
        """Returns (next_draft_len [B] int32, choice [1] int32) on the device."""
        B = self._ids(seq_ids)
        if next_draft_len is None:
            next_draft_len = torch.empty(B, dtype=torch.int32, device=self.device)
        if choice is None:
            choice = torch.empty(1, dtype=torch.int32, device=self.device)
        _check_dev("next_draft_len", next_draft_len, torch.int32, (B,), self.device)
        _check_dev("choice", choice, torch.int32, (1,), self.device)
        self._ok(self.lib.spec_ctrl_choose(self._c, B, _ptr(seq_ids), _ptr(next_draft_len), _ptr(choice),
                                           _stream_handle(stream)), "spec_ctrl_choose")
        return next_draft_len, choice

    def alpha(self, seq_ids, stream=None):
        B = self._ids(seq_ids)
        out = torch.empty(B, dtype=torch.float64, device=self.device)
        self._ok(self.lib.spec_ctrl_alpha(self._c, B, _ptr(seq_ids), _ptr(out), _stream_handle(stream)),
                 "spec_ctrl_alpha")
        return out

    def status(self, stream=None):
        """The sticky device error (SV_OK, SV_ERR_INVALID_ARG or
        SV_ERR_BAD_DRAFT_LEN); synchronises the stream."""
        return self.lib.spec_ctrl_status(self._c, _stream_handle(stream))


SV_TREE_MAX_NODES = 64


def verify_tree(target, draft, parents, tokens, n_nodes, uniforms, temperature, out_tokens=None, out_nodes=None,
                out_len=None, status=None, alpha=None, stream=None):
    """Tree verification (``spec_verify_tree`` in include/specverify.h).

    target, draft [B, M, V] (float32 or bfloat16), parents, tokens [B, M]
    int32, n_nodes [B] int32, uniforms [B, M] float32 (column 0 samples).
    Returns (out_tokens [B, M], out_nodes [B, M], out_len [B], status [B])
    int32 and, if given, fills alpha [B, M] float32."""
    lib = load_library()
    B, M, V = target.shape
    dtype = target.dtype
    if dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("logits must be float32 or bfloat16")
    dev = target.device
    _check_dev("target", target, dtype, (B, M, V), dev)
    _check_dev("draft", draft, dtype, (B, M, V), dev)
    _check_dev("parents", parents, torch.int32, (B, M), dev)
    _check_dev("tokens", tokens, torch.int32, (B, M), dev)
    _check_dev("n_nodes", n_nodes, torch.int32, (B,), dev)
    _check_dev("uniforms", uniforms, torch.float32, (B, M), dev)
    mk = lambda t, shape: t if t is not None else torch.empty(shape, dtype=torch.int32, device=dev)
    out_tokens, out_nodes = mk(out_tokens, (B, M)), mk(out_nodes, (B, M))
    out_len, status = mk(out_len, (B,)), mk(status, (B,))
    for name, t, shape in (("out_tokens", out_tokens, (B, M)), ("out_nodes", out_nodes, (B, M)),
                           ("out_len", out_len, (B,)), ("status", status, (B,))):
        _check_dev(name, t, torch.int32, shape, dev)
    if alpha is not None:
        _check_dev("alpha", alpha, torch.float32, (B, M), dev)
    st = lib.spec_verify_tree(B, M, V, SV_BF16 if dtype == torch.bfloat16 else SV_F32, _ptr(target), _ptr(draft),
                              _ptr(parents), _ptr(tokens), _ptr(n_nodes), _ptr(uniforms), float(temperature),
                              _ptr(out_tokens), _ptr(out_nodes), _ptr(out_len), _ptr(status), _ptr(alpha),
                              _stream_handle(stream))
    if st != SV_OK:
        raise SpecVerifyError(st, "spec_verify_tree")
    return out_tokens, out_nodes, out_len, status
