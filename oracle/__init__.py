"""ctypes wrapper around the fp64 C oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__``'s
smoke check and by the CPU-baseline leg of ``bench.py``.  The library in
``speculative_decoding_verification_71_gb300`` never imports this package,
and this package never imports the library.

``build()`` compiles ``oracle.c`` with gcc (-O2, no fast-math, no contraction of
a multiply and an add into one rounding, OpenMP) into
``liboracle.so`` beside it.  ``verify(...)`` takes numpy arrays or CPU torch
tensors with the same layout as the library's entry point and returns the
outputs plus the diagnostics the parity tests use.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

STATUS_OK = 0
STATUS_BAD_DRAFT_LEN = 2
STATUS_BAD_TOKEN = 3
STATUS_NONFINITE = 4
FLAG_ZERO_RESIDUAL = 256


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH, extra=()) -> str:
    """Compile the oracle (or, for mutation tests, another source file)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-Wall", *extra, src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def _bind(lib):
    c = ctypes
    P = c.c_void_p
    lib.oracle_verify.restype = c.c_int
    lib.oracle_verify.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int, P, P, P, P, P, c.c_double,
                                  P, P, P, P, P, P, P, P, P, P, c.c_double, P, P, P, c.c_int]
    lib.oracle_row_lse.restype = c.c_double
    lib.oracle_row_lse.argtypes = [c.c_int, c.c_int, P, c.c_double]
    lib.oracle_row_probs.restype = None
    lib.oracle_row_probs.argtypes = [c.c_int, c.c_int, P, c.c_double, P]
    lib.oracle_logit_value.restype = c.c_double
    lib.oracle_logit_value.argtypes = [P, c.c_int, c.c_longlong]
    lib.oracle_num_threads.restype = c.c_int
    lib.oracle_kd.restype = c.c_int
    lib.oracle_kd.argtypes = [c.c_int, c.c_int, c.c_int, c.c_int, P, P, P, c.c_double, P, P, P, P, c.c_int]
    D, I = c.c_double, c.c_int
    lib.oracle_ctrl_observe.restype = I
    lib.oracle_ctrl_observe.argtypes = [I, P, P, I, P, P, P, I, D, P]
    lib.oracle_ctrl_alpha.restype = D
    lib.oracle_ctrl_alpha.argtypes = [D, D, D, D]
    lib.oracle_ctrl_expected_tokens.restype = D
    lib.oracle_ctrl_expected_tokens.argtypes = [D, I]
    lib.oracle_ctrl_round_time.restype = D
    lib.oracle_ctrl_round_time.argtypes = [I, P, P, I, I, I]
    lib.oracle_ctrl_choose.restype = I
    lib.oracle_ctrl_choose.argtypes = [I, P, P, I, P, I, D, D, I, I, P, P, P, P, P, P, P]
    lib.oracle_tree_verify.restype = I
    lib.oracle_tree_verify.argtypes = [I, I, I, I, P, P, P, P, P, P, D, P, P, P, P, P, P, P, P, D, P, P, P, I]
    return lib


def load(path: str | None = None):
    """Load (building if needed) the oracle library.  ``path`` loads another
    build, e.g. a mutant compiled by the tests."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _as_np(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu()
            if x.dtype == torch.bfloat16:
                return x.contiguous().view(torch.int16).numpy().view(np.uint16), 1
            return x.contiguous().numpy(), (0 if x.dtype == torch.float32 else None)
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, 0
    if x.dtype == np.uint16:  # raw bf16 bits
        return x, 1
    return x, None


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


TIE_BAND = 1e-5


def verify(target, draft, tokens, draft_len, uniforms, T, nthreads=0, lib=None, tie_band=TIE_BAND):
    """Run the oracle on one batch.

    target [B,k+1,V] and draft [B,k,V]: float32 arrays, uint16 arrays of
    bf16 bits, or CPU/GPU torch tensors (fp32 or bf16).  Returns a dict with
    out_tokens, out_len, status and the fp64 diagnostics; sample_lo and
    sample_hi bound the tokens a draw could give with its uniform moved by at
    most ``tie_band`` (in units of the normalised CDF).
    """
    lib = lib or load()
    t, dt = _as_np(target)
    d, dd = _as_np(draft)
    if dt is None or dt != dd:
        raise TypeError("target and draft must both be float32 or both be bfloat16")
    B, k1, V = t.shape
    k = k1 - 1
    if d.shape != (B, k, V) and not (k == 0 and d.size == 0):
        raise ValueError(f"draft shape {d.shape} != {(B, k, V)}")
    tok = np.ascontiguousarray(_as_np(tokens)[0], dtype=np.int32).reshape(B, max(k, 0))
    kl = np.ascontiguousarray(_as_np(draft_len)[0], dtype=np.int32).reshape(B)
    u = np.ascontiguousarray(_as_np(uniforms)[0], dtype=np.float32).reshape(B, k + 1)
    if not (T >= 0.0) or not np.isfinite(T):
        raise ValueError("temperature must be finite and >= 0")
    out_tokens = np.empty((B, k + 1), np.int32)
    out_len = np.empty(B, np.int32)
    lse_t = np.empty((B, k + 1))
    lse_d = np.empty((B, max(k, 1)))
    p_x = np.empty((B, max(k, 1)))
    q_x = np.empty((B, max(k, 1)))
    alpha = np.empty((B, max(k, 1)))
    mass = np.empty(B)
    atie = np.empty(B)
    stie = np.empty(B)
    slo = np.empty(B, np.int32)
    shi = np.empty(B, np.int32)
    status = np.empty(B, np.int32)
    d_arr = d if d.size else np.zeros(1, t.dtype)
    lib.oracle_verify(B, k, V, dt, _ptr(t), _ptr(d_arr), _ptr(tok), _ptr(kl), _ptr(u), float(T),
                      _ptr(out_tokens), _ptr(out_len), _ptr(lse_t), _ptr(lse_d), _ptr(p_x),
                      _ptr(q_x), _ptr(alpha), _ptr(mass), _ptr(atie), _ptr(stie), float(tie_band),
                      _ptr(slo), _ptr(shi), _ptr(status), int(nthreads))
    return {
        "out_tokens": out_tokens, "out_len": out_len, "status": status,
        "lse_t": lse_t, "lse_d": lse_d[:, :k], "p_x": p_x[:, :k], "q_x": q_x[:, :k],
        "alpha": alpha[:, :k], "resid_mass": mass, "accept_tie": atie, "sample_tie": stie,
        "sample_lo": slo, "sample_hi": shi, "tie_band": float(tie_band),
    }


def row_lse(row, T, lib=None):
    lib = lib or load()
    r, dt = _as_np(row)
    return lib.oracle_row_lse(r.size, dt, _ptr(r), float(T))


def row_probs(row, T, lib=None):
    lib = lib or load()
    r, dt = _as_np(row)
    p = np.empty(r.size)
    lib.oracle_row_probs(r.size, dt, _ptr(r), float(T), _ptr(p))
    return p


def logit_values(arr, lib=None):
    lib = lib or load()
    a, dt = _as_np(arr)
    flat = a.reshape(-1)
    return np.array([lib.oracle_logit_value(_ptr(flat), dt, i) for i in range(flat.size)])


def num_threads(lib=None):
    return (lib or load()).oracle_num_threads()


def kd(target, draft, weights, T=1.0, grad=True, nthreads=0, lib=None):
    """Reward-weighted distillation loss of the draft (see ``oracle_kd`` in
    oracle.c).  target, draft: [n_seq, t_len, V] fp32 or bf16; weights:
    [n_seq] (w(r) per rollout).  Returns row_kl [n_seq, t_len], loss [n_seq],
    grad [n_seq, t_len, V] (float64, or None) and status [n_seq, t_len]."""
    lib = lib or load()
    t, dt = _as_np(target)
    d, dd = _as_np(draft)
    if dt is None or dd != dt:
        raise TypeError("target and draft must both be float32 or both bfloat16")
    n_seq, t_len, V = t.shape
    t = np.ascontiguousarray(t)
    d = np.ascontiguousarray(d)
    w = np.ascontiguousarray(np.asarray(weights, dtype=np.float64).reshape(n_seq))
    row_kl = np.empty((n_seq, t_len), np.float64)
    loss = np.empty(n_seq, np.float64)
    g = np.empty((n_seq, t_len, V), np.float64) if grad else None
    status = np.empty((n_seq, t_len), np.int32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p) if a is not None else None
    rc = lib.oracle_kd(n_seq, t_len, V, dt, ptr(t), ptr(d), ptr(w), float(T), ptr(row_kl), ptr(loss),
                       ptr(g), ptr(status), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle_kd failed ({rc})")
    return {"row_kl": row_kl, "loss": loss, "grad": g, "status": status}


CTRL_USED, CTRL_SKIPPED, CTRL_BAD_LEN, CTRL_BAD_ID = 0, 1, 2, 5


class Controller:
    """The draft-length controller of ``oracle_ctrl_*`` in oracle.c: decayed
    acceptance counts per sequence slot and the round-time table.  Mirrors
    the library's controller call for call (observe, choose, alpha)."""

    def __init__(self, n_slots, max_k, batch_sizes, table, decay=0.9, prior_alpha=0.5,
                 prior_weight=2.0, mode=0, lib=None):
        self.lib = lib or load()
        self.n_slots, self.max_k = int(n_slots), int(max_k)
        self.A = np.zeros(self.n_slots)
        self.N = np.zeros(self.n_slots)
        self.set_cost(batch_sizes, table)
        self.decay, self.prior_alpha, self.prior_weight, self.mode = float(decay), float(prior_alpha), \
            float(prior_weight), int(mode)

    def set_cost(self, batch_sizes, table):
        self.batch_sizes = np.ascontiguousarray(batch_sizes, dtype=np.int32).reshape(-1)
        self.table = np.ascontiguousarray(table, dtype=np.float64).reshape(self.batch_sizes.size, self.max_k + 1)

    def reset(self, seq_ids=None):
        if seq_ids is None:
            self.A[:] = 0.0
            self.N[:] = 0.0
        else:
            self.A[np.asarray(seq_ids)] = 0.0
            self.N[np.asarray(seq_ids)] = 0.0

    def observe(self, seq_ids, draft_len, out_len):
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        k = np.ascontiguousarray(draft_len, dtype=np.int32)
        n = np.ascontiguousarray(out_len, dtype=np.int32)
        st = np.empty(ids.size, np.int32)
        self.lib.oracle_ctrl_observe(self.n_slots, _ptr(self.A), _ptr(self.N), ids.size, _ptr(ids), _ptr(k),
                                     _ptr(n), self.max_k, self.decay, _ptr(st))
        return st

    def alpha(self, seq_ids):
        return np.array([self.lib.oracle_ctrl_alpha(self.A[i], self.N[i], self.prior_alpha, self.prior_weight)
                         for i in np.asarray(seq_ids)])

    def round_time(self, B, n):
        return self.lib.oracle_ctrl_round_time(self.batch_sizes.size, _ptr(self.batch_sizes), _ptr(self.table),
                                               self.max_k, int(B), int(n))

    def choose(self, seq_ids):
        """Returns next_len [B], choice, rates [max_k+1] (batch mode), margin
        ([1] batch mode, [B] per sequence) and the row status."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int32)
        B = ids.size
        nxt = np.empty(B, np.int32)
        choice = np.zeros(1, np.int32)
        rates = np.zeros(self.max_k + 1)
        margin = np.zeros(max(B, 1))
        st = np.empty(B, np.int32)
        rc = self.lib.oracle_ctrl_choose(self.n_slots, _ptr(self.A), _ptr(self.N), B, _ptr(ids), self.max_k,
                                         self.prior_alpha, self.prior_weight, self.mode, self.batch_sizes.size,
                                         _ptr(self.batch_sizes), _ptr(self.table), _ptr(nxt), _ptr(choice),
                                         _ptr(rates), _ptr(margin), _ptr(st))
        if rc != 0:
            raise ValueError(f"oracle_ctrl_choose failed ({rc})")
        return {"next_len": nxt, "choice": int(choice[0]), "rates": rates,
                "margin": margin[:1] if self.mode == 0 else margin[:B], "status": st}


def expected_tokens(alpha, n, lib=None):
    return (lib or load()).oracle_ctrl_expected_tokens(float(alpha), int(n))


def tree_verify(target, draft, parents, tokens, n_nodes, uniforms, T, final_w=False, nthreads=0, lib=None,
                tie_band=TIE_BAND):
    """Tree verification (see ``oracle_tree_verify`` in oracle.c).

    target, draft [B,M,V] (fp32 / bf16 as for ``verify``), parents, tokens
    [B,M] int32, n_nodes [B], uniforms [B,M] float32 (column 0 samples).
    Returns out_tokens, out_nodes [B,M], out_len [B], status and the fp64
    diagnostics (alpha [B,M], resid_mass, accept_tie, sample_tie; final_w
    [B,V] if asked for)."""
    lib = lib or load()
    t, dt = _as_np(target)
    d, dd = _as_np(draft)
    if dt is None or dt != dd:
        raise TypeError("target and draft must both be float32 or both be bfloat16")
    B, M, V = t.shape
    t, d = np.ascontiguousarray(t), np.ascontiguousarray(d)
    par = np.ascontiguousarray(_as_np(parents)[0], dtype=np.int32).reshape(B, M)
    tok = np.ascontiguousarray(_as_np(tokens)[0], dtype=np.int32).reshape(B, M)
    nn = np.ascontiguousarray(_as_np(n_nodes)[0], dtype=np.int32).reshape(B)
    u = np.ascontiguousarray(_as_np(uniforms)[0], dtype=np.float32).reshape(B, M)
    out_tokens = np.empty((B, M), np.int32)
    out_nodes = np.empty((B, M), np.int32)
    out_len = np.empty(B, np.int32)
    alpha = np.empty((B, M))
    fw = np.empty((B, V)) if final_w else None
    mass, atie, stie = np.empty(B), np.empty(B), np.empty(B)
    slo, shi = np.empty(B, np.int32), np.empty(B, np.int32)
    status = np.empty(B, np.int32)
    lib.oracle_tree_verify(B, M, V, dt, _ptr(t), _ptr(d), _ptr(par), _ptr(tok), _ptr(nn), _ptr(u), float(T),
                           _ptr(out_tokens), _ptr(out_nodes), _ptr(out_len), _ptr(alpha), _ptr(fw), _ptr(mass),
                           _ptr(atie), _ptr(stie), float(tie_band), _ptr(slo), _ptr(shi), _ptr(status),
                           int(nthreads))
    return {"out_tokens": out_tokens, "out_nodes": out_nodes, "out_len": out_len, "status": status,
            "alpha": alpha, "final_w": fw, "resid_mass": mass, "accept_tie": atie, "sample_tie": stie,
            "sample_lo": slo, "sample_hi": shi, "tie_band": float(tie_band)}
