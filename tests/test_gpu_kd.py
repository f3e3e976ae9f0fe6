"""Parity of the distillation-loss kernel (through the C ABI) with the fp64 oracle.

Tolerances, from the arithmetic: every exponential is ex2.approx and the
log-sums lg2.approx (relative error ~2^-22), summed in fp32 over the row.
  * KL = ln2 (c A / S^t - (K^t - K^d) - log2(S^t / S^d)): the error grows with
    the weighted mean |z^t - z^d| / T that A carries, so
    |dKL| <= 1e-5 (1 + E_p|z^t - z^d| / T) + 1e-6;
  * fp32 gradient w (q - p) / T: p and q carry ~1e-6 relative error each
    (ex2.approx, the rounding of z c - K), and the kernel's c = fl(log2 e / T)
    moves log p(x) by up to 6e-8 |z(x) - E_p z| / T (a few 1e-6 for tokens far
    below the mean); q - p may cancel, so |dg| <= 1e-5 w / T (p + q) + 1e-30;
  * bf16 gradient: the oracle's value rounded to nearest-even bf16, give or
    take one bf16 step of its magnitude plus the fp32 error above (the fp32
    value may sit on the other side of a rounding boundary).
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
import speculative_decoding_verification_71_gb300 as svp
from speculative_decoding_verification_71_gb300 import build as svbuild

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    svbuild.build()
    svp.load_library()


def make(n_seq, t_len, V, dtype, seed=0, scale=3.0, noise=0.7, peaks=True):
    g = torch.Generator(device="cpu").manual_seed(seed)
    t = torch.randn(n_seq, t_len, V, generator=g) * scale
    if peaks:
        idx = torch.randint(0, V, (n_seq, t_len, min(20, V)), generator=g)
        t.scatter_add_(2, idx, torch.full(idx.shape, 8.0))
    d = t + torch.randn(n_seq, t_len, V, generator=g) * noise
    w = torch.rand(n_seq, generator=g) * 2.0
    return t.to(dtype), d.to(dtype), w


def kl_tolerance(t, d, T):
    tt = t.double().numpy() / T
    dd = d.double().numpy() / T
    p = softmax(tt, axis=2)
    finite = np.isfinite(tt) & np.isfinite(dd)
    spread = np.where(finite & (p > 0), p * np.abs(np.where(finite, tt - dd, 0.0)), 0.0).sum(axis=2)
    return 1e-5 * (1.0 + spread) + 1e-6


def check(t, d, w, T, grad=True):
    tg, dg, wg = t.to(DEV), d.to(DEV), w.to(DEV).float()
    row_kl, loss, g = svp.kd_loss(tg, dg, wg, T, grad=grad)
    torch.cuda.synchronize()
    ref = oracle.kd(t, d, w.double().numpy(), T, grad=grad)
    kl = row_kl.cpu().double().numpy()
    ok = np.isfinite(ref["row_kl"])
    tol = kl_tolerance(t, d, T)
    assert np.array_equal(np.isnan(kl), np.isnan(ref["row_kl"])), "invalid rows differ"
    assert np.array_equal(np.isinf(kl), np.isinf(ref["row_kl"])), "infinite rows differ"
    err = np.abs(kl[ok] - ref["row_kl"][ok])
    assert (err <= tol[ok]).all(), (err.max(), tol[ok][np.argmax(err / tol[ok])])
    lref = ref["loss"]
    lg = loss.cpu().double().numpy()
    fin = np.isfinite(lref)
    ltol = w.double().numpy() * np.where(ok, tol, 0).sum(axis=1) + 1e-6
    assert (np.abs(lg[fin] - lref[fin]) <= ltol[fin]).all()
    assert np.array_equal(~np.isfinite(lg), ~fin)
    if grad:
        gg = g.cpu()
        gr = ref["grad"]
        ok = ~np.isnan(ref["row_kl"])          # KL = +inf rows have a finite gradient
        if t.dtype == torch.float32:
            p = softmax(t.double().numpy() / T, axis=2)
            q = softmax(d.double().numpy() / T, axis=2)
            gtol = 1e-5 * (w.double().numpy()[:, None, None] / T) * (p + q) + 1e-30
            diff = np.abs(gg.double().numpy() - gr)
            rows_ok = ok[:, :, None] & np.ones_like(diff, bool)
            assert (diff[rows_ok] <= gtol[rows_ok]).all(), diff[rows_ok].max()
        else:
            want = torch.from_numpy(gr).to(torch.bfloat16).double().numpy()
            got = gg.double().numpy()
            p = softmax(t.double().numpy() / T, axis=2)
            q = softmax(d.double().numpy() / T, axis=2)
            step = np.abs(want) * 2.0 ** -7 + 1e-5 * (w.double().numpy()[:, None, None] / T) * (p + q) + 1e-37
            rows_ok = np.broadcast_to(ok[:, :, None], got.shape)
            assert (np.abs(got - want)[rows_ok] <= step[rows_ok]).all()
        assert np.isnan(gg.double().numpy()[~ok]).all()
    return row_kl, loss, g


CASES = [
    (2, 3, 1000, torch.float32, 1.0),      # one CTA per row
    (3, 4, 4099, torch.float32, 0.8),      # unaligned rows: plain loads
    (2, 5, 20000, torch.bfloat16, 1.0),    # rows of 40 KB: clusters of two
    (2, 3, 40000, torch.bfloat16, 1.0),    # clusters of four
    (2, 3, 80000, torch.bfloat16, 0.9),    # clusters of eight
    (1, 3, 1001, torch.bfloat16, 1.3),     # unaligned bf16
    (2, 2, 151936, torch.bfloat16, 1.0),   # Qwen vocabulary: clusters of sixteen
    (2, 2, 65536, torch.float32, 0.6),     # fp32 rows of 256 KB
    (1, 2, 151936, torch.float32, 1.0),    # fp32 rows of 594 KB
]


@pytest.mark.parametrize("n_seq,t_len,V,dtype,T", CASES, ids=[f"{c[0]}x{c[1]}x{c[2]}-{str(c[3])[6:]}-T{c[4]}" for c in CASES])
def test_kd_matches_the_oracle(n_seq, t_len, V, dtype, T):
    t, d, w = make(n_seq, t_len, V, dtype, seed=V)
    check(t, d, w, T)


def test_loss_only_equals_loss_with_gradient():
    t, d, w = make(3, 4, 20000, torch.bfloat16, seed=3)
    kl1, l1, _ = svp.kd_loss(t.to(DEV), d.to(DEV), w.to(DEV), 1.0, grad=True)
    kl2, l2, g2 = svp.kd_loss(t.to(DEV), d.to(DEV), w.to(DEV), 1.0, grad=False)
    assert g2 is None
    torch.testing.assert_close(kl1, kl2, rtol=0, atol=0)
    torch.testing.assert_close(l1, l2, rtol=0, atol=0)
    check(t, d, w, 1.0, grad=False)


def test_masked_invalid_and_zero_weight_rows():
    t, d, w = make(4, 3, 5000, torch.float32, seed=4)
    t[0, 0, :100] = -float("inf")            # masked target tokens: fine
    d[0, 1, 7] = -float("inf")               # q = 0 where p > 0: KL = +inf
    t[1, 2, 9] = float("nan")                # invalid row
    d[2, 0, :] = -float("inf")               # all -inf draft row: invalid
    w[3] = 0.0                               # zero weight: zero gradient
    _, _, g = check(t, d, w, 1.0)
    assert (g[3] == 0).all()


def test_identical_rows_give_zero():
    t, _, w = make(2, 3, 30000, torch.bfloat16, seed=5)
    kl, loss, g = svp.kd_loss(t.to(DEV), t.to(DEV), w.to(DEV), 1.0)
    assert kl.abs().max().item() < 2e-6
    assert g.float().abs().max().item() < 1e-6


def test_repeated_calls_are_bitwise_identical():
    t, d, w = make(4, 8, 40000, torch.bfloat16, seed=6)
    a = svp.kd_loss(t.to(DEV), d.to(DEV), w.to(DEV), 1.0)
    for _ in range(5):
        b = svp.kd_loss(t.to(DEV), d.to(DEV), w.to(DEV), 1.0)
        for x, y in zip(a, b):
            assert torch.equal(x, y)


def test_full_size_batch_on_sampled_rollouts():
    # 64 rollouts x 64 positions of the Qwen vocabulary; the oracle checks two
    # rollouts, every row of the batch is checked for finiteness and sign
    n_seq, t_len, V = 64, 64, 151936
    g = torch.Generator(device=DEV).manual_seed(7)
    t = torch.randn(n_seq, t_len, V, generator=g, device=DEV) * 3.0
    d = (t + torch.randn(n_seq, t_len, V, generator=g, device=DEV) * 0.7).to(torch.bfloat16)
    t = t.to(torch.bfloat16)
    w = torch.rand(n_seq, generator=g, device=DEV)
    kl, loss, grad = svp.kd_loss(t, d, w, 1.0)
    torch.cuda.synchronize()
    assert torch.isfinite(kl).all() and (kl > 0).all()
    for b in (0, 37):
        check(t[b:b + 1].cpu(), d[b:b + 1].cpu(), w[b:b + 1].cpu(), 1.0)
        torch.testing.assert_close(kl[b:b + 1], svp.kd_loss(t[b:b + 1].contiguous(), d[b:b + 1].contiguous(),
                                                            w[b:b + 1].contiguous(), 1.0)[0], rtol=0, atol=0)
