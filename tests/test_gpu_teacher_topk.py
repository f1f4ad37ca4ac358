"""The teacher-side top-K cache producer (kd_teacher_topk) through the C ABI
against the fp64 oracle.

The selected indices are an integer decision taken on the kernel's fp32
logits, so: (1) the returned logits match the fp64 logits at the returned
indices; (2) the returned list is a valid top-K of the fp64 logits up to that
rounding (nothing left out is larger than the smallest kept by more than the
tolerance); (3) away from near-ties the index list equals the oracle's exactly.
Integer-valued inputs make every logit exact in fp32 as well as fp64, so there
the output must equal the oracle bit for bit, ties included."""

import math

import numpy as np
import pytest
import torch

import chunked_top_kl_logit_b300 as kd
from oracle import kd_residual_oracle as RO
from oracle import teacher_topk_oracle as TK
from tests.gpu_util import LSE_ATOL

pytestmark = pytest.mark.gpu

Z_ATOL = 1e-4


def run_producer(h, W, K, tau, chunk):
    dev = torch.device("cuda")
    T, d = h.shape
    V = W.shape[0]
    ws = torch.empty(kd.kd_teacher_topk_workspace_size(T, V, d, K, chunk), dtype=torch.uint8,
                     device=dev)
    idx = torch.full((T, K), -1, dtype=torch.int32, device=dev)
    val = torch.full((T, K), float("nan"), dtype=torch.float32, device=dev)
    lse = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    st = torch.full((1,), -1, dtype=torch.int32, device=dev)
    kd.kd_teacher_topk(h.to(dev).contiguous(), W.to(dev).contiguous(), K, tau, chunk, idx, val,
                       lse, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, kd.status_string(int(st.item()))
    return idx.cpu().numpy().astype(np.int64), val.double().cpu().numpy(), lse.double().cpu().numpy()


def check_against_oracle(h, W, K, tau, chunk):
    gi, gv, gl = run_producer(h, W, K, tau, chunk)
    h64, W64 = h.double().numpy(), W.double().numpy()
    oi, ov, ol = TK.teacher_topk(h64, W64, K, tau)
    z = h64 @ W64.T
    rows = np.arange(h.shape[0])[:, None]
    assert np.abs(gl - ol).max() <= LSE_ATOL
    # (1) values at the returned indices
    assert np.abs(gv - z[rows, gi]).max() <= Z_ATOL
    # descending, indices distinct and in range
    assert np.all(np.diff(gv, axis=1) <= 0)
    assert np.all((gi >= 0) & (gi < W.shape[0]))
    assert all(len(set(r)) == K for r in gi)
    # (2) valid top-K of the fp64 logits
    kept_min = z[rows, gi].min(axis=1)
    zz = z.copy()
    zz[rows, gi] = -np.inf
    assert np.all(zz.max(axis=1) <= kept_min + 2 * Z_ATOL)
    # (3) exact where the K-th and (K+1)-th fp64 logits are apart
    srt = -np.sort(-z, axis=1)
    gap = srt[:, K - 1] - srt[:, K] if z.shape[1] > K else np.full(z.shape[0], np.inf)
    clear = gap > 4 * Z_ATOL
    assert clear.mean() > 0.5
    np.testing.assert_array_equal(np.sort(gi[clear], axis=1), np.sort(oi[clear], axis=1))
    return gi, gv, gl


@pytest.mark.parametrize("T,V,d,K,tau,chunk", [(300, 5000, 256, 16, 1.0, 128),
                                               (130, 1000, 128, 10, 2.0, 1000),   # K > tiles
                                               (257, 8192, 384, 100, 1.0, 100),
                                               (64, 2048, 64, 1, 0.5, 64)])
def test_producer_parity(T, V, d, K, tau, chunk):
    g = torch.Generator().manual_seed(T + V)
    h = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    check_against_oracle(h, W, K, tau, chunk)


def test_producer_exact_ties_integer_logits():
    """Small-integer h and W: every logit is an exact small integer in fp32 and
    fp64, with many ties; the output must be the oracle's, bit for bit."""
    g = torch.Generator().manual_seed(7)
    T, V, d, K = 200, 3000, 64, 40
    h = torch.randint(-2, 3, (T, d), generator=g).to(torch.bfloat16)
    W = torch.randint(-1, 2, (V, d), generator=g).to(torch.bfloat16)
    gi, gv, gl = run_producer(h, W, K, 1.0, 96)
    oi, ov, ol = TK.teacher_topk(h.double().numpy(), W.double().numpy(), K, 1.0)
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov)


def test_producer_all_equal_logits():
    T, V, d, K = 50, 4096, 64, 100
    h = torch.randn(T, d).to(torch.bfloat16)
    W = torch.zeros(V, d, dtype=torch.bfloat16)
    gi, gv, gl = run_producer(h, W, K, 1.5, 32)
    np.testing.assert_array_equal(gi, np.tile(np.arange(K), (T, 1)))
    assert np.all(gv == 0.0)
    assert np.abs(gl - math.log(V)).max() <= 1e-5


def test_producer_full_vocab_sampled():
    """V = 201088, d = 2880, K = 100 on 192 rows (two chunks, the second ragged)."""
    g = torch.Generator().manual_seed(11)
    T, V, d, K = 192, 201088, 2880, 100
    h = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    check_against_oracle(h, W, K, 1.0, 128)


def test_producer_feeds_residual_loss_teacher_equals_student():
    """Cache the student's own top-K (with its full-vocabulary normaliser) and
    take the residual-variant loss against it: the two distributions are the
    same, so the loss and its gradient vanish."""
    g = torch.Generator().manual_seed(13)
    T, V, d, K, tau = 256, 6000, 192, 50, 1.0
    h = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    dev = torch.device("cuda")
    gi, gv, gl = run_producer(h, W, K, tau, 128)
    idx = torch.from_numpy(gi.astype(np.int32)).to(dev)
    tl = torch.from_numpy(gv.astype(np.float32)).to(dev)
    tlse = torch.from_numpy(gl.astype(np.float32)).to(dev)
    valid = torch.ones(T, dtype=torch.uint8, device=dev)
    hd, Wd = h.to(dev), W.to(dev)
    f, b = kd.kd_topk_kl_workspace_size(T, V, d, K, 128)
    ws = torch.empty(max(f, b), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    loss = torch.empty(1, device=dev)
    lse = torch.empty(T, device=dev)
    mass = torch.empty(T, device=dev)
    kd.kd_topk_kl_forward_residual(hd, Wd, idx, tl, tlse, valid, tau, 128, loss, lse, None, mass,
                                   ws=ws, dev_status=st)
    dh = torch.empty(T, d, device=dev)
    dW = torch.empty(V, d, device=dev)
    kd.kd_topk_kl_backward_residual(hd, Wd, idx, tl, tlse, valid, tau, 128, lse, mass, 1.0, dh, dW,
                                    ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert abs(float(loss.item())) <= 1e-5
    # the forward's own lse equals the producer's normaliser
    assert (lse - tlse).abs().max().item() <= 1e-5
    assert dh.abs().max().item() <= 1e-5 and dW.abs().max().item() <= 1e-5


def test_producer_k_larger_than_tile_count():
    """K = 1000 with 32 vocabulary tiles: every logit is a candidate and the
    selection orders 1000 of 8192 per row."""
    g = torch.Generator().manual_seed(17)
    T, V, d, K = 64, 8192, 128, 1000
    h = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    check_against_oracle(h, W, K, 1.0, 64)


KD_ERR_NONFINITE = 9


def test_producer_nonfinite_rows_are_reported():
    """Rows of h holding NaN or inf (host-made inputs, so their logits hold
    NaN and +-inf): the call reports KD_ERR_NONFINITE, writes those rows as
    index -1, logit NaN and lse NaN, and every other row is still the oracle's
    result bit for bit (integer inputs).  The bad rows sit in both chunks."""
    g = torch.Generator().manual_seed(19)
    T, V, d, K, chunk = 96, 3000, 64, 20, 64
    h = torch.randint(-2, 3, (T, d), generator=g).to(torch.bfloat16)
    W = torch.randint(-1, 2, (V, d), generator=g).to(torch.bfloat16)
    h[3, 5] = float("nan")
    h[40, :] = float("inf")
    h[95, 0] = float("-inf")
    bad = np.array([3, 40, 95])
    dev = torch.device("cuda")
    ws = torch.empty(kd.kd_teacher_topk_workspace_size(T, V, d, K, chunk), dtype=torch.uint8,
                     device=dev)
    # stale candidates from a clean run must not leak into the flagged rows
    clean = h.clone()
    clean[bad] = 1.0
    st = torch.full((1,), -1, dtype=torch.int32, device=dev)
    idx = torch.full((T, K), -7, dtype=torch.int32, device=dev)
    val = torch.zeros((T, K), dtype=torch.float32, device=dev)
    lse = torch.zeros(T, dtype=torch.float32, device=dev)
    kd.kd_teacher_topk(clean.to(dev), W.to(dev), K, 1.0, chunk, idx, val, lse, ws=ws,
                       dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kd.kd_teacher_topk(h.to(dev), W.to(dev), K, 1.0, chunk, idx, val, lse, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == KD_ERR_NONFINITE, kd.status_string(int(st.item()))
    gi, gv, gl = idx.cpu().numpy(), val.cpu().numpy(), lse.cpu().numpy()
    assert np.all(gi[bad] == -1) and np.all(np.isnan(gv[bad])) and np.all(np.isnan(gl[bad]))
    good = np.setdiff1d(np.arange(T), bad)
    oi, ov, ol = TK.teacher_topk(h[good].double().numpy(), W.double().numpy(), K, 1.0)
    np.testing.assert_array_equal(gi[good], oi)
    np.testing.assert_array_equal(gv[good], ov)
    assert np.abs(gl[good] - ol).max() <= LSE_ATOL


def test_producer_signed_zero_logits():
    """Integer inputs whose top logits are exact zeros of either sign (h >= 0,
    W in {-1, 0}, mostly 0): -0 and +0 are one value, so the top-K are the
    lowest indices among the zero logits, exactly as the oracle orders them."""
    g = torch.Generator().manual_seed(23)
    T, V, d, K = 128, 4096, 64, 100
    h = torch.randint(0, 3, (T, d), generator=g).to(torch.bfloat16)
    W = -(torch.rand(V, d, generator=g) < 0.02).to(torch.bfloat16)
    gi, gv, gl = run_producer(h, W, K, 1.0, 64)
    oi, ov, ol = TK.teacher_topk(h.double().numpy(), W.double().numpy(), K, 1.0)
    z = h.double().numpy() @ W.double().numpy().T
    assert np.all((z == 0).sum(axis=1) >= K)  # the top-K of every row are zeros
    np.testing.assert_array_equal(gi, oi)
    np.testing.assert_array_equal(gv, ov)
    assert np.abs(gl - ol).max() <= LSE_ATOL
