"""The teacher-entropy token filter (kd_entropy_filter) through the C ABI.

Entropies are compared with the fp64 oracle within fp32 rounding; the mask,
an integer decision taken on the kernel's own fp32 entropies, must equal the
oracle's selection run on those same values bit for bit (and it is checked
against the selection on the oracle's fp64 entropies away from near-ties)."""

import numpy as np
import pytest
import torch

import chunked_top_kl_logit_b300 as kd
from oracle import entropy_filter as EF
from synth import make_inputs, workload

pytestmark = pytest.mark.gpu

H_ATOL = 2e-5


def run_filter(tl, valid, tau, num, den):
    T = tl.shape[0]
    dev = torch.device("cuda")
    out = torch.full((T,), 7, dtype=torch.uint8, device=dev)
    ent = torch.full((T,), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(kd.kd_entropy_filter_workspace_size(T), dtype=torch.uint8, device=dev)
    st = torch.full((1,), -1, dtype=torch.int32, device=dev)
    kd.kd_entropy_filter(tl.to(dev).contiguous(), valid.to(dev).contiguous(), tau, num, den, out,
                         ent, ws=ws, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out.cpu().numpy(), ent.double().cpu().numpy()


@pytest.mark.parametrize("T,K,tau,num,den", [(4096, 100, 1.0, 7, 10), (3001, 64, 2.0, 1, 3),
                                             (1, 5, 1.0, 1, 1), (2500, 1, 1.0, 1, 2),
                                             (32768, 100, 1.0, 3, 4)])
def test_filter_matches_oracle(T, K, tau, num, den):
    x = make_inputs(workload("small_4k", T=T, d=64, V=max(256, K), K=K, tau=tau,
                             idx_kind="uniform"))
    tl, valid = x["teacher_logits"], x["valid"]
    out, ent = run_filter(tl, valid, tau, num, den)
    H = EF.teacher_entropy(tl.double().numpy(), tau)
    assert np.abs(ent - H).max() <= H_ATOL
    # the integer decision, on the kernel's own entropies
    np.testing.assert_array_equal(out, EF.entropy_filter(ent, valid.numpy(), num, den))
    # and on the oracle's fp64 entropies, up to rows within the tolerance of the threshold
    ref = EF.entropy_filter(H, valid.numpy(), num, den)
    diff = np.nonzero(out != ref)[0]
    if diff.size:
        kept = H[(ref == 1)]
        theta = kept.min() if kept.size else np.inf
        assert np.all(np.abs(H[diff] - theta) <= 2 * H_ATOL)


def test_filter_ties_and_extremes():
    T, K = 3000, 16
    g = torch.Generator().manual_seed(9)
    # four distinct teacher rows repeated: entropies tie in large groups
    base = torch.randn(4, K, generator=g) * 2
    tl = base[torch.randint(0, 4, (T,), generator=g)].contiguous()
    valid = (torch.rand(T, generator=g) < 0.8).to(torch.uint8)
    for num, den in ((0, 1), (1, 1), (1, 2), (37, 100), (999, 1000)):
        out, ent = run_filter(tl, valid, 1.0, num, den)
        np.testing.assert_array_equal(out, EF.entropy_filter(ent, valid.numpy(), num, den))
    out, _ = run_filter(tl, valid, 1.0, 1, 1)
    np.testing.assert_array_equal(out, valid.numpy())
    out, _ = run_filter(tl, torch.zeros(T, dtype=torch.uint8), 1.0, 1, 2)
    assert out.sum() == 0
