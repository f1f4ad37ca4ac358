"""topk_kl_loss, the autograd adapter, runs the same kernels as the explicit
calls: the loss and both gradients are bit-identical to TopKKL's forward and
backward, with a scaled upstream gradient passed through as grad_loss."""

import pytest
import torch

import chunked_top_kl_logit_b300 as kd
from synth import make_inputs, workload

pytestmark = pytest.mark.gpu


def test_autograd_matches_explicit_calls():
    w = workload("small_4k", T=300, d=192, V=3000, K=40, tau=1.5, idx_kind="uniform")
    x = make_inputs(w)
    dev = torch.device("cuda")
    h = x["h"].to(dev).requires_grad_(True)
    W = x["W"].to(dev).requires_grad_(True)
    idx, tl, valid = (x[k].to(dev) for k in ("teacher_idx", "teacher_logits", "valid"))
    chunk = 128
    loss = kd.topk_kl_loss(h, W, idx, tl, valid, w.tau, chunk)
    (2.5 * loss).backward()
    m = kd.TopKKL(w.T, w.V, w.d, w.K, chunk, device=dev)
    m.forward(h.detach(), W.detach(), idx, tl, valid, w.tau)
    m.backward(h.detach(), W.detach(), idx, tl, valid, w.tau, 2.5)
    torch.cuda.synchronize()
    kd.check_device_status(m.status, "explicit calls")
    assert loss.dtype == torch.float32 and loss.dim() == 0
    assert torch.equal(loss.detach().view(1), m.loss)
    assert h.grad.dtype == torch.bfloat16 and W.grad.dtype == torch.bfloat16
    assert torch.equal(h.grad, m.dh.to(torch.bfloat16))
    assert torch.equal(W.grad, m.dW.to(torch.bfloat16))
