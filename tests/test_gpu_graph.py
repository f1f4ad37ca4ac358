"""The training step can be captured in a CUDA graph: the library's calls are
stream-ordered, allocate nothing and never synchronise the host, so a captured
forward + backward replays with results bit-identical to eager execution."""

import pytest
import torch

import chunked_top_kl_logit_b300 as kd
from synth import make_inputs, workload
from tests.gpu_util import to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [False, True])
def test_step_replays_from_a_cuda_graph(fused):
    x = make_inputs(workload("small_4k", T=700, d=256, V=6000, K=50, tau=1.5))
    g = to_device(x)
    T, d = g["h"].shape
    V, K = g["W"].shape[0], g["teacher_idx"].shape[1]
    args = (g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"])

    eager = kd.TopKKL(T, V, d, K, 256)
    if fused:
        eager.forward_backward(*args, 1.0)
    else:
        eager.forward(*args)
        eager.backward(*args, 1.0)
    torch.cuda.synchronize()
    kd.check_device_status(eager.status, "eager")

    m = kd.TopKKL(T, V, d, K, 256)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm up on the capture stream (first-use set-up)
        if fused:
            m.forward_backward(*args, 1.0, stream=s)
        else:
            m.forward(*args, stream=s)
            m.backward(*args, 1.0, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        if fused:
            m.forward_backward(*args, 1.0, stream=s)
        else:
            m.forward(*args, stream=s)
            m.backward(*args, 1.0, stream=s)
    for _ in range(2):
        for t in (m.loss, m.lse, m.row_kl, m.dh, m.dW):
            t.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        kd.check_device_status(m.status, "graph replay")
        for name in ("loss", "lse", "row_kl", "dh", "dW"):
            assert torch.equal(getattr(m, name), getattr(eager, name)), name
