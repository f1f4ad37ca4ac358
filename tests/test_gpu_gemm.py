"""The tcgen05/TMA contraction pipeline on its own (C = A B^T, fp32 out) for
all four operand layouts, against a plain PyTorch fp64 product; and the
bounded pipeline wait, which must time out cleanly on a barrier nothing
arrives on."""

import pytest
import torch

import chunked_top_kl_logit_b300 as kd

pytestmark = pytest.mark.gpu


def _operands(M, N, Kd, a_mn, b_mn, seed):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn(M, Kd, generator=g).to(torch.bfloat16)
    B = torch.randn(N, Kd, generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T
    Ad = (A.T.contiguous() if a_mn else A).cuda()
    Bd = (B.T.contiguous() if b_mn else B).cuda()
    return Ad, Bd, ref


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 0), (1, 1)])
@pytest.mark.parametrize("M,N,Kd", [(128, 256, 64), (256, 512, 640), (200, 136, 200),
                                    (384, 192, 1024), (136, 64, 72)])
def test_gemm_layouts(M, N, Kd, a_mn, b_mn):
    Ad, Bd, ref = _operands(M, N, Kd, a_mn, b_mn, seed=M * 7 + N + Kd)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd.kd_gemm_bf16_diag(Ad, Bd, C, M, N, Kd, a_mn, b_mn, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    err = (C.double().cpu() - ref).abs().max().item()
    # bf16 products are exact in fp32; only the fp32 summation order differs
    assert err <= 1e-4 * (Kd ** 0.5) * 4, err


@pytest.mark.parametrize("M,N,Kd", [(256, 256, 64), (512, 512, 640), (200, 136, 200),
                                    (1024, 768, 1024), (136, 64, 72), (128, 256, 2880)])
def test_gemm_cta_pair(M, N, Kd):
    """The cta_group::2 pipeline (clusters of two CTAs, 256-row tiles)."""
    Ad, Bd, ref = _operands(M, N, Kd, 0, 0, seed=M * 5 + N + Kd)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd.kd_gemm_bf16_diag_pair(Ad, Bd, C, M, N, Kd, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, kd.status_string(int(st.item()))
    err = (C.double().cpu() - ref).abs().max().item()
    assert err <= 1e-4 * (Kd ** 0.5) * 4, err


def test_bounded_wait_times_out():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kd.kd_pipeline_wait_selftest(20_000_000, dev_status=st)  # 20 ms
    torch.cuda.synchronize()
    assert int(st.item()) == 6  # KD_ERR_TIMEOUT
    # the context is still usable afterwards
    x = torch.ones(1024, device="cuda")
    assert float(x.sum().item()) == 1024.0
