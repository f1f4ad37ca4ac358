"""The allocation-free forward, kd_topk_kl_forward_noalloc.

Some callers cannot call cudaMalloc at all, for example code that runs
inside another framework's memory manager, which owns the whole device pool.
For them the library offers a forward whose workspace is a fixed 32 MiB array
built into the library.  These tests call it through the C ABI and hold it to
the regular kd_topk_kl_forward and to the fp64 oracle (same tolerances as
every parity test), on two calls in a row with different inputs, so that
contents left in the shared array by the first call cannot leak into the
second.

The file is named so that pytest collects it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import chunked_top_kl_logit_b300 as kd
from oracle import kd_oracle as O
from synth import make_inputs, workload
from tests.gpu_util import LOSS_RTOL, LSE_ATOL, oracle_inputs, to_device

KD_ERR_SCRATCH_LIMIT = 7


def test_rejects_shapes_beyond_the_builtin_scratch():
    # host-side check, before any CUDA call: 8192 rows at V=201088 need > 32 MiB
    A = ctypes.c_void_p(0x10000)
    rc = kd.lib().kd_topk_kl_forward_noalloc(A, A, A, A, A, 8192, 201088, 2880, 100, 1.0,
                                             A, A, None, None, A, None)
    assert rc == KD_ERR_SCRATCH_LIMIT
    assert "32 MiB" in kd.status_string(rc)


def _both(x):
    g = to_device(x)
    T, d = g["h"].shape
    V, K = g["W"].shape[0], g["teacher_idx"].shape[1]
    dev = torch.device("cuda")
    ref = kd.TopKKL(T, V, d, K, T, device=dev)
    ref_gidx = torch.full((T, K), -1, dtype=torch.int32, device=dev)
    ref.forward(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"], g["valid"], g["tau"],
                gathered_idx=ref_gidx)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    row_kl = torch.empty(T, dtype=torch.float32, device=dev)
    gidx = torch.full((T, K), -1, dtype=torch.int32, device=dev)
    st = torch.full((1,), -1, dtype=torch.int32, device=dev)
    kd.kd_topk_kl_forward_noalloc(g["h"], g["W"], g["teacher_idx"], g["teacher_logits"],
                                  g["valid"], g["tau"], loss, lse, row_kl, gidx, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(ref.status.item()) == 0
    return ((float(loss.item()), lse.cpu().numpy(), row_kl.cpu().numpy(), gidx.cpu().numpy()),
            (float(ref.loss.item()), ref.lse.cpu().numpy(), ref.row_kl.cpu().numpy(),
             ref_gidx.cpu().numpy()))


@pytest.mark.gpu
def test_matches_regular_forward_on_two_calls_in_a_row():
    first = make_inputs(workload("small_4k", T=4096, tau=1.0))  # full vocabulary, 17.8 MiB of scratch
    second = make_inputs(workload("small_4k", T=1500, d=512, V=40000, K=64, tau=2.0,
                                  mask_kind="packed", seq_len=500, pad=120), seed=3)
    for x in (first, second):
        (loss, lse, row_kl, gidx), (rloss, rlse, rrow, rgidx) = _both(x)
        assert abs(loss - rloss) <= LOSS_RTOL * abs(rloss)
        assert np.abs(lse - rlse).max() <= LSE_ATOL
        assert np.abs(row_kl - rrow).max() <= LSE_ATOL
        np.testing.assert_array_equal(gidx, rgidx)
        # and the oracle, which shares no code with either kernel path
        P = oracle_inputs(x)
        f = O.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"],
                      P["tau"], block=1024)
        assert abs(loss - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
        assert np.abs(lse - f["lse"]).max() <= LSE_ATOL
        assert np.abs(row_kl - f["row_kl"]).max() <= LSE_ATOL
        np.testing.assert_array_equal(gidx, f["gathered_idx"])
