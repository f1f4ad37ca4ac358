"""GPU path (through the C ABI) against the fp64 oracle, element by element,
on seeded inputs that span several tiles with ragged tails in every
dimension, plus the closed forms, edge cases and exact metamorphic checks."""

import math

import numpy as np
import pytest
import torch

import chunked_top_kl_logit_b300 as kd
from oracle import kd_oracle as O
from synth import make_inputs, workload
from tests.gpu_util import (GRAD_RL2, LSE_ATOL, assert_forward_parity, oracle_inputs, rel_l2,
                            run_gpu)

pytestmark = pytest.mark.gpu


def oracle_all(x, grad_loss=1.0):
    P = oracle_inputs(x)
    f = O.forward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    dh, dW = O.backward(P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"],
                        P["tau"], grad_loss, lse=f["lse"])
    f["dh"], f["dW"] = dh, dW
    return f


# (name, workload overrides, chunk); each spans several tiles and has ragged tails
CASES = [
    ("teacher_T300_V5000_d256", dict(T=300, d=256, V=5000, tau=1.0), 128),
    ("packed_T520_V3000_d320_tau2", dict(T=520, d=320, V=3000, K=64, tau=2.0,
                                         mask_kind="packed", seq_len=130, pad=30), 200),
    ("uniform_T128_V2048_d192", dict(T=128, d=192, V=2048, K=16, tau=0.5, idx_kind="uniform",
                                     mask_kind="all"), 1000),
    ("teacher_T1000_V8192_d384", dict(T=1000, d=384, V=8192, tau=1.5), 512),
]


@pytest.mark.parametrize("name,over,chunk", CASES, ids=[c[0] for c in CASES])
def test_parity_small(name, over, chunk):
    x = make_inputs(workload("small_4k", **over))
    gpu = run_gpu(x, chunk, grad_loss=1.0)
    ref = oracle_all(x)
    assert_forward_parity(gpu, ref)
    assert gpu["bwd_status"] == 0
    assert rel_l2(gpu["dh"], ref["dh"]) <= GRAD_RL2
    assert rel_l2(gpu["dW"], ref["dW"]) <= GRAD_RL2
    inval = x["valid"].numpy() == 0
    assert np.all(gpu["dh"][inval] == 0.0)


def test_tiny_workload_chunk64():
    x = make_inputs(workload("tiny_fp32"))
    gpu = run_gpu(x, 64, grad_loss=1.0)
    ref = oracle_all(x)
    assert_forward_parity(gpu, ref)
    assert rel_l2(gpu["dh"], ref["dh"]) <= GRAD_RL2
    assert rel_l2(gpu["dW"], ref["dW"]) <= GRAD_RL2


def test_w_zero_closed_form():
    """W = 0: lse = log V, row_kl = sum p log p + log V, dh exactly 0."""
    x = make_inputs(workload("tiny_fp32"))
    x["W"] = torch.zeros_like(x["W"])
    x["valid"] = x["valid"].clone()
    x["valid"][::7] = 0
    gpu = run_gpu(x, 64, grad_loss=0.5)
    tl = x["teacher_logits"].double().numpy()
    a = tl / x["tau"]
    logp = a - (a.max(1, keepdims=True) + np.log(np.exp(a - a.max(1, keepdims=True)).sum(1, keepdims=True)))
    V = x["W"].shape[0]
    assert np.abs(gpu["lse"] - math.log(V)).max() <= 1e-5
    valid = x["valid"].numpy() > 0
    expect = np.where(valid, (np.exp(logp) * logp).sum(1) + math.log(V), 0.0)
    assert np.abs(gpu["row_kl"] - expect).max() <= LSE_ATOL
    assert np.all(gpu["dh"] == 0.0)
    ref = oracle_all(x, grad_loss=0.5)
    assert rel_l2(gpu["dW"], ref["dW"]) <= GRAD_RL2


def test_teacher_equals_student_is_zero():
    """K = V = 64, tau = 1, teacher logits = student logits: KL = 0, G = 0.
    Also exercises a vocabulary smaller than one logit tile."""
    g = torch.Generator().manual_seed(5)
    T, d, V = 200, 128, 64
    h = torch.randn(T, d, generator=g).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g) / math.sqrt(d)).to(torch.bfloat16)
    z = (h.double() @ W.double().T)
    perm = torch.stack([torch.randperm(V, generator=g) for _ in range(T)]).to(torch.int32)
    tl = torch.gather(z, 1, perm.long()).float()
    x = dict(h=h, W=W, teacher_idx=perm, teacher_logits=tl, valid=torch.ones(T, dtype=torch.uint8),
             tau=1.0)
    gpu = run_gpu(x, 96)
    assert abs(gpu["loss"]) <= 1e-5
    assert np.abs(gpu["row_kl"]).max() <= 1e-5
    assert np.abs(gpu["dh"]).max() <= 1e-5 and np.abs(gpu["dW"]).max() <= 1e-5
    np.testing.assert_array_equal(gpu["gathered_idx"], perm.numpy())


def test_teacher_covers_whole_vocabulary():
    """K = V = 1000 over four vocabulary tiles (the last one ragged): every
    tile holds 256 cached entries per row, the most the gather and scatter
    walks ever see, and the top-K softmax is the full-vocabulary one."""
    g = torch.Generator().manual_seed(17)
    T, d, V = 150, 128, 1000
    x = make_inputs(workload("small_4k", T=T, d=d, V=V, K=8, tau=1.25, idx_kind="uniform"))
    x["teacher_idx"] = torch.stack([torch.randperm(V, generator=g) for _ in range(T)]).to(torch.int32)
    x["teacher_logits"] = (2.0 * torch.randn(T, V, generator=g)).float()
    gpu = run_gpu(x, 64)
    ref = oracle_all(x)
    assert_forward_parity(gpu, ref)
    assert rel_l2(gpu["dh"], ref["dh"]) <= GRAD_RL2
    assert rel_l2(gpu["dW"], ref["dW"]) <= GRAD_RL2
    np.testing.assert_array_equal(gpu["gathered_idx"], x["teacher_idx"].numpy())


def test_duplicate_indices():
    x = make_inputs(workload("small_4k", T=200, d=128, V=1024, K=32, tau=1.0, idx_kind="uniform"))
    idx = x["teacher_idx"].clone()
    idx[::3, 5] = idx[::3, 0]
    idx[1::3, 31] = idx[1::3, 30]
    x["teacher_idx"] = idx
    gpu = run_gpu(x, 64)
    ref = oracle_all(x)
    assert_forward_parity(gpu, ref)
    assert rel_l2(gpu["dh"], ref["dh"]) <= GRAD_RL2
    assert rel_l2(gpu["dW"], ref["dW"]) <= GRAD_RL2


def test_no_valid_rows():
    x = make_inputs(workload("small_4k", T=130, d=128, V=1024, K=20, idx_kind="uniform"))
    x["valid"] = torch.zeros_like(x["valid"])
    gpu = run_gpu(x, 64)
    assert gpu["loss"] == 0.0
    assert np.all(gpu["row_kl"] == 0) and np.all(gpu["dh"] == 0) and np.all(gpu["dW"] == 0)
    ref = oracle_all(x)
    assert np.abs(gpu["lse"] - ref["lse"]).max() <= LSE_ATOL


def test_heavy_masking_leaves_empty_chunks():
    """70% of rows masked and small chunks: the backward runs over the valid
    rows only, so the last chunks hold no row at all (their kernels find no
    work on the device and dW keeps the earlier chunks' sum)."""
    x = make_inputs(workload("small_4k", T=600, d=128, V=2000, K=24, tau=1.0, idx_kind="uniform"))
    g = torch.Generator().manual_seed(11)
    x["valid"] = (torch.rand(600, generator=g) < 0.3).to(torch.uint8)
    gpu = run_gpu(x, 96)
    ref = oracle_all(x)
    assert_forward_parity(gpu, ref)
    assert rel_l2(gpu["dh"], ref["dh"]) <= GRAD_RL2
    assert rel_l2(gpu["dW"], ref["dW"]) <= GRAD_RL2
    assert np.all(gpu["dh"][x["valid"].numpy() == 0] == 0.0)


def test_single_row_and_k1():
    x = make_inputs(workload("small_4k", T=1, d=64, V=8, K=1, idx_kind="uniform", mask_kind="all"))
    gpu = run_gpu(x, 1)
    ref = oracle_all(x)
    assert_forward_parity(gpu, ref)
    assert rel_l2(gpu["dh"], ref["dh"]) <= GRAD_RL2
    assert rel_l2(gpu["dW"], ref["dW"]) <= GRAD_RL2


def test_index_out_of_range_sets_status():
    x = make_inputs(workload("small_4k", T=64, d=64, V=512, K=8, idx_kind="uniform"))
    x["teacher_idx"] = x["teacher_idx"].clone()
    x["teacher_idx"][3, 2] = 512
    x["teacher_idx"][7, 0] = -1
    gpu = run_gpu(x, 64)
    assert gpu["fwd_status"] == 5 and gpu["bwd_status"] == 5


def test_power_of_two_scaling_bitwise():
    """(h, teacher_logits, tau) -> (2h, 2 teacher_logits, 2 tau) is exact in bf16
    and fp32, so lse, row_kl and loss are bit-identical; dh halves exactly and
    dW is unchanged bit for bit."""
    x = make_inputs(workload("small_4k", T=260, d=192, V=2000, K=40, tau=1.25, idx_kind="uniform"))
    a = run_gpu(x, 128, grad_loss=1.0)
    y = dict(x, h=(x["h"].float() * 2).to(torch.bfloat16), teacher_logits=x["teacher_logits"] * 2,
             tau=2 * x["tau"])
    b = run_gpu(y, 128, grad_loss=1.0)
    np.testing.assert_array_equal(a["lse"], b["lse"])
    np.testing.assert_array_equal(a["row_kl"], b["row_kl"])
    assert a["loss"] == b["loss"]
    np.testing.assert_array_equal(b["dh"], a["dh"] / 2)
    np.testing.assert_array_equal(b["dW"], a["dW"])


def test_permutation_invariance():
    x = make_inputs(workload("small_4k", T=150, d=128, V=3000, K=50, tau=1.0))
    a = run_gpu(x, 64)
    g = torch.Generator().manual_seed(1)
    perm = torch.stack([torch.randperm(50, generator=g) for _ in range(150)])
    y = dict(x, teacher_idx=torch.gather(x["teacher_idx"], 1, perm).contiguous(),
             teacher_logits=torch.gather(x["teacher_logits"], 1, perm).contiguous())
    b = run_gpu(y, 64)
    assert np.abs(a["lse"] - b["lse"]).max() == 0.0  # the student side does not see the order
    assert np.abs(a["row_kl"] - b["row_kl"]).max() <= 1e-5
    assert rel_l2(b["dh"], a["dh"]) <= 1e-3 and rel_l2(b["dW"], a["dW"]) <= 1e-3
    np.testing.assert_array_equal(b["gathered_idx"], y["teacher_idx"].numpy())


def test_chunk_invariance():
    x = make_inputs(workload("small_4k", T=700, d=256, V=4000, tau=2.0))
    outs = [run_gpu(x, c) for c in (128, 300, 700)]
    for o in outs[1:]:
        np.testing.assert_array_equal(o["lse"], outs[0]["lse"])
        assert rel_l2(o["dh"], outs[0]["dh"]) <= 1e-6
        assert rel_l2(o["dW"], outs[0]["dW"]) <= 1e-5


def test_grad_loss_scales():
    x = make_inputs(workload("small_4k", T=200, d=128, V=1504, K=30, idx_kind="uniform"))
    a = run_gpu(x, 100, grad_loss=1.0)
    b = run_gpu(x, 100, grad_loss=-0.25)
    assert rel_l2(b["dh"], -0.25 * a["dh"]) <= 1e-2
    assert rel_l2(b["dW"], -0.25 * a["dW"]) <= 1e-2


def test_large_k():
    """K = 2048 cached entries per row (a quarter of the vocabulary): the rank
    sort of the teacher entries and the gather / scatter walk over many entries
    per vocabulary tile."""
    x = make_inputs(workload("small_4k", T=96, d=128, V=8192, K=2048, tau=1.0,
                             idx_kind="uniform"))
    gpu = run_gpu(x, 64)
    ref = oracle_all(x)
    assert_forward_parity(gpu, ref)
    assert rel_l2(gpu["dh"], ref["dh"]) <= GRAD_RL2
    assert rel_l2(gpu["dW"], ref["dW"]) <= GRAD_RL2


def test_wide_hidden_and_ragged_vocab():
    """d = 4096 (64 contraction steps) with V = 3000 (a ragged last vocabulary
    tile) and a chunk that is not a multiple of the tile height."""
    x = make_inputs(workload("small_4k", T=333, d=4096, V=3000, K=24, tau=0.75,
                             idx_kind="uniform"))
    gpu = run_gpu(x, 150)
    ref = oracle_all(x)
    assert_forward_parity(gpu, ref)
    assert rel_l2(gpu["dh"], ref["dh"]) <= GRAD_RL2
    assert rel_l2(gpu["dW"], ref["dW"]) <= GRAD_RL2
