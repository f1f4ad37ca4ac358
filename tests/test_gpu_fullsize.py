"""Full-size workloads in the launch configuration the benchmark times.

small_4k (T=4096, V=201088, d=2880, K=100): the oracle runs the full forward
(lse of every row, hence the exact loss), dh on sampled rows and dW on sampled
vocabulary rows.

ctx_32k (T=32768, same V, d; the headline workload): the oracle checks
sampled rows one by one (lse, row_kl, dh), the gathered indices are compared
in full, and dW is held to properties that hold at any size.
"""

import numpy as np
import pytest

from oracle import kd_oracle as O
from synth import make_inputs, workload
from tests.gpu_util import (GRAD_RL2, LOSS_RTOL, LSE_ATOL, assert_forward_parity, oracle_inputs,
                            rel_l2, run_gpu)

pytestmark = pytest.mark.gpu


def test_small_4k_full_size():
    w = workload("small_4k")
    x = make_inputs(w)
    gpu = run_gpu(x, w.chunk)
    P = oracle_inputs(x)
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    f = O.forward(*args)
    assert_forward_parity(gpu, f)
    assert gpu["bwd_status"] == 0
    rng = np.random.default_rng(1)
    inval = np.nonzero(P["valid"] == 0)[0]
    rows = np.concatenate([rng.choice(w.T, 24, replace=False), inval[:4]])
    dh_ref = O.dh_rows(*args, 1.0, f["lse"], f["n_valid"], rows)
    assert rel_l2(gpu["dh"][rows], dh_ref) <= GRAD_RL2
    assert np.all(gpu["dh"][inval] == 0.0)
    hit = np.unique(P["teacher_idx"][rng.choice(w.T, 8, replace=False), :3])
    vrows = np.unique(np.concatenate([rng.choice(w.V, 40, replace=False), hit, [w.V - 1]]))
    dW_ref = O.dW_rows(*args, 1.0, f["lse"], f["n_valid"], vrows)
    assert rel_l2(gpu["dW"][vrows], dW_ref) <= GRAD_RL2


def test_ctx_32k_sampled():
    w = workload("ctx_32k")
    x = make_inputs(w)
    gpu = run_gpu(x, w.chunk)
    assert gpu["fwd_status"] == 0 and gpu["bwd_status"] == 0
    P = oracle_inputs(x)
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    np.testing.assert_array_equal(gpu["gathered_idx"], P["teacher_idx"])
    rng = np.random.default_rng(2)
    inval = np.nonzero(P["valid"] == 0)[0]
    rows = np.concatenate([rng.choice(w.T, 20, replace=False), inval[:4], [w.T - 1]])
    lse_r = O.student_lse(P["h"], P["W"], P["tau"], rows)
    assert np.abs(gpu["lse"][rows] - lse_r).max() <= LSE_ATOL
    lse_full = np.zeros(w.T)
    lse_full[rows] = lse_r
    kl_r = O.row_kl_rows(*args, rows, lse=lse_full)
    assert np.abs(gpu["row_kl"][rows] - kl_r).max() <= LSE_ATOL
    n_valid = int((P["valid"] > 0).sum())
    # the loss is the mean of the per-row values over valid rows
    assert abs(gpu["loss"] - gpu["row_kl"].sum() / n_valid) <= LOSS_RTOL * abs(gpu["loss"])
    dh_ref = O.dh_rows(*args, 1.0, lse_full, n_valid, rows)
    assert rel_l2(gpu["dh"][rows], dh_ref) <= GRAD_RL2
    assert np.all(gpu["dh"][inval] == 0.0)
    # every row of G sums to zero, so the column sums of dW vanish up to the
    # bf16 rounding of G
    col = gpu["dW"].sum(axis=0)
    assert np.linalg.norm(col) <= 1e-2 * np.linalg.norm(gpu["dW"])
    assert np.all(np.isfinite(gpu["dW"]))


def _sampled_checks(w, gpu, P, seed, n_rows=16, n_vrows=24, check_dw=True):
    """Oracle on sampled rows (lse, row_kl, dh) and vocabulary rows (dW), with
    the exact full-row lse of the sampled rows; loss = mean of row_kl."""
    args = (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])
    rng = np.random.default_rng(seed)
    inval = np.nonzero(P["valid"] == 0)[0]
    rows = np.unique(np.concatenate([rng.choice(w.T, n_rows, replace=False), inval[:3],
                                     [w.T - 1]]))
    lse_r = O.student_lse(P["h"], P["W"], P["tau"], rows)
    assert np.abs(gpu["lse"][rows] - lse_r).max() <= LSE_ATOL
    lse_full = np.zeros(w.T)
    lse_full[rows] = lse_r
    kl_r = O.row_kl_rows(*args, rows, lse=lse_full)
    assert np.abs(gpu["row_kl"][rows] - kl_r).max() <= LSE_ATOL
    n_valid = int((P["valid"] > 0).sum())
    assert abs(gpu["loss"] - gpu["row_kl"].sum() / n_valid) <= LOSS_RTOL * abs(gpu["loss"])
    dh_ref = O.dh_rows(*args, 1.0, lse_full, n_valid, rows)
    assert rel_l2(gpu["dh"][rows], dh_ref) <= GRAD_RL2
    assert np.all(gpu["dh"][inval] == 0.0)
    if check_dw:
        # dW rows need the lse of every row: use the GPU's, checked above on samples
        hit = np.unique(P["teacher_idx"][rng.choice(w.T, 4, replace=False), :2])
        vrows = np.unique(np.concatenate([rng.choice(w.V, n_vrows, replace=False), hit,
                                          [w.V - 1]]))
        dW_ref = O.dW_rows(*args, 1.0, gpu["lse"], n_valid, vrows)
        assert rel_l2(gpu["dW"][vrows], dW_ref) <= GRAD_RL2


@pytest.mark.parametrize("chunk", [1024, 2048, 4096])
def test_ctx_8k_chunk_sweep(chunk):
    """T=8192, V=201088, d=2880, tau=2: the chunk sizes of the 8k-context
    workload give the same results (within the tolerances) and match the oracle
    on sampled rows."""
    w = workload("ctx_8k")
    x = make_inputs(w)
    gpu = run_gpu(x, chunk)
    assert gpu["fwd_status"] == 0 and gpu["bwd_status"] == 0
    P = oracle_inputs(x)
    np.testing.assert_array_equal(gpu["gathered_idx"], P["teacher_idx"])
    _sampled_checks(w, gpu, P, seed=chunk, check_dw=(chunk == 2048))


def test_vocab_152k_packed_mask():
    """T=16384, d=4096, V=151936 (593.5 vocabulary tiles), four packed
    sequences with their last 1024 rows masked."""
    w = workload("vocab_152k")
    x = make_inputs(w)
    gpu = run_gpu(x, w.chunk)
    assert gpu["fwd_status"] == 0 and gpu["bwd_status"] == 0
    P = oracle_inputs(x)
    valid = P["valid"]
    assert valid.sum() == 3 * 4096 and np.all(valid.reshape(4, 4096)[:, 3072:] == 0)
    np.testing.assert_array_equal(gpu["gathered_idx"], P["teacher_idx"])
    assert np.all(gpu["row_kl"][valid == 0] == 0.0)
    _sampled_checks(w, gpu, P, seed=5)
