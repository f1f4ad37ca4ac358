"""Full-size workloads in the launch configuration the benchmark times, held to
the fp64 oracle.

small_4k (T=4096, V=201088, d=2880) and vocab_152k (T=16384, V=151936,
d=4096, packed mask): the full oracle, forward and backward; every element of
lse, row_kl, dh and dW is compared.

ctx_8k (T=8192, tau=2, chunk sizes 1024 / 2048 / 4096) and ctx_32k (T=32768,
the headline workload): the oracle's full forward gives the exact loss and the
lse and row_kl of every row; dh is compared on seeded rows and dW on seeded
vocabulary rows, both computed by the oracle from its own lse; the gathered
indices are compared in full.  Nothing the oracle uses comes from the GPU.
At ctx_32k the one-call training step (the single sweep the benchmark times)
must also give the separate calls' loss, lse and row_kl bit for bit, and dh
and dW within the oracle's tolerance on the same sampled rows.

The oracle's row blocks are larger here than its defaults only to make fewer,
larger BLAS calls; a block is the plain definition applied to a set of rows.
"""

import numpy as np
import pytest

from oracle import kd_oracle as O
from synth import make_inputs, workload
from tests.gpu_util import (GRAD_RL2, LOSS_RTOL, LSE_ATOL, assert_forward_parity,
                            oracle_inputs, rel_l2, run_gpu, run_sweep)

pytestmark = pytest.mark.gpu

_ORACLE_BLOCK = 1024
_cache = {}


def _args(P):
    return (P["h"], P["W"], P["teacher_idx"], P["teacher_logits"], P["valid"], P["tau"])


def _inputs_and_forward(name):
    """Seeded inputs of a workload and the oracle's full forward on them (cached
    per workload: the chunk sweep reuses them)."""
    if name not in _cache:
        _cache.clear()
        w = workload(name)
        x = make_inputs(w)
        P = oracle_inputs(x)
        f = O.forward(*_args(P), block=_ORACLE_BLOCK)
        _cache[name] = (w, x, P, f)
    return _cache[name]


def _check_full(name):
    w, x, P, f = _inputs_and_forward(name)
    gpu = run_gpu(x, w.chunk)
    assert_forward_parity(gpu, f)
    assert gpu["bwd_status"] == 0
    dh_ref, dW_ref = O.backward(*_args(P), 1.0, lse=f["lse"], block=_ORACLE_BLOCK)
    assert rel_l2(gpu["dh"], dh_ref) <= GRAD_RL2
    assert rel_l2(gpu["dW"], dW_ref) <= GRAD_RL2
    inval = P["valid"] == 0
    assert np.all(gpu["dh"][inval] == 0.0) and np.all(gpu["row_kl"][inval] == 0.0)
    return w, gpu, P, f


def test_small_4k_full_oracle():
    """T=4096, V=201088, d=2880, K=100, tau=1, 10% of rows masked at random."""
    _check_full("small_4k")


def test_vocab_152k_full_oracle():
    """T=16384, d=4096, V=151936 (593.5 vocabulary tiles), four packed
    sequences with their last 1024 rows masked."""
    w, gpu, P, f = _check_full("vocab_152k")
    valid = P["valid"]
    assert valid.sum() == 3 * 4096 and np.all(valid.reshape(4, 4096)[:, 3072:] == 0)


def _sampled_grads(w, gpu, P, f, seed, n_rows, n_vrows, slab=0):
    """dh on seeded rows (with every kind of row: random, masked, the last) and
    dW on seeded vocabulary rows (random, a contiguous slab, entries of the
    teacher cache, the last), from the oracle's own lse."""
    args = _args(P)
    rng = np.random.default_rng(seed)
    inval = np.nonzero(P["valid"] == 0)[0]
    rows = np.unique(np.concatenate([rng.choice(w.T, n_rows - 5, replace=False), inval[:4],
                                     [w.T - 1]]))
    dh_ref = O.dh_rows(*args, 1.0, f["lse"], f["n_valid"], rows)
    assert rel_l2(gpu["dh"][rows], dh_ref) <= GRAD_RL2
    assert np.all(gpu["dh"][inval] == 0.0)
    hit = np.unique(P["teacher_idx"][rng.choice(w.T, 64, replace=False), :4])
    parts = [rng.choice(w.V, n_vrows, replace=False), hit, [w.V - 1]]
    if slab:
        s0 = int(rng.integers(0, w.V - slab))
        parts.append(np.arange(s0, s0 + slab))
    vrows = np.unique(np.concatenate(parts))
    dW_ref = O.dW_rows(*args, 1.0, f["lse"], f["n_valid"], vrows)
    assert rel_l2(gpu["dW"][vrows], dW_ref) <= GRAD_RL2
    return rows, vrows


@pytest.mark.parametrize("chunk", [1024, 2048, 4096])
def test_ctx_8k_chunk_sweep(chunk):
    """T=8192, V=201088, d=2880, tau=2: every chunk size of the 8k-context
    workload matches the oracle's full forward and its sampled gradients."""
    w, x, P, f = _inputs_and_forward("ctx_8k")
    gpu = run_gpu(x, chunk)
    assert_forward_parity(gpu, f)
    assert gpu["bwd_status"] == 0
    _sampled_grads(w, gpu, P, f, seed=chunk, n_rows=128, n_vrows=256)


def test_ctx_32k_full_forward_sampled_grads():
    """The headline workload (T=32768, V=201088, d=2880, K=100, tau=1, chunk
    8192): the oracle's loss and the lse / row_kl of all 32768 rows, the
    gathered indices in full, dh on 512 seeded rows and dW on more than 1024
    seeded vocabulary rows."""
    w, x, P, f = _inputs_and_forward("ctx_32k")
    gpu = run_gpu(x, w.chunk)
    assert_forward_parity(gpu, f)
    assert gpu["bwd_status"] == 0
    rows, vrows = _sampled_grads(w, gpu, P, f, seed=2, n_rows=512, n_vrows=640, slab=256)
    assert len(rows) >= 500 and len(vrows) >= 1024
    sw = run_sweep(x, w.chunk)
    assert sw["status"] == 0
    for k in ("loss", "lse", "row_kl"):
        np.testing.assert_array_equal(sw[k], gpu[k], err_msg=k)
    _sampled_grads(w, sw, P, f, seed=2, n_rows=512, n_vrows=640, slab=256)
    assert rel_l2(sw["dh"], gpu["dh"]) <= 5e-3 and rel_l2(sw["dW"], gpu["dW"]) <= 5e-3
    del sw
    # every row of G sums to zero, so the column sums of dW vanish up to the
    # bf16 rounding of G (a property beside the oracle comparison above)
    col = gpu["dW"].sum(axis=0)
    assert np.linalg.norm(col) <= 1e-2 * np.linalg.norm(gpu["dW"])
    assert np.all(np.isfinite(gpu["dW"]))


def test_ctx_32k_single_sweep_chunk_4096():
    """The one-call training step at ctx_32k with 4096-row chunks: loss, lse and
    row_kl bit for bit those of the separate forward and backward at the same
    chunk size, and held to the oracle's full forward and its sampled
    gradients."""
    w, x, P, f = _inputs_and_forward("ctx_32k")
    sw = run_sweep(x, 4096)
    assert sw["status"] == 0
    gpu = run_gpu(x, 4096)
    for k in ("loss", "lse", "row_kl"):
        np.testing.assert_array_equal(sw[k], gpu[k], err_msg=k)
    assert abs(sw["loss"] - f["loss"]) <= LOSS_RTOL * abs(f["loss"])
    assert np.abs(sw["lse"] - f["lse"]).max() <= LSE_ATOL
    assert np.abs(sw["row_kl"] - f["row_kl"]).max() <= LSE_ATOL
    _sampled_grads(w, sw, P, f, seed=3, n_rows=256, n_vrows=512, slab=128)
    _cache.clear()
