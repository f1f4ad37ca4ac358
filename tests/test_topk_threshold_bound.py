"""The candidate bound of the teacher top-K producer, checked on the CPU.

Every logit z_v has the unique key (z_v, -v): larger logit first, then the
lower vocabulary index.  The producer takes, per row, the largest key of every
256-wide vocabulary tile and the K-th largest of those tile maxima, theta.
Two facts make its candidate set exact and bounded:

- the K tiles with the largest maxima hold K distinct keys >= theta, so the
  row's K-th largest key is >= theta and every top-K key is a candidate;
- a key >= theta lies in one of the fewer than K tiles whose maximum is above
  theta, or is theta itself, so there are at most (K - 1) * 256 + 1 candidates.

When the row has fewer than K tiles, every logit is a candidate.  This test
restates that rule with numpy ranks (independent of the CUDA code) and checks
both facts on random, tied and adversarial rows.
"""

import numpy as np
import pytest

TILE = 256


def key_ranks(z: np.ndarray) -> np.ndarray:
    """Rank 0 = the largest key (largest z, then the lowest index)."""
    order = np.lexsort((np.arange(z.shape[0]), -z))
    rank = np.empty(z.shape[0], dtype=np.int64)
    rank[order] = np.arange(z.shape[0])
    return rank


def candidates(z: np.ndarray, K: int) -> np.ndarray:
    V = z.shape[0]
    n_tiles = -(-V // TILE)
    if K > n_tiles:
        return np.arange(V)
    rank = key_ranks(z)
    tile_best = np.array([rank[t * TILE:(t + 1) * TILE].min() for t in range(n_tiles)])
    theta = np.sort(tile_best)[K - 1]  # the K-th largest tile maximum
    return np.nonzero(rank <= theta)[0]


def check(z: np.ndarray, K: int):
    V = z.shape[0]
    cand = candidates(z, K)
    top = np.nonzero(key_ranks(z) < K)[0]
    assert set(top.tolist()) <= set(cand.tolist())
    if K <= -(-V // TILE):
        assert cand.shape[0] <= (K - 1) * TILE + 1
    return cand


@pytest.mark.parametrize("V,K", [(5000, 1), (5000, 16), (201088 // 8, 100), (1000, 4),
                                 (1024, 4), (1000, 5), (300, 16)])
def test_random_rows(V, K):
    rng = np.random.default_rng(V + K)
    for _ in range(5):
        check(rng.standard_normal(V).astype(np.float32), K)


def test_all_equal_logits():
    """Every key differs only by index: the top-K is the K lowest indices."""
    for V, K in [(5000, 16), (2048, 8), (999 * 8, 100)]:
        cand = check(np.zeros(V, dtype=np.float32), K)
        assert cand.shape[0] <= (K - 1) * TILE + 1


def test_bound_is_reached():
    """The K - 1 best tiles hold all-larger logits and theta is a lone tile
    maximum: exactly (K - 1) * 256 + 1 candidates."""
    K, V = 8, 64 * TILE
    z = np.full(V, -10.0, dtype=np.float32)
    z[:(K - 1) * TILE] = 5.0           # K - 1 full tiles above theta
    z[(K - 1) * TILE] = 1.0            # theta: the K-th tile's maximum
    cand = check(z, K)
    assert cand.shape[0] == (K - 1) * TILE + 1


def test_top_k_in_one_tile_and_ascending_rows():
    V, K = 40 * TILE, 100
    z = np.linspace(-1.0, 1.0, V).astype(np.float32)  # the best tiles are the last ones
    check(z, K)
    z = np.zeros(V, dtype=np.float32)
    z[3 * TILE:3 * TILE + K] = 1.0 + np.arange(K, dtype=np.float32)  # all top-K in one tile
    cand = check(z, K)
    assert cand.shape[0] <= (K - 1) * TILE + 1


def test_fewer_tiles_than_k_takes_the_whole_row():
    z = np.random.default_rng(3).standard_normal(700).astype(np.float32)
    assert candidates(z, 16).shape[0] == 700


def test_signed_zeros_count_as_one_value():
    """-0.0 and +0.0 are one logit value (the producer folds -0 into +0 before
    forming keys, and numpy's ordering treats them as equal): mixed signed
    zeros at the top of a row order by index alone, and the bound holds."""
    rng = np.random.default_rng(5)
    for V, K in [(64 * TILE, 8), (201088 // 8, 100)]:
        z = np.where(rng.random(V) < 0.5, np.float32(-0.0), np.float32(0.0))
        z[rng.random(V) < 0.3] = -1.0
        assert np.signbit(z[z == 0]).any() and (~np.signbit(z[z == 0])).any()
        cand = check(z, K)
        top = np.nonzero(key_ranks(z) < K)[0]
        np.testing.assert_array_equal(top, np.nonzero(z == 0)[0][:K])
        assert cand.shape[0] <= (K - 1) * TILE + 1
