"""The arithmetic behind the packed calls' 1-D grid (no GPU): CTA k takes tile k - Q(b) of the last
sequence b with Q(b) = floor(cu_seqlens[b] / tile) + b <= k. For non-decreasing cu_seqlens inside
[0, T], Q increases strictly and leaves room for every tile of every sequence, so a grid of
floor(T / tile) + B CTAs gives each tile exactly one CTA and leaves at most one CTA per sequence
(plus those before Q(0)) without tokens."""
import numpy as np
import pytest


def _assign(cu, T, tile):
    B = len(cu) - 1
    Q = np.floor_divide(cu[:B], tile) + np.arange(B)
    owner = {}
    for k in range(T // tile + B):
        b = int(np.searchsorted(Q, k, side="right")) - 1  # the last sequence with Q(b) <= k
        if b < 0:
            continue
        j = k - int(Q[b])
        if j * tile < cu[b + 1] - cu[b]:
            assert (b, j) not in owner
            owner[(b, j)] = k
    return Q, owner


@pytest.mark.parametrize("tile", [4, 8, 32, 64])
@pytest.mark.parametrize("seed", range(25))
def test_every_tile_has_one_cta(tile, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 300))
    lens = rng.choice([0, 0, 1, 2, 3, tile - 1, tile, tile + 1, 3 * tile, 200], size=B)
    lead, trail = int(rng.integers(0, 3 * tile)), int(rng.integers(0, 3 * tile))
    cu = lead + np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1]) + trail
    Q, owner = _assign(cu, T, tile)
    assert np.all(np.diff(Q) >= 1)  # strictly increasing
    assert np.all(np.diff(Q) >= -(-lens[:-1] // tile))  # room for each sequence's tiles
    n_tiles = -(-lens // tile)
    assert len(owner) == int(n_tiles.sum())
    for b in range(B):
        for j in range(int(n_tiles[b])):
            assert (b, j) in owner
    # CTAs from Q(0) up to Q(B) = floor(cu[B] / tile) + B: those without tokens are at most one per sequence
    q_end = int(cu[-1]) // tile + B
    idle = q_end - int(Q[0]) - len(owner)
    assert 0 <= idle <= B
    assert q_end <= T // tile + B  # the grid covers them
