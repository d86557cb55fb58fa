"""The threshold's two-level form, checked on the CPU.

The fused sampling grid, when blocks x (t + 1) <= 2048, lets each block of
512 draws keep its own t largest and ranks only their union.  That is exact
because every draw among the t largest of all S draws is also among the t
largest of its own block (fewer draws of its block outrank it than of all
S).  With draws made with replacement a position can appear twice; equal
keys then take consecutive ranks in slot order.  Here the draws come from
the oracle's Philox sampler on rows small enough for many repeats, and the
union's t-th largest is compared with the oracle's order statistic of all
draws.
"""
import numpy as np
import pytest

from oracle import philox, plain

BLOCK_DRAWS = 512


def _block_top(keys, t):
    """The t largest of one block, equal keys ranked in slot order (a stable sort)."""
    order = np.argsort(-keys.astype(np.float64), kind="stable")
    return keys[order[:t]]


@pytest.mark.parametrize("n,S,t", [(65600, 32768, 22), (70000, 32768, 9), (1 << 20, 86966, 7), (65600, 4096, 3)])
@pytest.mark.parametrize("counter", [0, 1, 2])
def test_union_of_block_tops_holds_the_t_th_largest_draw(n, S, t, counter):
    x = np.random.default_rng(counter).integers(0, 1 << 20, size=n).astype(np.float32)
    pos = philox.sample_positions(n, S, seed=0x243F6A8885A308D3, counter=counter)
    assert np.unique(pos).size < pos.size or S < 8192  # repeats are common on these rows
    # a draw's key: its value, then the lower position first (the engine's composite order)
    keys = x[pos].astype(np.float64) * n + (n - 1 - pos)
    union = np.concatenate([_block_top(keys[b:b + BLOCK_DRAWS], t) for b in range(0, S, BLOCK_DRAWS)])
    assert union.size <= (S + BLOCK_DRAWS - 1) // BLOCK_DRAWS * t
    kth = np.sort(union)[::-1][t - 1]
    want = plain.sample_order_stat(x, pos, t)          # position of the t-th largest draw
    assert kth == float(x[want]) * n + (n - 1 - want)


def _union_kth(keys, t):
    union = np.concatenate([_block_top(keys[b:b + BLOCK_DRAWS], t) for b in range(0, keys.size, BLOCK_DRAWS)])
    return np.sort(union)[::-1][t - 1]


@pytest.mark.parametrize("t", [1, 7, 93, 512])
def test_one_block_holding_all_of_the_t_largest(t):
    # the t largest draws all sit in block 0 (each block must keep a full t),
    # and equal keys (a position drawn twice) straddle the t-th place
    rng = np.random.default_rng(t)
    keys = rng.integers(0, 1 << 30, size=4 * BLOCK_DRAWS).astype(np.float64)
    top = np.sort(rng.integers(1 << 31, 1 << 32, size=t).astype(np.float64))[::-1]
    if t >= 2:
        top[t - 1] = top[t - 2]                   # a repeated draw at places t-1 and t
    keys[:t] = top                                 # block 0
    want = np.sort(keys)[::-1][t - 1]
    assert _union_kth(keys, t) == want
    if t >= 2:
        # one key fewer per block would lose the t-th largest draw
        short = np.concatenate([_block_top(keys[b:b + BLOCK_DRAWS], t - 1)
                                for b in range(0, keys.size, BLOCK_DRAWS)])
        assert np.sort(short)[::-1][t - 1] < want


def test_single_block_union_is_the_block():
    keys = np.random.default_rng(5).permutation(500).astype(np.float64)
    assert _union_kth(keys, 7) == 493.0   # 499, 498, ..., 493
