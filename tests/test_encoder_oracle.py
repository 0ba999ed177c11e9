"""Pins of the trellis encoder's CPU oracle (exl3_encoder_oracle.c).

The pages show no encoder (their weights come from trained checkpoints); the
encoder follows QTIP's Viterbi search over the bit-shift trellis with its
two-pass tail-biting approximation, on integer targets of the value grid.
Nothing here reuses the oracle's DP: the DP is checked against brute force
over every path of small trellises, and the encoded tiles are decoded by the
oracle's decoder (exl3_oracle.c, pinned in test_oracle.py) to recompute
their error.
"""
import itertools

import numpy as np
import pytest

import oracle


def brute_force(W, bits, val, T, constrain=False, c=0):
    """Cheapest state path by enumeration: a start state and the new bits of
    every later step determine the path."""
    n = len(T)
    m = (1 << (W - bits)) - 1
    best = None
    for s0 in range(1 << W):
        if constrain and (s0 & m) != c:
            continue
        for us in itertools.product(range(1 << bits), repeat=n - 1):
            s, cost = s0, (val[s0] - T[0]) ** 2
            for j, u in enumerate(us, start=1):
                s = (s >> bits) | (u << (W - bits))
                cost += (val[s] - T[j]) ** 2
            if constrain and (s >> bits) != c:
                continue
            if best is None or cost < best:
                best = cost
    return best


def path_cost_and_validity(W, bits, val, T, states):
    m = (1 << (W - bits)) - 1
    for j in range(1, len(states)):
        assert (int(states[j]) & m) == (int(states[j - 1]) >> bits), "not a trellis path"
    return sum((val[int(s)] - t) ** 2 for s, t in zip(states, T))


@pytest.mark.parametrize("W,bits,n", [(4, 1, 6), (4, 2, 4), (5, 2, 4), (6, 3, 3), (5, 1, 7)])
def test_viterbi_equals_brute_force(W, bits, n):
    rng = np.random.default_rng(W * 100 + bits * 10 + n)
    m = (1 << (W - bits)) - 1
    for trial in range(4):
        val = rng.integers(-20, 21, size=1 << W)
        T = rng.integers(-20, 21, size=n)
        cost, st = oracle.viterbi(W, bits, val, T)
        assert cost == brute_force(W, bits, val, T)
        assert path_cost_and_validity(W, bits, val, T, st) == cost
        for c in (0, m, int(rng.integers(0, m + 1))):
            cost_c, st_c = oracle.viterbi(W, bits, val, T, constrain=True, c=c)
            bf = brute_force(W, bits, val, T, constrain=True, c=c)
            assert cost_c == bf, (trial, c)
            assert path_cost_and_validity(W, bits, val, T, st_c) == cost_c
            assert (int(st_c[0]) & m) == c and (int(st_c[-1]) >> bits) == c


def test_viterbi_ties_take_the_smaller_predecessor_and_state():
    # all values equal: every path costs the same; the DP keeps v = 0 at every
    # step and the smallest end state, so the path is the all-zero one
    W, bits = 6, 2
    val = np.zeros(1 << W, dtype=np.int64)
    cost, st = oracle.viterbi(W, bits, val, np.zeros(5, dtype=np.int64))
    assert cost == 0 and np.all(st == 0)


def decode_tile_grid(words, bits):
    """Grid values (units of 1/128) of a tile's 256 weights in stream order,
    by the oracle's decoder."""
    return np.array([oracle.code_sum(oracle.state(words, bits, j)) - 510 for j in range(256)])


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_encoded_tile_error_recomputed_by_the_decoder(bits):
    rng = np.random.default_rng(bits)
    T = np.clip(np.rint(rng.normal(0.0, 1.155, 256) * 128), -1024, 1023).astype(np.int64)
    words, err = oracle.encode_tile(T, bits)
    got = decode_tile_grid(words, bits)
    assert int(((got - T) ** 2).sum()) == err


def test_representable_targets_reach_zero_in_the_unconstrained_pass():
    # targets that ARE the decoded values of a random tail-biting code: the
    # first (rotated, unconstrained) pass finds a path of zero error
    rng = np.random.default_rng(7)
    val = oracle.state_values()
    for bits in (2, 4):
        words = rng.integers(0, 1 << 32, size=8 * bits, dtype=np.uint64).astype(np.uint32)
        T = decode_tile_grid(words, bits)
        R = np.roll(T, -128)
        cost, _ = oracle.viterbi(16, bits, val, R)
        assert cost == 0


def test_error_falls_with_bits():
    rng = np.random.default_rng(11)
    T = np.clip(np.rint(rng.normal(0.0, 1.155, 256) * 128), -1024, 1023).astype(np.int64)
    errs = [oracle.encode_tile(T, b)[1] for b in (1, 2, 3, 4, 5)]
    assert all(a > b for a, b in zip(errs, errs[1:])), errs
    # 4 bits per weight: mean squared error well under 1 % of the target variance
    assert errs[3] / 256 / 128 ** 2 < 0.01 * 1.155 ** 2


def test_encode_places_tiles_like_the_decoder_reads_them():
    # a 32 x 48 weight (6 tiles): decoding the encoded words with the oracle's
    # layer decoder gives values whose error against the targets is the
    # reported one, tile by tile
    K, N, bits = 32, 48, 3
    rng = np.random.default_rng(5)
    Tg = np.clip(np.rint(rng.normal(0.0, 1.155, (K, N)) * 128), -1024, 1023).astype(np.int16)
    trellis, err = oracle.encode(Tg, K, N, bits)
    W = oracle.decode(trellis, K, N, bits)
    assert int(((np.rint(W * 128) - Tg) ** 2).sum()) == err
    # a subrange of tiles leaves the others zero and reports their error only
    part, err2 = oracle.encode(Tg, K, N, bits, tile0=2, ntiles=3)
    tiles = part.reshape(K // 16, N // 16, 8 * bits)
    assert np.all(tiles.reshape(-1, 8 * bits)[[0, 1, 5]] == 0)
    assert np.array_equal(tiles.reshape(-1, 8 * bits)[2:5], trellis.reshape(K // 16, N // 16, 8 * bits).reshape(-1, 8 * bits)[2:5])
    assert 0 < err2 < err
