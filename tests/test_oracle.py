"""Pins of the CPU oracle against facts fixed outside it.

Each test checks the oracle against something it does not compute itself:
the window behaviour the pages state (PR #1467, gate 4), closed forms of the
rotation and of structured weights, library routines (scipy's Hadamard,
numpy's float16 rounding), distribution facts of the Irwin-Hall sum, an
independent shift-register encoder, and a pure-Python brute force on a tiny
layer.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def tile_of(word, bits):
    return np.full(8 * bits, word, dtype=np.uint32)


def decode_tile(words, bits):
    """Decoded 16x16 tile (k, n) through the oracle's full decode."""
    return oracle.decode(np.asarray(words, dtype=np.uint32).reshape(1, -1), 16, 16, bits)


# ---------------------------------------------------------------- decode rule

def test_window_invariants_from_pages():
    g = json.load(open(os.path.join(GOLDEN, "window_invariants.json")))
    for b in range(1, 9):
        W1 = decode_tile(tile_of(g["all_ones_word"], b), b)
        assert np.unique(W1).size == g["all_ones_distinct_values_per_width"][str(b)]
        Wa = decode_tile(tile_of(g["aaaa_word"], b), b)
        assert np.unique(Wa).size == g["aaaa_distinct_values_per_width"][str(b)], b
        if b % 2 == 1:
            vals = [oracle.value(oracle.state(tile_of(g["aaaa_word"], b), b, j)) for j in range(256)]
            assert all(vals[j] != vals[j + 1] for j in range(255))
            assert all(vals[j] == vals[j + 2] for j in range(254))


def test_single_bit_windows_and_wrap():
    # Only stream bit p set: state_j = 2^((p - j*b) mod L) when that is < 16, else 0.
    rng = np.random.default_rng(5)
    for b in range(1, 9):
        L = 256 * b
        for p in [0, 1, 15, 16, L - 1, L - 16] + list(rng.integers(0, L, 4)):
            p = int(p)
            t = np.zeros(8 * b, dtype=np.uint32)
            t[p // 32] = np.uint32(1 << (p % 32))
            for j in range(256):
                d = (p - j * b) % L
                want = (1 << d) if d < 16 else 0
                assert oracle.state(t, b, j) == want, (b, p, j)


def _encode_walk(stream_bits, b):
    """Independent encoder view: the shift register walk of a tail-biting trellis.

    state_0 is the first 16 stream bits; each step drops the b oldest bits and
    shifts in the next b bits (taken circularly)."""
    L = len(stream_bits)
    s = sum(stream_bits[t] << t for t in range(16))
    out = [s]
    for j in range(1, 256):
        s >>= b
        for q in range(b):
            s |= stream_bits[(j * b + 16 - b + q) % L] << (16 - b + q)
        out.append(s)
    return out


def test_encode_decode_round_trip():
    rng = np.random.default_rng(11)
    for b in range(1, 9):
        L = 256 * b
        bits_ = [int(v) for v in rng.integers(0, 2, L)]
        words = np.zeros(8 * b, dtype=np.uint64)
        for i, v in enumerate(bits_):
            words[i // 32] |= np.uint64(v) << np.uint64(i % 32)
        words = words.astype(np.uint32)
        want = _encode_walk(bits_, b)
        got = [oracle.state(words, b, j) for j in range(256)]
        assert got == want, b


def test_positions_are_the_mma_a_fragment():
    seen = set()
    for lane in range(32):
        g, t = lane >> 2, lane & 3
        mine = {oracle.position(8 * lane + i) for i in range(8)}
        assert mine == {(k, n) for n in (g, g + 8) for k in (2 * t, 2 * t + 1, 2 * t + 8, 2 * t + 9)}
        # consecutive weights pair up along k (the half2 an MMA register holds)
        for i in (0, 2, 4, 6):
            (k0, n0), (k1, n1) = oracle.position(8 * lane + i), oracle.position(8 * lane + i + 1)
            assert n0 == n1 and k1 == k0 + 1
        seen |= mine
    assert seen == {(k, n) for k in range(16) for n in range(16)}


def test_value_set_and_distribution():
    vals = np.array([oracle.value(s) for s in range(1 << 16)])
    sums = np.array([oracle.code_sum(s) for s in range(0, 1 << 16, 97)])
    assert sums.min() >= 0 and sums.max() <= 1020
    # exact FP16: multiples of 2^-7 with |numerator| <= 510
    assert np.all(vals * 128 == np.round(vals * 128)) and np.abs(vals).max() <= 510 / 128
    assert np.all(vals.astype(np.float16).astype(np.float64) == vals)
    # Irwin-Hall sum of four uniform bytes: mean 510, variance 4*(256^2-1)/12
    m, sd = vals.mean(), vals.std()
    sd_ih = math.sqrt(4 * (256 ** 2 - 1) / 12) / 128
    assert abs(m) < 0.01 and abs(sd - sd_ih) < 0.01
    z = (vals - m) / sd
    assert abs((z ** 3).mean()) < 0.02
    assert abs((z ** 4).mean() - (3 - 6 / (5 * 4))) < 0.05  # kurtosis of IH(4) = 3 - 1.2/4
    assert np.unique(vals).size > 800  # a real codebook, not a handful of levels


def test_code_sum_cross_check_python_ints():
    # Same rule through Python big integers and bytes (guards C wrap-around and shifts).
    for s in [0, 1, 2, 0x5555, 0xAAAA, 0x7FFF, 0x8000, 0xFFFF, 12345, 54321]:
        h = (s * 0x9E3779B1 + 0x7F4A7C15) % (1 << 32)
        assert oracle.code_sum(s) == sum(h.to_bytes(4, "little"))


def test_within_tile_positions_b8_byte_probe():
    # b = 8: all-ones tile except stream byte m = 0 changes exactly weights m-1 and m.
    b = 8
    for m in (1, 9, 100, 255):
        words = np.full(8 * b, 0xFFFFFFFF, dtype=np.uint32)
        words[m // 4] &= np.uint32(~(0xFF << (8 * (m % 4))) & 0xFFFFFFFF)
        W = decode_tile(words, b)
        base = oracle.value(0xFFFF)
        special = {oracle.position(m - 1): oracle.value(0x00FF), oracle.position(m): oracle.value(0xFF00)}
        for k in range(16):
            for n in range(16):
                assert W[k, n] == special.get((k, n), base)


def test_tile_addressing_and_orientation():
    K, N, b = 64, 128, 3
    c0, c1 = oracle.value(0), oracle.value(0xFFFF)
    stride = (N // 16) * 8 * b
    # one tile-column of all-ones tiles
    t = np.zeros((K // 16, stride), dtype=np.uint32)
    t[:, 5 * 8 * b:6 * 8 * b] = 0xFFFFFFFF
    W = oracle.decode(t, K, N, b)
    want = np.full((K, N), c0)
    want[:, 80:96] = c1
    assert np.array_equal(W, want)
    # one tile-row of all-ones tiles
    t = np.zeros((K // 16, stride), dtype=np.uint32)
    t[2, :] = 0xFFFFFFFF
    W = oracle.decode(t, K, N, b)
    want = np.full((K, N), c0)
    want[32:48, :] = c1
    assert np.array_equal(W, want)
    # a column view keeps the parent's stride and starts at its first block
    full = synth.codes(3, K, 256, b)
    Wf = oracle.decode(full, K, 256, b)
    Wv = oracle.decode(full, K, 128, b, tile_row_stride=(256 // 16) * 8 * b, col_from=128)
    assert np.array_equal(Wv, Wf[:, 128:])


# ---------------------------------------------------------------- rotation

def test_hadamard_matrix():
    scipy_linalg = pytest.importorskip("scipy.linalg")
    H = oracle.hadamard()
    assert np.array_equal(H, scipy_linalg.hadamard(128).astype(np.float64))
    assert np.array_equal(H @ H.T, 128 * np.eye(128))
    Hn = H / math.sqrt(128)
    e0 = np.zeros(128)
    e0[0] = 1
    assert np.allclose(Hn @ e0, np.full(128, 1 / math.sqrt(128)), rtol=0, atol=1e-15)
    assert np.allclose(Hn @ Hn, np.eye(128), rtol=0, atol=1e-14)


def test_round_f16_matches_numpy():
    rng = np.random.default_rng(1)
    v = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-9, 6, 2000),
                        [65504.0, 65519.99, 65520.0, 70000.0, -65520.0, 2.0 ** -24, 2.0 ** -25,
                         3 * 2.0 ** -26, 2.0 ** -14, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 0.0, -0.0]])
    got = np.array([oracle.round_f16(float(a)) for a in v])
    with np.errstate(over="ignore"):  # the cases past 65520 round to infinity on purpose
        want = v.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, want)


def test_round_bf16_matches_bit_rounding():
    rng = np.random.default_rng(2)
    v32 = (rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000)).astype(np.float32)
    v32 = np.concatenate([v32, np.float32([1 + 2 ** -8, 1 + 3 * 2 ** -8, 3.3895314e38, -1e-40])])
    want = synth.bf16_bits_to_f64(synth.f32_to_bf16_bits(v32))
    got = np.array([oracle.round_bf16(float(a)) for a in v32.astype(np.float64)])
    assert np.array_equal(got, want)


def test_rot_in_equals_block_hadamard_then_fp16():
    rng = np.random.default_rng(3)
    K = 384
    x = rng.standard_normal((3, K)).astype(np.float16).astype(np.float64)
    s = np.where(rng.integers(0, 2, K) == 1, 1.0, -1.0)
    from scipy.linalg import hadamard
    B = np.kron(np.eye(K // 128), hadamard(128)) / math.sqrt(128)
    want = ((x * s) @ B.T).astype(np.float16).astype(np.float64)
    got = oracle.rot_in(x, s)
    # identical up to FP64 summation order deciding an FP16 tie (never on random data)
    assert np.mean(got == want) > 0.999
    assert np.max(np.abs(got - want) / np.maximum(np.abs(want), 1e-3)) < 2 ** -10


# ---------------------------------------------------------------- whole layer

def _dense_expected(t, K, N, b, su, sv, x):
    from scipy.linalg import hadamard
    W = oracle.decode(t, K, N, b)
    HK = np.kron(np.eye(K // 128), hadamard(128)) / math.sqrt(128)
    HN = np.kron(np.eye(N // 128), hadamard(128)) / math.sqrt(128)
    xr = ((x * su) @ HK.T).astype(np.float16).astype(np.float64)
    return ((xr @ W) @ HN.T) * sv


def test_linear_dense_closed_form():
    K, N, b = 256, 384, 5
    t = synth.codes(7, K, N, b)
    su = synth.suh(7, K).astype(np.float64)
    sv = synth.svh(7, N).astype(np.float64)
    x = synth.as_f64(synth.activations(7, 4, K), "f16")
    y = oracle.linear(t, K, N, b, su, sv, x)
    want = _dense_expected(t, K, N, b, su, sv, x)
    assert np.linalg.norm(y - want) / np.linalg.norm(want) < 1e-12


def test_linear_constant_weight_closed_form():
    # all-ones codes: W == c everywhere, so z[n] = c * sum_k xr[k] for every n and
    # rot_out leaves only the first output of each 128-block: y = svh * sqrt(128) * z.
    K, N, b = 512, 256, 4
    rng = np.random.default_rng(9)
    t = np.full((K // 16, (N // 16) * 8 * b), 0xFFFFFFFF, dtype=np.uint32)
    su = np.where(rng.integers(0, 2, K) == 1, 1.0, -1.0)
    sv = np.where(rng.integers(0, 2, N) == 1, 1.0, -1.0)
    x = rng.standard_normal((2, K)).astype(np.float16).astype(np.float64)
    c = (388 - 510) / 128  # code sum of state 0xFFFF is 388 under the rule
    assert oracle.value(0xFFFF) == c
    xr = oracle.rot_in(x, su)
    y = oracle.linear(t, K, N, b, su, sv, x)
    for r in range(2):
        z = c * xr[r].sum()
        for blk in range(N // 128):
            assert abs(y[r, 128 * blk] - sv[128 * blk] * math.sqrt(128) * z) < 1e-9 * abs(z) + 1e-12
            assert np.max(np.abs(y[r, 128 * blk + 1:128 * blk + 128])) < 1e-12 * abs(z) + 1e-12
    # and without rounding the rotated x, the first column is svh * 128 * c * sum_b suh*x at 128b
    xs = x * su
    exact = c * 128 * xs[:, ::128].sum(axis=1)
    assert np.allclose(y[:, 0] * sv[0], exact, rtol=2e-3, atol=1e-3)


def test_linear_structured_columns_closed_form():
    # all-ones tiles in tile-column 3 only: z[n] = c(n) * sum_k xr[k]
    K, N, b = 256, 128, 2
    c0, c1 = oracle.value(0), oracle.value(0xFFFF)
    t = np.zeros((K // 16, (N // 16) * 8 * b), dtype=np.uint32)
    t[:, 3 * 8 * b:4 * 8 * b] = 0xFFFFFFFF
    rng = np.random.default_rng(4)
    su = np.ones(K)
    sv = np.ones(N)
    x = rng.standard_normal((1, K)).astype(np.float16).astype(np.float64)
    xr = oracle.rot_in(x, su)
    cvec = np.full(N, c0)
    cvec[48:64] = c1
    z = cvec * xr[0].sum()
    from scipy.linalg import hadamard
    want = hadamard(128) @ z / math.sqrt(128)
    y = oracle.linear(t, K, N, b, su, sv, x)
    assert np.allclose(y[0], want, rtol=0, atol=1e-10 * np.abs(z).max())


def _brute_force(words2d, K, N, b, su, sv, x):
    """Pure-Python restatement on tiny sizes: bit loop, popcount Hadamard, plain sums."""
    stride = (N // 16) * 8 * b
    flat = [int(w) for w in np.asarray(words2d).reshape(-1)]
    W = [[0.0] * N for _ in range(K)]
    for tk in range(K // 16):
        for tn in range(N // 16):
            base = tk * stride + tn * 8 * b
            tile = flat[base:base + 8 * b]
            stream = sum(w << (32 * i) for i, w in enumerate(tile))
            L = 256 * b
            for j in range(256):
                st = sum(((stream >> ((j * b + q) % L)) & 1) << q for q in range(16))
                h = (st * 0x9E3779B1 + 0x7F4A7C15) & 0xFFFFFFFF
                v = sum((h >> (8 * q)) & 255 for q in range(4))
                lane, i = j // 8, j % 8
                n = lane // 4 + 8 * ((i // 2) % 2)
                k = 2 * (lane % 4) + i % 2 + 8 * (i // 4)
                W[16 * tk + k][16 * tn + n] = (v - 510) / 128
    out = []
    for row in x:
        xr = []
        for blk in range(K // 128):
            for i in range(128):
                s = 0.0
                for j in range(128):
                    sign = -1.0 if bin(i & j).count("1") % 2 else 1.0
                    s += sign * su[128 * blk + j] * row[128 * blk + j]
                xr.append(float(np.float16(s / math.sqrt(128))))
        z = [sum(xr[k] * W[k][n] for k in range(K)) for n in range(N)]
        y = []
        for blk in range(N // 128):
            for i in range(128):
                s = 0.0
                for j in range(128):
                    sign = -1.0 if bin(i & j).count("1") % 2 else 1.0
                    s += sign * z[128 * blk + j]
                y.append(sv[128 * blk + i] * s / math.sqrt(128))
        out.append(y)
    return np.array(out)


def test_linear_brute_force_tiny():
    K = N = 128
    for b in (3, 4):
        t = synth.codes(1, K, N, b)
        su = synth.suh(1, K).astype(np.float64)
        sv = synth.svh(1, N).astype(np.float64)
        x = synth.as_f64(synth.activations(1, 2, K), "f16")
        y = oracle.linear(t, K, N, b, su, sv, x)
        want = _brute_force(t, K, N, b, su, sv, x)
        assert np.max(np.abs(y - want)) < 1e-9 * np.abs(want).max()


def test_rows_independent_and_linear_in_x():
    K, N, b = 256, 256, 4
    t = synth.codes(2, K, N, b)
    su = synth.suh(2, K).astype(np.float64)
    sv = synth.svh(2, N).astype(np.float64)
    x = synth.as_f64(synth.activations(2, 5, K), "f16")
    y = oracle.linear(t, K, N, b, su, sv, x)
    for r in range(5):
        assert np.array_equal(oracle.linear(t, K, N, b, su, sv, x[r:r + 1])[0], y[r])
    # linear up to the FP16 rounding of the rotated x
    y2 = oracle.linear(t, K, N, b, su, sv, 2 * x)
    assert np.array_equal(y2, 2 * y)  # doubling is exact through every step
    ysum = oracle.linear(t, K, N, b, su, sv, x[:1] + x[1:2])
    rel = np.linalg.norm(ysum[0] - (y[0] + y[1])) / np.linalg.norm(y[0] + y[1])
    assert rel < 2e-3


def test_golden_tiny_config_regression():
    # The stored y of the tiny 256x256 layer was written by tests/golden/make_golden.py,
    # which calls only the oracle; it guards against silent drift of the oracle.
    path = os.path.join(GOLDEN, "tiny_k256_n256_b4_seed0.txt")
    want = np.loadtxt(path)
    K = N = 256
    b = 4
    t = synth.codes(0, K, N, b)
    y = oracle.linear(t, K, N, b, synth.suh(0, K).astype(np.float64), synth.svh(0, N).astype(np.float64),
                      synth.as_f64(synth.activations(0, 1, K), "f16"))
    assert np.allclose(y[0], want, rtol=1e-12, atol=1e-12)
