"""GPU parity: the CUDA path through the C ABI against the CPU oracle, and the
byte-identity invariants of TensorFold PR #1467 ("The arithmetic": every
variant returns the bytes of the one-weight launch) and PR #1475 (a repeated
call needs no counter memset)."""
import math

import numpy as np
import pytest
import torch

import exl3_trellis_quantized_rot_gb300 as tfx
import oracle
import synth
from gpu_helpers import (DEV, HostWeight, assert_close, make, oracle_y, same_bytes, to_f64, upload, x_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build_library()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tfx.set_variant(tfx.VARIANT_AUTO)
    yield
    tfx.set_variant(tfx.VARIANT_AUTO)


# ------------------------------------------------------------------ decode

@pytest.mark.parametrize("bits", range(1, 9))
def test_debug_decode_bit_exact(bits):
    hw, w = make(100 + bits, 256, 384, bits)
    got = tfx.debug_decode(w).cpu().numpy()
    want = oracle.decode(hw.codes, 256, 384, bits).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), want.view(np.uint16))
    v = tfx.columns(w, 128, 256)
    gv = tfx.debug_decode(v).cpu().numpy()
    assert np.array_equal(gv.view(np.uint16), want[:, 128:].view(np.uint16))


# ------------------------------------------------------------------ config 1

def test_tiny_layer_matches_oracle():
    hw, w = make(0, 256, 256, 4, max_rows=1)
    x64, x = x_of(0, 1, 256)
    y = tfx.linear(w, x)
    assert_close(to_f64(y), oracle_y(hw, x64), what="tiny")
    assert tfx.plan(w) == (4, 4)


# ------------------------------------------------------------------ config 2

@pytest.mark.parametrize("rows", [1, 7, 16])
def test_decode_rows_single_matches_oracle(rows):
    hw, w = make(1, 5120, 5120, 4)
    x64, x = x_of(1, rows, 5120)
    y = tfx.linear(w, x)
    assert_close(to_f64(y), oracle_y(hw, x64), what=f"5120x5120 rows={rows}")


@pytest.fixture(scope="module")
def qkv():
    out = []
    for m, N in enumerate((6144, 1024, 1024)):
        out.append(make(2, 5120, N, 4, member=m))
    return out


@pytest.mark.parametrize("rows", [1, 7, 16])
def test_group_equals_single_and_oracle(qkv, rows):
    x64, x = x_of(2, rows, 5120)
    ws = [w for _, w in qkv]
    ys = tfx.group(ws, x)
    for (hw, w), yg in zip(qkv, ys):
        ys1 = tfx.linear(w, x)
        assert same_bytes(yg, ys1)
        assert_close(to_f64(yg), oracle_y(hw, x64), what=f"group N={hw.N} rows={rows}")


@pytest.mark.parametrize("rows", [2, 7])
def test_group_planted_controls_go_red(qkv, rows):
    # one member's suh swapped (rot_group, or the in-kernel rotation at 2 rows)
    # and one member's svh swapped must change bytes
    x64, x = x_of(3, rows, 5120)
    (hq, q), (hk, k), (hv, v) = qkv
    ref = tfx.group([q, k, v], x)
    k_bad = tfx.Weight(k._keep[0], q._keep[1], k._keep[2], 5120, 1024, 4)
    tfx.reserve(k_bad, 16)
    bad = tfx.group([q, k_bad, v], x)
    assert same_bytes(bad[0], ref[0]) and same_bytes(bad[2], ref[2])
    assert not same_bytes(bad[1], ref[1])
    v_bad = tfx.Weight(v._keep[0], v._keep[1], k._keep[2], 5120, 1024, 4)
    tfx.reserve(v_bad, 16)
    bad = tfx.group([q, k, v_bad], x)
    assert not same_bytes(bad[2], ref[2])


@pytest.mark.parametrize("variant", [tfx.VARIANT_ROWS, tfx.VARIANT_AUTO, tfx.VARIANT_WARP_GLOBAL])
def test_repeated_calls_need_no_memset(variant):
    # VARIANT_ROWS: every block goes through the in-kernel arrival counters (8 splits);
    # VARIANT_AUTO: the cluster of a block folds its chunk sums in shared memory;
    # VARIANT_WARP_GLOBAL (8 rows): the decode-rows kernel's 16 chunk slabs per
    # block, summed by the last CTA to arrive on the block's counter
    hw, w = make(4, 5120, 1024, 4)
    x64, x = x_of(4, 8 if variant == tfx.VARIANT_WARP_GLOBAL else 16, 5120)
    tfx.set_variant(variant)
    try:
        first = tfx.linear(w, x)
        allocs, memsets = tfx.stats(w)
        y = torch.empty_like(first)
        for _ in range(100):
            tfx.linear(w, x, y=y)
            assert same_bytes(y, first)
    finally:
        tfx.set_variant(tfx.VARIANT_AUTO)
    assert tfx.stats(w) == (allocs, memsets) == (3, 1)
    assert tfx.device_error(w) == 0
    assert_close(to_f64(first), oracle_y(hw, x64), what="repeat")


def test_repeated_tensor_core_calls_need_no_memset():
    hw, w = make(14, 5120, 1024, 4, max_rows=128)
    x64, x = x_of(14, 100, 5120)
    first = tfx.linear(w, x)
    allocs, memsets = tfx.stats(w)
    y = torch.empty_like(first)
    for _ in range(20):
        tfx.linear(w, x, y=y)
        assert same_bytes(y, first)
    assert tfx.stats(w) == (allocs, memsets)
    assert tfx.device_error(w) == 0
    assert_close(to_f64(first), oracle_y(hw, x64), what="tensor-core repeat")


def test_reset_counters_then_same_bytes():
    hw, w = make(5, 5120, 1024, 4)
    x64, x = x_of(5, 3, 5120)
    tfx.set_variant(tfx.VARIANT_ROWS)
    try:
        a = tfx.linear(w, x)
        tfx.reset_counters(w)
        b = tfx.linear(w, x)
    finally:
        tfx.set_variant(tfx.VARIANT_AUTO)
    assert same_bytes(a, b)
    assert same_bytes(a, tfx.linear(w, x))


# ------------------------------------------------------------------ row independence, variants

def test_row_bytes_do_not_depend_on_other_rows():
    hw, w = make(6, 5120, 5120, 4, max_rows=128)
    x64, x = x_of(6, 128, 5120)
    full = tfx.linear(w, x[:16])
    for r in range(16):
        assert same_bytes(tfx.linear(w, x[r:r + 1])[0], full[r])
    rev = tfx.linear(w, torch.flip(x[:16], [0]))
    assert same_bytes(torch.flip(rev, [0]), full)


@pytest.mark.parametrize("K,N,act", [(5120, 5120, tfx.F16), (5120, 17408, tfx.BF16), (17408, 5120, tfx.BF16)])
def test_variants_and_row_counts_byte_identical(K, N, act):
    hw, w = make(7, K, N, 4, act=act, max_rows=128)
    x64, x = x_of(7, 128, K, act)
    tfx.set_variant(tfx.VARIANT_AUTO)
    ref = tfx.linear(w, x)  # 128 rows: mid kernel, NR = 16
    try:
        for rows in (1, 3, 4, 5, 7, 16, 17, 24, 32, 33, 48, 49, 64, 100, 128):
            for var in (tfx.VARIANT_AUTO, tfx.VARIANT_ROWS, tfx.VARIANT_MID, tfx.VARIANT_WARP,
                        tfx.VARIANT_WARP_GLOBAL):
                tfx.set_variant(var)
                y = tfx.linear(w, x[:rows])
                assert same_bytes(y, ref[:rows]), (rows, var)
    finally:
        tfx.set_variant(tfx.VARIANT_AUTO)
    # sampled 128-column blocks against the oracle, all 128 rows
    for blk in (0, N // 256, N // 128 - 1):
        want = oracle_y(hw, x64, col_from=128 * blk, n=128)
        assert_close(to_f64(ref[:, 128 * blk:128 * blk + 128]), want, act, what=f"K={K} N={N} blk={blk}")


@pytest.mark.parametrize("K", [384, 640, 1152])
def test_tensor_core_partial_stages_and_unequal_chunk_pairs(K):
    """K whose chunks are not a whole number of 4-k-step stages (384: C = 4
    chunks of 6 k-steps; 640: C = 8 chunks of 5) or differ in length inside a
    chunk pair (1152: C = 16 chunks of 4 and 5 k-steps alternately, so a pair's
    second stage holds no k-step of its first chunk): every family and row
    count gives the same bytes, and every block matches the oracle."""
    N = 512
    C = 16
    while C > 1 and (K // 16) // C < 4:
        C //= 2
    sizes = [((c + 1) * (K // 16)) // C - (c * (K // 16)) // C for c in range(C)]
    assert any(n % 4 for n in sizes)
    hw, w = make(31, K, N, 4, act=tfx.BF16, max_rows=200)
    x64, x = x_of(31, 200, K, tfx.BF16)
    tfx.set_variant(tfx.VARIANT_AUTO)
    ref = tfx.linear(w, x)  # 200 rows: two 128-row tensor-core passes
    try:
        for rows in (1, 16, 33, 40, 64, 100, 128, 129, 200):
            for var in (tfx.VARIANT_AUTO, tfx.VARIANT_MID, tfx.VARIANT_WARP, tfx.VARIANT_ROWS,
                        tfx.VARIANT_WARP_GLOBAL):
                tfx.set_variant(var)
                y = tfx.linear(w, x[:rows])
                assert same_bytes(y, ref[:rows]), (K, rows, var)
    finally:
        tfx.set_variant(tfx.VARIANT_AUTO)
    want = oracle_y(hw, x64)
    assert_close(to_f64(ref), want, tfx.BF16, what=f"K={K}")
    assert tfx.device_error(w) == 0


@pytest.mark.parametrize("rows", [40, 100])
def test_mid_rows_every_block_against_oracle(rows):
    # every 128-column block of a 2048 x 1024 layer against the oracle, in every
    # kernel family that serves the row count (the byte-identity tests compare
    # families with each other; this checks each of them against the definition)
    hw, w = make(17, 2048, 1024, 4, act=tfx.BF16, max_rows=128)
    x64, x = x_of(17, rows, 2048, tfx.BF16)
    want = oracle_y(hw, x64)
    try:
        for var in (tfx.VARIANT_AUTO, tfx.VARIANT_MID, tfx.VARIANT_WARP, tfx.VARIANT_ROWS):
            tfx.set_variant(var)
            y = tfx.linear(w, x)
            assert_close(to_f64(y), want, tfx.BF16, what=f"rows={rows} variant={var}")
    finally:
        tfx.set_variant(tfx.VARIANT_AUTO)


def test_gate_up_group_mid_rows():
    gate = make(8, 5120, 17408, 4, act=tfx.BF16, member=0, max_rows=128)
    up = make(8, 5120, 17408, 4, act=tfx.BF16, member=1, max_rows=128)
    for rows in (17, 33, 64, 100, 128):
        x64, x = x_of(8, rows, 5120, tfx.BF16)
        yg = tfx.group([gate[1], up[1]], x)
        for (hw, w), y in zip((gate, up), yg):
            assert same_bytes(y, tfx.linear(w, x))
        for (hw, w), y in zip((gate, up), yg):
            blk = 77
            assert_close(to_f64(y[:, 128 * blk:128 * blk + 128]), oracle_y(hw, x64, 128 * blk, 128), tfx.BF16,
                         what=f"gate/up rows={rows}")


@pytest.mark.parametrize("rows", [40, 128, 200])
def test_qkv_group_at_tensor_core_rows(rows):
    """q/k/v (N = 6144, 1024, 1024) as one group at tensor-core row counts: the
    persistent grid walks units of three members of unequal N (and 200 rows
    take two passes); each member's bytes equal its own call, and its first
    and last blocks match the oracle."""
    ws = [make(2, 5120, N, 4, member=m, max_rows=200) for m, N in enumerate((6144, 1024, 1024))]
    x64, x = x_of(41, rows, 5120)
    ys = tfx.group([w for _, w in ws], x)
    for (hw, w), y in zip(ws, ys):
        assert same_bytes(y, tfx.linear(w, x)), (hw.N, rows)
        for blk in (0, hw.N // 128 - 1):
            assert_close(to_f64(y[:, 128 * blk:128 * blk + 128]), oracle_y(hw, x64, 128 * blk, 128),
                         what=f"q/k/v group N={hw.N} rows={rows} blk={blk}")
        assert tfx.device_error(w) == 0


@pytest.mark.parametrize("rows", [40, 128, 200])
def test_column_view_at_tensor_core_rows(rows):
    """A view of blocks [4, 12) of a 1024 x 2048 6-bit weight at tensor-core row
    counts gives the bytes of the same columns of the full call (the view keeps
    the parent's strides and plan), and its first block matches the oracle."""
    hw, w = make(43, 1024, 2048, 6, act=tfx.BF16, max_rows=200)
    v = tfx.columns(w, 512, 1024)
    tfx.reserve(v, 200)
    x64, x = x_of(43, rows, 1024, tfx.BF16)
    full = tfx.linear(w, x)
    yv = tfx.linear(v, x)
    assert same_bytes(yv, full[:, 512:1536]), rows
    assert_close(to_f64(yv[:, :128]), oracle_y(hw, x64, 512, 128), tfx.BF16, what=f"view rows={rows}")


def test_prefill_4096_rows():
    hw, w = make(9, 5120, 17408, 4, act=tfx.BF16, max_rows=4096)
    x64, x = x_of(9, 4096, 5120, tfx.BF16)
    y = tfx.linear(w, x)
    # a pass's rows equal the same rows in their own call
    for r0 in (0, 128, 2048, 3968):
        assert same_bytes(y[r0:r0 + 128], tfx.linear(w, x[r0:r0 + 128]))
    rows = [0, 127, 128, 1000, 2047, 4095]
    for blk in (0, 37, 100, 135):
        want = oracle_y(hw, x64[rows], 128 * blk, 128)
        assert_close(to_f64(y[rows][:, 128 * blk:128 * blk + 128]), want, tfx.BF16, what=f"prefill blk={blk}")


def test_ragged_last_pass():
    hw, w = make(10, 1024, 2048, 3, max_rows=300)
    x64, x = x_of(10, 300, 1024)
    y = tfx.linear(w, x)
    assert_close(to_f64(y), oracle_y(hw, x64), what="300 rows")
    assert same_bytes(y[256:], tfx.linear(w, x[256:]))


# ------------------------------------------------------------------ bit widths

@pytest.mark.parametrize("bits", range(1, 9))
def test_bit_sweep(bits):
    hw, w = make(20 + bits, 5120, 5120, bits, max_rows=64)
    for rows in (1, 64):
        x64, x = x_of(20 + bits, rows, 5120)
        y = tfx.linear(w, x)
        if rows == 1:
            assert_close(to_f64(y), oracle_y(hw, x64), what=f"bits={bits} rows=1")
        else:
            for blk in (0, 39):
                assert_close(to_f64(y[:, 128 * blk:128 * blk + 128]), oracle_y(hw, x64, 128 * blk, 128),
                             what=f"bits={bits} rows=64 blk={blk}")


# ------------------------------------------------------------------ lm head views

def test_lm_head_views_equal_full_head():
    K, N, bits = 5120, 248320, 6
    hw, w = make(11, K, N, bits)
    first = tfx.columns(w, 0, 98304)
    tail = tfx.columns(w, 240128, 8192)
    tfx.reserve(first, 16)
    tfx.reserve(tail, 16)
    assert tfx.plan(first) == tfx.plan(tail) == tfx.plan(w) == (16, 20)
    for rows in (1, 8, 16):
        x64, x = x_of(11, rows, K)
        full = tfx.linear(w, x)
        assert same_bytes(tfx.linear(first, x), full[:, :98304])
        assert same_bytes(tfx.linear(tail, x), full[:, 240128:])
        for blk in (0, 1000, 1939):
            assert_close(to_f64(full[:, 128 * blk:128 * blk + 128]), oracle_y(hw, x64, 128 * blk, 128),
                         what=f"head rows={rows} blk={blk}")


def test_lm_head_span_packing_equals_full_head():
    """The drafter's head over two vocabulary spans (PR #1507, "What this
    changes"): the view [0, 98304) and the last 64 blocks, packed into one
    logits buffer without the tail's first 7,904 columns, in one group_into
    call; every packed element has the bytes of the same column of the full
    head."""
    K, N, bits = 5120, 248320, 6
    hw, w = make(11, K, N, bits)
    first = tfx.columns(w, 0, 98304)
    tail = tfx.columns(w, 240128, 8192)
    tfx.reserve(first, 16)
    tfx.reserve(tail, 16)
    keep = 248320 - 240128 - 7904  # 288 columns of the tail
    for rows in (1, 8, 16):
        x64, x = x_of(11, rows, K)
        full = tfx.linear(w, x)
        packed = torch.full((rows, 98304 + keep), float("nan"), dtype=torch.float16, device=DEV)
        tfx.pack_spans([first, tail], x, packed, [0, 7904])
        assert same_bytes(packed[:, :98304], full[:, :98304])
        assert same_bytes(packed[:, 98304:], full[:, 240128 + 7904:])


@pytest.mark.parametrize("variant", [tfx.VARIANT_AUTO, tfx.VARIANT_ROWS, tfx.VARIANT_MID, tfx.VARIANT_WARP,
                                     tfx.VARIANT_WARP_GLOBAL])
def test_output_window_bytes_equal_plain_call(variant):
    # a member's output window (row stride, first stored column) changes where
    # elements land, never their bytes; columns below col0 and the padding of
    # each row stay untouched
    hw, w = make(15, 1024, 768, 4, max_rows=128)
    hk, k = make(15, 1024, 256, 4, member=1, max_rows=128)
    tfx.set_variant(variant)
    try:
        for rows in (1, 7, 16, 40, 128):
            x64, x = x_of(15, rows, 1024)
            ref_w, ref_k = tfx.linear(w, x), tfx.linear(k, x)
            out = torch.full((rows, 1000), 3.0, dtype=torch.float16, device=DEV)
            ld = 1000
            tfx.group_into([w, k], x, [out.data_ptr(), out.data_ptr() + 2 * (768 - 136)], [ld, ld], [136, 8])
            assert same_bytes(out[:, :768 - 136], ref_w[:, 136:]), rows
            assert same_bytes(out[:, 768 - 136:768 - 136 + 248], ref_k[:, 8:]), rows
            assert bool((out[:, 768 - 136 + 248:] == 3.0).all()), rows
    finally:
        tfx.set_variant(tfx.VARIANT_AUTO)


def test_output_window_validation():
    hw, w = make(16, 256, 256, 4)
    x64, x = x_of(16, 1, 256)
    y = torch.empty((1, 512), dtype=torch.float16, device=DEV)
    for ld, c0 in ((256, 4), (256, 256), (248, 0), (300, 0), (256, -8)):
        with pytest.raises(tfx.TfxError) as e:
            tfx.group_into([w], x, [y], [ld], [c0])
        assert e.value.code == tfx.EINVAL, (ld, c0)


# ------------------------------------------------------------------ edge cases and stress

def test_zero_rows_is_a_no_op():
    hw, w = make(12, 256, 256, 4)
    y = torch.full((1, 256), 7.0, dtype=torch.float16, device=DEV)
    x = torch.zeros((1, 256), dtype=torch.float16, device=DEV)
    tfx.linear(w, x, rows=0, y=y)
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


def test_nan_and_inf_reach_their_rows_only():
    hw, w = make(13, 1024, 1024, 4)
    x64, x = x_of(13, 8, 1024)
    clean = tfx.linear(w, x)
    xb = x.clone()
    xb[2, 5] = float("nan")
    xb[3, 700] = float("inf")
    xb[5, 1] = float("-inf")
    for var in (tfx.VARIANT_AUTO, tfx.VARIANT_ROWS, tfx.VARIANT_MID, tfx.VARIANT_WARP, tfx.VARIANT_WARP_GLOBAL):
        tfx.set_variant(var)
        try:
            y = tfx.linear(w, xb)
        finally:
            tfx.set_variant(tfx.VARIANT_AUTO)
        yf = y.float()
        for r in (2, 3, 5):
            assert not bool(torch.isfinite(yf[r]).any()), r
        for r in (0, 1, 4, 6, 7):
            assert same_bytes(y[r], clean[r])
    xb64 = x64.copy()
    xb64[2, 5] = np.nan
    xb64[3, 700] = np.inf
    xb64[5, 1] = -np.inf
    want = oracle_y(hw, xb64)
    assert np.array_equal(np.isfinite(want), np.isfinite(to_f64(y)))


def test_constant_weight_closed_form_and_fp32_accumulation():
    # all-ones codes decode to one weight c at every width; with rotated inputs of
    # ~4096 every FP16 running sum would overflow, the FP32 one stays in range.
    K, N = 5120, 256
    c = (388 - 510) / 128
    for bits in (3, 4, 5, 6):
        codes = np.full((K // 16, (N // 16) * 8 * bits), 0xFFFFFFFF, dtype=np.uint32)
        hw = HostWeight(30, K, N, bits, codes=codes)
        w = upload(hw, tfx.BF16)
        tfx.reserve(w, 4)
        v = 46336.0  # bf16-exact, rotates to ~4096 in every position of its block
        xs = np.zeros((2, K))
        xs[0, ::128] = v
        xs[1, ::128] = -v / 2
        x64 = xs * hw.suh.astype(np.float64)
        xt = torch.from_numpy(x64.astype(np.float32)).to(DEV).to(torch.bfloat16)
        y = to_f64(tfx.linear(w, xt))
        xr = oracle.rot_in(x64, hw.suh.astype(np.float64))
        assert np.abs(xr[0]).max() > 4000
        for r in range(2):
            z = c * xr[r].sum()
            assert abs(z) > 65504 * 100
            for blk in range(N // 128):
                lead = hw.svh[128 * blk] * math.sqrt(128) * z
                assert abs(y[r, 128 * blk] - lead) <= 2 ** -7 * abs(lead)
                assert np.all(y[r, 128 * blk + 1:128 * blk + 128] == 0.0)
