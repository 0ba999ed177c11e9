"""Host logic of the C ABI, run without a GPU.

The allocator and memset of reserve/release are replaced by a counting fake
(tfx_exl3_debug_set_driver) so the grow-only zeroing can be checked on CPU;
every other check stops at validation, before any CUDA call.
"""
import ctypes as C
import os
import re

import pytest

import exl3_trellis_quantized_rot_gb300 as tfx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build_library()
    return tfx.lib()


def header_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"\b(tfx_exl3_[a-z0-9_]+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol(L):
    names = header_symbols()
    assert "tfx_exl3_linear" in names and "tfx_exl3_group" in names
    for n in sorted(names):
        assert hasattr(L, n), n
    assert set(tfx.ABI_SYMBOLS) <= names


class FakeDriver:
    """Counting stand-in for cudaMallocAsync / cudaFreeAsync / cudaMemsetAsync."""

    def __init__(self):
        self.allocs, self.frees, self.memsets = [], [], []
        self.next = 1 << 20
        self.s = tfx.DriverStruct(tfx.ALLOC_FN(self._alloc), tfx.FREE_FN(self._free), tfx.MEMSET_FN(self._memset))

    def _alloc(self, pp, nbytes, stream):
        p = self.next
        self.next += (nbytes + 4095) // 4096 * 4096 + 4096
        pp[0] = p
        self.allocs.append((p, nbytes, stream))
        return 0

    def _free(self, p, stream):
        self.frees.append((p, stream))
        return 0

    def _memset(self, p, nbytes, stream):
        self.memsets.append((p, nbytes, stream))
        return 0


@pytest.fixture
def drv(L):
    d = FakeDriver()
    tfx.set_driver(d.s)
    yield d
    tfx.set_driver(None)


FAKE = 0x7F0000000000  # aligned stand-in device addresses (never dereferenced on the host)


def fake_weight(K, N, bits, act=tfx.F16):
    return tfx.Weight(FAKE, FAKE + (1 << 30), FAKE + (2 << 30), K, N, bits, act)


def test_plan_rule(L):
    # the plan is the number of K chunks whose tree-ordered sum defines the bits:
    # a power of two <= 16 with at least 4 tiles per chunk; rows, N and bits never enter
    for N in (128, 384, 1024, 5120, 8192, 17408, 248320):
        assert tfx.plan(fake_weight(5120, N, 4)) == (16, 20)
    assert tfx.plan(fake_weight(17408, 5120, 4)) == (16, 68)
    assert tfx.plan(fake_weight(256, 256, 4)) == (4, 4)
    assert tfx.plan(fake_weight(128, 256, 4)) == (2, 4)
    assert tfx.plan(fake_weight(5120, 1024, 1)) == tfx.plan(fake_weight(5120, 1024, 8))
    for K in range(128, 20000, 128):
        C, tiles = tfx.plan(fake_weight(K, 256, 4))
        assert C & (C - 1) == 0 and 1 <= C <= 16 and (K // 16) // C >= 4
        assert C == 16 or 2 * C > (K // 16) // 4


def test_head_views_plan_like_the_head(L):
    # the pages' tail view had to take 64 blocks so that it planned like the head;
    # here the plan depends on K alone, so every whole-block view plans like its parent
    head = fake_weight(5120, 248320, 6)
    for start, n in [(0, 98304), (240128, 8192), (247936, 384), (128, 128)]:
        assert tfx.plan(tfx.columns(head, start, n)) == tfx.plan(head)


def test_columns_view_keeps_strides_and_moves_to_first_block(L):
    K, N, b = 512, 1024, 3
    w = fake_weight(K, N, b)
    v = tfx.columns(w, 256, 512)
    assert v.s.tile_row_stride == w.s.tile_row_stride == (N // 16) * 8 * b
    assert v.s.trellis == w.s.trellis + (256 // 16) * 8 * b * 4
    assert v.s.svh == w.s.svh + 256 * 2
    assert v.s.suh == w.s.suh and v.s.K == K and v.s.N == 512 and v.s.bits == b
    assert not v.s.priv
    # a view of a view composes
    vv = tfx.columns(v, 128, 256)
    assert vv.s.trellis == w.s.trellis + (384 // 16) * 8 * b * 4
    for bad in [(1, 128), (0, 100), (896, 256), (-128, 128), (0, 0)]:
        with pytest.raises(tfx.TfxError) as e:
            tfx.columns(w, *bad)
        assert e.value.code == tfx.EINVAL


def test_reserve_grows_only_and_zeroes_counters_once_per_growth(L, drv):
    w = fake_weight(5120, 5120, 4)
    stream = 0x1234
    tfx.reserve(w, 16, stream)
    assert len(drv.allocs) == 3 and len(drv.memsets) == 1
    cnt_ptr = drv.memsets[0][0]
    assert drv.memsets[0][2] == stream  # on the call's stream, not the legacy stream
    assert all(a[2] == stream for a in drv.allocs)
    # counter buffer: the device error word (padded to 4 ints), then 1 pass x 40 blocks
    assert drv.memsets[0][1] == (4 + 40) * 4 and cnt_ptr in [a[0] for a in drv.allocs]
    # same or fewer rows: nothing
    for r in (1, 7, 16):
        tfx.reserve(w, r, stream)
    assert len(drv.allocs) == 3 and len(drv.memsets) == 1
    assert tfx.stats(w) == (3, 1)
    # more rows within one 64-row pass: scratch grows, counters do not
    tfx.reserve(w, 64, stream)
    assert len(drv.memsets) == 1
    # more passes: the counter buffer grows and is zeroed once, on the stream
    tfx.reserve(w, 200, 0x99)
    assert len(drv.memsets) == 2 and drv.memsets[1][2] == 0x99 and drv.memsets[1][1] == (4 + 4 * 40) * 4
    freed = {p for p, _ in drv.frees}
    assert cnt_ptr in freed
    tfx.release(w)
    assert not w.s.priv


def test_group_reserve_sizes_each_member(L, drv):
    q, k, v = fake_weight(5120, 6144, 4), fake_weight(5120, 1024, 4), fake_weight(5120, 1024, 4)
    for m in (q, k, v):
        tfx.reserve(m, 16, 7)
    n_alloc = len(drv.allocs)
    # a reserved group call at 1..16 rows would allocate and zero nothing: reserve again is a no-op
    for m in (q, k, v):
        tfx.reserve(m, 16, 7)
    assert len(drv.allocs) == n_alloc


def test_validation_errors_before_any_launch(L, drv):
    w = fake_weight(256, 256, 4)
    x = FAKE + (3 << 30)
    y = FAKE + (4 << 30)
    # not reserved
    assert L.tfx_exl3_linear(w.ref(), x, 1, y, None) == tfx.ENOTRESERVED
    tfx.reserve(w, 8, 0)
    assert L.tfx_exl3_linear(w.ref(), x, 9, y, None) == tfx.ENOTRESERVED
    assert "reserved for 8" in tfx.last_error()
    # rows == 0 is a no-op
    assert L.tfx_exl3_linear(w.ref(), x, 0, y, None) == 0
    assert L.tfx_exl3_linear(w.ref(), x, -1, y, None) == tfx.EINVAL
    # alignment
    assert L.tfx_exl3_linear(w.ref(), x + 2, 1, y, None) == tfx.EALIGN
    assert L.tfx_exl3_linear(w.ref(), x, 1, y + 8, None) == tfx.EALIGN
    # shapes and bits
    for K, N, b in [(100, 256, 4), (256, 200, 4), (256, 256, 0), (256, 256, 9)]:
        bad = fake_weight(K, N, b)
        assert L.tfx_exl3_reserve(bad.ref(), 4, None) == tfx.EINVAL
    # stride below the weight's own
    bad = tfx.Weight(FAKE, FAKE, FAKE, 256, 256, 4, tile_row_stride=10)
    assert L.tfx_exl3_plan(bad.ref(), None, None) == tfx.EINVAL
    # group members must share K and bits; count within 1..3
    a, b2 = fake_weight(256, 256, 4), fake_weight(512, 256, 4)
    tfx.reserve(a, 4, 0)
    tfx.reserve(b2, 4, 0)
    arr = (C.POINTER(tfx.WeightStruct) * 2)(C.pointer(a.s), C.pointer(b2.s))
    ys = (C.c_void_p * 2)(y, y)
    assert L.tfx_exl3_group(arr, 2, x, 1, ys, None) == tfx.EUNSUPPORTED
    assert L.tfx_exl3_group(arr, 4, x, 1, ys, None) == tfx.EINVAL
    assert L.tfx_exl3_group(arr, 0, x, 1, ys, None) == tfx.EINVAL
    # reset_counters on an unreserved weight
    assert L.tfx_exl3_reset_counters(fake_weight(256, 256, 4).ref(), None) == tfx.ENOTRESERVED


def test_reset_counters_goes_to_the_stream(L, drv):
    w = fake_weight(256, 384, 2)
    tfx.reserve(w, 4, 0x55)
    tfx.reset_counters(w, 0x66)
    assert drv.memsets[-1][2] == 0x66 and drv.memsets[-1][1] == (4 + 3) * 4
    assert tfx.stats(w) == (3, 2)


def test_variant_and_pdl_switches(L):
    old = tfx.set_variant(tfx.VARIANT_MID)
    assert tfx.set_variant(old) == tfx.VARIANT_MID
    old = tfx.set_pdl(False)
    assert tfx.set_pdl(old) == 0
    # three modes; the default (unless TFX_EXL3_PDL overrides it) is automatic
    if os.environ.get("TFX_EXL3_PDL") not in ("0", "1"):
        assert old == 2
    assert tfx.set_pdl(1) == old and tfx.set_pdl(2) == 1 and tfx.set_pdl(old) == 2
    with pytest.raises(tfx.TfxError):
        tfx.set_pdl(3)
    assert tfx.set_pdl(old) == old


def test_kernel_choice_and_tensor_core_unit_size(L):
    """The launch-shape rules (host only): auto sends 1..16 rows to the
    warp-granular decode-rows kernel and every longer call to the tensor-core
    kernel; the tensor-core unit size G (chunks of K per unit) is the measured
    best for the 27B shapes on 152 SMs and always fits TMEM; forced variants
    serve the row counts they cover. None of this changes the bits (the GPU
    parity tests compare the families byte for byte)."""
    shape = tfx.debug_launch_shape
    old = tfx.set_variant(tfx.VARIANT_AUTO)
    try:
        for rows in (1, 7, 8, 9, 16):
            assert shape(5120, 4, rows, 40, 152) == (tfx.FAMILY_ROWS_WARP, 0), rows
        for rows in (17, 31, 32, 33, 48, 64, 65, 100, 128, 129, 4096):
            assert shape(5120, 4, rows, 40, 152)[0] == tfx.FAMILY_TENSOR, rows
        # G on 152 SMs, K = 5120 (16 chunks): 5120 x 5120 (40 blocks), the q/k/v group (64 blocks), gate+up (272)
        want = {(40, 64): 2, (40, 128): 2, (64, 64): 8, (64, 128): 8, (272, 64): 16, (272, 128): 16}
        for (blocks, rows), g in want.items():
            assert shape(5120, 4, rows, blocks, 152) == (tfx.FAMILY_TENSOR, g), (blocks, rows)
        # above 128 rows every unit holds all C chunks of a 128-row pass (no slabs)
        assert shape(5120, 4, 4096, 136, 152) == (tfx.FAMILY_TENSOR, 16)
        assert shape(1024, 4, 200, 8, 152) == (tfx.FAMILY_TENSOR, 16)
        # G is a power of two dividing C, at least 2 (units hold whole chunk
        # pairs), whose chunk-tree levels above the pairs fit: the TMEM levels
        # next to four accumulator regions of rows16 columns, plus at most
        # three levels parked in global scratch
        for K in (256, 1024, 5120, 17408):
            c = min(16, K // 64)
            c = 1 << (c.bit_length() - 1)
            for rows in (33, 40, 64, 96, 128):
                for blocks in (1, 8, 40, 64, 272, 1940):
                    for sms in (1, 152, 1000):
                        f, g = shape(K, 4, rows, blocks, sms)
                        assert f == tfx.FAMILY_TENSOR
                        assert g >= 2 and g & (g - 1) == 0 and c % g == 0, (K, rows, blocks, sms, g)
                        tmem_levels = min(3, 512 // ((rows + 15) // 16 * 16) - 4)
                        assert g.bit_length() - 2 <= tmem_levels + 3
        # forced families
        tfx.set_variant(tfx.VARIANT_MID)
        assert shape(5120, 4, 1, 40, 152)[0] == tfx.FAMILY_TENSOR
        tfx.set_variant(tfx.VARIANT_WARP)
        assert shape(5120, 4, 64, 40, 152) == (tfx.FAMILY_ROWS_WARP, 0)
        assert shape(5120, 4, 65, 40, 152)[0] == tfx.FAMILY_TENSOR
        tfx.set_variant(tfx.VARIANT_ROWS)
        assert shape(5120, 4, 64, 40, 152) == (tfx.FAMILY_ROWS_CTA, 0)
        assert shape(5120, 4, 65, 40, 152)[0] == tfx.FAMILY_TENSOR
        tfx.set_variant(tfx.VARIANT_WARP_GLOBAL)
        assert shape(5120, 4, 8, 40, 152) == (tfx.FAMILY_ROWS_WARP, 0)
        assert shape(5120, 4, 65, 40, 152)[0] == tfx.FAMILY_TENSOR
        # a value outside 0..4 changes nothing
        assert tfx.set_variant(5) == tfx.VARIANT_WARP_GLOBAL
    finally:
        tfx.set_variant(old)
    for bad in ((100, 4, 1, 1, 152), (5120, 0, 1, 1, 152), (5120, 9, 1, 1, 152), (5120, 4, 0, 1, 152),
                (5120, 4, 1, 0, 152), (5120, 4, 1, 1, -1)):
        with pytest.raises(tfx.TfxError) as e:
            shape(*bad)
        assert e.value.code == tfx.EINVAL, bad


def test_output_window_validation_before_any_launch(L, drv):
    # group_into's window checks run before anything is enqueued
    w = fake_weight(256, 256, 4)
    tfx.reserve(w, 4, 0)
    x = FAKE + (3 << 30)
    y = FAKE + (4 << 30)
    arr = (C.POINTER(tfx.WeightStruct) * 1)(C.pointer(w.s))
    ys = (C.c_void_p * 1)(y)
    for ld, c0 in ((256, 4), (256, 256), (248, 0), (300, 0), (256, -8), (112, 136)):
        rc = L.tfx_exl3_group_into(arr, 1, x, 1, ys, (C.c_int64 * 1)(ld), (C.c_int * 1)(c0), None)
        assert rc == tfx.EINVAL, (ld, c0)
    assert L.tfx_exl3_group_into(arr, 1, x, 1, ys, None, (C.c_int * 1)(0), None) == tfx.EINVAL
    # a valid window still needs a reserve large enough
    rc = L.tfx_exl3_group_into(arr, 1, x, 9, ys, (C.c_int64 * 1)(128), (C.c_int * 1)(128), None)
    assert rc == tfx.ENOTRESERVED


def test_launch_count_moves_only_with_launches(L, drv):
    # the count the benchmark reads around a captured step: calls rejected on
    # the host and zero-row calls enqueue nothing
    w = fake_weight(256, 256, 4)
    tfx.reserve(w, 4, 0)
    n0 = tfx.launch_count()
    assert n0 >= 0
    arr = (C.POINTER(tfx.WeightStruct) * 1)(C.pointer(w.s))
    ys = (C.c_void_p * 1)(FAKE + (4 << 30))
    assert L.tfx_exl3_group(arr, 1, FAKE + (3 << 30), 0, ys, None) == 0
    assert L.tfx_exl3_group(arr, 1, FAKE + (3 << 30), 9, ys, None) == tfx.ENOTRESERVED
    assert L.tfx_exl3_group(arr, 1, FAKE + 3, 1, ys, None) == tfx.EALIGN
    assert tfx.launch_count() == n0


def test_spin_limit_and_decode_rate_query(L):
    old = tfx.set_spin_limit(7)
    assert old == 2_000_000_000
    assert tfx.set_spin_limit(-1) == 7
    assert tfx.set_spin_limit(0) == 2_000_000_000
    # the probe's size query launches nothing: 8 CTAs of 8 warps per SM (152
    # when no device is visible), 256 weights per tile
    weights, floats = tfx.decode_rate(4, 1000)
    assert floats % 64 == 0 and weights == floats * 1000 * 256
    with pytest.raises(tfx.TfxError):
        tfx.decode_rate(9, 10)


def test_switches_are_safe_across_threads(L):
    import threading
    old = tfx.set_variant(tfx.VARIANT_AUTO)
    seen = []

    def flip(v):
        for _ in range(2000):
            seen.append(tfx.set_variant(v))

    ts = [threading.Thread(target=flip, args=(v,)) for v in (0, 1, 2, 3)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert set(seen) <= {0, 1, 2, 3}
    assert tfx.set_variant(9) in (0, 1, 2, 3)  # out of range: unchanged
    tfx.set_variant(old)
