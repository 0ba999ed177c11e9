"""Bounded waits in the decode-rows and tensor-core kernels, made to give up on a healthy GPU.

Every wait of a kernel on a copy into shared memory polls for at most the
launch's spin limit (about 1 s by default). Lowering the limit to one clock
cycle makes the first waits give up before the copies land (at 5 or more
rows: calls of at most 4 rows rotate x inside the kernel, which takes longer
than the copies of trellis words, so their first poll already succeeds): the CTA then
records device error 3, waits for its own copies in flight, skips its work
and still meets its cluster at both barriers, so the launch ends and the
context stays usable. No fault, trap or endless loop is involved: the copies
are valid and complete; only the waiting side stops early. After
reset_counters and with the default limit back, the next call gives the
bytes of a call made before.
"""
import pytest
import torch

import exl3_trellis_quantized_rot_gb300 as tfx
from gpu_helpers import make, same_bytes, x_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build_library()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    tfx.set_spin_limit(0)
    tfx.set_variant(tfx.VARIANT_AUTO)


@pytest.mark.parametrize("rows", [7, 16])
def test_decode_rows_waits_give_up_and_recover(rows):
    hw, w = make(70, 5120, 1024, 4, max_rows=16)
    x64, x = x_of(70, rows, 5120)
    tfx.set_variant(tfx.VARIANT_WARP)
    try:
        good = tfx.linear(w, x)
        torch.cuda.synchronize()
        assert tfx.device_error(w) == 0
        old = tfx.set_spin_limit(1)
        assert old == 2_000_000_000
        err = 0
        for _ in range(5):  # one launch of 128 CTAs practically always has a copy in flight at its first poll
            tfx.linear(w, x)
            torch.cuda.synchronize()
            err = tfx.device_error(w)
            if err:
                break
        assert err == 3
        assert tfx.set_spin_limit(0) == 1
        tfx.reset_counters(w)
        assert tfx.device_error(w) == 0
        again = tfx.linear(w, x)
        torch.cuda.synchronize()
        assert same_bytes(again, good)
        assert tfx.device_error(w) == 0
    finally:
        tfx.set_spin_limit(0)
        tfx.set_variant(tfx.VARIANT_AUTO)


def test_tensor_core_waits_give_up_and_recover():
    # the tensor-core kernel: every hand-off is an mbarrier polled for at most
    # the spin limit; a wait that gives up aborts the CTA (device error 1), every
    # role leaves its loop at its next wait, copies and MMAs in flight land, TMEM
    # is freed and the launch ends
    hw, w = make(71, 5120, 1024, 4, max_rows=128)
    x64, x = x_of(71, 100, 5120)
    tfx.set_variant(tfx.VARIANT_MID)
    try:
        good = tfx.linear(w, x)
        torch.cuda.synchronize()
        assert tfx.device_error(w) == 0
        tfx.set_spin_limit(1)
        err = 0
        for _ in range(5):
            tfx.linear(w, x)
            torch.cuda.synchronize()
            err = tfx.device_error(w)
            if err:
                break
        assert err == 1
        tfx.set_spin_limit(0)
        tfx.reset_counters(w)  # an aborted launch may leave split-K counters behind
        assert tfx.device_error(w) == 0
        for _ in range(3):
            again = tfx.linear(w, x)
            torch.cuda.synchronize()
            assert same_bytes(again, good)
        assert tfx.device_error(w) == 0
    finally:
        tfx.set_spin_limit(0)
        tfx.set_variant(tfx.VARIANT_AUTO)
