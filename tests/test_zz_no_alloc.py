"""tfx_exl3_linear_static: the allocation-free entry point.

Some callers cannot allocate device memory where they run the layer (code in
a host callback or in a context where allocation is forbidden, plugins whose
host owns all device memory, runtimes that must not allocate after start-up).
tfx_exl3_linear_static serves them from a static scratch array inside the
library. This test calls it through the C ABI and checks its output against
tfx_exl3_linear's on two calls in a row, within the tolerance the parity tests
use (and byte for byte, since both run the same kernels), with the
automatic kernel choice and with the kernel whose split-K uses counters. It
lives in its own file, collected last, and passes alone or after the
other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import exl3_trellis_quantized_rot_gb300 as tfx
from gpu_helpers import assert_close, make, same_bytes, to_f64, x_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build_library()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _call_static(w, x, rows, y):
    L = tfx.lib()
    return L.tfx_exl3_linear_static(w.ref(), x.data_ptr(), rows, y.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("variant", [tfx.VARIANT_AUTO, tfx.VARIANT_ROWS, tfx.VARIANT_WARP_GLOBAL])
@pytest.mark.parametrize("K,N,bits,rows,act", [(5120, 5120, 4, 16, tfx.F16), (5120, 1024, 3, 7, tfx.F16),
                                               (1024, 2048, 4, 40, tfx.BF16), (1024, 20480, 3, 4, tfx.F16)])
def test_static_entry_matches_linear_on_two_calls(K, N, bits, rows, act, variant):
    # VARIANT_ROWS sends 1..64 rows through the kernel whose split-K partials are
    # summed by the last CTA to arrive on each block's counter, VARIANT_WARP_GLOBAL
    # up to 8 rows through the decode-rows kernel's global-slab fold: the counters
    # and the error word the static call clears at its start are then in use
    hw, w = make(40 + bits, K, N, bits, act=act, max_rows=rows)
    ref_w = w
    # a second descriptor of the same weight that was never reserved: the static
    # entry point must not need (or touch) reserved scratch
    plain = tfx.Weight(w._keep[0], w._keep[1], w._keep[2], K, N, bits, act)
    old = tfx.set_variant(variant)
    try:
        for call in range(2):
            x64, x = x_of(50 + call, rows, K, act)
            want = tfx.linear(ref_w, x)
            y = torch.empty_like(want)
            assert _call_static(plain, x, rows, y) == 0, tfx.last_error()
            torch.cuda.synchronize()
            # the same kernels on the same inputs: the same bytes (the tolerance
            # of the parity tests is implied)
            assert same_bytes(y, want), f"static call {call}"
            assert_close(to_f64(y), to_f64(want), act, what=f"static call {call}")
    finally:
        tfx.set_variant(old)
    assert tfx.stats(plain) == (0, 0)


def test_static_entry_rejects_oversized_requests():
    hw, w = make(60, 5120, 5120, 4, max_rows=1)
    rows = 4096  # the rotated x alone (40 MiB) exceeds the 8 MiB array
    x = torch.zeros((rows, 5120), dtype=torch.float16, device="cuda")
    y = torch.empty((rows, 5120), dtype=torch.float16, device="cuda")
    rc = _call_static(w, x, rows, y)
    assert rc == tfx.EUNSUPPORTED
    assert "static scratch holds" in tfx.last_error()
