"""Layer-level chaining (tfx_exl3_chain): q/k/v -> o and gate/up -> down.

The pages chain the rotations and the decode-row linears with programmatic
dependent launch so that each launch hides behind the previous one (PR #1467,
"What this changes") and reserve every weight at load, so that a captured
decode step allocates and clears nothing (PR #1475, "What this changes").
Here the second layer of each chain consumes an output of the first (o takes
q's output, down takes gate's: stand-ins for the attention output and the MLP
activation, which are not part of this layer), so the chain carries a real
data dependency. Checked: chained bytes (with and without dependent launch,
eager and replayed from a CUDA graph) equal the same calls made one by one,
and capture allocates and clears nothing.
"""
import pytest
import torch

import exl3_trellis_quantized_rot_gb300 as tfx
from gpu_helpers import DEV, make, same_bytes, x_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build_library()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    tfx.set_variant(tfx.VARIANT_AUTO)


def _chains(rows):
    q = make(80, 5120, 6144, 4, member=0, max_rows=rows)[1]
    k = make(80, 5120, 1024, 4, member=1, max_rows=rows)[1]
    v = make(80, 5120, 1024, 4, member=2, max_rows=rows)[1]
    o = make(81, 6144, 5120, 4, max_rows=rows)[1]
    g = make(82, 5120, 17408, 4, member=0, max_rows=rows)[1]
    u = make(82, 5120, 17408, 4, member=1, max_rows=rows)[1]
    d = make(83, 17408, 5120, 4, max_rows=rows)[1]
    return (q, k, v, o), (g, u, d)


def _outs(rows, ns):
    return [torch.empty((rows, n), dtype=torch.float16, device=DEV) for n in ns]


@pytest.mark.parametrize("rows", [16, 64])
def test_chain_bytes_equal_unchained_calls(rows):
    (q, k, v, o), (g, u, d) = _chains(rows)
    x64, x = x_of(84, rows, 5120)
    # one by one
    yq, yk, yv = tfx.group([q, k, v], x)
    yo = tfx.linear(o, yq)
    yg, yu = tfx.group([g, u], x)
    yd = tfx.linear(d, yg)
    for pdl in (0, 1, 2):
        a = _outs(rows, (6144, 1024, 1024, 5120))
        b = _outs(rows, (17408, 17408, 5120))
        tfx.chain([([q, k, v], x, a[:3]), ([o], a[0], a[3:])], rows, pdl=pdl)
        tfx.chain([([g, u], x, b[:2]), ([d], b[0], b[2:])], rows, pdl=pdl)
        torch.cuda.synchronize()
        for got, want in zip(a + b, (yq, yk, yv, yo, yg, yu, yd)):
            assert same_bytes(got, want), pdl
    for w in (q, k, v, o, g, u, d):
        assert tfx.device_error(w) == 0


@pytest.mark.parametrize("pdl", [0, 1, 2])
def test_captured_chain_allocates_nothing(pdl):
    rows = 16
    (q, k, v, o), (g, u, d) = _chains(rows)
    x64, x = x_of(85, rows, 5120)
    yq, yk, yv = tfx.group([q, k, v], x)
    yo = tfx.linear(o, yq)
    yg, yu = tfx.group([g, u], x)
    yd = tfx.linear(d, yg)
    before = [tfx.stats(w) for w in (q, k, v, o, g, u, d)]
    a = _outs(rows, (6144, 1024, 1024, 5120))
    b = _outs(rows, (17408, 17408, 5120))
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        tfx.chain([([q, k, v], x, a[:3]), ([o], a[0], a[3:]), ([g, u], x, b[:2]), ([d], b[0], b[2:])], rows,
                  pdl=pdl, stream=s)
    for _ in range(3):
        for t in a + b:
            t.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        for got, want in zip(a + b, (yq, yk, yv, yo, yg, yu, yd)):
            assert same_bytes(got, want)
    assert [tfx.stats(w) for w in (q, k, v, o, g, u, d)] == before


def test_chain_validates_every_step_first():
    (q, k, v, o), _ = _chains(16)
    # the first step's weights are reserved for 32 rows, the second step's for
    # 16: a 32-row chain fails before the (valid) first step is enqueued
    for w in (q, k, v):
        tfx.reserve(w, 32)
    a = _outs(32, (6144, 1024, 1024, 5120))
    sentinel = torch.full_like(a[0], 5.0)
    a[0].copy_(sentinel)
    x32 = torch.zeros((32, 5120), dtype=torch.float16, device=DEV)
    with pytest.raises(tfx.TfxError) as e:
        tfx.chain([([q, k, v], x32, a[:3]), ([o], a[0], a[3:])], 32)
    assert e.value.code == tfx.ENOTRESERVED
    torch.cuda.synchronize()
    assert same_bytes(a[0], sentinel)
