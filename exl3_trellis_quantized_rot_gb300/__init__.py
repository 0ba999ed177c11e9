"""Python binding of the tfx_exl3 C ABI (argument marshalling only).

Every step of the layer runs in the CUDA kernels of ``libtfx_exl3.so``; this
module only turns tensors into device pointers and streams into handles.
If the library is missing the import of any entry point raises: there is no
CPU fallback.

Names follow the C ABI: ``linear``, ``group``, ``columns``, ``reserve``,
``release``, ``reset_counters``, ``debug_decode``, ``plan``, ``stats``,
``set_variant``, ``set_pdl``, ``last_error``.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtfx_exl3.so")

OK, EINVAL, ENOTRESERVED, EUNSUPPORTED, EALIGN, ECUDA = 0, -1, -2, -3, -4, -5
F16, BF16 = 0, 1
VARIANT_AUTO, VARIANT_ROWS, VARIANT_MID, VARIANT_WARP, VARIANT_WARP_GLOBAL = 0, 1, 2, 3, 4

ABI_SYMBOLS = ("tfx_exl3_linear", "tfx_exl3_group", "tfx_exl3_columns", "tfx_exl3_reserve",
               "tfx_exl3_release", "tfx_exl3_reset_counters", "tfx_exl3_debug_decode", "tfx_exl3_plan",
               "tfx_exl3_stats", "tfx_exl3_set_variant", "tfx_exl3_set_pdl", "tfx_exl3_debug_set_driver",
               "tfx_exl3_debug_mark_events", "tfx_exl3_linear_static", "tfx_exl3_debug_error",
               "tfx_exl3_debug_launch_shape", "tfx_exl3_group_into", "tfx_exl3_debug_set_spin_limit",
               "tfx_exl3_debug_decode_rate", "tfx_exl3_chain", "tfx_exl3_encode", "tfx_exl3_encode_scratch_bytes",
               "tfx_exl3_debug_launch_count", "tfx_exl3_last_error")


class WeightStruct(C.Structure):
    _fields_ = [("trellis", C.c_void_p), ("suh", C.c_void_p), ("svh", C.c_void_p), ("K", C.c_int),
                ("N", C.c_int), ("bits", C.c_int), ("tile_row_stride", C.c_int64), ("act", C.c_int),
                ("priv", C.c_void_p)]


class StepStruct(C.Structure):
    _fields_ = [("ws", C.POINTER(C.POINTER(WeightStruct))), ("count", C.c_int), ("x", C.c_void_p),
                ("ys", C.POINTER(C.c_void_p))]


ALLOC_FN = C.CFUNCTYPE(C.c_int, C.POINTER(C.c_void_p), C.c_size_t, C.c_void_p)
FREE_FN = C.CFUNCTYPE(C.c_int, C.c_void_p, C.c_void_p)
MEMSET_FN = C.CFUNCTYPE(C.c_int, C.c_void_p, C.c_size_t, C.c_void_p)


class DriverStruct(C.Structure):
    _fields_ = [("alloc", ALLOC_FN), ("free", FREE_FN), ("memset0", MEMSET_FN)]


class TfxError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"tfx_exl3 error {code}: {msg}")
        self.code = code


_lib = None


def lib() -> C.CDLL:
    """Load libtfx_exl3.so (built by ``exl3_trellis_quantized_rot_gb300.build``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run the build (python -m "
                              "exl3_trellis_quantized_rot_gb300.build); there is no CPU fallback")
        L = C.CDLL(LIB_PATH)
        W = C.POINTER(WeightStruct)
        vp, i = C.c_void_p, C.c_int
        L.tfx_exl3_linear.argtypes = [W, vp, i, vp, vp]
        L.tfx_exl3_group.argtypes = [C.POINTER(W), i, vp, i, C.POINTER(vp), vp]
        L.tfx_exl3_columns.argtypes = [W, i, i, W]
        L.tfx_exl3_reserve.argtypes = [W, i, vp]
        L.tfx_exl3_release.argtypes = [W]
        L.tfx_exl3_reset_counters.argtypes = [W, vp]
        L.tfx_exl3_debug_decode.argtypes = [W, vp, vp]
        L.tfx_exl3_plan.argtypes = [W, C.POINTER(i), C.POINTER(i)]
        L.tfx_exl3_stats.argtypes = [W, C.POINTER(C.c_int64), C.POINTER(C.c_int64)]
        L.tfx_exl3_set_variant.argtypes = [i]
        L.tfx_exl3_set_pdl.argtypes = [i]
        L.tfx_exl3_debug_set_driver.argtypes = [C.POINTER(DriverStruct)]
        L.tfx_exl3_debug_mark_events.argtypes = [vp, vp]
        L.tfx_exl3_linear_static.argtypes = [W, vp, i, vp, vp]
        L.tfx_exl3_debug_error.argtypes = [W, C.POINTER(i)]
        L.tfx_exl3_debug_launch_shape.argtypes = [i, i, i, C.c_int64, i, C.POINTER(i), C.POINTER(i)]
        L.tfx_exl3_group_into.argtypes = [C.POINTER(W), i, vp, i, C.POINTER(vp), C.POINTER(C.c_int64),
                                          C.POINTER(i), vp]
        L.tfx_exl3_debug_set_spin_limit.argtypes = [C.c_int64]
        L.tfx_exl3_debug_decode_rate.argtypes = [i, i, vp, C.POINTER(i), C.POINTER(C.c_int64), vp]
        L.tfx_exl3_chain.argtypes = [C.POINTER(StepStruct), i, i, i, vp]
        L.tfx_exl3_encode_scratch_bytes.argtypes = [i, i, i, i, C.POINTER(C.c_size_t)]
        L.tfx_exl3_encode.argtypes = [vp, i, i, i, vp, vp, vp, C.c_size_t, i, vp]
        L.tfx_exl3_last_error.restype = C.c_char_p
        for n in ABI_SYMBOLS[:-1]:
            getattr(L, n).restype = C.c_int
        L.tfx_exl3_debug_set_spin_limit.restype = C.c_int64
        L.tfx_exl3_debug_launch_count.argtypes = []
        L.tfx_exl3_debug_launch_count.restype = C.c_int64
        _lib = L
    return _lib


def last_error() -> str:
    return lib().tfx_exl3_last_error().decode()


def _check(rc: int) -> int:
    if rc != 0:
        raise TfxError(rc, last_error())
    return rc


def _ptr(t) -> int:
    return 0 if t is None else (t if isinstance(t, int) else t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


class Weight:
    """A quantized weight: the C descriptor plus references keeping its tensors alive.

    trellis: uint32 words (int32 tensor), shape (K/16, tile_row_stride) or flat;
    suh: K FP16; svh: N FP16; all on the same CUDA device (or raw pointers).
    """

    def __init__(self, trellis, suh, svh, K: int, N: int, bits: int, act: int = F16,
                 tile_row_stride: int | None = None, _parent=None):
        self.s = WeightStruct()
        self.s.trellis, self.s.suh, self.s.svh = _ptr(trellis), _ptr(suh), _ptr(svh)
        self.s.K, self.s.N, self.s.bits, self.s.act = K, N, bits, act
        self.s.tile_row_stride = (N // 16) * 8 * bits if tile_row_stride is None else tile_row_stride
        self.s.priv = None
        self._keep = (trellis, suh, svh, _parent)

    @property
    def K(self):
        return self.s.K

    @property
    def N(self):
        return self.s.N

    @property
    def bits(self):
        return self.s.bits

    @property
    def act(self):
        return self.s.act

    def ref(self):
        return C.byref(self.s)

    def __del__(self):
        try:
            if self.s.priv and _lib is not None:
                _lib.tfx_exl3_release(C.byref(self.s))
        except Exception:
            pass


def reserve(w: Weight, max_rows: int, stream=None) -> None:
    _check(lib().tfx_exl3_reserve(w.ref(), max_rows, _stream(stream)))


def release(w: Weight) -> None:
    _check(lib().tfx_exl3_release(w.ref()))


def reset_counters(w: Weight, stream=None) -> None:
    _check(lib().tfx_exl3_reset_counters(w.ref(), _stream(stream)))


def linear(w: Weight, x, rows: int | None = None, y=None, stream=None):
    """y = layer(x); x is rows x K in the weight's act dtype. Returns y."""
    import torch
    if rows is None:
        rows = x.shape[0]
    if y is None:
        y = torch.empty((rows, w.N), dtype=x.dtype, device=x.device)
    _check(lib().tfx_exl3_linear(w.ref(), _ptr(x), rows, _ptr(y), _stream(stream)))
    return y


def linear_static(w: Weight, x, rows: int | None = None, y=None, stream=None):
    """tfx_exl3_linear with its scratch in the library's static device array:
    for callers that cannot allocate device memory where they run the layer.
    Needs no reserve(). Calls share the array: order them on one stream."""
    import torch
    if rows is None:
        rows = x.shape[0]
    if y is None:
        y = torch.empty((rows, w.N), dtype=x.dtype, device=x.device)
    _check(lib().tfx_exl3_linear_static(w.ref(), _ptr(x), rows, _ptr(y), _stream(stream)))
    return y


def group(ws, x, rows: int | None = None, ys=None, stream=None):
    """One rotation and one launch over up to 3 weights of the same K. Returns ys."""
    import torch
    if rows is None:
        rows = x.shape[0]
    if ys is None:
        ys = [torch.empty((rows, w.N), dtype=x.dtype, device=x.device) for w in ws]
    n = len(ws)
    arr = (C.POINTER(WeightStruct) * max(n, 1))(*[C.pointer(w.s) for w in ws])
    yarr = (C.c_void_p * max(n, 1))(*[_ptr(y) for y in ys])
    _check(lib().tfx_exl3_group(arr, n, _ptr(x), rows, yarr, _stream(stream)))
    return ys


def group_into(ws, x, ys, ldy, col0, rows: int | None = None, stream=None):
    """tfx_exl3_group with an output window per member: member i's element
    (r, n >= col0[i]) goes to ys[i] + r*ldy[i] + (n - col0[i]). ys are device
    pointers or tensors (a tensor's data_ptr is the window's first element)."""
    if rows is None:
        rows = x.shape[0]
    n = len(ws)
    arr = (C.POINTER(WeightStruct) * max(n, 1))(*[C.pointer(w.s) for w in ws])
    yarr = (C.c_void_p * max(n, 1))(*[_ptr(y) for y in ys])
    larr = (C.c_int64 * max(n, 1))(*ldy)
    carr = (C.c_int * max(n, 1))(*col0)
    _check(lib().tfx_exl3_group_into(arr, n, _ptr(x), rows, yarr, larr, carr, _stream(stream)))


def pack_spans(views, x, out, col0, rows: int | None = None, stream=None):
    """Several column views of one weight packed side by side into `out`
    (rows x sum of kept columns): view i keeps its columns from col0[i] on and
    lands right after view i-1's kept columns, all in one call."""
    ld = out.shape[1]
    ys, off = [], 0
    for v, c in zip(views, col0):
        ys.append(out.data_ptr() + off * out.element_size())
        off += v.N - c
    if off != ld:
        raise ValueError(f"kept columns {off} != out width {ld}")
    group_into(views, x, ys, [ld] * len(views), list(col0), rows, stream)
    return out


def _pdl_mode(pdl) -> int:
    return (1 if pdl else 0) if isinstance(pdl, bool) else int(pdl)


def chain(steps, rows: int, pdl=True, stream=None):
    """Run group calls back to back (tfx_exl3_chain). steps: list of
    (weights, x, ys); a step's x may be an earlier step's output. Outputs
    must be allocated by the caller (the chain allocates nothing). pdl:
    True/1 on every launch, False/0 off, 2 the automatic choice."""
    keep = []
    arr = (StepStruct * len(steps))()
    for st, (ws, x, ys) in zip(arr, steps):
        wa = (C.POINTER(WeightStruct) * len(ws))(*[C.pointer(w.s) for w in ws])
        ya = (C.c_void_p * len(ys))(*[_ptr(y) for y in ys])
        keep += [wa, ya]
        st.ws = C.cast(wa, C.POINTER(C.POINTER(WeightStruct)))
        st.count = len(ws)
        st.x = _ptr(x)
        st.ys = C.cast(ya, C.POINTER(C.c_void_p))
    _check(lib().tfx_exl3_chain(arr, len(steps), rows, _pdl_mode(pdl), _stream(stream)))


def encode_scratch_bytes(K: int, N: int, bits: int, max_ctas: int = 0) -> int:
    n = C.c_size_t()
    _check(lib().tfx_exl3_encode_scratch_bytes(K, N, bits, max_ctas, C.byref(n)))
    return n.value


def encode(targets, bits: int, max_ctas: int = 0, scratch=None, stream=None):
    """Trellis words of a K x N weight from int16 grid targets (W*128 rounded),
    on the GPU. Returns (trellis int32 tensor (K/16, (N/16)*8*bits), per-tile
    squared error int64 tensor)."""
    import torch
    K, N = targets.shape
    out = torch.empty((K // 16, (N // 16) * 8 * bits), dtype=torch.int32, device=targets.device)
    err = torch.empty(((K // 16) * (N // 16),), dtype=torch.int64, device=targets.device)
    need = encode_scratch_bytes(K, N, bits, max_ctas)
    if scratch is None:
        scratch = torch.empty(need, dtype=torch.uint8, device=targets.device)
    _check(lib().tfx_exl3_encode(_ptr(targets), K, N, bits, _ptr(out), _ptr(err), _ptr(scratch), scratch.numel(),
                                 max_ctas, _stream(stream)))
    return out, err


def columns(w: Weight, start: int, n: int) -> Weight:
    """View of whole 128-column blocks [start, start+n) sharing w's memory."""
    v = Weight.__new__(Weight)
    v.s = WeightStruct()
    _check(lib().tfx_exl3_columns(w.ref(), start, n, C.byref(v.s)))
    v._keep = (None, None, None, w)
    return v


def debug_decode(w: Weight, W_out=None, stream=None):
    import torch
    if W_out is None:
        W_out = torch.empty((w.K, w.N), dtype=torch.float16, device="cuda")
    _check(lib().tfx_exl3_debug_decode(w.ref(), _ptr(W_out), _stream(stream)))
    return W_out


def plan(w: Weight):
    s, k = C.c_int(), C.c_int()
    _check(lib().tfx_exl3_plan(w.ref(), C.byref(s), C.byref(k)))
    return s.value, k.value


def stats(w: Weight):
    a, m = C.c_int64(), C.c_int64()
    _check(lib().tfx_exl3_stats(w.ref(), C.byref(a), C.byref(m)))
    return a.value, m.value


def device_error(w: Weight) -> int:
    """The weight's device error word: 1 a tensor-core launch gave up a bounded
    wait, 2 a tensor-core launch had too little shared memory, 3 a decode-rows
    launch gave up waiting for a copy; 0 otherwise."""
    e = C.c_int()
    _check(lib().tfx_exl3_debug_error(w.ref(), C.byref(e)))
    return e.value


def set_variant(v: int) -> int:
    return lib().tfx_exl3_set_variant(v)


FAMILY_ROWS_CTA, FAMILY_ROWS_WARP, FAMILY_TENSOR = 0, 1, 2


def debug_launch_shape(K: int, bits: int, rows: int, blocks: int, sm_count: int = 0):
    """(family, chunks per tensor-core unit) that a call would launch; host only."""
    f, g = C.c_int(), C.c_int()
    _check(lib().tfx_exl3_debug_launch_shape(K, bits, rows, blocks, sm_count, C.byref(f), C.byref(g)))
    return f.value, g.value


def set_spin_limit(clocks: int) -> int:
    """Clock cycles a bounded wait in a kernel polls before it gives up (<= 0:
    the default, about 1 s). Returns the previous limit. For tests."""
    return lib().tfx_exl3_debug_set_spin_limit(clocks)


def decode_rate(bits: int, tiles_per_warp: int, sink=None, stream=None):
    """Launch the decode-rate probe (no global traffic); returns (weights decoded,
    floats the sink needs). With sink None nothing is launched."""
    nf, nw = C.c_int(), C.c_int64()
    _check(lib().tfx_exl3_debug_decode_rate(bits, tiles_per_warp, _ptr(sink) if sink is not None else None,
                                            C.byref(nf), C.byref(nw), _stream(stream) if sink is not None else None))
    return nw.value, nf.value


def launch_count() -> int:
    """Kernels the library has enqueued or captured since it was loaded."""
    return lib().tfx_exl3_debug_launch_count()


def set_pdl(mode) -> int:
    """0/False off, 1/True every launch, 2 automatic (the default). Returns the
    previous mode."""
    old = lib().tfx_exl3_set_pdl(_pdl_mode(mode))
    if old < 0:
        _check(old)
    return old


def mark_events(before, after) -> None:
    """Record torch.cuda.Event `before`/`after` around the next call's linear kernel."""
    _check(lib().tfx_exl3_debug_mark_events(before.cuda_event if before is not None else None,
                                             after.cuda_event if after is not None else None))


def set_driver(drv: DriverStruct | None) -> None:
    _check(lib().tfx_exl3_debug_set_driver(C.byref(drv) if drv is not None else None))
