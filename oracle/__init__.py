"""CPU oracle of the EXL3 trellis linear (FP64, single thread, plain C).

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. It is independent of the
CUDA path (no shared code); both follow the decode rule and rotation written
in ``oracle/exl3_oracle.c``'s header.

Every function takes and returns numpy arrays. Float inputs are FP64 copies
of the FP16/BF16 values the GPU side sees (exact conversions).
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        d, i, u32p, dp = C.c_double, C.c_int, C.POINTER(C.c_uint32), C.POINTER(C.c_double)
        ll = C.c_longlong
        _lib.exl3o_state.argtypes = [u32p, i, i]
        _lib.exl3o_state.restype = C.c_uint32
        _lib.exl3o_code_sum.argtypes = [C.c_uint32]
        _lib.exl3o_code_sum.restype = i
        _lib.exl3o_value.argtypes = [C.c_uint32]
        _lib.exl3o_value.restype = d
        _lib.exl3o_position.argtypes = [i, C.POINTER(i), C.POINTER(i)]
        _lib.exl3o_decode.argtypes = [u32p, ll, i, i, i, dp]
        _lib.exl3o_hadamard.argtypes = [dp]
        _lib.exl3o_round_f16.argtypes = [d]
        _lib.exl3o_round_f16.restype = d
        _lib.exl3o_round_bf16.argtypes = [d]
        _lib.exl3o_round_bf16.restype = d
        _lib.exl3o_rot_in.argtypes = [dp, dp, i, i, dp]
        _lib.exl3o_matmul.argtypes = [dp, dp, i, i, i, dp]
        _lib.exl3o_rot_out.argtypes = [dp, dp, i, i, dp]
        _lib.exl3o_linear.argtypes = [u32p, ll, i, i, i, dp, dp, dp, i, dp]
        for f in ("exl3o_decode", "exl3o_rot_in", "exl3o_matmul", "exl3o_rot_out", "exl3o_linear"):
            getattr(_lib, f).restype = i
        ip = C.POINTER(C.c_int)
        _lib.exl3o_viterbi.argtypes = [i, i, i, ip, ip, i, C.c_uint32, u32p]
        _lib.exl3o_viterbi.restype = ll
        _lib.exl3o_encode_tile.argtypes = [ip, i, ip, u32p]
        _lib.exl3o_encode_tile.restype = ll
        _lib.exl3o_encode.argtypes = [C.POINTER(C.c_int16), i, i, i, ll, ll, u32p, C.POINTER(ll)]
        _lib.exl3o_encode.restype = i
    return _lib


def _u32(a):
    a = np.ascontiguousarray(a, dtype=np.uint32)
    return a, a.ctypes.data_as(C.POINTER(C.c_uint32))


def _f64(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(C.POINTER(C.c_double))


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed ({rc})")


def state(tile_words, bits: int, j: int) -> int:
    t, p = _u32(tile_words)
    assert t.size == 8 * bits
    return int(lib().exl3o_state(p, bits, j))


def code_sum(state_: int) -> int:
    return int(lib().exl3o_code_sum(state_))


def value(state_: int) -> float:
    return float(lib().exl3o_value(state_))


def position(j: int):
    k, n = C.c_int(), C.c_int()
    lib().exl3o_position(j, C.byref(k), C.byref(n))
    return k.value, n.value


def decode(trellis, K: int, N: int, bits: int, tile_row_stride: int | None = None,
           col_from: int = 0) -> np.ndarray:
    """Decoded weight W[k][n] (K x N, FP64) of the columns [col_from, col_from+N)."""
    t = np.ascontiguousarray(trellis, dtype=np.uint32).reshape(-1)
    if tile_row_stride is None:
        tile_row_stride = (N // 16) * 8 * bits
    off = (col_from // 16) * 8 * bits
    t = t[off:]
    W = np.empty((K, N), dtype=np.float64)
    _, p = _u32(t)
    _check(lib().exl3o_decode(p, tile_row_stride, K, N, bits,
                              W.ctypes.data_as(C.POINTER(C.c_double))), "decode")
    return W


def hadamard() -> np.ndarray:
    H = np.empty((128, 128), dtype=np.float64)
    lib().exl3o_hadamard(H.ctypes.data_as(C.POINTER(C.c_double)))
    return H


def round_f16(v: float) -> float:
    return float(lib().exl3o_round_f16(v))


def round_bf16(v: float) -> float:
    return float(lib().exl3o_round_bf16(v))


def rot_in(x, suh) -> np.ndarray:
    x, px = _f64(np.atleast_2d(x))
    s, ps = _f64(suh)
    rows, K = x.shape
    xr = np.empty_like(x)
    _check(lib().exl3o_rot_in(px, ps, rows, K, xr.ctypes.data_as(C.POINTER(C.c_double))), "rot_in")
    return xr


def matmul(xr, W) -> np.ndarray:
    xr, px = _f64(np.atleast_2d(xr))
    W, pw = _f64(W)
    rows, K = xr.shape
    N = W.shape[1]
    z = np.empty((rows, N), dtype=np.float64)
    _check(lib().exl3o_matmul(px, pw, rows, K, N, z.ctypes.data_as(C.POINTER(C.c_double))), "matmul")
    return z


def rot_out(z, svh) -> np.ndarray:
    z, pz = _f64(np.atleast_2d(z))
    s, ps = _f64(svh)
    rows, N = z.shape
    y = np.empty_like(z)
    _check(lib().exl3o_rot_out(pz, ps, rows, N, y.ctypes.data_as(C.POINTER(C.c_double))), "rot_out")
    return y


def linear(trellis, K: int, N: int, bits: int, suh, svh, x, tile_row_stride: int | None = None,
           col_from: int = 0) -> np.ndarray:
    """y (rows x N, FP64) of the columns [col_from, col_from+N) of a weight.

    ``svh`` is the vector of those N columns; ``x`` is rows x K (FP64 copy).
    """
    t = np.ascontiguousarray(trellis, dtype=np.uint32).reshape(-1)
    if tile_row_stride is None:
        tile_row_stride = (N // 16) * 8 * bits
    t = t[(col_from // 16) * 8 * bits:]
    _, pt = _u32(t)
    x, px = _f64(np.atleast_2d(x))
    su, psu = _f64(suh)
    sv, psv = _f64(svh)
    rows = x.shape[0]
    y = np.empty((rows, N), dtype=np.float64)
    _check(lib().exl3o_linear(pt, tile_row_stride, K, N, bits, psu, psv, px, rows,
                              y.ctypes.data_as(C.POINTER(C.c_double))), "linear")
    return y


# ---------------------------------------------------------------- trellis encoder

VITERBI_INF = 1 << 30


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(C.POINTER(C.c_int))


def viterbi(W: int, bits: int, val, T, constrain: bool = False, c: int = 0):
    """Best path of a W-bit shift-register trellis (see exl3_encoder_oracle.c):
    returns (cost, states)."""
    v, pv = _i32(val)
    t, pt = _i32(T)
    assert v.size == 1 << W
    st = np.zeros(t.size, dtype=np.uint32)
    cost = lib().exl3o_viterbi(W, bits, t.size, pv, pt, 1 if constrain else 0, c,
                               st.ctypes.data_as(C.POINTER(C.c_uint32)))
    if cost < 0:
        raise ValueError("oracle viterbi failed")
    return int(cost), st


def state_values() -> np.ndarray:
    """code_sum(s) - 510 for every 16-bit state (the integer value, units of 1/128)."""
    return np.array([code_sum(s) - 510 for s in range(1 << 16)], dtype=np.int32)


def encode_tile(T, bits: int, val=None):
    """256 grid targets (stream order) -> (8*bits words, squared error)."""
    v, pv = _i32(state_values() if val is None else val)
    t, pt = _i32(T)
    assert t.size == 256
    w = np.zeros(8 * bits, dtype=np.uint32)
    e = lib().exl3o_encode_tile(pt, bits, pv, w.ctypes.data_as(C.POINTER(C.c_uint32)))
    if e < 0:
        raise ValueError("oracle encode_tile failed")
    return w, int(e)


def encode(Tgrid, K: int, N: int, bits: int, tile0: int = 0, ntiles: int = 0):
    """K x N grid targets (int16, units of 1/128) -> (trellis words in the tile
    layout, squared error over the encoded tiles). Only tiles [tile0, tile0 +
    ntiles) of the row-major tile order are encoded when ntiles > 0 (the other
    words stay zero)."""
    g = np.ascontiguousarray(Tgrid, dtype=np.int16)
    assert g.shape == (K, N)
    out = np.zeros((K // 16, (N // 16) * 8 * bits), dtype=np.uint32)
    err = C.c_longlong()
    rc = lib().exl3o_encode(g.ctypes.data_as(C.POINTER(C.c_int16)), K, N, bits, tile0, ntiles,
                            out.ctypes.data_as(C.POINTER(C.c_uint32)), C.byref(err))
    if rc != 0:
        raise ValueError(f"oracle encode failed ({rc})")
    return out, int(err.value)


def round_out(y: np.ndarray, dtype: str) -> np.ndarray:
    """Round the FP64 output to the activation dtype (nearest even), kept as FP64."""
    f = lib().exl3o_round_f16 if dtype == "f16" else lib().exl3o_round_bf16
    return np.vectorize(lambda v: f(float(v)), otypes=[np.float64])(y)
