"""Shared set-up for the GPU parity tests: seeded inputs uploaded to cuda:0,
oracle references and the tolerance check.

Tolerance (stated once): relative L2 <= 2e-3 and, per element,
|gpu - oracle| <= 1e-2 * rms(oracle); for BF16 outputs the per-element bound
is max(1e-2 * rms, one BF16 ulp of the oracle value), because rounding to
BF16 alone can exceed 1e-2 * rms at |y| above ~2.6 rms.
"""
from __future__ import annotations

import numpy as np
import torch

import exl3_trellis_quantized_rot_gb300 as tfx
import oracle
import synth

DEV = torch.device("cuda:0")
REL_L2 = 2e-3
MAX_REL_RMS = 1e-2


class HostWeight:
    def __init__(self, seed, K, N, bits, member=0, codes=None):
        self.K, self.N, self.bits = K, N, bits
        self.codes = synth.codes(seed, K, N, bits, member) if codes is None else codes
        self.suh = synth.suh(seed, K, member)
        self.svh = synth.svh(seed, N, member)


def upload(hw: HostWeight, act=tfx.F16):
    t_codes = torch.from_numpy(np.ascontiguousarray(hw.codes).view(np.int32)).to(DEV)
    t_suh = torch.from_numpy(hw.suh.view(np.int16)).to(DEV)
    t_svh = torch.from_numpy(hw.svh.view(np.int16)).to(DEV)
    return tfx.Weight(t_codes, t_suh, t_svh, hw.K, hw.N, hw.bits, act)


def make(seed, K, N, bits, act=tfx.F16, member=0, max_rows=16):
    hw = HostWeight(seed, K, N, bits, member)
    w = upload(hw, act)
    tfx.reserve(w, max_rows)
    return hw, w


def act_name(act):
    return "f16" if act == tfx.F16 else "bf16"


def x_of(seed, rows, K, act=tfx.F16):
    """(FP64 host copy, device tensor) of seeded activations."""
    a = synth.activations(seed, rows, K, act_name(act))
    if act == tfx.F16:
        t = torch.from_numpy(a).to(DEV)
    else:
        t = torch.from_numpy(a.view(np.int16)).to(DEV).view(torch.bfloat16)
    return synth.as_f64(a, act_name(act)), t


def to_f64(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def bits16(y: torch.Tensor) -> torch.Tensor:
    return y.view(torch.int16)


def same_bytes(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(bits16(a), bits16(b))


def oracle_y(hw: HostWeight, x64, col_from=0, n=None):
    n = hw.N if n is None else n
    return oracle.linear(hw.codes, hw.K, n, hw.bits, hw.suh.astype(np.float64),
                         hw.svh[col_from:col_from + n].astype(np.float64), x64,
                         tile_row_stride=(hw.N // 16) * 8 * hw.bits, col_from=col_from)


def assert_close(got: np.ndarray, want: np.ndarray, act=tfx.F16, what=""):
    assert got.shape == want.shape, (got.shape, want.shape)
    rms = np.sqrt(np.mean(want ** 2))
    err = np.abs(got - want)
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    bound = np.full(want.shape, MAX_REL_RMS * rms)
    if act == tfx.BF16:
        with np.errstate(divide="ignore"):
            ulp = np.where(want != 0, 2.0 ** (np.floor(np.log2(np.abs(want) + 1e-300)) - 7), 0)
        bound = np.maximum(bound, ulp)
    bad = err > bound
    assert rel <= REL_L2, f"{what}: relative L2 {rel:.3e} > {REL_L2}"
    assert not bad.any(), f"{what}: {bad.sum()} elements over the bound; worst {err.max():.3e} (rms {rms:.3e})"
    return rel, float(err.max() / rms)
