"""Helpers shared by the GPU parity tests (comparison rules, sharding via the C ABI).

Tolerances (stated once, used everywhere):
  * fp32 inputs:      max |y - y_ref| <= 1e-5 * (|y_ref| + 1), elementwise.
  * bf16 inputs with fp32 accumulation, fp32 output:
                      max |y - y_ref| <= 5e-3 * RMS(y_ref).
  * a bf16-stored intermediate (the FFN's h) against the oracle's exact fp64
    value: |h - h_exact| <= 2^-8 |h_exact| + 1e-3 RMS(h_exact), i.e. within
    half a bf16 ulp of the exact value plus fp32 accumulation error.  (Two
    independent bf16 roundings of nearly equal values may differ by a whole
    ulp, so h is never compared bf16 against bf16.)
  * bf16 output:      bit-identical to round-to-nearest-even(bf16) of the
                      fp32-output run of the same call.
  * column-parallel:  bit-identical to the same call with tp = 1.
The oracle rounds the FFN intermediate h to bf16 where the kernels store it
in bf16, so the bf16 tolerance measures accumulation error only.
"""
from __future__ import annotations

import numpy as np
import torch

from tensor_column_linear_gelu_b300 import tpla

TOL_F32 = 1e-5
TOL_BF16_RMS = 5e-3
# unit roundoff of the wire dtypes of the ring-ordered shard sum
U_BF16 = 2.0 ** -8
U_F32 = 2.0 ** -24


def np64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def rms(a: np.ndarray) -> float:
    return float(np.sqrt(np.mean(np.asarray(a, np.float64) ** 2)))


def assert_close_fp32(y: torch.Tensor, ref: np.ndarray):
    y = np64(y)
    bound = TOL_F32 * (np.abs(ref) + 1.0)
    err = np.abs(y - ref)
    assert np.all(err <= bound), f"fp32 max err {err.max():.3e}"


def assert_close_bf16(y: torch.Tensor, ref: np.ndarray, tol: float = TOL_BF16_RMS) -> float:
    y = np64(y)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    r = rms(ref)
    err = float(np.max(np.abs(y - ref))) if y.size else 0.0
    assert np.all(np.isfinite(y)), "non-finite output"
    assert err <= tol * r, f"max err {err:.4e} > {tol} * RMS {r:.4e} (ratio {err / r:.3e})"
    return err / r if r > 0 else 0.0


def assert_h_bf16(h: torch.Tensor, h_exact: np.ndarray):
    """h stored in bf16 is the exact value rounded once (plus accumulation error)."""
    hv = np64(h)
    assert hv.shape == h_exact.shape
    bound = 2.0 ** -8 * np.abs(h_exact) + 1e-3 * rms(h_exact)
    err = np.abs(hv - h_exact)
    assert np.all(err <= bound), \
        f"h: {int(np.sum(err > bound))} elements off by more than half a bf16 ulp (+ slack)"


def assert_bf16_is_rounded_fp32(y_bf16: torch.Tensor, y_f32: torch.Tensor):
    want = y_f32.to(torch.bfloat16)
    assert torch.equal(y_bf16.view(torch.int16), want.view(torch.int16)), \
        "bf16 output differs from RNE(fp32 output)"


def assert_bitwise_equal(a: torch.Tensor, b: torch.Tensor, what: str = ""):
    assert a.dtype == b.dtype and a.shape == b.shape
    ia = a.contiguous().view(torch.int16 if a.element_size() == 2 else torch.int32)
    ib = b.contiguous().view(torch.int16 if b.element_size() == 2 else torch.int32)
    ne = (ia != ib).sum().item()
    assert ne == 0, f"{what}: {ne} of {a.numel()} elements differ bitwise"


def shard(split, tp, W, W_up=None, b=None, **heads):
    return tpla.tp_shard_weights(split, tp, W, W_up=W_up, b=b, **heads)
