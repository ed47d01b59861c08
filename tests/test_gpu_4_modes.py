"""The two variants of the split beyond the fused path, against the oracle.

* row_parallel_linear_ring: the shard sum done the way a ring all-reduce adds
  the partials ("Tensor parallel serving", "Communication cost"): partials
  held in the wire dtype, chunk c summed from rank c around the ring, rounded
  to the wire dtype after every hop, bias once.  The oracle does the same
  from its fp64 partials.  The two can differ where a partial or a running sum
  sits on a rounding boundary, so the bound per element is 2 * tp roundings
  of the wire dtype at the size of the partials, S_e = sum_i |P_i[e]|, plus
  fp32 accumulation error.
* column_parallel_linear_uneven: explicit per-shard widths ("Tensor parallel
  serving", "Try it yourself": 9 outputs as 5 + 4).  Each shard runs as a
  one-shard call, so the result is bit-identical to tp = 1.
All three kernels are covered: GEMV (M <= 2), decode (3..128), prefill (> 128).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import (U_BF16, U_F32, assert_bf16_is_rounded_fp32, assert_bitwise_equal,
                         assert_close_bf16, assert_close_fp32, assert_h_bf16, np64, shard)
from tensor_column_linear_gelu_b300 import inputs, tpla

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = {torch.bfloat16: U_BF16, torch.float32: U_F32}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


# M, K, N, tp, bias
RING_CASES = [(1, 128, 40, 2, True), (2, 192, 24, 3, False), (5, 264, 72, 3, True),
              (64, 1024, 300, 4, False), (200, 1024, 520, 4, True), (129, 512, 256, 8, False)]


@pytest.mark.parametrize("wire", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("M,K,N,tp,bias", RING_CASES)
def test_ring_allreduce_mode(orc, M, K, N, tp, bias, wire):
    seed = 13 * M + K + N + tp
    X = inputs.normal((M, K), 1.0, seed, torch.bfloat16, DEV)
    W = inputs.normal((N, K), 0.05, seed + 3, torch.bfloat16, DEV)
    b = inputs.normal((N,), 0.1, seed + 5, torch.float32, DEV) if bias else None
    ws, _ = shard("row", tp, W)
    y32, parts = tpla.row_parallel_linear_ring(tp, X, ws, b, wire_dtype=wire,
                                               out_dtype=torch.float32)
    y16, parts2 = tpla.row_parallel_linear_ring(tp, X, ws, b, wire_dtype=wire,
                                                out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert_bitwise_equal(parts, parts2, "partials of two identical calls")
    assert_bf16_is_rounded_fp32(y16, y32)
    # the oracle's own partials (fp64) and its ring sum
    ks = K // tp
    Xh, Wh = np64(X), np64(W)
    P = np.stack([orc.linear(Xh[:, i * ks:(i + 1) * ks], Wh[:, i * ks:(i + 1) * ks])
                  for i in range(tp)])
    for i in range(tp):
        if wire == torch.bfloat16:
            assert_h_bf16(parts[i], P[i])
        else:
            assert_close_fp32(parts[i], P[i])
    ref = orc.row_parallel_ring(tp, X, W, b, "bf16" if wire == torch.bfloat16 else "f32")
    S = np.sum(np.abs(P), axis=0)
    bound = (2 * tp * U[wire] + 1e-5) * S + 1e-6
    err = np.abs(np64(y32) - ref)
    assert np.all(err <= bound), f"max err / bound {np.max(err / bound):.3f}"
    # against the fused sum: the ring mode is the fused result plus the wire's roundings
    fused = orc.row_parallel(tp, X, W, b)
    assert np.all(np.abs(np64(y32) - fused) <= (2 * tp * U[wire] + 1e-5) * S + 1e-6)
    assert tpla.tp_device_status() == tpla.TP_OK


def test_ring_mode_rounds_at_every_hop():
    """The hand-worked case of the oracle's pins, on the GPU: tp=3, x = 1s,
    W rows [256, 1, 1] -> partials 256, 1, 1; bf16 ring: [256, 258, 258, 256, 256]."""
    X = torch.ones(1, 3 * 8, dtype=torch.bfloat16, device=DEV)
    W = torch.zeros(5, 3 * 8, dtype=torch.bfloat16, device=DEV)
    W[:, 0], W[:, 8], W[:, 16] = 256.0, 1.0, 1.0
    ws, _ = shard("row", 3, W)
    y, _ = tpla.row_parallel_linear_ring(3, X, ws, None, wire_dtype=torch.bfloat16,
                                         out_dtype=torch.float32)
    assert y.cpu().tolist() == [[256.0, 258.0, 258.0, 256.0, 256.0]]
    yf, _ = tpla.row_parallel_linear_ring(3, X, ws, None, wire_dtype=torch.float32,
                                          out_dtype=torch.float32)
    assert yf.cpu().tolist() == [[258.0] * 5]


# M, K, widths, act, xdt, bias
UNEVEN_CASES = [(1, 8, [5, 4], "none", torch.float32, True),
                (3, 64, [5, 4], "gelu", torch.float32, False),
                (1, 64, [300, 200, 500], "gelu", torch.bfloat16, True),
                (7, 520, [300, 200, 500], "none", torch.bfloat16, False),
                (200, 256, [136, 8, 256, 40], "gelu", torch.bfloat16, True)]


@pytest.mark.parametrize("M,K,widths,act,xdt,bias", UNEVEN_CASES)
def test_uneven_column_split(orc, M, K, widths, act, xdt, bias):
    N = sum(widths)
    seed = 17 * M + K + N
    X = inputs.normal((M, K), 1.0, seed, xdt, DEV)
    W = inputs.normal((N, K), 0.05, seed + 1, xdt, DEV)
    b = inputs.normal((N,), 0.1, seed + 4, torch.float32, DEV) if bias else None
    ws, bs = tpla.tp_shard_weights_uneven(widths, W, b)
    off = 0
    for i, w in enumerate(widths):
        assert torch.equal(ws[i], W[off:off + w])
        if bias:
            assert torch.equal(bs[i], b[off:off + w])
        off += w
    y = tpla.column_parallel_linear_uneven(widths, X, ws, bs, act, out_dtype=torch.float32)
    ref = orc.column_parallel_uneven(widths, X, W, b, act)
    if xdt == torch.float32:
        assert_close_fp32(y, ref)
    else:
        assert_close_bf16(y, ref)
    w1, b1 = shard("column", 1, W, b=b)
    y1 = tpla.column_parallel_linear(1, X, w1, b1, act, out_dtype=torch.float32)
    assert_bitwise_equal(y, y1, "uneven split vs tp=1")
    assert tpla.tp_device_status() == tpla.TP_OK
