"""tp_mlp_block_noalloc: the FFN block for callers that cannot allocate device memory.

Such callers (a serving engine that owns all device memory from start-up, a
plugin whose host hands out no device memory, a path where cudaMalloc's
implicit synchronisation is not allowed) cannot provide tp_mlp_block's [M, d_ff]
workspace; this entry point keeps that workspace in a fixed buffer built into
the library.  Each test calls it twice in a row through the C ABI and checks
both results against tp_mlp_block on the same inputs: the two run the same
kernels in the same order, so the outputs must be bit-identical.  The first
result is also checked against the fp64 oracle with the tolerances of every
parity test (bf16 inputs: 5e-3 x RMS; fp32 inputs: 1e-5 x (|y| + 1)).  The
cases reach every kernel family with h in the fixed buffer: the
weight-streaming GEMV (one token, and the fp32 path), the tensor-core decode
kernel (3..128 tokens) and the prefill GEMM on CTA pairs (more than 128
tokens), all within the buffer's 8 MiB.  This file is collected last so that
a run stopping at its first failure has already run every other test; it
needs nothing from them and also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

from gpu_helpers import assert_bitwise_equal, assert_close_bf16, assert_close_fp32
from tensor_column_linear_gelu_b300 import inputs, tpla

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def _noalloc_abi(tp, X, w1, b1, w2, b2, act, d_ff, Y):
    """Call the entry point through the C ABI (ctypes), on the current stream."""
    M, d_model = X.shape
    return tpla.lib.tp_mlp_block_noalloc(
        tp, M, d_model, d_ff, tpla.ACTS[act], tpla.dtype_code(X.dtype), X.data_ptr(),
        tpla.ptr_array(w1), tpla.ptr_array(b1), tpla.ptr_array(w2),
        None if b2 is None else b2.data_ptr(), Y.data_ptr(), tpla.dtype_code(Y.dtype),
        tpla.stream_handle(None))


# M, d_model, d_ff, tp, act, input dtype; h = M * d_ff elements of the input
# dtype, at most 2 MiB here (the buffer holds 8 MiB)
CASES = [
    (1, 256, 1024, 4, "swiglu", torch.bfloat16),   # weight-streaming GEMV
    (3, 256, 512, 2, "gelu", torch.float32),       # fp32 path (GEMV), h in fp32
    (4, 256, 1024, 4, "swiglu", torch.bfloat16),   # tensor-core decode kernel
    (96, 512, 2048, 2, "gelu", torch.bfloat16),    # tensor-core decode kernel
    (512, 512, 2048, 2, "gelu", torch.bfloat16),   # prefill GEMM on CTA pairs
]


@pytest.mark.parametrize("M,d,dff,tp,act,dt", CASES)
def test_noalloc_matches_tp_mlp_block_twice(orc, M, d, dff, tp, act, dt):
    bias = act != "swiglu"
    f = inputs.ffn(seed=500 + M, M=M, d_model=d, d_ff=dff, act=act, bias=bias, device=DEV,
                   dtype=dt)
    split = "gate_up" if act == "swiglu" else "column"
    w1, b1 = tpla.tp_shard_weights(split, tp, f.W1, W_up=f.W_up, b=f.b1)
    w2, _ = tpla.tp_shard_weights("row", tp, f.W2)
    X2 = inputs.normal((M, d), 1.0, 900 + M, dt, DEV)   # second call: new tokens
    for k, X in enumerate((f.X, X2)):
        ref, _ = tpla.tp_mlp_block(tp, X, w1, b1, w2, f.b2, act, d_ff=dff,
                                   out_dtype=torch.float32)
        Y = torch.full((M, d), float("nan"), dtype=torch.float32, device=DEV)
        st = _noalloc_abi(tp, X, w1, b1, w2, f.b2, act, dff, Y)
        assert st == tpla.TP_OK, tpla.status_string(st)
        torch.cuda.synchronize()
        assert_bitwise_equal(Y, ref, f"call {k + 1}: noalloc vs tp_mlp_block")
        if k == 0:
            y_ref, _ = orc.mlp_block(tp, X, f.W1, f.b1, f.W2, f.b2, act, W1u=f.W_up,
                                     round_h=(dt == torch.bfloat16))
            if dt == torch.bfloat16:
                assert_close_bf16(Y, y_ref)
            else:
                assert_close_fp32(Y, y_ref)
    assert tpla.tp_device_status() == tpla.TP_OK


def test_noalloc_rejects_calls_beyond_its_workspace():
    M, d, dff, tp = 8, 256, 1024, 2
    W1 = inputs.normal((dff, d), 0.02, 1, torch.bfloat16, DEV)
    W2 = inputs.normal((d, dff), 0.02, 2, torch.bfloat16, DEV)
    w1, _ = tpla.tp_shard_weights("column", tp, W1)
    w2, _ = tpla.tp_shard_weights("row", tp, W2)
    # h would need M * d_ff * 2 bytes: one token-row more than the limit allows
    too_many = tpla.TP_NOALLOC_SCRATCH_BYTES // (dff * 2) + 1
    X = torch.zeros(too_many, d, dtype=torch.bfloat16, device=DEV)
    Y = torch.full((too_many, d), 7.0, dtype=torch.float32, device=DEV)
    st = _noalloc_abi(tp, X, w1, None, w2, None, "gelu", dff, Y)
    assert st == tpla.TP_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(Y == 7.0)           # nothing was launched or written
    assert ctypes.sizeof(ctypes.c_int) == 4  # the status travels as a C int
