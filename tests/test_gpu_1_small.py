"""GPU parity on small and ragged shapes: every entry point against the oracle.

Shapes span several kernel tiles with ragged tails in M, N and K, every tp the
pages use (1, 2, 4, 8) and some they do not (3, 5), fp32 and bf16, each
activation, with and without bias, on all three kernels: the weight-streaming
GEMV (fp32, and bf16 with M <= 2), the tcgen05 decode kernel (bf16,
3 <= M <= 128; the cases below put its per-SM feature ranges across shard and
gate/up-group boundaries and give shards widths that are not multiples of 8)
and the tcgen05 prefill GEMM (bf16, M > 128).  All calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle_pin_checks as pins
from gpu_helpers import (assert_bf16_is_rounded_fp32, assert_bitwise_equal, assert_close_bf16,
                         assert_close_fp32, assert_h_bf16, np64, shard)
from tensor_column_linear_gelu_b300 import inputs, tpla

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


# --------------------------------------------------------------- worked example

def test_worked_example_fp32_tp2(orc):
    """x [1,8] . W [6,8]^T + b split 3 + 3 ("Tensor parallel serving", the demo)."""
    x, W, b = inputs.worked_example()
    xd, Wd, bd = x.to(DEV), W.to(DEV), b.to(DEV)
    w2, b2 = shard("column", 2, Wd, b=bd)
    assert [t.numel() for t in w2] == [24, 24]          # 24 of 48 weights each
    y2 = tpla.column_parallel_linear(2, xd, w2, b2, "none")
    ref = orc.linear(x, W, b)
    assert_close_fp32(y2, ref)
    vals, _ = pins.read_golden()
    assert np.array_equal(np.round(np64(y2)[0], 4), vals["combined"])
    w1, b1 = shard("column", 1, Wd, b=bd)
    y1 = tpla.column_parallel_linear(1, xd, w1, b1, "none")
    assert np.array_equal(np.round(np64(y1)[0], 4), vals["full"])
    assert_bitwise_equal(y2, y1, "tp=2 vs tp=1")


# --------------------------------------------------------------- column

COLUMN_CASES = [
    # M, K, N, tp, act, xdt, bias
    (1, 8, 6, 2, "none", torch.float32, True),
    (5, 64, 48, 3, "gelu", torch.float32, True),
    (20, 32, 16, 4, "gelu", torch.float32, False),
    (1, 64, 96, 2, "gelu", torch.bfloat16, True),
    (2, 264, 136, 2, "swiglu", torch.bfloat16, False),
    (3, 520, 200, 4, "gelu", torch.bfloat16, True),
    (8, 256, 384, 8, "none", torch.bfloat16, False),
    (128, 64, 256, 1, "none", torch.bfloat16, False),      # exactly one GEMM tile
    (13, 136, 72, 2, "gelu", torch.bfloat16, True),
    (130, 264, 320, 2, "gelu", torch.bfloat16, True),
    (200, 512, 1024, 4, "none", torch.bfloat16, True),
    (300, 1032, 640, 8, "gelu", torch.bfloat16, False),
    (4, 1024, 256, 2, "swiglu", torch.bfloat16, False),
    (5, 136, 300, 2, "swiglu", torch.bfloat16, False),
    (150, 264, 520, 4, "swiglu", torch.bfloat16, False),
    (333, 512, 1280, 2, "swiglu", torch.bfloat16, False),
    (96, 200, 3000, 3, "swiglu", torch.bfloat16, False),   # partial gate/up groups
    (64, 1000, 2600, 4, "gelu", torch.bfloat16, True),     # 650 outputs per shard
    (16, 256, 40000, 2, "none", torch.bfloat16, False),    # several chunks per SM
    (128, 64, 1000, 5, "none", torch.bfloat16, True),
    (6, 72, 136, 1, "swiglu", torch.bfloat16, False),
    # decode column launches with too few weight rows per SM and long K
    # loops split K over clusters: ten 20-feature shards need two tiles per
    # cluster range; a gate/up tile of 128 features runs across a shard
    # boundary
    (8, 4096, 200, 10, "gelu", torch.bfloat16, True),
    (12, 4096, 360, 3, "swiglu", torch.bfloat16, False),
    (32, 8192, 2560, 4, "none", torch.bfloat16, False),
    # prefill GEMM with more tiles (9 x 20 = 180) than clusters that run at
    # once: the running clusters take over the others' tiles; ragged M and N
    (2300, 256, 4100, 4, "gelu", torch.bfloat16, True),
]


def _column_inputs(M, K, N, act, xdt, bias, seed):
    X = inputs.normal((M, K), 1.0, seed, xdt, DEV)
    W = inputs.normal((N, K), 0.05, seed + 1, xdt, DEV)
    Wu = inputs.normal((N, K), 0.05, seed + 2, xdt, DEV) if act == "swiglu" else None
    b = inputs.normal((N,), 0.1, seed + 4, torch.float32, DEV) if bias else None
    return X, W, Wu, b


@pytest.mark.parametrize("M,K,N,tp,act,xdt,bias", COLUMN_CASES)
def test_column_parallel(orc, M, K, N, tp, act, xdt, bias):
    X, W, Wu, b = _column_inputs(M, K, N, act, xdt, bias, seed=M * 7 + K + N + tp)
    split = "gate_up" if act == "swiglu" else "column"
    ws, bs = shard(split, tp, W, W_up=Wu, b=b)
    y32 = tpla.column_parallel_linear(tp, X, ws, bs, act, out_dtype=torch.float32, N=N)
    ref = orc.column_parallel(tp, X, W, b, act, Wu=Wu)
    if xdt == torch.float32:
        assert_close_fp32(y32, ref)
    else:
        assert_close_bf16(y32, ref)
        y16 = tpla.column_parallel_linear(tp, X, ws, bs, act, out_dtype=torch.bfloat16, N=N)
        assert_bf16_is_rounded_fp32(y16, y32)
    # bit-exact against the same kernel unsharded
    w1, b1 = shard(split, 1, W, W_up=Wu, b=b)
    y1 = tpla.column_parallel_linear(1, X, w1, b1, act, out_dtype=torch.float32, N=N)
    assert_bitwise_equal(y32, y1, "sharded vs tp=1")


def test_column_output_strided(orc):
    """Y with a leading dimension larger than N (a column block of a wider buffer)."""
    M, K, N, tp = 37, 128, 96, 2
    X, W, _, b = _column_inputs(M, K, N, "gelu", torch.bfloat16, True, seed=5)
    ws, bs = shard("column", tp, W, b=b)
    big = torch.full((M, N + 40), 7.0, dtype=torch.float32, device=DEV)
    tpla.column_parallel_linear(tp, X, ws, bs, "gelu", Y=big[:, 8:8 + N], N=N)
    assert_close_bf16(big[:, 8:8 + N], orc.column_parallel(tp, X, W, b, "gelu"))
    assert torch.all(big[:, :8] == 7.0) and torch.all(big[:, 8 + N:] == 7.0)


def test_empty_batch():
    W = torch.randn(64, 64, device=DEV).to(torch.bfloat16)
    ws, _ = shard("column", 2, W)
    X = torch.empty(0, 64, dtype=torch.bfloat16, device=DEV)
    Y = tpla.column_parallel_linear(2, X, ws, None, "none")
    assert Y.shape == (0, 64)
    w2, _ = shard("row", 2, W)
    Y = tpla.row_parallel_linear(2, X, w2, None)
    assert Y.shape == (0, 64)


# --------------------------------------------------------------- row

ROW_CASES = [
    # M, K, N, tp, xdt, bias
    (1, 16, 8, 2, torch.float32, True),
    (9, 96, 40, 3, torch.float32, False),
    (1, 64, 32, 2, torch.bfloat16, True),
    (7, 1056, 100, 4, torch.bfloat16, True),
    (8, 512, 64, 8, torch.bfloat16, False),
    (130, 2048, 96, 8, torch.bfloat16, True),
    (257, 768, 520, 2, torch.bfloat16, True),
    (64, 4096, 256, 4, torch.bfloat16, False),
    (100, 3000, 1000, 3, torch.bfloat16, True),   # K/tp = 1000: ragged k-block per shard
    (128, 1024, 4000, 2, torch.bfloat16, False),
    (5, 4096, 3000, 4, torch.bfloat16, True),
    # prefill GEMM, 9 x 11 = 99 tiles (more than run at once), ragged M and N
    (2300, 1024, 2600, 4, torch.bfloat16, True),
]


@pytest.mark.parametrize("M,K,N,tp,xdt,bias", ROW_CASES)
def test_row_parallel(orc, M, K, N, tp, xdt, bias):
    seed = 3 * M + K + N + tp
    X = inputs.normal((M, K), 1.0, seed, xdt, DEV)
    W = inputs.normal((N, K), 0.05, seed + 3, xdt, DEV)
    b = inputs.normal((N,), 0.1, seed + 5, torch.float32, DEV) if bias else None
    ws, _ = shard("row", tp, W)
    y32 = tpla.row_parallel_linear(tp, X, ws, b, out_dtype=torch.float32)
    ref = orc.row_parallel(tp, X, W, b)
    if xdt == torch.float32:
        assert_close_fp32(y32, ref)
    else:
        assert_close_bf16(y32, ref)
        y16 = tpla.row_parallel_linear(tp, X, ws, b, out_dtype=torch.bfloat16)
        assert_bf16_is_rounded_fp32(y16, y32)


# --------------------------------------------------------------- FFN block

def test_gelu_ffn_block_tp2(orc):
    """GELU FFN block, tp=2: X bf16 [16,512]; W1 [2048,512]; W2 [512,2048]; fp32 biases."""
    f = inputs.gelu_ffn_small(seed=1234, device=DEV)
    w1, b1 = shard("column", 2, f.W1, b=f.b1)
    w2, _ = shard("row", 2, f.W2)
    y32, h = tpla.tp_mlp_block(2, f.X, w1, b1, w2, f.b2, "gelu", out_dtype=torch.float32)
    Yref, _ = orc.mlp_block(2, f.X, f.W1, f.b1, f.W2, f.b2, "gelu", round_h=True)
    assert_h_bf16(h, orc.column_parallel(2, f.X, f.W1, f.b1, "gelu"))
    assert_close_bf16(y32, Yref)
    y16, _ = tpla.tp_mlp_block(2, f.X, w1, b1, w2, f.b2, "gelu", out_dtype=torch.bfloat16)
    assert_bf16_is_rounded_fp32(y16, y32)
    # the column half alone is bit-identical to tp=1
    w11, b11 = shard("column", 1, f.W1, b=f.b1)
    h1 = tpla.column_parallel_linear(1, f.X, w11, b11, "gelu")
    assert_bitwise_equal(h, h1, "h sharded vs tp=1")


@pytest.mark.parametrize("M,d,dff,tp,act", [(3, 256, 512, 4, "swiglu"), (70, 128, 640, 2, "swiglu"),
                                            (129, 256, 1024, 8, "gelu"), (5, 64, 96, 3, "none")])
def test_ffn_block_shapes(orc, M, d, dff, tp, act):
    f = inputs.ffn(seed=M + d + dff, M=M, d_model=d, d_ff=dff, act=act,
                   bias=(act != "swiglu"), device=DEV)
    split = "gate_up" if act == "swiglu" else "column"
    w1, b1 = shard(split, tp, f.W1, W_up=f.W_up, b=f.b1)
    w2, _ = shard("row", tp, f.W2)
    y32, h = tpla.tp_mlp_block(tp, f.X, w1, b1, w2, f.b2, act, d_ff=dff, out_dtype=torch.float32)
    Yref, _ = orc.mlp_block(tp, f.X, f.W1, f.b1, f.W2, f.b2, act, W1u=f.W_up, round_h=True)
    assert_h_bf16(h, orc.column_parallel(tp, f.X, f.W1, f.b1 if act != "swiglu" else None, act,
                                         Wu=f.W_up))
    assert_close_bf16(y32, Yref)


# --------------------------------------------------------------- attention projections

@pytest.mark.parametrize("M,d,H,Hkv,hd,tp,bias", [(5, 64, 8, 2, 16, 2, True),
                                                  (140, 256, 8, 4, 32, 4, False),
                                                  (33, 128, 16, 8, 16, 8, True)])
def test_attn_proj(orc, M, d, H, Hkv, hd, tp, bias):
    a = inputs.attn(seed=M + d + H, M=M, d_model=d, n_heads=H, n_kv_heads=Hkv, head_dim=hd,
                    bias=bias, device=DEV)
    heads = dict(n_heads=H, n_kv_heads=Hkv, head_dim=hd)
    wq, bq = shard("qkv_heads", tp, a.Wqkv, b=a.bqkv, **heads)
    wo, _ = shard("row", tp, a.Wo)
    qkv, y = tpla.tp_attn_proj(tp, a.X, wq, bq, a.ctx, wo, a.bo, H, Hkv, hd,
                               qkv_dtype=torch.float32, out_dtype=torch.float32)
    ref_qkv = orc.qkv_proj(tp, a.X, a.Wqkv, a.bqkv, H, Hkv, hd)
    ref_y = orc.o_proj(tp, a.ctx, a.Wo, a.bo, H, hd)
    assert_close_bf16(qkv, ref_qkv)
    assert_close_bf16(y, ref_y)


# --------------------------------------------------------------- sharding

def test_shard_weights_bytes():
    """Every split against host slicing, bit for bit."""
    torch.manual_seed(0)
    W = torch.randn(48, 40).to(torch.bfloat16)
    Wu = torch.randn(48, 40).to(torch.bfloat16)
    b = torch.randn(48)
    for tp in (1, 2, 4):
        ns = 48 // tp
        ws, bs = shard("column", tp, W.to(DEV), b=b.to(DEV))
        for i in range(tp):
            assert torch.equal(ws[i].cpu(), W[i * ns:(i + 1) * ns])
            assert torch.equal(bs[i].cpu(), b[i * ns:(i + 1) * ns])
        ks = 40 // tp
        if (ks * 2) % 16 == 0:
            ws, _ = shard("row", tp, W.to(DEV))
            for i in range(tp):
                assert torch.equal(ws[i].cpu(), W[:, i * ks:(i + 1) * ks])
        ws, _ = shard("gate_up", tp, W.to(DEV), W_up=Wu.to(DEV))
        G = tpla.TP_GATE_UP_GROUP
        for i in range(tp):
            got = ws[i].cpu()
            for j in range(0, ns, G):
                g = min(G, ns - j)
                base = (j // G) * 2 * G
                assert torch.equal(got[base:base + g], W[i * ns + j:i * ns + j + g])
                assert torch.equal(got[base + G:base + G + g], Wu[i * ns + j:i * ns + j + g])
                assert torch.all(got[base + g:base + G] == 0)
                assert torch.all(got[base + G + g:base + 2 * G] == 0)
    H, Hkv, hd = 8, 4, 8
    Wq = torch.randn((H + 2 * Hkv) * hd, 40).to(torch.bfloat16)
    bq = torch.randn((H + 2 * Hkv) * hd)
    for tp in (1, 2, 4):
        ws, bs = shard("qkv_heads", tp, Wq.to(DEV), b=bq.to(DEV), n_heads=H, n_kv_heads=Hkv,
                       head_dim=hd)
        hq, hk = H // tp, Hkv // tp
        for i in range(tp):
            rows = (list(range(i * hq * hd, (i + 1) * hq * hd)) +
                    list(range(H * hd + i * hk * hd, H * hd + (i + 1) * hk * hd)) +
                    list(range((H + Hkv) * hd + i * hk * hd, (H + Hkv) * hd + (i + 1) * hk * hd)))
            assert torch.equal(ws[i].cpu(), Wq[rows])
            assert torch.equal(bs[i].cpu(), bq[rows])


# --------------------------------------------------------------- bounded waits

def test_bounded_wait_reports_timeout_and_context_survives(orc):
    s = torch.cuda.current_stream()
    assert tpla.tp_device_status(s) == tpla.TP_OK
    tpla.tp_selftest_bounded_wait(2_000_000, s)      # 2 ms limit on a barrier nobody completes
    assert tpla.tp_device_status(s) == tpla.TP_ERR_DEVICE_TIMEOUT
    assert tpla.tp_device_status(s) == tpla.TP_OK    # the word was cleared
    # the context is still usable
    x, W, b = inputs.worked_example()
    ws, bs = shard("column", 2, W.to(DEV), b=b.to(DEV))
    y = tpla.column_parallel_linear(2, x.to(DEV), ws, bs, "none")
    assert_close_fp32(y, orc.linear(x, W, b))
