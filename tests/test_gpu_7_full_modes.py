"""GPU parity at the Llama-2-70B widths for the variants beyond the fused path,
in the launch configurations the benchmark times.

The decode kernels choose their cluster sizes, per-SM feature ranges and
weight-box shapes from the problem size, so only the full-size launch runs
the tilings the benchmark measures.  Each case below is one benchmarked
workload, checked against the fp64 oracle:

  * FP8 (e4m3) SwiGLU FFN decode, tp=4 (d_model 8192, d_ff 28672), tokens in
    {1, 8, 64, 100}: the FP8 GEMV, the kernel that widens the codes into
    tensor memory, and the decode kernel in its FP8 mode.  The oracle
    quantizes the same bf16 weights itself ("Model Parallelism", opening
    section: about one byte per parameter in FP8).
  * The FFN down projection of the 4096-token prefill, tp=8, with the shard
    sum done the way a ring all-reduce adds bf16 partials ("Tensor parallel
    serving", "Communication cost"): 64 sampled rows (always 0 and M-1),
    checked with the oracle's ring on the full call's chunks.
  * The uneven tp=3 column split of the 8-token decode (9558 + 9557 + 9557 of
    d_ff 28672; "Tensor parallel serving", "Try it yourself"): every row,
    bit-identical to tp=1.
  * One decoder layer's linear algebra at 8 tokens, tp=4 (64 query heads, 8
    KV heads of dim 128, SwiGLU FFN): tp_layer_forward and its CUDA-graph
    replay, every row ("What is tensor parallelism?", "How a layer is
    split").  The projections against the oracle; the FFN bit-identical to
    the MLP block on the layer's own attention output, and against the
    oracle on the oracle's attention output rounded to bf16.
Tolerances are those of gpu_helpers (bf16 inputs, fp32 output: 5e-3 x RMS).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import (U_BF16, U_F32, assert_bitwise_equal, assert_close_bf16, assert_h_bf16,
                         np64, shard)
from tensor_column_linear_gelu_b300 import inputs, tpla

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"
D, DFF = 8192, 28672


@pytest.fixture(scope="module")
def weights():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    f = inputs.llama70b_ffn(77_000, M=1, device=DEV)
    yield f
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def fp8_setup(orc, weights):
    f = weights
    tp = 4
    w1, _ = shard("gate_up", tp, f.W1, W_up=f.W_up)
    w2, _ = shard("row", tp, f.W2)
    q1, s1 = tpla.quantize_shards_fp8(w1)
    q2, s2 = tpla.quantize_shards_fp8(w2)
    del w1, w2
    torch.cuda.synchronize()
    # the oracle's own quantization of the same bf16 weights
    ref = {}
    ref["qg"], ref["sg"] = orc.quantize_rows_fp8(f.W1)
    ref["qu"], ref["su"] = orc.quantize_rows_fp8(f.W_up)
    ref["qd"], ref["sd"] = orc.quantize_row_shards_fp8(tp, f.W2)
    # the GPU quantizer's scales equal the oracle's (integer decisions, both in fp32)
    assert np.array_equal(np.stack([s.cpu().numpy() for s in s2]), ref["sd"])
    yield tp, q1, s1, q2, s2, ref
    del q1, q2
    torch.cuda.empty_cache()


@pytest.mark.parametrize("B,n_sample", [(1, 1), (8, 8), (64, 24), (100, 24)])
def test_fp8_swiglu_decode_tp4_full(orc, fp8_setup, B, n_sample):
    tp, q1, s1, q2, s2, ref = fp8_setup
    X = inputs.normal((B, D), 1.0, 78_000 + B, torch.bfloat16, DEV)
    y, h = tpla.tp_mlp_block_fp8(tp, X, q1, s1, None, q2, s2, None, "swiglu", d_ff=DFF,
                                 out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = inputs.sample_rows(B, n_sample, 78_000 + B)
    Xs = X[rows]
    h_exact = orc.column_parallel_fp8(tp, Xs, ref["qg"], ref["sg"], None, "swiglu",
                                      Qu=ref["qu"], Su=ref["su"])
    assert_h_bf16(h[rows], h_exact)
    h_ref = np.vectorize(orc.round_bf16)(h_exact)
    y_ref = orc.row_parallel_fp8(tp, h_ref, ref["qd"], ref["sd"], None)
    assert_close_bf16(y[rows], y_ref)


def test_row_ring_prefill_tp8_full(orc, weights):
    """The benchmarked ring-ordered down projection: M 4096, K 28672, N 8192."""
    tp, M = 8, 4096
    hX = inputs.normal((M, DFF), 1.0, 79_000, torch.bfloat16, DEV)
    ws, _ = shard("row", tp, weights.W2)
    y32, parts = tpla.row_parallel_linear_ring(tp, hX, ws, None, wire_dtype=torch.bfloat16,
                                               out_dtype=torch.float32)
    torch.cuda.synchronize()
    rows = inputs.sample_rows(M, 64, 79_000)
    Xs = np64(hX[rows])
    Wh = weights.W2.float().cpu().numpy()
    ref = orc.row_parallel_ring_rows(tp, M, rows.numpy(), Xs, Wh, None, "bf16")
    # per-element bound: 2 * tp wire roundings at the size of the partials
    ks = DFF // tp
    P = np.stack([orc.linear(Xs[:, i * ks:(i + 1) * ks], Wh[:, i * ks:(i + 1) * ks])
                  for i in range(tp)])
    for i in range(tp):
        assert_h_bf16(parts[i][rows], P[i])
    S = np.sum(np.abs(P), axis=0)
    bound = (2 * tp * U_BF16 + 1e-5) * S + 1e-6
    err = np.abs(np64(y32[rows]) - ref)
    assert np.all(err <= bound), f"max err / bound {np.max(err / bound):.3f}"


def test_column_uneven_decode_tp3_full(orc, weights):
    """The benchmarked uneven split: 8 tokens, widths 9558/9557/9557."""
    widths = (9558, 9557, 9557)
    X = inputs.normal((8, D), 1.0, 80_000, torch.bfloat16, DEV)
    ws, _ = tpla.tp_shard_weights_uneven(widths, weights.W1)
    for act in ("none", "gelu"):
        y = tpla.column_parallel_linear_uneven(widths, X, ws, None, act, out_dtype=torch.float32)
        y1 = tpla.column_parallel_linear(1, X, [weights.W1], None, act, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert_bitwise_equal(y, y1, f"uneven tp=3 vs tp=1 ({act})")
        ref = orc.column_parallel_uneven(list(widths), X, weights.W1, None, act)
        assert_close_bf16(y, ref)


def test_layer_decode_tp4_full(orc):
    """The benchmarked decoder layer at 8 tokens: direct call, graph replay, oracle."""
    M, tp, H, Hkv, hd = 8, 4, 64, 8, 128
    a = inputs.llama70b_attn(81_000, M, device=DEV)
    f = inputs.llama70b_ffn(81_100, M, device=DEV)
    heads = dict(n_heads=H, n_kv_heads=Hkv, head_dim=hd)
    wq, _ = shard("qkv_heads", tp, a.Wqkv, **heads)
    wo, _ = shard("row", tp, a.Wo)
    w1, _ = shard("gate_up", tp, f.W1, W_up=f.W_up)
    w2, _ = shard("row", tp, f.W2)
    kw = dict(X=a.X, wqkv_shards=wq, bqkv_shards=None, ctx=a.ctx, wo_shards=wo, bo=None,
              w1_shards=w1, b1_shards=None, w2_shards=w2, b2=None, ffn_act="swiglu", d_ff=DFF,
              **heads)
    qkv, ya, h, yf = tpla.tp_layer_forward(tp, **kw, out_dtype=torch.float32,
                                           qkv_dtype=torch.float32)
    g = tpla.LayerGraph(tp, **kw)
    outs = [o.clone() for o in g.replay()]
    direct = tpla.tp_layer_forward(tp, **kw)
    torch.cuda.synchronize()
    for x, y in zip(outs, direct):
        assert_bitwise_equal(x, y, "graph replay vs direct call")
    ref_qkv = orc.qkv_proj(tp, a.X, a.Wqkv, None, H, Hkv, hd)
    assert_close_bf16(qkv, ref_qkv)
    ref_ya = orc.o_proj(tp, a.ctx, a.Wo, None, H, hd)
    assert_h_bf16(ya, ref_ya)
    # The layer feeds its own bf16 attention output to the FFN: its h and FFN
    # output are those of the MLP block called on that tensor.
    yf2, h2 = tpla.tp_mlp_block(tp, ya, w1, None, w2, None, "swiglu", d_ff=DFF,
                                out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert_bitwise_equal(h, h2, "layer h vs MLP block on the layer's attention output")
    assert_bitwise_equal(yf, yf2, "layer FFN output vs MLP block")
    # The FFN against the oracle, on the oracle's attention output in bf16.  (An
    # element of ya within rounding slack of a bf16 midpoint may round either
    # way, which changes h there by more than half an ulp; so h is compared on
    # the oracle's own input, not chained through ya.)
    ya_bf16 = np.vectorize(orc.round_bf16)(ref_ya)
    x_ref = torch.tensor(ya_bf16, dtype=torch.float32).to(torch.bfloat16).to(DEV)
    yf3, h3 = tpla.tp_mlp_block(tp, x_ref, w1, None, w2, None, "swiglu", d_ff=DFF,
                                out_dtype=torch.float32)
    torch.cuda.synchronize()
    ref_yf, h_exact = orc.mlp_block(tp, ya_bf16, f.W1, None, f.W2, None, "swiglu", W1u=f.W_up,
                                    round_h=False)
    assert_h_bf16(h3, h_exact)
    ref_yf, _ = orc.mlp_block(tp, ya_bf16, f.W1, None, f.W2, None, "swiglu", W1u=f.W_up,
                              round_h=True)
    assert_close_bf16(yf3, ref_yf)
    assert_close_bf16(yf, ref_yf)
