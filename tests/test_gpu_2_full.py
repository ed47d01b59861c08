"""GPU parity at the full Llama-2-70B-shaped sizes, in the benchmark's launch path.

  * SwiGLU FFN decode, tp=4: X [B, 8192], B in {1, 8, 32, 64}; W_gate/W_up
    [28672, 8192], W_down [8192, 28672], N(0, 0.02), no bias.
  * SwiGLU FFN prefill, tp=8: X [4096, 8192], same weights.
  * Attention projections, tp=8: X [2048, 8192], 64 query heads, 8 KV heads of
    dim 128; W_qkv [10240, 8192] split by head group, W_o [8192, 8192] split by
    head.
The oracle checks every row of the decode calls, and 64 seeded rows (always
rows 0 and M-1) of the 4096-token prefill and the 2048-token attention
projections: each output row depends only on its own input row, so a sampled
row is checked exactly as in the full call.  Column outputs are checked bit
for bit against tp = 1 on every row.
"""
import pytest
import torch

from gpu_helpers import (assert_bf16_is_rounded_fp32, assert_bitwise_equal, assert_close_bf16,
                         assert_h_bf16, shard)
from tensor_column_linear_gelu_b300 import inputs, tpla

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"
D, DFF = 8192, 28672
WEIGHT_SEED = 70_000


@pytest.fixture(scope="module")
def ffn_weights():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    f = inputs.llama70b_ffn(WEIGHT_SEED, M=1, device=DEV)
    host = {"Wg": f.W1.float().cpu().numpy(), "Wu": f.W_up.float().cpu().numpy(),
            "Wd": f.W2.float().cpu().numpy()}
    shards = {}
    for tp in (1, 4, 8):
        shards[tp] = (shard("gate_up", tp, f.W1, W_up=f.W_up)[0], shard("row", tp, f.W2)[0])
    yield f, host, shards
    del shards
    torch.cuda.empty_cache()


def _run_ffn(orc, ffn_weights, M, tp, n_sample, x_seed):
    f, host, shards = ffn_weights
    X = inputs.normal((M, D), 1.0, x_seed, torch.bfloat16, DEV)
    w1, w2 = shards[tp]
    y32, h = tpla.tp_mlp_block(tp, X, w1, None, w2, None, "swiglu", d_ff=DFF,
                               out_dtype=torch.float32)
    y16, h16 = tpla.tp_mlp_block(tp, X, w1, None, w2, None, "swiglu", d_ff=DFF,
                                 out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert_bf16_is_rounded_fp32(y16, y32)
    assert_bitwise_equal(h16, h, "h of the bf16-out run")
    # column half bit-exact against tp = 1 (every row)
    h1 = tpla.column_parallel_linear(1, X, shards[1][0], None, "swiglu", N=DFF)
    assert_bitwise_equal(h, h1, f"h tp={tp} vs tp=1")
    rows = inputs.sample_rows(M, n_sample, x_seed)
    Xs = X[rows]
    Yref, _ = orc.mlp_block(tp, Xs, host["Wg"], None, host["Wd"], None, "swiglu",
                            W1u=host["Wu"], round_h=True)
    h_exact = orc.column_parallel(tp, Xs, host["Wg"], None, "swiglu", Wu=host["Wu"])
    assert_h_bf16(h[rows], h_exact)
    return assert_close_bf16(y32[rows], Yref)


@pytest.mark.parametrize("B", [1, 8, 32, 64])
def test_swiglu_decode_tp4(orc, ffn_weights, B):
    _run_ffn(orc, ffn_weights, B, 4, n_sample=B, x_seed=71_000 + B)


def test_swiglu_prefill_tp8(orc, ffn_weights):
    _run_ffn(orc, ffn_weights, 4096, 8, n_sample=64, x_seed=72_000)


def test_attn_proj_tp8(orc):
    H, Hkv, hd, M, tp = 64, 8, 128, 2048, 8
    a = inputs.llama70b_attn(73_000, M, device=DEV)
    heads = dict(n_heads=H, n_kv_heads=Hkv, head_dim=hd)
    wq, _ = shard("qkv_heads", tp, a.Wqkv, **heads)
    wo, _ = shard("row", tp, a.Wo)
    qkv, y32 = tpla.tp_attn_proj(tp, a.X, wq, None, a.ctx, wo, None, H, Hkv, hd,
                                 qkv_dtype=torch.float32, out_dtype=torch.float32)
    qkv16, y16 = tpla.tp_attn_proj(tp, a.X, wq, None, a.ctx, wo, None, H, Hkv, hd)
    torch.cuda.synchronize()
    assert_bf16_is_rounded_fp32(y16, y32)
    assert_bf16_is_rounded_fp32(qkv16, qkv)
    # QKV shards re-gathered == the unsharded projection, bit for bit
    wq1, _ = shard("qkv_heads", 1, a.Wqkv, **heads)
    full = tpla.column_parallel_linear(1, a.X, wq1, None, "none", out_dtype=torch.float32)
    hq, hk = H // tp, Hkv // tp
    for i in range(tp):
        cols = (list(range(i * hq * hd, (i + 1) * hq * hd)) +
                list(range(H * hd + i * hk * hd, H * hd + (i + 1) * hk * hd)) +
                list(range((H + Hkv) * hd + i * hk * hd, (H + Hkv) * hd + (i + 1) * hk * hd)))
        assert_bitwise_equal(qkv[i], full[:, cols].contiguous(), f"qkv shard {i}")
    rows = inputs.sample_rows(M, 64, 73_000)
    ref_qkv = orc.qkv_proj(tp, a.X[rows], a.Wqkv.float().cpu().numpy(), None, H, Hkv, hd)
    assert_close_bf16(qkv[:, rows], ref_qkv)
    ref_y = orc.o_proj(tp, a.ctx[rows], a.Wo.float().cpu().numpy(), None, H, hd)
    assert_close_bf16(y32[rows], ref_y)
