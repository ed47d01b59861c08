"""tp_layer_forward: one layer's linear algebra in one call, and its CUDA-graph replay.

The call issues the attention projections (QKV by head group, O by head with
the shard sum) and then the FFN block (column with the activation per shard,
row with the shard sum).  Checks:
  * its outputs are bit-identical to tp_attn_proj followed by tp_mlp_block on
    the same inputs (the same kernels in the same order);
  * against the oracle: QKV (fp32 output) within the bf16 tolerance; the
    attention output, stored in bf16, within half a bf16 ulp of the exact
    value; the FFN output computed by the oracle from its own attention output
    rounded to bf16 (the FFN reads the attention block's output);
  * a CUDA graph of the call replays to the same bits, and replays on new
    inputs copied into the captured buffers.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_bitwise_equal, assert_close_bf16, assert_h_bf16, shard
from tensor_column_linear_gelu_b300 import inputs, tpla

pytestmark = pytest.mark.gpu
DEV = "cuda"

# M, d_model, H, Hkv, hd, d_ff, tp, FFN activation
CASES = [(8, 256, 8, 4, 32, 1024, 4, "swiglu"),
         (200, 512, 16, 8, 32, 2048, 2, "gelu")]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def _layer(M, d, H, Hkv, hd, dff, tp, act, seed):
    a = inputs.attn(seed=seed, M=M, d_model=d, n_heads=H, n_kv_heads=Hkv, head_dim=hd,
                    bias=(act != "swiglu"), device=DEV)
    f = inputs.ffn(seed=seed + 50, M=M, d_model=d, d_ff=dff, act=act, bias=(act != "swiglu"),
                   device=DEV)
    heads = dict(n_heads=H, n_kv_heads=Hkv, head_dim=hd)
    wq, bq = shard("qkv_heads", tp, a.Wqkv, b=a.bqkv, **heads)
    wo, _ = shard("row", tp, a.Wo)
    split = "gate_up" if act == "swiglu" else "column"
    w1, b1 = shard(split, tp, f.W1, W_up=f.W_up, b=f.b1)
    w2, _ = shard("row", tp, f.W2)
    kw = dict(X=a.X, wqkv_shards=wq, bqkv_shards=bq, ctx=a.ctx, wo_shards=wo, bo=a.bo,
              n_heads=H, n_kv_heads=Hkv, head_dim=hd, w1_shards=w1, b1_shards=b1, w2_shards=w2,
              b2=f.b2, ffn_act=act, d_ff=dff)
    return a, f, kw


@pytest.mark.parametrize("M,d,H,Hkv,hd,dff,tp,act", CASES)
def test_layer_forward_matches_blocks_and_oracle(orc, M, d, H, Hkv, hd, dff, tp, act):
    a, f, kw = _layer(M, d, H, Hkv, hd, dff, tp, act, seed=7 * M + d)
    qkv, ya, h, yf = tpla.tp_layer_forward(tp, **kw, out_dtype=torch.float32,
                                           qkv_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ya.dtype == torch.bfloat16  # the FFN reads it: kept in the input dtype
    # the same kernels, called block by block
    qkv2, ya2 = tpla.tp_attn_proj(tp, a.X, kw["wqkv_shards"], kw["bqkv_shards"], a.ctx,
                                  kw["wo_shards"], a.bo, H, Hkv, hd, qkv_dtype=torch.float32)
    yf2, h2 = tpla.tp_mlp_block(tp, ya2, kw["w1_shards"], kw["b1_shards"], kw["w2_shards"], f.b2,
                                act, d_ff=dff, out_dtype=torch.float32)
    torch.cuda.synchronize()
    for x, y, what in [(qkv, qkv2, "qkv"), (ya, ya2, "attention output"), (h, h2, "h"),
                       (yf, yf2, "FFN output")]:
        assert_bitwise_equal(x, y, what)
    # the oracle, chained the same way: FFN input = its attention output in bf16
    ref_qkv = orc.qkv_proj(tp, a.X, a.Wqkv, a.bqkv, H, Hkv, hd)
    ref_ya = orc.o_proj(tp, a.ctx, a.Wo, a.bo, H, hd)
    assert_close_bf16(qkv, ref_qkv)
    assert_h_bf16(ya, ref_ya)  # stored in bf16: within half an ulp of the exact value
    ya_bf16 = np.vectorize(orc.round_bf16)(ref_ya)
    ref_yf, _ = orc.mlp_block(tp, ya_bf16, f.W1, f.b1, f.W2, f.b2, act, W1u=f.W_up, round_h=True)
    assert_close_bf16(yf, ref_yf)
    assert tpla.tp_device_status() == tpla.TP_OK


@pytest.mark.parametrize("M,d,H,Hkv,hd,dff,tp,act", CASES[:1])
def test_layer_graph_replays_bitwise(M, d, H, Hkv, hd, dff, tp, act):
    a, f, kw = _layer(M, d, H, Hkv, hd, dff, tp, act, seed=11)
    g = tpla.LayerGraph(tp, **kw)
    outs = [o.clone() for o in g.replay()]
    torch.cuda.synchronize()
    direct = tpla.tp_layer_forward(tp, **kw)
    torch.cuda.synchronize()
    for x, y in zip(outs, direct):
        assert_bitwise_equal(x, y, "graph replay vs direct call")
    # new inputs, copied into the captured buffers
    X2 = inputs.normal((M, d), 1.0, 991, torch.bfloat16, DEV)
    c2 = inputs.normal(tuple(a.ctx.shape), 1.0, 992, torch.bfloat16, DEV)
    kw["X"].copy_(X2)
    kw["ctx"].copy_(c2)
    outs2 = [o.clone() for o in g.replay()]
    torch.cuda.synchronize()
    direct2 = tpla.tp_layer_forward(tp, **dict(kw, X=X2, ctx=c2))
    torch.cuda.synchronize()
    for x, y in zip(outs2, direct2):
        assert_bitwise_equal(x, y, "graph replay on new inputs vs direct call")
    assert not torch.equal(outs2[3], outs[3])
    assert tpla.tp_device_status() == tpla.TP_OK
