"""The C-ABI library: loads, exports every declared symbol, validates arguments.

CPU only.  The error-path calls run in a child process with no visible CUDA
device, so even a validation bug could not turn a fake pointer into a kernel
launch on a real GPU.
"""
import json
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tpla.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for must in ("tp_shard_weights", "column_parallel_linear", "row_parallel_linear",
                 "tp_mlp_block", "tp_attn_proj", "tp_layer_forward", "tp_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol():
    from tensor_column_linear_gelu_b300 import tpla
    out = subprocess.run(["nm", "-D", "--defined-only", tpla.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(tpla.lib, name)
    assert set(tpla.EXPORTS) == set(declared_functions())


def test_checked_build_exports_the_same_symbols():
    """libtpla_checked.so (the kernels with index checks, loaded when
    TPLA_CHECKED=1) is built beside the release library and exports the same
    entry points."""
    from tensor_column_linear_gelu_b300 import build
    path = build.build(checked=True)
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, name
    code = ("import os; os.environ['TPLA_CHECKED'] = '1'\n"
            "from tensor_column_linear_gelu_b300 import tpla\n"
            "assert tpla.CHECKED and tpla.LIB_PATH.endswith('libtpla_checked.so')\n"
            "print(tpla.status_string(tpla.TP_ERR_DEVICE_CHECK))")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr
    assert r.stdout.startswith("TP_ERR_DEVICE_CHECK")


def test_shard_shape():
    from tensor_column_linear_gelu_b300 import tpla
    assert tpla.tp_shard_shape("column", 2, 6, 8) == (3, 8)
    assert tpla.tp_shard_shape("row", 4, 8192, 28672) == (8192, 7168)
    assert tpla.tp_shard_shape("qkv_heads", 8, 10240, 8192, 64, 8, 128) == (1280, 8192)
    assert tpla.tp_shard_shape("gate_up", 4, 28672, 8192) == (14336, 8192)
    assert tpla.tp_shard_shape("gate_up", 2, 300, 64) == (2 * 128 * 2, 64)  # 150 -> 2 groups
    for args, code in [(("column", 4, 6, 8), tpla.TP_ERR_NOT_DIVISIBLE),
                       (("row", 3, 6, 8), tpla.TP_ERR_NOT_DIVISIBLE),
                       (("qkv_heads", 3, 96, 8, 4, 2, 12), tpla.TP_ERR_NOT_DIVISIBLE),
                       (("qkv_heads", 2, 100, 8, 4, 2, 12), tpla.TP_ERR_BAD_SHAPE),
                       (("column", 0, 6, 8), tpla.TP_ERR_BAD_SHAPE),
                       (("column", 17, 34, 8), tpla.TP_ERR_BAD_SHAPE),
                       (("row", 2, 0, 8), tpla.TP_ERR_BAD_SHAPE)]:
        with pytest.raises(tpla.TplaError) as e:
            tpla.tp_shard_shape(*args)
        assert e.value.status == code, args


CHILD = r'''
import ctypes, json, sys
from tensor_column_linear_gelu_b300 import tpla as t
L = t.lib
A = 0x7f0000000000          # fake, 16-byte aligned "device" addresses: never dereferenced
def arr(*p): return ctypes.cast((ctypes.c_void_p * len(p))(*p), t._vpp)
w2 = arr(A + 0x1000, A + 0x2000)
res = {}
def rec(name, got): res[name] = got
BF, F32 = t.TP_BF16, t.TP_F32
# column_parallel_linear(tp, M, K, N, X, ldx, xdt, w, b, act, Y, ldy, ydt, s)
C = L.column_parallel_linear
rec("col_ok_M0", C(2, 0, 64, 64, None, 64, BF, None, None, 0, None, 64, BF, None))
rec("col_tp0", C(0, 4, 64, 64, A, 64, BF, w2, None, 0, A, 64, BF, None))
rec("col_tp17", C(17, 4, 64, 68, A, 64, BF, w2, None, 0, A, 68, BF, None))
rec("col_negM", C(2, -1, 64, 64, A, 64, BF, w2, None, 0, A, 64, BF, None))
rec("col_K0", C(2, 4, 0, 64, A, 64, BF, w2, None, 0, A, 64, BF, None))
rec("col_notdiv", C(2, 4, 64, 63, A, 64, BF, w2, None, 0, A, 63, BF, None))
rec("col_dtype_f32_to_bf16", C(2, 4, 64, 64, A, 64, F32, w2, None, 0, A, 64, BF, None))
rec("col_dtype_bad", C(2, 4, 64, 64, A, 64, 7, w2, None, 0, A, 64, BF, None))
rec("col_act_bad", C(2, 4, 64, 64, A, 64, BF, w2, None, 9, A, 64, BF, None))
rec("col_swiglu_bias", C(2, 4, 64, 64, A, 64, BF, w2, w2, 2, A, 64, BF, None))
rec("col_ldx_small", C(2, 4, 64, 64, A, 32, BF, w2, None, 0, A, 64, BF, None))
rec("col_ldy_small", C(2, 4, 64, 64, A, 64, BF, w2, None, 0, A, 32, BF, None))
rec("col_null_X", C(2, 4, 64, 64, None, 64, BF, w2, None, 0, A, 64, BF, None))
rec("col_null_Y", C(2, 4, 64, 64, A, 64, BF, w2, None, 0, None, 64, BF, None))
rec("col_null_warr", C(2, 4, 64, 64, A, 64, BF, None, None, 0, A, 64, BF, None))
rec("col_null_shard", C(2, 4, 64, 64, A, 64, BF, arr(A, None), None, 0, A, 64, BF, None))
rec("col_null_bias_shard", C(2, 4, 64, 64, A, 64, BF, w2, arr(A, None), 0, A, 64, BF, None))
rec("col_misaligned_X", C(2, 4, 64, 64, A + 8, 64, BF, w2, None, 0, A, 64, BF, None))
rec("col_misaligned_ldx", C(2, 4, 64, 64, A, 68, BF, w2, None, 0, A, 64, BF, None))
rec("col_misaligned_K", C(2, 4, 60, 64, A, 64, BF, w2, None, 0, A, 64, BF, None))
rec("col_misaligned_w", C(2, 4, 64, 64, A, 64, BF, arr(A, A + 4), None, 0, A, 64, BF, None))
rec("col_misaligned_Y", C(2, 4, 64, 64, A, 64, BF, w2, None, 0, A + 1, 64, BF, None))
# row_parallel_linear(tp, M, K, N, X, ldx, xdt, w, b, Y, ldy, ydt, s)
R = L.row_parallel_linear
rec("row_notdiv", R(3, 4, 64, 64, A, 64, BF, arr(A, A, A), None, A, 64, BF, None))
rec("row_shard_K_misaligned", R(2, 4, 40, 64, A, 40, BF, w2, None, A, 64, BF, None))
rec("row_null_Y", R(2, 4, 64, 64, A, 64, BF, w2, None, None, 64, BF, None))
rec("row_misaligned_bias", R(2, 4, 64, 64, A, 64, BF, w2, A + 2, A, 64, BF, None))
rec("row_M0", R(2, 0, 64, 64, None, 64, BF, None, None, None, 64, BF, None))
# tp_mlp_block(tp, M, d, dff, act, xdt, X, w1, b1, w2, b2, h, Y, ydt, s)
B = L.tp_mlp_block
rec("mlp_notdiv", B(3, 4, 64, 64, 1, BF, A, arr(A, A, A), None, arr(A, A, A), None, A, A, BF, None))
rec("mlp_null_h", B(2, 4, 64, 64, 1, BF, A, w2, None, w2, None, None, A, BF, None))
rec("mlp_swiglu_bias", B(2, 4, 64, 64, 2, BF, A, w2, w2, w2, None, A, A, BF, None))
rec("mlp_misaligned_shardK", B(2, 4, 64, 72, 1, BF, A, w2, None, w2, None, A, A, BF, None))
# tp_attn_proj(tp, M, d, H, Hkv, hd, xdt, X, wqkv, bqkv, qkv, qdt, ctx, wo, bo, Y, ydt, s)
P = L.tp_attn_proj
rec("attn_heads_notdiv", P(3, 4, 64, 4, 2, 8, BF, A, arr(A, A, A), None, A, BF, A, arr(A, A, A), None, A, BF, None))
rec("attn_kv_notdiv", P(4, 4, 64, 8, 2, 8, BF, A, arr(A, A, A, A), None, A, BF, A, arr(A, A, A, A), None, A, BF, None))
rec("attn_hd0", P(2, 4, 64, 4, 2, 0, BF, A, w2, None, A, BF, A, w2, None, A, BF, None))
rec("attn_null_ctx", P(2, 4, 64, 4, 2, 8, BF, A, w2, None, A, BF, None, w2, None, A, BF, None))
rec("attn_qkv_dtype", P(2, 4, 64, 4, 2, 8, F32, A, w2, None, A, BF, A, w2, None, A, F32, None))
# tp_shard_weights(split, tp, wdt, W, Wup, out, in, b, H, Hkv, hd, w_sh, b_sh, s)
S = L.tp_shard_weights
rec("shard_row_bias", S(1, 2, BF, A, None, 64, 64, A, 0, 0, 0, w2, w2, None))
rec("shard_gateup_no_up", S(3, 2, BF, A, None, 64, 64, None, 0, 0, 0, w2, None, None))
rec("shard_bias_no_dst", S(0, 2, BF, A, None, 64, 64, A, 0, 0, 0, w2, None, None))
rec("shard_null_W", S(0, 2, BF, None, None, 64, 64, None, 0, 0, 0, w2, None, None))
rec("shard_notdiv", S(0, 3, BF, A, None, 64, 64, None, 0, 0, 0, arr(A, A, A), None, None))
rec("shard_row_cols_misaligned", S(1, 2, BF, A, None, 64, 40, None, 0, 0, 0, w2, None, None))
rec("shard_dtype", S(0, 2, 5, A, None, 64, 64, None, 0, 0, 0, w2, None, None))
rec("selftest_bad_limit", L.tp_selftest_bounded_wait(0, None))
# tp_layer_forward(args, s): validation of both blocks before any launch
rec("layer_null_args", L.tp_layer_forward(None, None))
def layer(**over):
    f = dict(tp=2, M=4, d_model=64, xdt=BF, n_heads=4, n_kv_heads=2, head_dim=8, X=A,
             wqkv_shards=w2, bqkv_shards=None, qkv_out=A, qkv_dt=BF, ctx=A, wo_shards=w2, bo=None,
             Y_attn=A + 0x100, attn_ydt=BF, d_ff=128, ffn_act=2, X_ffn=A + 0x100, w1_shards=w2,
             b1_shards=None, w2_shards=w2, b2=None, h=A, Y_ffn=A, ffn_ydt=BF)
    f.update(over)
    a = t.LayerArgs(**f)
    return L.tp_layer_forward(ctypes.byref(a), None)
rec("layer_M0", layer(M=0, X=None, qkv_out=None, ctx=None, Y_attn=None, X_ffn=None, h=None, Y_ffn=None))
rec("layer_ffn_notdiv", layer(d_ff=129))
rec("layer_ffn_null_h", layer(h=None))
rec("layer_attn_kv_notdiv", layer(n_kv_heads=1))
rec("layer_feed_dtype", layer(attn_ydt=F32))
rec("layer_swiglu_bias", layer(b1_shards=w2))
# row_parallel_linear_ring(tp, M, K, N, X, ldx, xdt, w, b, wire, partials, Y, ldy, ydt, s)
RR = L.row_parallel_linear_ring
rec("ring_null_partials", RR(2, 4, 64, 64, A, 64, BF, w2, None, BF, None, A, 64, BF, None))
rec("ring_wire_bf16_from_f32", RR(2, 4, 64, 64, A, 64, F32, w2, None, BF, A, A, 64, F32, None))
rec("ring_notdiv", RR(3, 4, 64, 64, A, 64, BF, arr(A, A, A), None, BF, A, A, 64, BF, None))
rec("ring_M0", RR(2, 0, 64, 64, None, 64, BF, None, None, BF, None, None, 64, BF, None))
rec("ring_bad_wire", RR(2, 4, 64, 64, A, 64, BF, w2, None, 9, A, A, 64, BF, None))
# uneven split
W64 = lambda *v: ctypes.cast((ctypes.c_int64 * len(v))(*v), t._i64p)
US = L.tp_shard_weights_uneven
rec("uneven_shard_sum", US(2, W64(5, 3), BF, A, 9, 64, None, w2, None, None))
rec("uneven_shard_zero", US(2, W64(9, 0), BF, A, 9, 64, None, w2, None, None))
rec("uneven_shard_null_widths", US(2, None, BF, A, 9, 64, None, w2, None, None))
UC = L.column_parallel_linear_uneven
rec("uneven_col_swiglu", UC(2, W64(5, 4), 4, 64, A, 64, BF, w2, None, 2, A, 9, BF, None))
rec("uneven_col_ldy", UC(2, W64(5, 4), 4, 64, A, 64, BF, w2, None, 0, A, 8, BF, None))
rec("uneven_col_M0", UC(2, W64(5, 4), 0, 64, None, 64, BF, None, None, 0, None, 9, BF, None))
rec("uneven_col_width0", UC(2, W64(9, 0), 4, 64, A, 64, BF, w2, None, 0, A, 9, BF, None))
# FP8 weights
QZ = L.tp_quantize_fp8
rec("fp8_quant_rows0", QZ(0, 64, None, None, None, None))
rec("fp8_quant_null", QZ(4, 64, A, None, A, None))
rec("fp8_quant_cols0", QZ(4, 0, A, A, A, None))
CF = L.column_parallel_linear_fp8
rec("fp8_col_f32_x", CF(2, 4, 64, 64, A, 64, F32, w2, w2, None, 0, A, 64, F32, None))
rec("fp8_col_too_many_tokens", CF(2, 129, 64, 64, A, 64, BF, w2, w2, None, 0, A, 64, BF, None))
rec("fp8_col_null_scales", CF(2, 4, 64, 64, A, 64, BF, w2, None, None, 0, A, 64, BF, None))
rec("fp8_col_K_not16", CF(2, 4, 72, 64, A, 72, BF, w2, w2, None, 0, A, 64, BF, None))
rec("fp8_col_swiglu_bias", CF(2, 4, 64, 64, A, 64, BF, w2, w2, w2, 2, A, 64, BF, None))
RF = L.row_parallel_linear_fp8
rec("fp8_row_shardK_not16", RF(2, 4, 48, 64, A, 48, BF, w2, w2, None, A, 64, BF, None))
rec("fp8_row_notdiv", RF(3, 4, 64, 64, A, 64, BF, arr(A, A, A), arr(A, A, A), None, A, 64, BF, None))
rec("fp8_row_M0", RF(2, 0, 64, 64, None, 64, BF, None, None, None, None, 64, BF, None))
MF = L.tp_mlp_block_fp8
rec("fp8_mlp_null_h", MF(2, 4, 64, 128, 2, A, w2, w2, None, w2, w2, None, None, A, BF, None))
rec("fp8_mlp_too_many", MF(2, 129, 64, 128, 2, A, w2, w2, None, w2, w2, None, A, A, BF, None))
json.dump(res, sys.stdout)
'''

EXPECT = {
    "col_ok_M0": 0, "col_tp0": 3, "col_tp17": 3, "col_negM": 3, "col_K0": 3, "col_notdiv": 2,
    "col_dtype_f32_to_bf16": 4, "col_dtype_bad": 4, "col_act_bad": 3, "col_swiglu_bias": 8,
    "col_ldx_small": 3, "col_ldy_small": 3, "col_null_X": 1, "col_null_Y": 1,
    "col_null_warr": 1, "col_null_shard": 1, "col_null_bias_shard": 1, "col_misaligned_X": 5,
    "col_misaligned_ldx": 5, "col_misaligned_K": 5, "col_misaligned_w": 5,
    "col_misaligned_Y": 5, "row_notdiv": 2, "row_shard_K_misaligned": 5, "row_null_Y": 1,
    "row_misaligned_bias": 5, "row_M0": 0, "mlp_notdiv": 2, "mlp_null_h": 1,
    "mlp_swiglu_bias": 8, "mlp_misaligned_shardK": 5, "attn_heads_notdiv": 2,
    "attn_kv_notdiv": 2, "attn_hd0": 3, "attn_null_ctx": 1, "attn_qkv_dtype": 4,
    "shard_row_bias": 8, "shard_gateup_no_up": 1, "shard_bias_no_dst": 1, "shard_null_W": 1,
    "shard_notdiv": 2, "shard_row_cols_misaligned": 5, "shard_dtype": 4,
    "selftest_bad_limit": 3, "layer_null_args": 1, "layer_M0": 0, "layer_ffn_notdiv": 2,
    "layer_ffn_null_h": 1, "layer_attn_kv_notdiv": 2, "layer_feed_dtype": 4,
    "layer_swiglu_bias": 8, "ring_null_partials": 1, "ring_wire_bf16_from_f32": 4,
    "ring_notdiv": 2, "ring_M0": 0, "ring_bad_wire": 4, "uneven_shard_sum": 3,
    "uneven_shard_zero": 3, "uneven_shard_null_widths": 1, "uneven_col_swiglu": 8,
    "uneven_col_ldy": 3, "uneven_col_M0": 0, "uneven_col_width0": 3,
    "fp8_quant_rows0": 0, "fp8_quant_null": 1, "fp8_quant_cols0": 3, "fp8_col_f32_x": 4,
    "fp8_col_too_many_tokens": 8, "fp8_col_null_scales": 1, "fp8_col_K_not16": 5,
    "fp8_col_swiglu_bias": 8, "fp8_row_shardK_not16": 5, "fp8_row_notdiv": 2, "fp8_row_M0": 0,
    "fp8_mlp_null_h": 1, "fp8_mlp_too_many": 8,
}


def test_validation_error_paths():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=300)
    assert r.returncode == 0, r.stderr
    got = json.loads(r.stdout)
    bad = {k: (got.get(k), v) for k, v in EXPECT.items() if got.get(k) != v}
    assert not bad, bad
