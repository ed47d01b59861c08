"""Python binding of libtpla.so (include/tpla.h): argument marshalling only.

Every step of the path runs in the library's CUDA kernels.  PyTorch supplies
device memory and the current stream; this module turns tensors into
pointers, sizes and dtype codes, calls the C entry point of the same name,
and raises ``TplaError`` on any status other than TP_OK.  There is no CPU
fallback: if the compiled library is missing, importing this module fails.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtpla.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m tensor_column_linear_gelu_b300.build` "
        "(nvcc, sm_103a). There is no fallback path.")

lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------- constants
TP_OK = 0
TP_ERR_NULL, TP_ERR_NOT_DIVISIBLE, TP_ERR_BAD_SHAPE, TP_ERR_DTYPE = 1, 2, 3, 4
TP_ERR_ALIGNMENT, TP_ERR_CUDA, TP_ERR_DEVICE_TIMEOUT, TP_ERR_UNSUPPORTED = 5, 6, 7, 8
TP_F32, TP_BF16 = 0, 1
TP_ACT_NONE, TP_ACT_GELU_ERF, TP_ACT_SWIGLU = 0, 1, 2
TP_SPLIT_COLUMN, TP_SPLIT_ROW, TP_SPLIT_QKV_HEADS, TP_SPLIT_GATE_UP = 0, 1, 2, 3
TP_MAX_TP = 16
TP_GATE_UP_GROUP = 128
TP_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024

ACTS = {"none": TP_ACT_NONE, "gelu": TP_ACT_GELU_ERF, "swiglu": TP_ACT_SWIGLU}
SPLITS = {"column": TP_SPLIT_COLUMN, "row": TP_SPLIT_ROW, "qkv_heads": TP_SPLIT_QKV_HEADS,
          "gate_up": TP_SPLIT_GATE_UP}
_DT = {torch.float32: TP_F32, torch.bfloat16: TP_BF16}

# Every symbol include/tpla.h declares.
EXPORTS = ("tp_status_string", "tp_shard_shape", "tp_shard_weights", "column_parallel_linear",
           "row_parallel_linear", "tp_mlp_block", "tp_attn_proj", "tp_device_status",
           "tp_selftest_bounded_wait", "tp_mlp_block_noalloc")

# ----------------------------------------------------------------- prototypes
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int
_vpp = ctypes.POINTER(ctypes.c_void_p)
_i64p = ctypes.POINTER(ctypes.c_int64)

lib.tp_status_string.restype = ctypes.c_char_p
lib.tp_status_string.argtypes = [_int]
lib.tp_shard_shape.argtypes = [_int, _int, _i64, _i64, _int, _int, _int, _i64p, _i64p]
lib.tp_shard_weights.argtypes = [_int, _int, _int, _vp, _vp, _i64, _i64, _vp, _int, _int, _int,
                                 _vpp, _vpp, _vp]
lib.column_parallel_linear.argtypes = [_int, _i64, _i64, _i64, _vp, _i64, _int, _vpp, _vpp, _int,
                                       _vp, _i64, _int, _vp]
lib.row_parallel_linear.argtypes = [_int, _i64, _i64, _i64, _vp, _i64, _int, _vpp, _vp, _vp, _i64,
                                    _int, _vp]
lib.tp_mlp_block.argtypes = [_int, _i64, _i64, _i64, _int, _int, _vp, _vpp, _vpp, _vpp, _vp, _vp,
                             _vp, _int, _vp]
lib.tp_attn_proj.argtypes = [_int, _i64, _i64, _int, _int, _int, _int, _vp, _vpp, _vpp, _vp, _int,
                             _vp, _vpp, _vp, _vp, _int, _vp]
lib.tp_mlp_block_noalloc.argtypes = [_int, _i64, _i64, _i64, _int, _int, _vp, _vpp, _vpp, _vpp,
                                     _vp, _vp, _int, _vp]
lib.tp_device_status.argtypes = [_vp]
lib.tp_selftest_bounded_wait.argtypes = [_i64, _vp]
for _name in EXPORTS[1:]:
    getattr(lib, _name).restype = _int


class TplaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib.tp_status_string(status).decode()
        super().__init__(f"{where}: {msg}")


def _check(status: int, where: str):
    if status != TP_OK:
        raise TplaError(status, where)


def status_string(status: int) -> str:
    return lib.tp_status_string(status).decode()


# ----------------------------------------------------------------- marshalling
def ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def ptr_array(ts: Optional[Sequence[Optional[torch.Tensor]]]):
    """Host array of device pointers (NULL for a None list)."""
    if ts is None:
        return None
    arr = (ctypes.c_void_p * len(ts))(*[ptr(t) for t in ts])
    return ctypes.cast(arr, _vpp)


def dtype_code(dt: torch.dtype) -> int:
    if dt not in _DT:
        raise TplaError(TP_ERR_DTYPE, f"dtype {dt}")
    return _DT[dt]


def stream_handle(stream: Optional[torch.cuda.Stream]) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _act(act) -> int:
    return ACTS[act] if isinstance(act, str) else int(act)


def _split(split) -> int:
    return SPLITS[split] if isinstance(split, str) else int(split)


# ----------------------------------------------------------------- entry points
def tp_shard_shape(split, tp: int, out_f: int, in_f: int, n_heads: int = 0,
                   n_kv_heads: int = 0, head_dim: int = 0):
    rows, cols = ctypes.c_int64(), ctypes.c_int64()
    _check(lib.tp_shard_shape(_split(split), tp, out_f, in_f, n_heads, n_kv_heads, head_dim,
                              ctypes.byref(rows), ctypes.byref(cols)), "tp_shard_shape")
    return rows.value, cols.value


def tp_shard_weights(split, tp: int, W: torch.Tensor, W_up: Optional[torch.Tensor] = None,
                     b: Optional[torch.Tensor] = None, n_heads: int = 0, n_kv_heads: int = 0,
                     head_dim: int = 0, stream=None):
    """Shard W (and b) on W's device.  Returns (w_shards, b_shards or None)."""
    out_f, in_f = W.shape
    rows, cols = tp_shard_shape(split, tp, out_f, in_f, n_heads, n_kv_heads, head_dim)
    w_sh = [torch.empty(rows, cols, dtype=W.dtype, device=W.device) for _ in range(tp)]
    b_sh = None
    if b is not None:
        b_sh = [torch.empty(rows, dtype=torch.float32, device=W.device) for _ in range(tp)]
    wa, ba = ptr_array(w_sh), ptr_array(b_sh)
    _check(lib.tp_shard_weights(_split(split), tp, dtype_code(W.dtype), ptr(W), ptr(W_up), out_f,
                                in_f, ptr(b), n_heads, n_kv_heads, head_dim, wa, ba,
                                stream_handle(stream)), "tp_shard_weights")
    return w_sh, b_sh


def column_parallel_linear(tp: int, X: torch.Tensor, w_shards, b_shards=None, act="none",
                           out_dtype: Optional[torch.dtype] = None, Y: Optional[torch.Tensor] = None,
                           N: Optional[int] = None, stream=None) -> torch.Tensor:
    """Y_i = act(X . W_i^T + b_i) for all shards; Y's column block i is shard i."""
    M, K = X.shape
    if N is None:
        if _act(act) == TP_ACT_SWIGLU:
            raise ValueError("pass N (d_ff) for SwiGLU: packed shards are padded")
        N = w_shards[0].shape[0] * tp
    if Y is None:
        Y = torch.empty(M, N, dtype=out_dtype or X.dtype, device=X.device)
    _check(lib.column_parallel_linear(tp, M, K, N, ptr(X), X.stride(0), dtype_code(X.dtype),
                                      ptr_array(w_shards), ptr_array(b_shards), _act(act), ptr(Y),
                                      Y.stride(0), dtype_code(Y.dtype), stream_handle(stream)),
           "column_parallel_linear")
    return Y


def row_parallel_linear(tp: int, X: torch.Tensor, w_shards, b: Optional[torch.Tensor] = None,
                        out_dtype: Optional[torch.dtype] = None, Y: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """Y = sum_i X_i . W_i^T + b, X_i = columns [i*K/tp, (i+1)*K/tp) of X."""
    M, K = X.shape
    N = w_shards[0].shape[0]
    if Y is None:
        Y = torch.empty(M, N, dtype=out_dtype or X.dtype, device=X.device)
    _check(lib.row_parallel_linear(tp, M, K, N, ptr(X), X.stride(0), dtype_code(X.dtype),
                                   ptr_array(w_shards), ptr(b), ptr(Y), Y.stride(0),
                                   dtype_code(Y.dtype), stream_handle(stream)),
           "row_parallel_linear")
    return Y


def tp_mlp_block(tp: int, X: torch.Tensor, w1_shards, b1_shards, w2_shards,
                 b2: Optional[torch.Tensor], act="gelu", d_ff: Optional[int] = None,
                 out_dtype: Optional[torch.dtype] = None, h: Optional[torch.Tensor] = None,
                 Y: Optional[torch.Tensor] = None, stream=None):
    """FFN block: column (act per shard) -> h -> row (+ b2 once).  Returns (Y, h)."""
    M, d_model = X.shape
    if d_ff is None:
        d_ff = w2_shards[0].shape[1] * tp
    if h is None:
        h = torch.empty(M, d_ff, dtype=X.dtype, device=X.device)
    if Y is None:
        Y = torch.empty(M, d_model, dtype=out_dtype or X.dtype, device=X.device)
    _check(lib.tp_mlp_block(tp, M, d_model, d_ff, _act(act), dtype_code(X.dtype), ptr(X),
                            ptr_array(w1_shards), ptr_array(b1_shards), ptr_array(w2_shards),
                            ptr(b2), ptr(h), ptr(Y), dtype_code(Y.dtype), stream_handle(stream)),
           "tp_mlp_block")
    return Y, h


def tp_attn_proj(tp: int, X: torch.Tensor, wqkv_shards, bqkv_shards, ctx: torch.Tensor, wo_shards,
                 bo: Optional[torch.Tensor], n_heads: int, n_kv_heads: int, head_dim: int,
                 qkv_dtype: Optional[torch.dtype] = None, out_dtype: Optional[torch.dtype] = None,
                 qkv_out: Optional[torch.Tensor] = None, Y: Optional[torch.Tensor] = None,
                 stream=None):
    """QKV by head group and O by head.  Returns (qkv_out [tp, M, ws], Y [M, d_model])."""
    M, d_model = X.shape
    ws = (n_heads // tp + 2 * (n_kv_heads // tp)) * head_dim if tp > 0 else 0
    if qkv_out is None:
        qkv_out = torch.empty(tp, M, ws, dtype=qkv_dtype or X.dtype, device=X.device)
    if Y is None:
        Y = torch.empty(M, d_model, dtype=out_dtype or X.dtype, device=X.device)
    _check(lib.tp_attn_proj(tp, M, d_model, n_heads, n_kv_heads, head_dim, dtype_code(X.dtype),
                            ptr(X), ptr_array(wqkv_shards), ptr_array(bqkv_shards), ptr(qkv_out),
                            dtype_code(qkv_out.dtype), ptr(ctx), ptr_array(wo_shards), ptr(bo),
                            ptr(Y), dtype_code(Y.dtype), stream_handle(stream)),
           "tp_attn_proj")
    return qkv_out, Y


def tp_mlp_block_noalloc(tp: int, X: torch.Tensor, w1_shards, b1_shards, w2_shards,
                         b2: Optional[torch.Tensor], act="gelu", d_ff: Optional[int] = None,
                         out_dtype: Optional[torch.dtype] = None, Y: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """The FFN block with h kept in the library's built-in workspace, for callers
    that cannot allocate device memory (M * d_ff * element size must fit
    TP_NOALLOC_SCRATCH_BYTES).  Returns Y; Y must be preallocated by such callers."""
    M, d_model = X.shape
    if d_ff is None:
        d_ff = w2_shards[0].shape[1] * tp
    if Y is None:
        Y = torch.empty(M, d_model, dtype=out_dtype or X.dtype, device=X.device)
    _check(lib.tp_mlp_block_noalloc(tp, M, d_model, d_ff, _act(act), dtype_code(X.dtype), ptr(X),
                                    ptr_array(w1_shards), ptr_array(b1_shards),
                                    ptr_array(w2_shards), ptr(b2), ptr(Y), dtype_code(Y.dtype),
                                    stream_handle(stream)),
           "tp_mlp_block_noalloc")
    return Y


def tp_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device-side status code."""
    return lib.tp_device_status(stream_handle(stream))


def tp_selftest_bounded_wait(limit_ns: int, stream=None):
    _check(lib.tp_selftest_bounded_wait(int(limit_ns), stream_handle(stream)),
           "tp_selftest_bounded_wait")
