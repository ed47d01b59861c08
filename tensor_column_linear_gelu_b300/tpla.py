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
# TPLA_CHECKED=1 loads the checked build of the same library (index checks in
# the kernels, reported as TP_ERR_DEVICE_CHECK); it must have been built.
CHECKED = os.environ.get("TPLA_CHECKED") == "1"
LIB_PATH = os.path.join(_PKG, "libtpla_checked.so" if CHECKED else "libtpla.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m tensor_column_linear_gelu_b300.build"
        f"{' --checked' if CHECKED else ''}` (nvcc, sm_103a). There is no fallback path.")

lib = ctypes.CDLL(LIB_PATH)

# ----------------------------------------------------------------- constants
TP_OK = 0
TP_ERR_NULL, TP_ERR_NOT_DIVISIBLE, TP_ERR_BAD_SHAPE, TP_ERR_DTYPE = 1, 2, 3, 4
TP_ERR_ALIGNMENT, TP_ERR_CUDA, TP_ERR_DEVICE_TIMEOUT, TP_ERR_UNSUPPORTED = 5, 6, 7, 8
TP_ERR_DEVICE_CHECK = 9
TP_F32, TP_BF16 = 0, 1
TP_ACT_NONE, TP_ACT_GELU_ERF, TP_ACT_SWIGLU = 0, 1, 2
TP_SPLIT_COLUMN, TP_SPLIT_ROW, TP_SPLIT_QKV_HEADS, TP_SPLIT_GATE_UP = 0, 1, 2, 3
TP_MAX_TP = 16
TP_GATE_UP_GROUP = 128
TP_NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024
TP_FP8_MAX_TOKENS = 128

ACTS = {"none": TP_ACT_NONE, "gelu": TP_ACT_GELU_ERF, "swiglu": TP_ACT_SWIGLU}
SPLITS = {"column": TP_SPLIT_COLUMN, "row": TP_SPLIT_ROW, "qkv_heads": TP_SPLIT_QKV_HEADS,
          "gate_up": TP_SPLIT_GATE_UP}
_DT = {torch.float32: TP_F32, torch.bfloat16: TP_BF16}

# Every symbol include/tpla.h declares.
EXPORTS = ("tp_status_string", "tp_shard_shape", "tp_shard_weights", "column_parallel_linear",
           "row_parallel_linear", "row_parallel_linear_ring", "tp_shard_weights_uneven",
           "column_parallel_linear_uneven", "tp_quantize_fp8", "column_parallel_linear_fp8",
           "row_parallel_linear_fp8", "tp_mlp_block_fp8", "tp_mlp_block", "tp_attn_proj",
           "tp_layer_forward", "tp_device_status", "tp_selftest_bounded_wait",
           "tp_mlp_block_noalloc")

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
lib.row_parallel_linear_ring.argtypes = [_int, _i64, _i64, _i64, _vp, _i64, _int, _vpp, _vp,
                                         _int, _vp, _vp, _i64, _int, _vp]
lib.tp_shard_weights_uneven.argtypes = [_int, _i64p, _int, _vp, _i64, _i64, _vp, _vpp, _vpp, _vp]
lib.column_parallel_linear_uneven.argtypes = [_int, _i64p, _i64, _i64, _vp, _i64, _int, _vpp,
                                              _vpp, _int, _vp, _i64, _int, _vp]
lib.tp_quantize_fp8.argtypes = [_i64, _i64, _vp, _vp, _vp, _vp]
lib.column_parallel_linear_fp8.argtypes = [_int, _i64, _i64, _i64, _vp, _i64, _int, _vpp, _vpp,
                                           _vpp, _int, _vp, _i64, _int, _vp]
lib.row_parallel_linear_fp8.argtypes = [_int, _i64, _i64, _i64, _vp, _i64, _int, _vpp, _vpp, _vp,
                                        _vp, _i64, _int, _vp]
lib.tp_mlp_block_fp8.argtypes = [_int, _i64, _i64, _i64, _int, _vp, _vpp, _vpp, _vpp, _vpp, _vpp,
                                 _vp, _vp, _vp, _int, _vp]
lib.tp_mlp_block.argtypes = [_int, _i64, _i64, _i64, _int, _int, _vp, _vpp, _vpp, _vpp, _vp, _vp,
                             _vp, _int, _vp]
lib.tp_attn_proj.argtypes = [_int, _i64, _i64, _int, _int, _int, _int, _vp, _vpp, _vpp, _vp, _int,
                             _vp, _vpp, _vp, _vp, _int, _vp]
lib.tp_mlp_block_noalloc.argtypes = [_int, _i64, _i64, _i64, _int, _int, _vp, _vpp, _vpp, _vpp,
                                     _vp, _vp, _int, _vp]


class LayerArgs(ctypes.Structure):
    """tp_layer_args of include/tpla.h (same field order and C types)."""
    _fields_ = [("tp", _int), ("M", _i64), ("d_model", _i64), ("xdt", _int),
                ("n_heads", _int), ("n_kv_heads", _int), ("head_dim", _int),
                ("X", _vp), ("wqkv_shards", _vpp), ("bqkv_shards", _vpp), ("qkv_out", _vp),
                ("qkv_dt", _int), ("ctx", _vp), ("wo_shards", _vpp), ("bo", _vp),
                ("Y_attn", _vp), ("attn_ydt", _int),
                ("d_ff", _i64), ("ffn_act", _int), ("X_ffn", _vp), ("w1_shards", _vpp),
                ("b1_shards", _vpp), ("w2_shards", _vpp), ("b2", _vp), ("h", _vp),
                ("Y_ffn", _vp), ("ffn_ydt", _int)]


lib.tp_layer_forward.argtypes = [ctypes.POINTER(LayerArgs), _vp]
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


def row_parallel_linear_ring(tp: int, X: torch.Tensor, w_shards, b: Optional[torch.Tensor] = None,
                             wire_dtype: torch.dtype = torch.bfloat16,
                             out_dtype: Optional[torch.dtype] = None,
                             Y: Optional[torch.Tensor] = None,
                             partials: Optional[torch.Tensor] = None, stream=None):
    """Row-parallel linear whose shard sum follows a ring all-reduce: partials
    held in wire_dtype, chunk c summed from rank c around the ring, rounded to
    wire_dtype after every hop, + b once.  Returns (Y, partials [tp, M, N])."""
    M, K = X.shape
    N = w_shards[0].shape[0]
    if Y is None:
        Y = torch.empty(M, N, dtype=out_dtype or X.dtype, device=X.device)
    if partials is None:
        partials = torch.empty(tp, M, N, dtype=wire_dtype, device=X.device)
    _check(lib.row_parallel_linear_ring(tp, M, K, N, ptr(X), X.stride(0), dtype_code(X.dtype),
                                        ptr_array(w_shards), ptr(b), dtype_code(partials.dtype),
                                        ptr(partials), ptr(Y), Y.stride(0), dtype_code(Y.dtype),
                                        stream_handle(stream)),
           "row_parallel_linear_ring")
    return Y, partials


def _widths(widths):
    return (ctypes.c_int64 * len(widths))(*[int(w) for w in widths])


def tp_shard_weights_uneven(widths: Sequence[int], W: torch.Tensor,
                            b: Optional[torch.Tensor] = None, stream=None):
    """Column shards of explicit widths (rows of W).  Returns (w_shards, b_shards or None)."""
    tp = len(widths)
    out_f, in_f = W.shape
    w_sh = [torch.empty(int(w), in_f, dtype=W.dtype, device=W.device) for w in widths]
    b_sh = None if b is None else [torch.empty(int(w), dtype=torch.float32, device=W.device)
                                   for w in widths]
    _check(lib.tp_shard_weights_uneven(tp, _widths(widths), dtype_code(W.dtype), ptr(W), out_f,
                                       in_f, ptr(b), ptr_array(w_sh), ptr_array(b_sh),
                                       stream_handle(stream)),
           "tp_shard_weights_uneven")
    return w_sh, b_sh


def column_parallel_linear_uneven(widths: Sequence[int], X: torch.Tensor, w_shards,
                                  b_shards=None, act="none",
                                  out_dtype: Optional[torch.dtype] = None,
                                  Y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Column split with explicit widths; shard i writes its column block of Y."""
    M, K = X.shape
    N = int(sum(widths))
    if Y is None:
        Y = torch.empty(M, N, dtype=out_dtype or X.dtype, device=X.device)
    _check(lib.column_parallel_linear_uneven(len(widths), _widths(widths), M, K, ptr(X),
                                             X.stride(0), dtype_code(X.dtype),
                                             ptr_array(w_shards), ptr_array(b_shards), _act(act),
                                             ptr(Y), Y.stride(0), dtype_code(Y.dtype),
                                             stream_handle(stream)),
           "column_parallel_linear_uneven")
    return Y


def tp_quantize_fp8(W: torch.Tensor, stream=None):
    """Per-row e4m3 quantization of a bf16 [rows, cols] tensor: (codes uint8, scales fp32)."""
    rows, cols = W.shape
    Q = torch.empty(rows, cols, dtype=torch.uint8, device=W.device)
    S = torch.empty(rows, dtype=torch.float32, device=W.device)
    _check(lib.tp_quantize_fp8(rows, cols, ptr(W.contiguous()), ptr(Q), ptr(S),
                               stream_handle(stream)), "tp_quantize_fp8")
    return Q, S


def quantize_shards_fp8(w_shards, stream=None):
    """Quantize every shard of a tp_shard_weights result: (code shards, scale shards)."""
    qs = [tp_quantize_fp8(w, stream) for w in w_shards]
    return [q for q, _ in qs], [s for _, s in qs]


def column_parallel_linear_fp8(tp: int, X: torch.Tensor, q_shards, s_shards, b_shards=None,
                               act="none", out_dtype: Optional[torch.dtype] = None,
                               Y: Optional[torch.Tensor] = None, N: Optional[int] = None,
                               stream=None) -> torch.Tensor:
    """column_parallel_linear with FP8 weight shards (codes + row scales)."""
    M, K = X.shape
    if N is None:
        if _act(act) == TP_ACT_SWIGLU:
            raise ValueError("pass N (d_ff) for SwiGLU: packed shards are padded")
        N = q_shards[0].shape[0] * tp
    if Y is None:
        Y = torch.empty(M, N, dtype=out_dtype or X.dtype, device=X.device)
    _check(lib.column_parallel_linear_fp8(tp, M, K, N, ptr(X), X.stride(0), dtype_code(X.dtype),
                                          ptr_array(q_shards), ptr_array(s_shards),
                                          ptr_array(b_shards), _act(act), ptr(Y), Y.stride(0),
                                          dtype_code(Y.dtype), stream_handle(stream)),
           "column_parallel_linear_fp8")
    return Y


def row_parallel_linear_fp8(tp: int, X: torch.Tensor, q_shards, s_shards,
                            b: Optional[torch.Tensor] = None,
                            out_dtype: Optional[torch.dtype] = None,
                            Y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """row_parallel_linear with FP8 weight shards (codes + row scales)."""
    M, K = X.shape
    N = q_shards[0].shape[0]
    if Y is None:
        Y = torch.empty(M, N, dtype=out_dtype or X.dtype, device=X.device)
    _check(lib.row_parallel_linear_fp8(tp, M, K, N, ptr(X), X.stride(0), dtype_code(X.dtype),
                                       ptr_array(q_shards), ptr_array(s_shards), ptr(b), ptr(Y),
                                       Y.stride(0), dtype_code(Y.dtype), stream_handle(stream)),
           "row_parallel_linear_fp8")
    return Y


def tp_mlp_block_fp8(tp: int, X: torch.Tensor, q1_shards, s1_shards, b1_shards, q2_shards,
                     s2_shards, b2: Optional[torch.Tensor], act="swiglu",
                     d_ff: Optional[int] = None, out_dtype: Optional[torch.dtype] = None,
                     h: Optional[torch.Tensor] = None, Y: Optional[torch.Tensor] = None,
                     stream=None):
    """The FFN block with FP8 weights.  Returns (Y, h)."""
    M, d_model = X.shape
    if d_ff is None:
        d_ff = q2_shards[0].shape[1] * tp
    if h is None:
        h = torch.empty(M, d_ff, dtype=torch.bfloat16, device=X.device)
    if Y is None:
        Y = torch.empty(M, d_model, dtype=out_dtype or X.dtype, device=X.device)
    _check(lib.tp_mlp_block_fp8(tp, M, d_model, d_ff, _act(act), ptr(X), ptr_array(q1_shards),
                                ptr_array(s1_shards), ptr_array(b1_shards), ptr_array(q2_shards),
                                ptr_array(s2_shards), ptr(b2), ptr(h), ptr(Y),
                                dtype_code(Y.dtype), stream_handle(stream)),
           "tp_mlp_block_fp8")
    return Y, h


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


def tp_layer_forward(tp: int, X: torch.Tensor, wqkv_shards, bqkv_shards, ctx: torch.Tensor,
                     wo_shards, bo: Optional[torch.Tensor], n_heads: int, n_kv_heads: int,
                     head_dim: int, w1_shards, b1_shards, w2_shards, b2: Optional[torch.Tensor],
                     ffn_act="swiglu", d_ff: Optional[int] = None, X_ffn="attn",
                     qkv_out: Optional[torch.Tensor] = None, Y_attn: Optional[torch.Tensor] = None,
                     h: Optional[torch.Tensor] = None, Y_ffn: Optional[torch.Tensor] = None,
                     out_dtype: Optional[torch.dtype] = None, qkv_dtype: Optional[torch.dtype] = None,
                     stream=None):
    """One layer's linear algebra: QKV and O projections, then the FFN block.

    X_ffn is the FFN block's input; "attn" (the default) feeds it the attention
    block's output Y_attn, which is then kept in X's dtype.  Returns
    (qkv_out, Y_attn, h, Y_ffn)."""
    M, d_model = X.shape
    if d_ff is None:
        d_ff = w2_shards[0].shape[1] * tp
    ws = (n_heads // tp + 2 * (n_kv_heads // tp)) * head_dim if tp > 0 else 0
    if qkv_out is None:
        qkv_out = torch.empty(tp, M, ws, dtype=qkv_dtype or X.dtype, device=X.device)
    feed = isinstance(X_ffn, str) and X_ffn == "attn"
    if Y_attn is None:
        Y_attn = torch.empty(M, d_model, dtype=X.dtype if feed else (out_dtype or X.dtype),
                             device=X.device)
    if feed:
        X_ffn = Y_attn
    if h is None:
        h = torch.empty(M, d_ff, dtype=X.dtype, device=X.device)
    if Y_ffn is None:
        Y_ffn = torch.empty(M, d_model, dtype=out_dtype or X.dtype, device=X.device)
    keep = [ptr_array(wqkv_shards), ptr_array(bqkv_shards), ptr_array(wo_shards),
            ptr_array(w1_shards), ptr_array(b1_shards), ptr_array(w2_shards)]
    a = LayerArgs(tp, M, d_model, dtype_code(X.dtype), n_heads, n_kv_heads, head_dim,
                  ptr(X), keep[0], keep[1], ptr(qkv_out), dtype_code(qkv_out.dtype), ptr(ctx),
                  keep[2], ptr(bo), ptr(Y_attn), dtype_code(Y_attn.dtype),
                  d_ff, _act(ffn_act), ptr(X_ffn), keep[3], keep[4], keep[5], ptr(b2), ptr(h),
                  ptr(Y_ffn), dtype_code(Y_ffn.dtype))
    _check(lib.tp_layer_forward(ctypes.byref(a), stream_handle(stream)), "tp_layer_forward")
    return qkv_out, Y_attn, h, Y_ffn


class LayerGraph:
    """One tp_layer_forward call captured in a CUDA graph.

    The call runs once outside the capture (one-time set-up), then once under
    torch.cuda.graph; replay() re-runs the four launches with no host work
    between them.  Inputs are read from, and outputs written to, the tensors
    given at construction: copy new inputs into them before a replay."""

    def __init__(self, tp: int, **kw):
        self.tp, self.kw = tp, kw
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self.outputs = tp_layer_forward(tp, **kw, stream=side)
        torch.cuda.current_stream().wait_stream(side)
        qkv, ya, h, yf = self.outputs
        kw = dict(kw, qkv_out=qkv, Y_attn=ya, h=h, Y_ffn=yf)
        if isinstance(kw.get("X_ffn", "attn"), str):
            kw["X_ffn"] = "attn"
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            tp_layer_forward(tp, **kw)

    def replay(self):
        self.graph.replay()
        return self.outputs


def tp_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device-side status code."""
    return lib.tp_device_status(stream_handle(stream))


def tp_selftest_bounded_wait(limit_ns: int, stream=None):
    _check(lib.tp_selftest_bounded_wait(int(limit_ns), stream_handle(stream)),
           "tp_selftest_bounded_wait")
