"""fp64 CPU oracle for the tensor-parallel linear path (ctypes binding).

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never does, and this package imports nothing from it: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over output
elements).  This module only marshals numpy arrays: every input is passed as
float32 (bf16 and fp32 values widen to float32 exactly), every output comes
back as float64.

Sources, by page title and section:
  * "Understanding Tensor Parallelism for Multi-GPU LLM Serving" -- "How Tensor
    Parallelism Works Under the Hood"; the ColumnParallelLinear and
    RowParallelLinear modules of "Implementing Tensor Parallelism with Hugging
    Face Accelerate".
  * "What is tensor parallelism?" -- "How a layer is split", "Why it helps when
    serving".
  * "Tensor parallel serving" -- "Simulating the split, and proving it is
    correct", "Try it yourself", "Column-parallel and row-parallel layers,
    paired".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

ACT_NONE, ACT_GELU, ACT_SWIGLU = 0, 1, 2
_ACTS = {"none": ACT_NONE, "gelu": ACT_GELU, "swiglu": ACT_SWIGLU}

_ERRORS = {1: "null pointer", 2: "not divisible by tp", 3: "bad shape",
           8: "out of memory"}


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"oracle {what}: {_ERRORS.get(code, code)}")
        self.code = code


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (fp64, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


_f = ctypes.POINTER(ctypes.c_float)
_d = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def _bind(lib):
    for name in ("orc_gelu", "orc_silu", "orc_round_bf16", "orc_round_f32", "orc_round_e4m3"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_double
        fn.argtypes = [ctypes.c_double]
    lib.orc_num_threads.restype = ctypes.c_int
    lib.orc_linear.argtypes = [_i64, _i64, _i64, _f, _i64, _f, _i64, _f,
                               ctypes.c_int, _d, _i64]
    lib.orc_swiglu.argtypes = [_i64, _i64, _i64, _f, _i64, _f, _f, _i64, _d, _i64]
    lib.orc_column_parallel.argtypes = [ctypes.c_int, _i64, _i64, _i64, _f, _i64,
                                        _f, _f, _i64, _f, ctypes.c_int, _d, _i64]
    lib.orc_column_parallel_uneven.argtypes = [
        ctypes.c_int, ctypes.POINTER(_i64), _i64, _i64, _i64, _f, _i64, _f, _i64,
        _f, ctypes.c_int, _d, _i64]
    lib.orc_row_parallel.argtypes = [ctypes.c_int, _i64, _i64, _i64, _f, _i64, _f,
                                     _i64, _f, _d, _i64]
    lib.orc_row_parallel_ring.argtypes = [ctypes.c_int, _i64, _i64, _i64, _f, _i64, _f,
                                          _i64, _f, ctypes.c_int, _d, _i64]
    lib.orc_row_parallel_ring_rows.argtypes = [ctypes.c_int, _i64, ctypes.POINTER(_i64), _i64,
                                               _i64, _i64, _f, _i64, _f, _i64, _f, ctypes.c_int,
                                               _d, _i64]
    lib.orc_quantize_fp8_rows.argtypes = [_i64, _i64, _f, _i64, _f, _f]
    lib.orc_column_parallel_fp8.argtypes = [ctypes.c_int, _i64, _i64, _i64, _f, _i64, _f, _f,
                                            _i64, _f, _f, _f, ctypes.c_int, _d, _i64]
    lib.orc_row_parallel_fp8.argtypes = [ctypes.c_int, _i64, _i64, _i64, _f, _i64, _f, _i64, _f,
                                         _f, _d, _i64]
    lib.orc_mlp_block.argtypes = [ctypes.c_int, _i64, _i64, _i64, ctypes.c_int, _f,
                                  _f, _f, _f, _f, _f, ctypes.c_int, _d, _d]
    lib.orc_qkv_proj.argtypes = [ctypes.c_int, _i64, _i64, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, _f, _f, _f, _d]
    lib.orc_o_proj.argtypes = [ctypes.c_int, _i64, _i64, ctypes.c_int, ctypes.c_int,
                               _f, _f, _f, _d]
    for name in ("orc_linear", "orc_swiglu", "orc_column_parallel",
                 "orc_column_parallel_uneven", "orc_row_parallel", "orc_row_parallel_ring",
                 "orc_row_parallel_ring_rows",
                 "orc_quantize_fp8_rows", "orc_column_parallel_fp8", "orc_row_parallel_fp8",
                 "orc_mlp_block",
                 "orc_qkv_proj", "orc_o_proj"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


def _f32(a):
    """C-contiguous float32 copy/view of an input (None passes through)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        a = a.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32))


def _pf(a):
    return None if a is None else a.ctypes.data_as(_f)


def _pd(a):
    return None if a is None else a.ctypes.data_as(_d)


def _check(rc: int, what: str):
    if rc != 0:
        raise OracleError(rc, what)


def _act(act) -> int:
    return _ACTS[act] if isinstance(act, str) else int(act)


class Oracle:
    """The oracle's functions, bound to one compiled copy of oracle.c."""

    def __init__(self, libpath: str):
        self.libpath = libpath
        self._lib = _bind(ctypes.CDLL(libpath))

    # ------------------------------------------------------------ scalars
    def gelu(self, z: float) -> float:
        return self._lib.orc_gelu(float(z))

    def silu(self, z: float) -> float:
        return self._lib.orc_silu(float(z))

    def round_bf16(self, x: float) -> float:
        return self._lib.orc_round_bf16(float(x))

    def num_threads(self) -> int:
        return self._lib.orc_num_threads()

    # ------------------------------------------------------------ unsharded
    def linear(self, X, W, b=None, act="none"):
        """Unsharded y = act(X . W^T + b); act in {none, gelu}."""
        X, W, b = _f32(X), _f32(W), _f32(b)
        M, K = X.shape
        N = W.shape[0]
        assert W.shape[1] == K
        Y = np.empty((M, N), dtype=np.float64)
        _check(self._lib.orc_linear(M, K, N, _pf(X), K, _pf(W), K, _pf(b), _act(act),
                                    _pd(Y), N), "linear")
        return Y

    def swiglu(self, X, Wg, Wu):
        """Unsharded y = silu(X . Wg^T) * (X . Wu^T)."""
        X, Wg, Wu = _f32(X), _f32(Wg), _f32(Wu)
        M, K = X.shape
        N = Wg.shape[0]
        Y = np.empty((M, N), dtype=np.float64)
        _check(self._lib.orc_swiglu(M, K, N, _pf(X), K, _pf(Wg), _pf(Wu), K, _pd(Y), N),
               "swiglu")
        return Y

    # ------------------------------------------------------------ sharded
    def column_parallel(self, tp, X, W, b=None, act="none", Wu=None):
        """Literal column split: shard i = W rows [i*N/tp, (i+1)*N/tp); concat."""
        X, W, Wu, b = _f32(X), _f32(W), _f32(Wu), _f32(b)
        M, K = X.shape
        N = W.shape[0]
        Y = np.empty((M, N), dtype=np.float64)
        _check(self._lib.orc_column_parallel(tp, M, K, N, _pf(X), K, _pf(W), _pf(Wu),
                                             K, _pf(b), _act(act), _pd(Y), N),
               "column_parallel")
        return Y

    def column_parallel_uneven(self, widths, X, W, b=None, act="none"):
        """Column split with explicit per-shard output widths (e.g. 9 -> 5 + 4)."""
        X, W, b = _f32(X), _f32(W), _f32(b)
        M, K = X.shape
        N = W.shape[0]
        w = (_i64 * len(widths))(*widths)
        Y = np.empty((M, N), dtype=np.float64)
        _check(self._lib.orc_column_parallel_uneven(len(widths), w, M, K, N, _pf(X), K,
                                                    _pf(W), K, _pf(b), _act(act),
                                                    _pd(Y), N),
               "column_parallel_uneven")
        return Y

    def row_parallel(self, tp, X, W, b=None):
        """Literal row split: partial_i = X_i . W_i^T, summed in shard order, + b once."""
        X, W, b = _f32(X), _f32(W), _f32(b)
        M, K = X.shape
        N = W.shape[0]
        assert W.shape[1] == K
        Y = np.empty((M, N), dtype=np.float64)
        _check(self._lib.orc_row_parallel(tp, M, K, N, _pf(X), K, _pf(W), K, _pf(b),
                                          _pd(Y), N), "row_parallel")
        return Y

    def row_parallel_ring(self, tp, X, W, b=None, wire="bf16"):
        """Row split whose all-reduce adds the partials as a ring all-reduce does:
        partials held in the wire dtype, chunk c summed from rank c around the
        ring, rounded to the wire dtype after every hop, + b once (fp64 out)."""
        X, W, b = _f32(X), _f32(W), _f32(b)
        M, K = X.shape
        N = W.shape[0]
        assert W.shape[1] == K and wire in ("bf16", "f32")
        Y = np.empty((M, N), dtype=np.float64)
        _check(self._lib.orc_row_parallel_ring(tp, M, K, N, _pf(X), K, _pf(W), K, _pf(b),
                                               1 if wire == "bf16" else 0, _pd(Y), N),
               "row_parallel_ring")
        return Y

    def row_parallel_ring_rows(self, tp, M_total, rows, X, W, b=None, wire="bf16"):
        """row_parallel_ring on some rows of a call of M_total rows: X holds the
        sampled input rows, rows[r] their row numbers in the full call; the
        chunks of the ring are those of the full [M_total, N] message."""
        X, W, b = _f32(X), _f32(W), _f32(b)
        n, K = X.shape
        N = W.shape[0]
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        assert W.shape[1] == K and r.shape == (n,) and wire in ("bf16", "f32")
        Y = np.empty((n, N), dtype=np.float64)
        _check(self._lib.orc_row_parallel_ring_rows(tp, M_total, r.ctypes.data_as(ctypes.POINTER(_i64)),
                                                    n, K, N, _pf(X), K, _pf(W), K, _pf(b),
                                                    1 if wire == "bf16" else 0, _pd(Y), N),
               "row_parallel_ring_rows")
        return Y

    # ------------------------------------------------------------ FP8 weights
    def round_e4m3(self, x: float) -> float:
        return self._lib.orc_round_e4m3(float(x))

    def quantize_rows_fp8(self, W):
        """Per-row e4m3 quantization: (Q as float32 e4m3 values, S fp32 row scales)."""
        W = _f32(W)
        R, C = W.shape
        Q = np.empty((R, C), dtype=np.float32)
        S = np.empty((R,), dtype=np.float32)
        _check(self._lib.orc_quantize_fp8_rows(R, C, _pf(W), C, _pf(Q), _pf(S)), "quantize_fp8")
        return Q, S

    def column_parallel_fp8(self, tp, X, Q, S, b=None, act="none", Qu=None, Su=None):
        """Column split with FP8 weights: act(S[n] * (x . Q[n]) + b[n]) (SwiGLU: gate/up)."""
        X, Q, Qu, S, Su, b = (_f32(a) for a in (X, Q, Qu, S, Su, b))
        M, K = X.shape
        N = Q.shape[0]
        Y = np.empty((M, N), dtype=np.float64)
        _check(self._lib.orc_column_parallel_fp8(tp, M, K, N, _pf(X), K, _pf(Q), _pf(Qu), K,
                                                 _pf(S), _pf(Su), _pf(b), _act(act), _pd(Y), N),
               "column_parallel_fp8")
        return Y

    def row_parallel_fp8(self, tp, X, Q, S, b=None):
        """Row split with FP8 weights: sum_i S_i[n] * (x_i . Q_i[n]) + b; S is [tp, N]."""
        X, Q, S, b = (_f32(a) for a in (X, Q, S, b))
        M, K = X.shape
        N = Q.shape[0]
        Y = np.empty((M, N), dtype=np.float64)
        _check(self._lib.orc_row_parallel_fp8(tp, M, K, N, _pf(X), K, _pf(Q), K, _pf(S),
                                              _pf(b), _pd(Y), N), "row_parallel_fp8")
        return Y

    def quantize_row_shards_fp8(self, tp, W):
        """Quantize each row-split shard [N, K/tp] of W on its own: (Q [N, K], S [tp, N])."""
        W = _f32(W)
        N, K = W.shape
        ks = K // tp
        Qs = np.empty((tp, N, ks), dtype=np.float32)
        S = np.empty((tp, N), dtype=np.float32)
        for i in range(tp):
            # shard i: columns [i*ks, (i+1)*ks) of every row, read in place (row stride K)
            Wi = W[:, i * ks:].ctypes.data_as(_f)
            _check(self._lib.orc_quantize_fp8_rows(N, ks, Wi, K, _pf(Qs[i]), _pf(S[i])),
                   "quantize_fp8")
        return np.ascontiguousarray(Qs.transpose(1, 0, 2).reshape(N, K)), S

    def round_f32(self, x: float) -> float:
        return self._lib.orc_round_f32(float(x))

    def mlp_block(self, tp, X, W1, b1, W2, b2, act="gelu", W1u=None, round_h=True):
        """FFN block: column (act per shard) -> [bf16 h] -> row (+ b2 once).

        Returns (Y, h), both float64.  For act='swiglu', W1 is the gate weight
        and W1u the up weight (b1 is ignored: the SwiGLU layers carry no bias).
        """
        X, W1, W1u, b1, W2, b2 = (_f32(a) for a in (X, W1, W1u, b1, W2, b2))
        M, d = X.shape
        dff = W1.shape[0]
        Y = np.empty((M, d), dtype=np.float64)
        h = np.empty((M, dff), dtype=np.float64)
        _check(self._lib.orc_mlp_block(tp, M, d, dff, _act(act), _pf(X), _pf(W1),
                                       _pf(W1u), _pf(b1), _pf(W2), _pf(b2),
                                       1 if round_h else 0, _pd(h), _pd(Y)),
               "mlp_block")
        return Y, h

    def qkv_proj(self, tp, X, Wqkv, bqkv, n_heads, n_kv_heads, head_dim):
        """QKV column-split by head group; returns [tp, M, (H+2Hkv)/tp*hd]."""
        X, Wqkv, bqkv = _f32(X), _f32(Wqkv), _f32(bqkv)
        M, d = X.shape
        if tp < 1 or n_heads % tp or n_kv_heads % tp:
            ws = 0
        else:
            ws = (n_heads // tp + 2 * (n_kv_heads // tp)) * head_dim
        out = np.empty((max(tp, 1), M, ws), dtype=np.float64)
        _check(self._lib.orc_qkv_proj(tp, M, d, n_heads, n_kv_heads, head_dim, _pf(X),
                                      _pf(Wqkv), _pf(bqkv), _pd(out)), "qkv_proj")
        return out

    def o_proj(self, tp, ctx, Wo, bo, n_heads, head_dim):
        """O projection row-split by head: sum_i ctx_i . Wo_i^T + bo."""
        ctx, Wo, bo = _f32(ctx), _f32(Wo), _f32(bo)
        M = ctx.shape[0]
        d = Wo.shape[0]
        Y = np.empty((M, d), dtype=np.float64)
        _check(self._lib.orc_o_proj(tp, M, d, n_heads, head_dim, _pf(ctx), _pf(Wo),
                                    _pf(bo), _pd(Y)), "o_proj")
        return Y


_default = None
_lock = threading.Lock()


def default() -> Oracle:
    """The oracle built from this directory's oracle.c."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def __getattr__(name):
    # module-level access (oracle.linear, oracle.gelu, ...) goes to default()
    if name in Oracle.__dict__ and not name.startswith("_"):
        return getattr(default(), name)
    raise AttributeError(name)
