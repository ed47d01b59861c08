"""Pins for the fp64 oracle: checks against facts that do not come from it.

Each ``check_*`` takes an oracle instance and raises AssertionError on a
mismatch.  They pin the oracle to
  * the values printed in "Tensor parallel serving" ("Simulating the split,
    and proving it is correct"), stored in tests/golden/;
  * closed forms (the normal CDF at +-1, the logistic function at 1, bf16
    rounding of exactly representable ties);
  * library routines that the oracle does not use (scipy's ndtr / expit,
    numpy's float64 matmul, torch's fp32->bf16 conversion);
  * brute force with exact integer arithmetic on tiny inputs;
  * the divisibility rules of "Understanding Tensor Parallelism for Multi-GPU
    LLM Serving" (ColumnParallelLinear / RowParallelLinear asserts) and
    "What is tensor parallelism?" ("Why it helps when serving": tp divides the
    head count).
tests/test_oracle_mutants.py plants mistakes in copies of the oracle and
checks that these pins catch every one.
"""
from __future__ import annotations

import math
import os

import numpy as np
import scipy.special
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _int_mat(rng, shape, lo=-3, hi=3):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float32)


def _brute_linear(X, W, b=None):
    """Exact integer triple loop (Python ints) for integer-valued inputs."""
    M, K = X.shape
    N = W.shape[0]
    Xi = [[int(v) for v in row] for row in X]
    Wi = [[int(v) for v in row] for row in W]
    out = [[0] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            s = 0
            for k in range(K):
                s += Xi[m][k] * Wi[n][k]
            if b is not None:
                s += int(b[n])
            out[m][n] = s
    return np.array(out, dtype=np.float64)


def _rel_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(float(np.sqrt(np.mean(b * b))), 1e-300)
    return float(np.max(np.abs(a - b))) / scale


# ------------------------------------------------------------------ golden

def read_golden():
    vals, held = {}, []
    with open(os.path.join(GOLDEN, "worked_example_column_tp2.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key == "held":
                held.append((int(rest[0]), int(rest[1])))
            else:
                vals[key] = np.array([float(v) for v in rest])
    return vals, held


def worked_example_inputs():
    g = torch.Generator(device="cpu")
    g.manual_seed(0)
    x = torch.randn(1, 8, generator=g)
    W = torch.randn(6, 8, generator=g)
    b = torch.randn(6, generator=g)
    return x.numpy(), W.numpy(), b.numpy()


def check_worked_example(orc):
    """The page's printed full and combined outputs, to 4 decimals."""
    vals, held = read_golden()
    x, W, b = worked_example_inputs()
    full = orc.linear(x, W, b)
    combined = orc.column_parallel(2, x, W, b)
    assert np.array_equal(np.round(full[0], 4), vals["full"]), (full, vals["full"])
    assert np.array_equal(np.round(combined[0], 4), vals["combined"]), combined
    # each of the 2 shards holds N/tp * K of the N * K weights
    ns = W.shape[0] // 2
    for (h, tot) in held:
        assert (ns * W.shape[1], W.size) == (h, tot)


# ------------------------------------------------------------------ scalars

def check_gelu_closed_form(orc):
    """GELU(z) = z * Phi(z): Phi(1) = 0.841344746068543, Phi(-1) = 1 - Phi(1)."""
    assert orc.gelu(0.0) == 0.0
    assert abs(orc.gelu(1.0) - 0.8413447460685429) < 1e-15
    assert abs(orc.gelu(-1.0) - (-0.15865525393145707)) < 1e-15
    assert orc.gelu(10.0) == 10.0                  # Phi(10) rounds to 1
    assert abs(orc.gelu(-10.0)) < 1e-20            # Phi(-10) ~ 7.6e-24
    for z in np.linspace(-8, 8, 97):
        ref = z * scipy.special.ndtr(z)            # independent library routine
        assert abs(orc.gelu(z) - ref) <= 1e-15 * max(1.0, abs(ref)), z


def check_silu_closed_form(orc):
    """silu(z) = z * logistic(z): silu(1) = 1 / (1 + e^-1)."""
    assert orc.silu(0.0) == 0.0
    assert abs(orc.silu(1.0) - 0.7310585786300049) < 1e-15
    for z in np.linspace(-30, 30, 121):
        ref = z * scipy.special.expit(z)
        assert abs(orc.silu(z) - ref) <= 1e-15 * max(1.0, abs(ref)), z


def check_round_bf16(orc):
    """Round-to-nearest-even at bf16 precision (8 significant bits)."""
    e = 2.0 ** -8
    cases = [
        (1.0 + e, 1.0),                    # tie, even neighbour is 1
        (1.0 + 3 * e, 1.0 + 4 * e),        # tie, even neighbour is 1 + 2^-6
        (-(1.0 + e), -1.0),
        (1.0 + 1.5 * e, 1.0 + 2 * e),      # above the tie
        (3.0, 3.0),
        ((2 - 2 ** -7) * 2.0 ** 127, (2 - 2 ** -7) * 2.0 ** 127),   # largest finite
        ((2 - 2 ** -8) * 2.0 ** 127, math.inf),                    # tie -> 2^128 -> inf
        (2.0 ** -133, 2.0 ** -133),        # smallest subnormal
        (1.5 * 2.0 ** -133, 2.0 ** -132),  # subnormal tie -> even
        (0.5 * 2.0 ** -133, 0.0),          # subnormal tie -> 0
        (0.0, 0.0),
    ]
    for x, want in cases:
        got = orc.round_bf16(x)
        assert got == want, (x, got, want)
    # agreement with torch's fp32 -> bf16 conversion on fp32 values
    v = _rng(3).standard_normal(20000).astype(np.float32) * np.float32(37.0)
    want = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.round_bf16(float(a)) for a in v])
    assert np.array_equal(got, want)


# ------------------------------------------------------------------ linear

def check_brute_force_integers(orc):
    """Integer inputs make fp64 exact: compare with a Python-int triple loop."""
    rng = _rng(11)
    M, K, N = 3, 12, 12
    X = _int_mat(rng, (M, K))
    W = _int_mat(rng, (N, K))
    b = _int_mat(rng, (N,))
    ref = _brute_linear(X, W, b)
    ref_nb = _brute_linear(X, W)
    assert np.array_equal(orc.linear(X, W, b), ref)
    for tp in (1, 2, 3, 4):
        assert np.array_equal(orc.column_parallel(tp, X, W, b), ref), tp
        assert np.array_equal(orc.row_parallel(tp, X, W, b), ref), tp
        assert np.array_equal(orc.row_parallel(tp, X, W), ref_nb), tp
    # a non-square case catches transposed operands
    X2 = _int_mat(rng, (2, 6))
    W2 = _int_mat(rng, (5, 6))
    assert np.array_equal(orc.linear(X2, W2), _brute_linear(X2, W2))
    assert np.array_equal(orc.row_parallel(3, X2, W2), _brute_linear(X2, W2))


def check_numpy_fp64(orc):
    """Against numpy's float64 matmul (a library routine the oracle never calls)."""
    rng = _rng(5)
    M, K, N = 7, 40, 24
    X = rng.standard_normal((M, K)).astype(np.float32)
    W = rng.standard_normal((N, K)).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    z = X.astype(np.float64) @ W.astype(np.float64).T + b.astype(np.float64)
    assert _rel_err(orc.linear(X, W, b), z) < 1e-13
    assert _rel_err(orc.linear(X, W, b, "gelu"), z * scipy.special.ndtr(z)) < 1e-13
    for tp in (2, 4, 8):
        assert _rel_err(orc.column_parallel(tp, X, W, b, "gelu"),
                        z * scipy.special.ndtr(z)) < 1e-13
        assert _rel_err(orc.row_parallel(tp, X[:, :40], W[:, :40], b), z) < 1e-13
    Wu = rng.standard_normal((N, K)).astype(np.float32)
    g = X.astype(np.float64) @ W.astype(np.float64).T
    u = X.astype(np.float64) @ Wu.astype(np.float64).T
    sw = g * scipy.special.expit(g) * u
    assert _rel_err(orc.swiglu(X, W, Wu), sw) < 1e-13
    for tp in (1, 2, 3):
        assert _rel_err(orc.column_parallel(tp, X, W, None, "swiglu", Wu), sw) < 1e-13


def check_shard_invariants(orc):
    """Concat of column shards == unsharded; sum of row partials + b == full."""
    rng = _rng(7)
    M, K, N = 5, 48, 36
    X = rng.standard_normal((M, K)).astype(np.float32)
    W = rng.standard_normal((N, K)).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    full = orc.linear(X, W, b, "gelu")
    for tp in (1, 2, 3, 4, 6):
        # same dot product per element, in the same order: bit-identical
        assert np.array_equal(orc.column_parallel(tp, X, W, b, "gelu"), full), tp
    full_lin = orc.linear(X, W, b)
    for tp in (1, 2, 3, 4, 6, 8):
        assert _rel_err(orc.row_parallel(tp, X, W, b), full_lin) < 1e-13, tp


def check_identity_weight(orc):
    """W = I gives y = x + b exactly."""
    rng = _rng(9)
    K = 16
    X = rng.standard_normal((4, K)).astype(np.float32)
    b = rng.standard_normal(K).astype(np.float32)
    I = np.eye(K, dtype=np.float32)
    want = X.astype(np.float64) + b.astype(np.float64)
    assert np.array_equal(orc.linear(X, I, b), want)
    assert np.array_equal(orc.column_parallel(4, X, I, b), want)
    assert np.array_equal(orc.row_parallel(4, X, I, b), want)


def check_uneven_split(orc):
    """9 outputs split 5 + 4 still concatenate to the unsharded result."""
    rng = _rng(13)
    X = rng.standard_normal((2, 8)).astype(np.float32)
    W = rng.standard_normal((9, 8)).astype(np.float32)
    b = rng.standard_normal(9).astype(np.float32)
    full = orc.linear(X, W, b)
    assert np.array_equal(orc.column_parallel_uneven([5, 4], X, W, b), full)
    Xi = _int_mat(rng, (2, 8))
    Wi = _int_mat(rng, (9, 8))
    bi = _int_mat(rng, (9,))
    assert np.array_equal(orc.column_parallel_uneven([5, 4], Xi, Wi, bi),
                          _brute_linear(Xi, Wi, bi))


def check_ring_allreduce(orc):
    """The ring-ordered all-reduce ("Tensor parallel serving", "Communication
    cost"): values worked out by hand from the algorithm, not from the oracle.

    Case A: tp=3, M=1, K=3, N=5, x = [1,1,1], every W row = [256, 1, 1], so the
    partials are P0 = 256, P1 = P2 = 1 at every element.  L = 5 splits into
    chunks [0,1), [1,3), [3,5).  In bf16, 256..512 are spaced by 2 and a tie
    rounds to the even significand (256, 260):
      chunk 0 starts at rank 0: 256+1=257 -> 256, +1 -> 256;
      chunk 1 starts at rank 1: 1+1=2, +256=258;
      chunk 2 starts at rank 2: 1+256=257 -> 256, +1 -> 256.
    So y = [256, 258, 258, 256, 256]; an fp32 wire is exact: 258 everywhere.
    Case B: tp=4, M=2, K=4, N=3, x rows [1,1,1,1], W rows [256,1,1,1]; P0 =
    256, P1..P3 = 1.  L = 6 splits into [0,1), [1,3), [3,4), [4,6):
      chunk 0: 256 +1 +1 +1, each 257 -> 256: 256;
      chunk 1: 1+1=2, +1=3, +256=259 -> 260 (tie between 258 and 260);
      chunk 2: 1+1=2, +256=258, +1=259 -> 260;
      chunk 3: 1+256=257 -> 256, +1 -> 256, +1 -> 256.
    Flattened [256, 260, 260, 260, 256, 256] -> [[256,260,260],[260,256,256]].
    The bias is added once after the all-reduce.  Case C (below) checks that
    the partials themselves are held in the wire dtype.
    """
    X = np.ones((1, 3), np.float32)
    W = np.tile(np.array([[256, 1, 1]], np.float32), (5, 1))
    y = orc.row_parallel_ring(3, X, W, None, "bf16")
    assert np.array_equal(y, [[256, 258, 258, 256, 256]]), y
    assert np.array_equal(orc.row_parallel_ring(3, X, W, None, "f32"), np.full((1, 5), 258.0))
    b = np.array([0.5, -1, 2, 0, 3], np.float32)
    assert np.array_equal(orc.row_parallel_ring(3, X, W, b, "bf16"),
                          [[256.5, 257, 260, 256, 259]])
    X = np.ones((2, 4), np.float32)
    W = np.tile(np.array([[256, 1, 1, 1]], np.float32), (3, 1))
    y = orc.row_parallel_ring(4, X, W, None, "bf16")
    assert np.array_equal(y, [[256, 260, 260], [260, 256, 256]]), y
    # Case C: a partial that bf16 cannot hold.  tp=2, x = [1,1], W rows
    # [257, 1]: P0 = 257 is held as 256 (a tie, to the even significand),
    # P1 = 1.  Both chunks: 256 + 1 = 257 -> 256.  (Unrounded partials would
    # give 258.)
    y = orc.row_parallel_ring(2, np.ones((1, 2), np.float32),
                              np.tile(np.array([[257, 1]], np.float32), (2, 1)), None, "bf16")
    assert np.array_equal(y, [[256, 256]]), y
    # small integers: every partial and running sum is exact in bf16, so the
    # ring equals the plain sum; checked against exact integer brute force
    rng = _rng(77)
    for tp in (1, 2, 3, 4):
        X = _int_mat(rng, (3, 4 * tp), -2, 2)
        W = _int_mat(rng, (5, 4 * tp), -2, 2)
        b = _int_mat(rng, (5,), -3, 3)
        assert np.array_equal(orc.row_parallel_ring(tp, X, W, b, "bf16"), _brute_linear(X, W, b))
    # Case D, fp32 wire, worked by hand: tp=3, M=1, K=3, N=3, x = [1,1,1], W
    # rows [2^24, 1, 1]: P0 = 2^24, P1 = P2 = 1; L = 3, chunk c = element c.
    # fp32 holds integers exactly up to 2^24 and is spaced by 2 in
    # [2^24, 2^25); 2^24 + 1 is a tie that rounds to the even significand,
    # 2^24:
    #   chunk 0 starts at rank 0: 2^24 + 1 -> 2^24, + 1 -> 2^24;
    #   chunk 1 starts at rank 1: 1 + 1 = 2, + 2^24 = 2^24 + 2 (exact);
    #   chunk 2 starts at rank 2: 1 + 2^24 -> 2^24, + 1 -> 2^24.
    # Without the rounding after each hop every element would be 2^24 + 2.
    t24 = 2.0 ** 24
    X = np.ones((1, 3), np.float32)
    W = np.tile(np.array([[t24, 1, 1]], np.float32), (3, 1))
    y = orc.row_parallel_ring(3, X, W, None, "f32")
    assert np.array_equal(y, [[t24, t24 + 2, t24]]), y
    # Case E, fp32 wire, a partial fp32 cannot hold: tp=2, x = [1,1,1,1], W
    # row [2^24, 1, 1, 1].  P0 = 2^24 + 1 is held as 2^24 (the tie, to even),
    # P1 = 2.  Both chunks: 2^24 + 2 (exact).  Unrounded partials would give
    # 2^24 + 3, a tie that rounds to 2^24 + 4.
    X = np.ones((1, 4), np.float32)
    W = np.tile(np.array([[t24, 1, 1, 1]], np.float32), (2, 1))
    y = orc.row_parallel_ring(2, X, W, None, "f32")
    assert np.array_equal(y, [[t24 + 2, t24 + 2]]), y
    # The sampled-rows form keeps the full call's chunks.  Case A with M=2:
    # L = 10 splits into [0,3), [3,6), [6,10).  Row 1 is elements 5..9:
    # element 5 lies in chunk 1 (starts at rank 1: 1+1=2, +256 = 258),
    # elements 6..9 in chunk 2 (starts at rank 2: 1+256=257 -> 256, +1 -> 256).
    X = np.ones((1, 3), np.float32)
    W = np.tile(np.array([[256, 1, 1]], np.float32), (5, 1))
    y = orc.row_parallel_ring_rows(3, 2, [1], X, W, None, "bf16")
    assert np.array_equal(y, [[258, 256, 256, 256, 256]]), y
    # and every sampled row equals that row of the full call
    Xf = rng.standard_normal((9, 48)).astype(np.float32) * 40
    Wf = rng.standard_normal((7, 48)).astype(np.float32)
    bf = rng.standard_normal(7).astype(np.float32)
    for tp, wire in ((3, "bf16"), (4, "f32"), (2, "bf16")):
        full = orc.row_parallel_ring(tp, Xf, Wf, bf, wire)
        rows = [0, 3, 4, 8]
        assert np.array_equal(orc.row_parallel_ring_rows(tp, 9, rows, Xf[rows], Wf, bf, wire),
                              full[rows])
    # fp32 wire: within a few fp32 roundings of the exact sum
    X = rng.standard_normal((4, 96)).astype(np.float32)
    W = rng.standard_normal((7, 96)).astype(np.float32)
    exact = X.astype(np.float64) @ W.astype(np.float64).T
    y = orc.row_parallel_ring(3, X, W, None, "f32")
    assert np.max(np.abs(y - exact)) <= 6 * 2.0 ** -24 * np.max(np.abs(exact)) * 3
    import oracle
    try:
        orc.row_parallel_ring(3, np.ones((1, 4), np.float32), np.ones((2, 4), np.float32))
    except oracle.OracleError as e:
        assert e.code == 2  # tp must divide in_features
    else:
        raise AssertionError("row_parallel_ring accepted tp=3 with K=4")


def check_fp8_weights(orc):
    """FP8 (e4m3) weights with per-row scales: rounding against torch's
    float8_e4m3fn conversion and hand-worked ties, the quantizer against its
    invariants, the FP8 column and row splits against numpy fp64 matmuls."""
    # e4m3: 4 significant bits, spacing 1/8 in [1,2) and 2 in [16,32),
    # subnormal quantum 2^-9, saturation at 448; ties to even
    for x, want in [(448.0, 448.0), (449.0, 448.0), (1e6, 448.0), (1.0625, 1.0), (1.1875, 1.25),
                    (17.0, 16.0), (19.0, 20.0), (2.0 ** -10, 0.0), (3 * 2.0 ** -10, 2.0 ** -8),
                    (-0.3, -0.3125), (0.0625, 0.0625)]:
        assert orc.round_e4m3(x) == want, (x, orc.round_e4m3(x), want)
    v = (torch.from_numpy(_rng(5).standard_normal(20000).astype(np.float32)) * 60).clamp(-448, 448)
    ref = v.to(torch.float8_e4m3fn).double().numpy()
    mine = np.array([orc.round_e4m3(float(x)) for x in v.double().numpy()])
    assert np.array_equal(mine, ref)
    # quantizer invariants
    rng = _rng(8)
    W = (rng.standard_normal((6, 40)) * rng.uniform(0.01, 3, (6, 1))).astype(np.float32)
    W[3] = 0.0
    Q, S = orc.quantize_rows_fp8(W)
    assert S[3] == 1.0 and not np.any(Q[3])
    for r in (0, 1, 2, 4, 5):
        assert np.max(np.abs(Q[r])) == 448.0             # the row maximum maps to 448
        err = np.abs(S[r].astype(np.float64) * Q[r] - W[r])
        assert np.all(err <= S[r] * (np.abs(Q[r]) * 2.0 ** -4 + 2.0 ** -10) * 1.0001)
    assert all(orc.round_e4m3(float(q)) == q for q in Q.ravel()[:200])
    Q2, S2 = orc.quantize_rows_fp8(2 * W)                # a power of 2 scales exactly
    assert np.array_equal(Q2, Q) and np.array_equal(S2[[0, 1, 2, 4, 5]], 2 * S[[0, 1, 2, 4, 5]])
    # the scale is the correctly rounded fp32 quotient amax / 448, bit for bit
    # (numpy's float32 division is IEEE), on rows of many magnitudes
    Wm = (rng.standard_normal((64, 33)) * np.exp(rng.uniform(-12, 12, (64, 1)))).astype(np.float32)
    _, Sm = orc.quantize_rows_fp8(Wm)
    want = np.abs(Wm).max(axis=1).astype(np.float32) / np.float32(448.0)
    assert want.dtype == np.float32
    assert np.array_equal(Sm.view(np.uint32), want.view(np.uint32))
    # The code is decided by the fp32 quotient W / s.  A hand-built row whose
    # fp32 quotient lands exactly on an e4m3 tie while the exact quotient lies
    # just above it: amax = 1 + 2^-20, s = fl32(amax / 448) = 0x1.24925cp-9,
    # w = 0x1.36db82p-9.  w / s = 1.0625 + 1.3e-8 exactly; the nearest fp32 is
    # 1.0625, the tie between the e4m3 values 1 (significand 1.000) and 1.125
    # (1.001), which rounds to the even one, 1.  The exact quotient would give
    # 1.125.
    amax, w = np.float32(1 + 2.0 ** -20), np.float32(float.fromhex("0x1.36db82p-9"))
    s32 = amax / np.float32(448.0)
    assert float(s32) == float.fromhex("0x1.24925cp-9")
    assert float(w / s32) == 1.0625 and float(w) / float(s32) > 1.0625   # the fixture itself
    Qt, St = orc.quantize_rows_fp8(np.array([[amax, w, -w]], np.float32))
    assert St[0] == s32
    assert Qt[0, 1] == 1.0 and Qt[0, 2] == -1.0, Qt
    # FP8 column split (none / GELU / SwiGLU) against numpy on the dequantized weight
    X = rng.standard_normal((3, 40)).astype(np.float32)
    b = rng.standard_normal(6).astype(np.float32)
    Wd = S.astype(np.float64)[:, None] * Q
    lin = X.astype(np.float64) @ Wd.T
    for tp in (1, 2, 3):
        assert _rel_err(orc.column_parallel_fp8(tp, X, Q, S, b), lin + b) < 1e-13
        g = orc.column_parallel_fp8(tp, X, Q, S, b, "gelu")
        z = lin + b
        assert _rel_err(g, z * scipy.special.ndtr(z)) < 1e-12
    Qu, Su = orc.quantize_rows_fp8(W[::-1].copy())
    up = X.astype(np.float64) @ (Su.astype(np.float64)[:, None] * Qu).T
    sw = orc.column_parallel_fp8(2, X, Q, S, act="swiglu", Qu=Qu, Su=Su)
    assert _rel_err(sw, lin * scipy.special.expit(lin) * up) < 1e-12
    # FP8 row split: every shard quantized on its own, scaled, summed, + b once
    W = rng.standard_normal((5, 48)).astype(np.float32)
    X = rng.standard_normal((2, 48)).astype(np.float32)
    b = rng.standard_normal(5).astype(np.float32)
    for tp in (1, 2, 3, 4):
        Q, S = orc.quantize_row_shards_fp8(tp, W)
        ks = 48 // tp
        want = sum(X[:, i * ks:(i + 1) * ks].astype(np.float64) @
                   (S[i].astype(np.float64)[:, None] * Q[:, i * ks:(i + 1) * ks]).T
                   for i in range(tp)) + b
        assert _rel_err(orc.row_parallel_fp8(tp, X, Q, S, b), want) < 1e-13


def check_divisibility_errors(orc):
    """tp must divide out_features (column), in_features (row) and the heads."""
    import oracle
    X = np.ones((2, 6), np.float32)
    W = np.ones((9, 6), np.float32)
    for call in (lambda: orc.column_parallel(2, X, W),
                 lambda: orc.row_parallel(4, X, np.ones((3, 6), np.float32)),
                 lambda: orc.qkv_proj(3, X, np.ones((8 * 2, 6), np.float32), None, 4, 2, 2),
                 lambda: orc.qkv_proj(4, X, np.ones((12 * 2, 6), np.float32), None, 8, 2, 2),
                 lambda: orc.o_proj(3, np.ones((2, 8), np.float32),
                                    np.ones((6, 8), np.float32), None, 4, 2),
                 lambda: orc.mlp_block(3, X, np.ones((8, 6), np.float32), None,
                                       np.ones((6, 8), np.float32), None)):
        try:
            call()
        except oracle.OracleError as e:
            assert e.code == 2, e
        else:
            raise AssertionError("non-divisible split was accepted")


# ------------------------------------------------------------------ blocks

def check_mlp_block(orc):
    """FFN block == W2 . act(W1 x + b1) + b2 (numpy), any tp; h rounding point."""
    rng = _rng(17)
    M, d, dff = 4, 24, 48
    X = rng.standard_normal((M, d)).astype(np.float32)
    W1 = (0.2 * rng.standard_normal((dff, d))).astype(np.float32)
    W1u = (0.2 * rng.standard_normal((dff, d))).astype(np.float32)
    W2 = (0.2 * rng.standard_normal((d, dff))).astype(np.float32)
    b1 = rng.standard_normal(dff).astype(np.float32)
    b2 = rng.standard_normal(d).astype(np.float32)
    X64, W164, W1u64, W264 = (a.astype(np.float64) for a in (X, W1, W1u, W2))
    z = X64 @ W164.T + b1.astype(np.float64)
    h = z * scipy.special.ndtr(z)
    y = h @ W264.T + b2.astype(np.float64)
    g = X64 @ W164.T
    hs = g * scipy.special.expit(g) * (X64 @ W1u64.T)
    ys = hs @ W264.T
    for tp in (1, 2, 4, 8):
        Y, H = orc.mlp_block(tp, X, W1, b1, W2, b2, "gelu", round_h=False)
        assert _rel_err(H, h) < 1e-13 and _rel_err(Y, y) < 1e-13, tp
        Y, H = orc.mlp_block(tp, X, W1, None, W2, None, "swiglu", W1u=W1u,
                             round_h=False)
        assert _rel_err(H, hs) < 1e-13 and _rel_err(Y, ys) < 1e-13, tp
    # with the bf16 storage point: h is h rounded to bf16, and y uses that h
    Y, H = orc.mlp_block(2, X, W1, b1, W2, b2, "gelu", round_h=True)
    hb = torch.from_numpy(h).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    # fp64 -> bf16 directly may differ from fp64 -> fp32 -> bf16 only on ties
    assert np.mean(H == hb) > 0.99
    assert np.array_equal(H, np.vectorize(orc.round_bf16)(h))
    assert _rel_err(Y, H @ W264.T + b2.astype(np.float64)) < 1e-13


def check_attention_projections(orc):
    """QKV by head group and O by head, against an explicit gather (integers)."""
    rng = _rng(19)
    H, Hkv, hd, d, M = 4, 2, 3, 5, 2
    X = _int_mat(rng, (M, d))
    Wqkv = _int_mat(rng, ((H + 2 * Hkv) * hd, d))
    bqkv = _int_mat(rng, ((H + 2 * Hkv) * hd,))
    full = _brute_linear(X, Wqkv, bqkv)          # [M, (H+2Hkv)hd], rows Q;K;V
    for tp in (1, 2):
        out = orc.qkv_proj(tp, X, Wqkv, bqkv, H, Hkv, hd)
        for i in range(tp):
            q_heads = range(i * H // tp, (i + 1) * H // tp)
            k_heads = range(i * Hkv // tp, (i + 1) * Hkv // tp)
            cols = []
            for hh in q_heads:
                cols += list(range(hh * hd, (hh + 1) * hd))
            for hh in k_heads:
                cols += list(range(H * hd + hh * hd, H * hd + (hh + 1) * hd))
            for hh in k_heads:
                cols += list(range((H + Hkv) * hd + hh * hd, (H + Hkv) * hd + (hh + 1) * hd))
            assert np.array_equal(out[i], full[:, cols]), (tp, i)
    ctx = _int_mat(rng, (M, H * hd))
    Wo = _int_mat(rng, (d, H * hd))
    bo = _int_mat(rng, (d,))
    for tp in (1, 2, 4):
        assert np.array_equal(orc.o_proj(tp, ctx, Wo, bo, H, hd), _brute_linear(ctx, Wo, bo))


ALL_CHECKS = [
    check_worked_example,
    check_gelu_closed_form,
    check_silu_closed_form,
    check_round_bf16,
    check_brute_force_integers,
    check_numpy_fp64,
    check_shard_invariants,
    check_identity_weight,
    check_uneven_split,
    check_divisibility_errors,
    check_ring_allreduce,
    check_fp8_weights,
    check_mlp_block,
    check_attention_projections,
]


def run_all(orc):
    """name -> None (passed) or the failure message."""
    res = {}
    for c in ALL_CHECKS:
        try:
            c(orc)
            res[c.__name__] = None
        except Exception as e:  # noqa: BLE001 - a mutant may fail any way
            res[c.__name__] = f"{type(e).__name__}: {e}"
    return res
