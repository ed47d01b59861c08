"""FP8 (e4m3) weights: the GPU quantizer and every FP8 compute kernel.

* tp_quantize_fp8 decides integer codes, so it must match the oracle's
  quantizer bit for bit: the scale (fp32) and every e4m3 code, for ordinary
  rows, a row of zeros and rows of very different magnitude.  Both sides
  decide in fp32.
* column_parallel_linear_fp8, row_parallel_linear_fp8 and tp_mlp_block_fp8
  against the oracle's FP8 splits.  The oracle quantizes the same bf16
  weights itself; nothing it uses comes from the GPU.  Tolerance: the bf16
  one (5e-3 x RMS, fp32 output); the FFN's h (bf16) within half a bf16 ulp.
* The FP8 column split is bit-identical to tp = 1, as the bf16 one is.
* Every FP8 kernel is covered: the e4m3 x e4m3 tensor-core kernel (1..32
  tokens: codes straight into the MMA, tokens split into three e4m3 planes),
  the kernel that widens the codes into tensor memory (33..64 tokens), the
  tensor-core decode kernel in its FP8 mode, which widens them into shared
  memory (65..128 tokens), and the FP8 GEMV (row splits wider than a
  cluster, tp > 8): every one of the 254 finite e4m3 codes goes through each
  kernel once and must come out as its exact value.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_bitwise_equal, assert_close_bf16, assert_h_bf16, np64, shard
from tensor_column_linear_gelu_b300 import inputs, tpla

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)


def codes_to_float(Q: torch.Tensor) -> np.ndarray:
    return Q.view(torch.float8_e4m3fn).float().cpu().numpy()


def test_quantizer_matches_oracle_bitwise(orc):
    rng = np.random.default_rng(3)
    W = rng.standard_normal((40, 4096)).astype(np.float32)
    W *= rng.uniform(1e-4, 50, (40, 1)).astype(np.float32)   # very different row magnitudes
    W[7] = 0.0                                                # a row of zeros
    W[11, ::97] *= 1000.0                                     # outliers
    Wb = torch.from_numpy(W).to(torch.bfloat16).to(DEV)
    Q, S = tpla.tp_quantize_fp8(Wb)
    torch.cuda.synchronize()
    q_ref, s_ref = orc.quantize_rows_fp8(Wb)
    assert np.array_equal(S.cpu().numpy(), s_ref)
    assert np.array_equal(codes_to_float(Q), q_ref)


# M, K, N, tp, act, bias
COLUMN_CASES = [(1, 256, 96, 2, "none", True), (2, 512, 384, 4, "gelu", True),
                (5, 1024, 600, 3, "gelu", False), (8, 256, 520, 4, "swiglu", False),
                (1, 4096, 2048, 8, "swiglu", False), (3, 320, 48, 1, "none", False),
                (16, 1024, 1000, 4, "gelu", True), (64, 512, 2304, 2, "swiglu", False),
                (128, 256, 384, 3, "none", True), (33, 2048, 4096, 8, "swiglu", False),
                (5, 272, 64, 2, "gelu", True), (70, 336, 512, 2, "swiglu", False)]


@pytest.mark.parametrize("M,K,N,tp,act,bias", COLUMN_CASES)
def test_fp8_column_parallel(orc, M, K, N, tp, act, bias):
    seed = 5 * M + K + N + tp
    X = inputs.normal((M, K), 1.0, seed, torch.bfloat16, DEV)
    W = inputs.normal((N, K), 0.05, seed + 1, torch.bfloat16, DEV)
    Wu = inputs.normal((N, K), 0.05, seed + 2, torch.bfloat16, DEV) if act == "swiglu" else None
    b = inputs.normal((N,), 0.1, seed + 4, torch.float32, DEV) if bias else None
    split = "gate_up" if act == "swiglu" else "column"
    ws, bs = shard(split, tp, W, W_up=Wu, b=b)
    qs, ss = tpla.quantize_shards_fp8(ws)
    y = tpla.column_parallel_linear_fp8(tp, X, qs, ss, bs, act, out_dtype=torch.float32, N=N)
    q_ref, s_ref = orc.quantize_rows_fp8(W)
    qu_ref = su_ref = None
    if act == "swiglu":
        qu_ref, su_ref = orc.quantize_rows_fp8(Wu)
    ref = orc.column_parallel_fp8(tp, X, q_ref, s_ref, b, act, Qu=qu_ref, Su=su_ref)
    assert_close_bf16(y, ref)
    # bit-identical to the same call unsharded
    w1, b1 = shard(split, 1, W, W_up=Wu, b=b)
    q1, s1 = tpla.quantize_shards_fp8(w1)
    y1 = tpla.column_parallel_linear_fp8(1, X, q1, s1, b1, act, out_dtype=torch.float32, N=N)
    assert_bitwise_equal(y, y1, "fp8 column sharded vs tp=1")
    assert tpla.tp_device_status() == tpla.TP_OK


# M, K, N, tp, bias  (tp = 16 row calls take the FP8 GEMV)
ROW_CASES = [(1, 512, 64, 2, True), (3, 1536, 200, 3, False), (8, 4096, 256, 8, True),
             (16, 1024, 520, 4, True), (64, 2048, 1024, 2, False), (128, 512, 300, 1, True),
             (5, 4096, 96, 16, True), (40, 3072, 768, 6, False), (4, 544, 320, 2, True),
             (90, 672, 136, 2, False)]


@pytest.mark.parametrize("M,K,N,tp,bias", ROW_CASES)
def test_fp8_row_parallel(orc, M, K, N, tp, bias):
    seed = 3 * M + K + N + tp
    X = inputs.normal((M, K), 1.0, seed, torch.bfloat16, DEV)
    W = inputs.normal((N, K), 0.05, seed + 3, torch.bfloat16, DEV)
    b = inputs.normal((N,), 0.1, seed + 5, torch.float32, DEV) if bias else None
    ws, _ = shard("row", tp, W)
    qs, ss = tpla.quantize_shards_fp8(ws)
    y = tpla.row_parallel_linear_fp8(tp, X, qs, ss, b, out_dtype=torch.float32)
    q_ref, s_ref = orc.quantize_row_shards_fp8(tp, W)
    assert np.array_equal(np.stack([s.cpu().numpy() for s in ss]), s_ref)
    ref = orc.row_parallel_fp8(tp, X, q_ref, s_ref, b)
    assert_close_bf16(y, ref)
    assert tpla.tp_device_status() == tpla.TP_OK


@pytest.mark.parametrize("M,tp", [(1, 4), (2, 4), (8, 2), (3, 4), (64, 8)])
def test_fp8_ffn_block(orc, M, tp):
    d, dff = 1024, 4096
    f = inputs.ffn(seed=40 + M, M=M, d_model=d, d_ff=dff, act="swiglu", bias=False, device=DEV)
    w1, _ = shard("gate_up", tp, f.W1, W_up=f.W_up)
    w2, _ = shard("row", tp, f.W2)
    q1, s1 = tpla.quantize_shards_fp8(w1)
    q2, s2 = tpla.quantize_shards_fp8(w2)
    y, h = tpla.tp_mlp_block_fp8(tp, f.X, q1, s1, None, q2, s2, None, "swiglu", d_ff=dff,
                                 out_dtype=torch.float32)
    torch.cuda.synchronize()
    qg, sg = orc.quantize_rows_fp8(f.W1)
    qu, su = orc.quantize_rows_fp8(f.W_up)
    h_exact = orc.column_parallel_fp8(tp, f.X, qg, sg, None, "swiglu", Qu=qu, Su=su)
    assert_h_bf16(h, h_exact)
    h_ref = np.vectorize(orc.round_bf16)(h_exact)
    qd, sd = orc.quantize_row_shards_fp8(tp, f.W2)
    y_ref = orc.row_parallel_fp8(tp, h_ref, qd, sd, None)
    assert_close_bf16(y, y_ref)
    # the FP8 weights hold the bf16 layer to within e4m3 rounding of the weights
    y_bf16, _ = orc.mlp_block(tp, f.X, f.W1, None, f.W2, None, "swiglu", W1u=f.W_up)
    rel = float(np.sqrt(np.mean((np64(y) - y_bf16) ** 2)) / np.sqrt(np.mean(y_bf16 ** 2)))
    assert rel < 0.08, rel
    assert tpla.tp_device_status() == tpla.TP_OK


def test_fp8_quantizer_full_size_sampled_rows(orc):
    """The 70B-shaped packed gate/up shard of tp=4 (14336 x 8192): codes and scales
    of sampled rows against the oracle, bit for bit."""
    f = inputs.llama70b_ffn(70_000, M=1, device=DEV)
    w1, _ = shard("gate_up", 4, f.W1, W_up=f.W_up)
    Q, S = tpla.tp_quantize_fp8(w1[1])
    torch.cuda.synchronize()
    rows = inputs.sample_rows(w1[1].shape[0], 48, 5)
    q_ref, s_ref = orc.quantize_rows_fp8(w1[1][rows])
    assert np.array_equal(S[rows].cpu().numpy(), s_ref)
    assert np.array_equal(codes_to_float(Q[rows]), q_ref)


def e4m3_table() -> np.ndarray:
    """Value of every e4m3 code (NaN for the two NaN codes), decoded by torch's
    CPU float8 type."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()


@pytest.mark.parametrize("M", [1, 4, 40, 100])
def test_every_e4m3_code_exact(orc, M):
    """W[n, k] = the value of code (n + k) mod 256 (NaN codes -> +-448), so every
    row holds 448, its scale is 1 and its codes are the table itself; token m is
    one-hot at column m, so Y[m, n] is the value of code (n + m) mod 256."""
    vals = e4m3_table()
    vals[0x7F], vals[0xFF] = 448.0, -448.0
    N = K = 256
    codes = (np.arange(N)[:, None] + np.arange(K)[None, :]) % 256
    W = torch.from_numpy(vals[codes]).to(torch.bfloat16).to(DEV)
    X = torch.zeros(M, K, dtype=torch.bfloat16, device=DEV)
    X[torch.arange(M), torch.arange(M)] = 1.0
    Q, S = tpla.tp_quantize_fp8(W)
    torch.cuda.synchronize()
    assert torch.all(S == 1.0)
    want = torch.from_numpy(codes.astype(np.uint8))
    want[want == 0x7F], want[want == 0xFF] = 0x7E, 0xFE
    assert torch.equal(Q.cpu(), want)
    y = tpla.column_parallel_linear_fp8(1, X, [Q], [S], None, "none", out_dtype=torch.float32)
    torch.cuda.synchronize()
    exact = vals[codes[:, :M].T]          # [M, N]
    assert np.array_equal(y.cpu().numpy(), exact)
    q_ref, s_ref = orc.quantize_rows_fp8(W)
    assert np.array_equal(orc.column_parallel_fp8(1, X, q_ref, s_ref), exact)


def test_every_e4m3_code_exact_row_gemv():
    """The same table through the FP8 GEMV: a row split with tp = 16 (wider than
    a cluster).  Every shard's 256 columns hold the whole table, so every row
    of every shard holds 448 and its scale is 1; token m is one-hot at column m
    of shard 0, so Y[m, n] is the value of code (n + m) mod 256."""
    vals = e4m3_table()
    vals[0x7F], vals[0xFF] = 448.0, -448.0
    tp, N, ks, M = 16, 256, 256, 3
    codes = (np.arange(N)[:, None] + np.arange(ks)[None, :]) % 256
    W = torch.from_numpy(np.tile(vals[codes], (1, tp))).to(torch.bfloat16).to(DEV)
    X = torch.zeros(M, tp * ks, dtype=torch.bfloat16, device=DEV)
    X[torch.arange(M), torch.arange(M)] = 1.0
    ws, _ = shard("row", tp, W)
    qs, ss = tpla.quantize_shards_fp8(ws)
    torch.cuda.synchronize()
    assert all(torch.all(sc == 1.0) for sc in ss)
    y = tpla.row_parallel_linear_fp8(tp, X, qs, ss, None, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), vals[codes[:, :M].T])
