// api.cu -- the C-ABI entry points of include/tpla.h: argument validation
// (before any launch; on error nothing is written) and kernel dispatch.
//
// Dispatch keys on (M, K, dtype, act) only -- never on N or tp -- and the
// kernels' own tilings never on tp (the decode kernel's K split depends on
// the total output count, K and M), so a column-parallel call computes every
// output with the same kernel and the same summation order whatever the
// shard count.
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "internal.h"

namespace tpla {

tp_status fire(const Launch& L, cudaStream_t stream) {
  if (!L.kernel) return TP_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = L.grid;
  cfg.blockDim = L.block;
  cfg.dynamicSmemBytes = L.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (L.cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = L.cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (L.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  void* args[1] = {const_cast<unsigned char*>(L.params)};
  if (cudaLaunchKernelExC(&cfg, L.kernel, args) != cudaSuccess) return TP_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

int sm_count() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  if (dev >= 64) dev = 63;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

int max_active_clusters(const void* kernel, int block, int smem, int cs) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, int, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  const auto key = std::make_tuple(dev, kernel, block, smem, cs);
  {
    std::lock_guard<std::mutex> g(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = 0;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cs * sm_count()));
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 0) n = 0;
  }
  (void)cudaGetLastError();  // a refused query leaves no error behind
  std::lock_guard<std::mutex> g(mu);
  cache[key] = n;
  return n;
}

void resident_clusters(const void* kernel, int block, int smem, int cs_max, int unit,
                       int* resident) {
  for (int c = 0; c <= cs_max; ++c) resident[c] = 0;
  for (int c = unit; c <= cs_max; c += unit) resident[c] = max_active_clusters(kernel, block, smem, c);
}

namespace {

#define TP_RET_IF(cond, code) \
  do {                        \
    if (cond) return (code);  \
  } while (0)

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al_to(const void* p, int64_t a) { return (reinterpret_cast<uintptr_t>(p) % (uintptr_t)a) == 0; }
int64_t esz(int dt) { return dt == TP_F32 ? 4 : 2; }
bool valid_dtype(int dt) { return dt == TP_F32 || dt == TP_BF16; }
// bf16 in -> bf16 or fp32 out; fp32 in -> fp32 out.
bool valid_io(int xdt, int ydt) {
  return valid_dtype(xdt) && valid_dtype(ydt) && !(xdt == TP_F32 && ydt == TP_BF16);
}
bool valid_act(int a) { return a == TP_ACT_NONE || a == TP_ACT_GELU_ERF || a == TP_ACT_SWIGLU; }
bool valid_tp(int tp) { return tp >= 1 && tp <= TP_MAX_TP; }

int64_t gate_up_rows(int64_t ns) {
  const int64_t G = TP_GATE_UP_GROUP;
  return 2 * G * ((ns + G - 1) / G);
}

tp_status check_ptr_array(const void* const* a, int tp) {
  TP_RET_IF(!a, TP_ERR_NULL);
  for (int i = 0; i < tp; ++i) TP_RET_IF(!a[i], TP_ERR_NULL);
  return TP_OK;
}

tp_status check_aligned_array(const void* const* a, int tp) {
  for (int i = 0; i < tp; ++i) TP_RET_IF(!al16(a[i]), TP_ERR_ALIGNMENT);
  return TP_OK;
}

tp_status check_bias_array(const float* const* b, int tp) {
  if (!b) return TP_OK;
  for (int i = 0; i < tp; ++i) {
    TP_RET_IF(!b[i], TP_ERR_NULL);
    TP_RET_IF(!al_to(b[i], 4), TP_ERR_ALIGNMENT);
  }
  return TP_OK;
}

// The one place a validated problem picks its kernel, and prepares its launch
// (launching nothing).  The choice depends on
// the dtype and the token count M only (never on N or tp):
//   fp32, or bf16 with M <= kGemvMaxTokens      weight-streaming GEMV (CUDA cores)
//   bf16, kGemvMaxTokens < M <= kSkinnyMaxTokens  tcgen05 decode kernel
//   bf16, M > kSkinnyMaxTokens                    tcgen05 prefill GEMM
//   FP8 weights, M <= kF8MmaMaxTokens             tcgen05 e4m3 x e4m3 decode kernel
//   FP8 weights, M <= kFp8TmemMaxTokens           tcgen05 FP8 decode kernel, weights in TMEM
//   FP8 weights, larger M                         tcgen05 decode kernel, FP8 mode
// (FP8 row-parallel calls with tp above the decode kernels' largest cluster
// take the FP8 GEMV: the tensor-core kernels' CTAs must each hold one
// shard's k-range.)
tp_status prepare(const LinearProblem& p, Launch* L) {
  L->kernel = nullptr;
  if (p.M == 0) return TP_OK;
  if (p.fp8) {
    if (p.M <= kFp8GemvMaxTokens || (p.row && p.tp > kSkinnyMaxCluster))
      return prepare_gemv_fp8(p, L);
    if (p.M <= kF8MmaMaxTokens) return prepare_f8mma(p, L);
    if (p.M <= kFp8TmemMaxTokens) return prepare_decode_fp8(p, L);
    return prepare_skinny(p, L);
  }
  if (p.xdt == TP_BF16 && p.M > kGemvMaxTokens) {
    if (p.M <= kSkinnyMaxTokens) return prepare_skinny(p, L);
    return prepare_gemm_pair(p, L);
  }
  return prepare_gemv(p, L);
}

tp_status run(const LinearProblem& p, cudaStream_t s) {
  Launch L;
  tp_status st = prepare(p, &L);
  if (st != TP_OK) return st;
  return fire(L, s);
}

// The prefill GEMM takes the problem (bf16, more tokens than the decode
// kernels take).
bool takes_gemm(const LinearProblem& p) {
  return !p.fp8 && p.xdt == TP_BF16 && p.M > kSkinnyMaxTokens;
}

// The attention projections: QKV and O are independent (O reads the
// caller's ctx, not the QKV output), so when both run on the prefill GEMM
// they share one launch and neither leaves a partial last wave of tiles.
tp_status prepare_attn_pair(const LinearProblem& qkv, const LinearProblem& o, Launch* Lq,
                            Launch* Lo) {
  if (takes_gemm(qkv) && takes_gemm(o)) {
    Lo->kernel = nullptr;
    return prepare_gemm_pair2(qkv, o, Lq);
  }
  const tp_status st = prepare(qkv, Lq);
  return st != TP_OK ? st : prepare(o, Lo);
}

// Launch prepared kernels in order.
tp_status fire_all(const Launch* L, int n, cudaStream_t s) {
  for (int i = 0; i < n; ++i) {
    const tp_status st = fire(L[i], s);
    if (st != TP_OK) return st;
  }
  return TP_OK;
}

// Prepare every problem of a call, then launch them in order: a host-side
// failure (a tensor map that cannot be encoded, a shape no kernel offers) is
// reported before anything runs, so the call writes nothing.  Only a launch
// that CUDA itself rejects can stop the sequence part-way (TP_ERR_CUDA).
tp_status run_seq(const LinearProblem* const* ps, int n, cudaStream_t s) {
  thread_local std::vector<Launch> launches;
  if ((int)launches.size() < n) launches.resize((size_t)n);
  for (int i = 0; i < n; ++i) {
    const tp_status st = prepare(*ps[i], &launches[(size_t)i]);
    if (st != TP_OK) return st;
  }
  for (int i = 0; i < n; ++i) {
    const tp_status st = fire(launches[(size_t)i], s);
    if (st != TP_OK) return st;
  }
  return TP_OK;
}

LinearProblem column_problem(int tp, int64_t M, int64_t K, int64_t N, const void* X,
                             int64_t ldx, int xdt, const void* const* w,
                             const float* const* b, int act, void* Y, int64_t ldy,
                             int ydt, int64_t y_shard_stride) {
  LinearProblem p;
  p.tp = tp;
  p.row = false;
  p.act = act;
  p.xdt = xdt;
  p.ydt = ydt;
  p.M = M;
  p.K = K;
  p.n_out = N;
  p.ns = N / tp;
  p.w_rows = (act == TP_ACT_SWIGLU) ? gate_up_rows(p.ns) : p.ns;
  p.X = X;
  p.ldx = ldx;
  p.Y = Y;
  p.ldy = ldy;
  p.y_shard_stride = y_shard_stride;
  for (int i = 0; i < tp; ++i) {
    p.W[i] = w[i];
    p.bias[i] = b ? b[i] : nullptr;
    p.fo[i] = (int64_t)i * p.ns;
    p.wr[i] = p.w_rows;
    p.yoff[i] = (int64_t)i * y_shard_stride;
  }
  p.fo[tp] = (int64_t)tp * p.ns;
  return p;
}

LinearProblem row_problem(int tp, int64_t M, int64_t K, int64_t N, const void* X, int64_t ldx,
                          int xdt, const void* const* w, const float* b, void* Y, int64_t ldy,
                          int ydt) {
  LinearProblem p;
  p.tp = tp;
  p.row = true;
  p.act = TP_ACT_NONE;
  p.xdt = xdt;
  p.ydt = ydt;
  p.M = M;
  p.K = K / tp;
  p.n_out = N;
  p.ns = N;
  p.w_rows = N;
  p.X = X;
  p.ldx = ldx;
  p.x_shard_off = K / tp;
  p.Y = Y;
  p.ldy = ldy;
  for (int i = 0; i < tp; ++i) p.W[i] = w[i];
  p.bias[0] = b;
  return p;
}

// Validation and problem set-up of the FFN block, before anything is
// launched.  *empty: no tokens, nothing to launch.
tp_status prepare_mlp(int tp, int64_t M, int64_t d_model, int64_t d_ff, int act, int xdt,
                      const void* X, const void* const* w1_shards, const float* const* b1_shards,
                      const void* const* w2_shards, const float* b2, void* h, void* Y, int ydt,
                      LinearProblem* up, LinearProblem* down, bool* empty) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(M < 0 || d_model <= 0 || d_ff <= 0, TP_ERR_BAD_SHAPE);
  TP_RET_IF(d_ff % tp, TP_ERR_NOT_DIVISIBLE);
  TP_RET_IF(!valid_io(xdt, ydt), TP_ERR_DTYPE);
  TP_RET_IF(!valid_act(act), TP_ERR_BAD_SHAPE);
  TP_RET_IF(act == TP_ACT_SWIGLU && b1_shards, TP_ERR_UNSUPPORTED);
  *empty = (M == 0);
  if (M == 0) return TP_OK;
  tp_status st;
  TP_RET_IF(!X || !h || !Y, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(w1_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_ptr_array(w2_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_bias_array(b1_shards, tp)) != TP_OK, st);
  const int64_t es = esz(xdt);
  TP_RET_IF(!al16(X) || !al16(h) || (d_model * es) % 16 || ((d_ff / tp) * es) % 16,
            TP_ERR_ALIGNMENT);
  TP_RET_IF(!al_to(Y, esz(ydt)) || (b2 && !al_to(b2, 4)), TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(w1_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_aligned_array(w2_shards, tp)) != TP_OK, st);
  // h = act(X . W1_i^T + b1_i), shard i in columns [i*d_ff/tp, ...): stored in
  // the input dtype (bf16 for bf16 inputs).
  *up = column_problem(tp, M, d_model, d_ff, X, d_model, xdt, w1_shards, b1_shards, act, h, d_ff,
                       xdt, d_ff / tp);
  // Y = sum_i h_i . W2_i^T + b2
  *down = row_problem(tp, M, d_ff, d_model, h, d_ff, xdt, w2_shards, b2, Y, d_model, ydt);
  return TP_OK;
}

// Validation and problem set-up of the attention projections.
tp_status prepare_attn(int tp, int64_t M, int64_t d_model, int n_heads, int n_kv_heads,
                       int head_dim, int xdt, const void* X, const void* const* wqkv_shards,
                       const float* const* bqkv_shards, void* qkv_out, int qkv_dt,
                       const void* ctx, const void* const* wo_shards, const float* bo, void* Y,
                       int ydt, LinearProblem* qkv, LinearProblem* o, bool* empty) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(M < 0 || d_model <= 0 || n_heads < 1 || n_kv_heads < 1 || head_dim < 1,
            TP_ERR_BAD_SHAPE);
  TP_RET_IF(n_heads % tp || n_kv_heads % tp, TP_ERR_NOT_DIVISIBLE);
  TP_RET_IF(!valid_io(xdt, ydt) || !valid_io(xdt, qkv_dt), TP_ERR_DTYPE);
  *empty = (M == 0);
  if (M == 0) return TP_OK;
  tp_status st;
  TP_RET_IF(!X || !qkv_out || !ctx || !Y, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(wqkv_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_ptr_array(wo_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_bias_array(bqkv_shards, tp)) != TP_OK, st);
  const int64_t es = esz(xdt);
  const int64_t kq = (int64_t)n_heads * head_dim;        // ctx width
  const int64_t ks = (int64_t)(n_heads / tp) * head_dim;  // ctx columns per shard
  const int64_t ws = (int64_t)(n_heads / tp + 2 * (n_kv_heads / tp)) * head_dim;
  TP_RET_IF(!al16(X) || !al16(ctx) || (d_model * es) % 16 || (kq * es) % 16 || (ks * es) % 16,
            TP_ERR_ALIGNMENT);
  TP_RET_IF(!al_to(qkv_out, esz(qkv_dt)) || !al_to(Y, esz(ydt)) || (bo && !al_to(bo, 4)),
            TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(wqkv_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_aligned_array(wo_shards, tp)) != TP_OK, st);
  // QKV: shard i -> qkv_out[i] = [M, ws]
  *qkv = column_problem(tp, M, d_model, ws * tp, X, d_model, xdt, wqkv_shards, bqkv_shards,
                        TP_ACT_NONE, qkv_out, ws, qkv_dt, M * ws);
  // O: Y = sum_i ctx_i . Wo_i^T + bo
  *o = row_problem(tp, M, kq, d_model, ctx, kq, xdt, wo_shards, bo, Y, d_model, ydt);
  return TP_OK;
}

}  // namespace
}  // namespace tpla

using namespace tpla;

extern "C" {

const char* tp_status_string(tp_status s) {
  switch (s) {
    case TP_OK: return "TP_OK";
    case TP_ERR_NULL: return "TP_ERR_NULL: a required pointer is NULL";
    case TP_ERR_NOT_DIVISIBLE: return "TP_ERR_NOT_DIVISIBLE: tp does not divide a split dimension";
    case TP_ERR_BAD_SHAPE: return "TP_ERR_BAD_SHAPE: invalid size, tp or leading dimension";
    case TP_ERR_DTYPE: return "TP_ERR_DTYPE: unsupported dtype combination";
    case TP_ERR_ALIGNMENT: return "TP_ERR_ALIGNMENT: pointer or stride not 16-byte aligned";
    case TP_ERR_CUDA: return "TP_ERR_CUDA: a CUDA call failed";
    case TP_ERR_DEVICE_TIMEOUT: return "TP_ERR_DEVICE_TIMEOUT: a bounded device wait gave up";
    case TP_ERR_UNSUPPORTED: return "TP_ERR_UNSUPPORTED: argument combination not offered";
    case TP_ERR_DEVICE_CHECK:
      return "TP_ERR_DEVICE_CHECK: a kernel index check failed (checked build; access skipped)";
  }
  return "unknown tp_status";
}

tp_status tp_shard_shape(tp_split split, int tp, int64_t out_f, int64_t in_f, int n_heads,
                         int n_kv_heads, int head_dim, int64_t* rows, int64_t* cols) {
  TP_RET_IF(!rows || !cols, TP_ERR_NULL);
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(out_f <= 0 || in_f <= 0, TP_ERR_BAD_SHAPE);
  switch (split) {
    case TP_SPLIT_COLUMN:
      TP_RET_IF(out_f % tp, TP_ERR_NOT_DIVISIBLE);
      *rows = out_f / tp;
      *cols = in_f;
      return TP_OK;
    case TP_SPLIT_ROW:
      TP_RET_IF(in_f % tp, TP_ERR_NOT_DIVISIBLE);
      *rows = out_f;
      *cols = in_f / tp;
      return TP_OK;
    case TP_SPLIT_QKV_HEADS:
      TP_RET_IF(n_heads < 1 || n_kv_heads < 1 || head_dim < 1, TP_ERR_BAD_SHAPE);
      TP_RET_IF(out_f != (int64_t)(n_heads + 2 * (int64_t)n_kv_heads) * head_dim,
                TP_ERR_BAD_SHAPE);
      TP_RET_IF(n_heads % tp || n_kv_heads % tp, TP_ERR_NOT_DIVISIBLE);
      *rows = (int64_t)(n_heads / tp + 2 * (n_kv_heads / tp)) * head_dim;
      *cols = in_f;
      return TP_OK;
    case TP_SPLIT_GATE_UP:
      TP_RET_IF(out_f % tp, TP_ERR_NOT_DIVISIBLE);
      *rows = gate_up_rows(out_f / tp);
      *cols = in_f;
      return TP_OK;
  }
  return TP_ERR_BAD_SHAPE;
}

tp_status tp_shard_weights(tp_split split, int tp, tp_dtype wdt, const void* W, const void* W_up,
                           int64_t out_f, int64_t in_f, const float* b, int n_heads,
                           int n_kv_heads, int head_dim, void* const* w_shards,
                           float* const* b_shards, tp_stream_t stream) {
  int64_t rows = 0, cols = 0;
  tp_status st = tp_shard_shape(split, tp, out_f, in_f, n_heads, n_kv_heads, head_dim, &rows, &cols);
  if (st != TP_OK) return st;
  TP_RET_IF(!valid_dtype(wdt), TP_ERR_DTYPE);
  TP_RET_IF(b && split != TP_SPLIT_COLUMN && split != TP_SPLIT_QKV_HEADS, TP_ERR_UNSUPPORTED);
  TP_RET_IF(!W, TP_ERR_NULL);
  TP_RET_IF(split == TP_SPLIT_GATE_UP && !W_up, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(w_shards, tp)) != TP_OK, st);
  if (b) {
    TP_RET_IF((st = check_ptr_array(reinterpret_cast<const void* const*>(b_shards), tp)) != TP_OK, st);
    TP_RET_IF(!al_to(b, 4), TP_ERR_ALIGNMENT);
    for (int i = 0; i < tp; ++i) TP_RET_IF(!al_to(b_shards[i], 4), TP_ERR_ALIGNMENT);
  }
  const int64_t es = esz(wdt);
  TP_RET_IF(!al16(W) || (W_up && split == TP_SPLIT_GATE_UP && !al16(W_up)), TP_ERR_ALIGNMENT);
  TP_RET_IF((in_f * es) % 16 || (cols * es) % 16, TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(w_shards, tp)) != TP_OK, st);

  ShardJob j;
  j.split = split;
  j.tp = tp;
  j.esize = (int)es;
  j.W = W;
  j.W_up = (split == TP_SPLIT_GATE_UP) ? W_up : nullptr;
  j.out_f = out_f;
  j.in_f = in_f;
  j.n_heads = n_heads;
  j.n_kv_heads = n_kv_heads;
  j.head_dim = head_dim;
  j.rows = rows;
  j.cols = cols;
  j.b = b;
  for (int i = 0; i < tp; ++i) {
    j.dst[i] = w_shards[i];
    j.b_dst[i] = b ? b_shards[i] : nullptr;
  }
  return launch_shard(j, reinterpret_cast<cudaStream_t>(stream));
}

tp_status column_parallel_linear(int tp, int64_t M, int64_t K, int64_t N, const void* X,
                                 int64_t ldx, tp_dtype xdt, const void* const* w_shards,
                                 const float* const* b_shards, tp_act act, void* Y, int64_t ldy,
                                 tp_dtype ydt, tp_stream_t stream) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(M < 0 || K <= 0 || N <= 0, TP_ERR_BAD_SHAPE);
  TP_RET_IF(N % tp, TP_ERR_NOT_DIVISIBLE);
  TP_RET_IF(!valid_io(xdt, ydt), TP_ERR_DTYPE);
  TP_RET_IF(!valid_act(act), TP_ERR_BAD_SHAPE);
  TP_RET_IF(act == TP_ACT_SWIGLU && b_shards, TP_ERR_UNSUPPORTED);
  TP_RET_IF(ldx < K || ldy < N, TP_ERR_BAD_SHAPE);
  if (M == 0) return TP_OK;
  tp_status st;
  TP_RET_IF(!X || !Y, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(w_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_bias_array(b_shards, tp)) != TP_OK, st);
  const int64_t es = esz(xdt);
  TP_RET_IF(!al16(X) || (ldx * es) % 16 || (K * es) % 16, TP_ERR_ALIGNMENT);
  TP_RET_IF(!al_to(Y, esz(ydt)), TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(w_shards, tp)) != TP_OK, st);
  LinearProblem p = column_problem(tp, M, K, N, X, ldx, xdt, w_shards, b_shards, act, Y, ldy,
                                   ydt, N / tp);
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

tp_status row_parallel_linear(int tp, int64_t M, int64_t K, int64_t N, const void* X, int64_t ldx,
                              tp_dtype xdt, const void* const* w_shards, const float* b, void* Y,
                              int64_t ldy, tp_dtype ydt, tp_stream_t stream) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(M < 0 || K <= 0 || N <= 0, TP_ERR_BAD_SHAPE);
  TP_RET_IF(K % tp, TP_ERR_NOT_DIVISIBLE);
  TP_RET_IF(!valid_io(xdt, ydt), TP_ERR_DTYPE);
  TP_RET_IF(ldx < K || ldy < N, TP_ERR_BAD_SHAPE);
  if (M == 0) return TP_OK;
  tp_status st;
  TP_RET_IF(!X || !Y, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(w_shards, tp)) != TP_OK, st);
  const int64_t es = esz(xdt);
  TP_RET_IF(!al16(X) || (ldx * es) % 16 || ((K / tp) * es) % 16, TP_ERR_ALIGNMENT);
  TP_RET_IF(!al_to(Y, esz(ydt)) || (b && !al_to(b, 4)), TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(w_shards, tp)) != TP_OK, st);
  LinearProblem p = row_problem(tp, M, K, N, X, ldx, xdt, w_shards, b, Y, ldy, ydt);
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

tp_status row_parallel_linear_ring(int tp, int64_t M, int64_t K, int64_t N, const void* X,
                                   int64_t ldx, tp_dtype xdt, const void* const* w_shards,
                                   const float* b, tp_dtype wire_dt, void* partials, void* Y,
                                   int64_t ldy, tp_dtype ydt, tp_stream_t stream) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(M < 0 || K <= 0 || N <= 0, TP_ERR_BAD_SHAPE);
  TP_RET_IF(K % tp, TP_ERR_NOT_DIVISIBLE);
  TP_RET_IF(!valid_io(xdt, ydt) || !valid_io(xdt, wire_dt), TP_ERR_DTYPE);
  TP_RET_IF(ldx < K || ldy < N, TP_ERR_BAD_SHAPE);
  if (M == 0) return TP_OK;
  tp_status st;
  TP_RET_IF(!X || !Y || !partials, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(w_shards, tp)) != TP_OK, st);
  const int64_t es = esz(xdt);
  const int64_t ks = K / tp;
  TP_RET_IF(!al16(X) || (ldx * es) % 16 || (ks * es) % 16, TP_ERR_ALIGNMENT);
  TP_RET_IF(!al_to(Y, esz(ydt)) || !al_to(partials, esz(wire_dt)) || (b && !al_to(b, 4)),
            TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(w_shards, tp)) != TP_OK, st);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // rank i's local partial X_i . W_i^T, rounded once to the wire dtype
  const int64_t L = M * N;
  LinearProblem parts[TP_MAX_TP];
  const LinearProblem* seq[TP_MAX_TP];
  for (int i = 0; i < tp; ++i) {
    const void* xi = static_cast<const char*>(X) + (int64_t)i * ks * es;
    void* pi = static_cast<char*>(partials) + (int64_t)i * L * esz(wire_dt);
    parts[i] = row_problem(1, M, ks, N, xi, ldx, xdt, &w_shards[i], nullptr, pi, N, wire_dt);
    seq[i] = &parts[i];
  }
  if ((st = run_seq(seq, tp, s)) != TP_OK) return st;
  return launch_ring_reduce(tp, M, N, partials, wire_dt, b, Y, ldy, ydt, s);
}

tp_status tp_shard_weights_uneven(int tp, const int64_t* widths, tp_dtype wdt, const void* W,
                                  int64_t out_f, int64_t in_f, const float* b,
                                  void* const* w_shards, float* const* b_shards,
                                  tp_stream_t stream) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(!widths, TP_ERR_NULL);
  TP_RET_IF(!valid_dtype(wdt), TP_ERR_DTYPE);
  TP_RET_IF(out_f <= 0 || in_f <= 0, TP_ERR_BAD_SHAPE);
  int64_t total = 0;
  for (int i = 0; i < tp; ++i) {
    TP_RET_IF(widths[i] < 1, TP_ERR_BAD_SHAPE);
    total += widths[i];
  }
  TP_RET_IF(total != out_f, TP_ERR_BAD_SHAPE);
  tp_status st;
  TP_RET_IF(!W, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(w_shards, tp)) != TP_OK, st);
  if (b) TP_RET_IF((st = check_ptr_array(reinterpret_cast<const void* const*>(b_shards), tp)) != TP_OK, st);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t row_bytes = in_f * esz(wdt);
  int64_t off = 0;
  for (int i = 0; i < tp; ++i) {
    // shard i = rows [off, off + widths[i]) of W: one contiguous block
    if (cudaMemcpyAsync(w_shards[i], static_cast<const char*>(W) + off * row_bytes,
                        (size_t)(widths[i] * row_bytes), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return TP_ERR_CUDA;
    if (b && cudaMemcpyAsync(b_shards[i], b + off, (size_t)widths[i] * sizeof(float),
                             cudaMemcpyDeviceToDevice, s) != cudaSuccess)
      return TP_ERR_CUDA;
    off += widths[i];
  }
  return TP_OK;
}

tp_status column_parallel_linear_uneven(int tp, const int64_t* widths, int64_t M, int64_t K,
                                        const void* X, int64_t ldx, tp_dtype xdt,
                                        const void* const* w_shards,
                                        const float* const* b_shards, tp_act act, void* Y,
                                        int64_t ldy, tp_dtype ydt, tp_stream_t stream) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(!widths, TP_ERR_NULL);
  TP_RET_IF(M < 0 || K <= 0, TP_ERR_BAD_SHAPE);
  int64_t N = 0;
  for (int i = 0; i < tp; ++i) {
    TP_RET_IF(widths[i] < 1, TP_ERR_BAD_SHAPE);
    N += widths[i];
  }
  TP_RET_IF(!valid_io(xdt, ydt), TP_ERR_DTYPE);
  TP_RET_IF(act != TP_ACT_NONE && act != TP_ACT_GELU_ERF, TP_ERR_UNSUPPORTED);
  TP_RET_IF(ldx < K || ldy < N, TP_ERR_BAD_SHAPE);
  if (M == 0) return TP_OK;
  tp_status st;
  TP_RET_IF(!X || !Y, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(w_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_bias_array(b_shards, tp)) != TP_OK, st);
  const int64_t es = esz(xdt);
  TP_RET_IF(!al16(X) || (ldx * es) % 16 || (K * es) % 16, TP_ERR_ALIGNMENT);
  TP_RET_IF(!al_to(Y, esz(ydt)), TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(w_shards, tp)) != TP_OK, st);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (xdt == TP_F32 || M <= kSkinnyMaxTokens) {
    // one launch over all shards: shard i owns output features [off_i,
    // off_i + widths[i]) and writes them to the same columns of Y
    LinearProblem p = column_problem(1, M, K, N, X, ldx, xdt, w_shards, nullptr, act, Y, ldy,
                                     ydt, 0);
    p.tp = tp;
    p.uneven = true;
    int64_t off = 0;
    for (int i = 0; i < tp; ++i) {
      p.W[i] = w_shards[i];
      p.bias[i] = b_shards ? b_shards[i] : nullptr;
      p.fo[i] = off;
      p.wr[i] = widths[i];
      p.yoff[i] = off;
      off += widths[i];
    }
    p.fo[tp] = off;
    return run(p, s);
  }
  int64_t off = 0;
  LinearProblem parts[TP_MAX_TP];
  const LinearProblem* seq[TP_MAX_TP];
  for (int i = 0; i < tp; ++i) {
    // many tokens: shard i as a one-shard call writing columns [off, off +
    // widths[i]) of Y -- the prefill GEMM's tiles need an equal split
    void* yi = static_cast<char*>(Y) + off * esz(ydt);
    parts[i] = column_problem(1, M, K, widths[i], X, ldx, xdt, &w_shards[i],
                              b_shards ? &b_shards[i] : nullptr, act, yi, ldy, ydt, 0);
    seq[i] = &parts[i];
    off += widths[i];
  }
  return run_seq(seq, tp, s);
}

tp_status tp_quantize_fp8(int64_t rows, int64_t cols, const void* W, void* Q, float* scales,
                          tp_stream_t stream) {
  TP_RET_IF(rows < 0 || cols <= 0, TP_ERR_BAD_SHAPE);
  if (rows == 0) return TP_OK;
  TP_RET_IF(!W || !Q || !scales, TP_ERR_NULL);
  TP_RET_IF(!al_to(W, 2) || !al_to(scales, 4), TP_ERR_ALIGNMENT);
  return launch_quantize_fp8(W, rows, cols, Q, scales, reinterpret_cast<cudaStream_t>(stream));
}

tp_status column_parallel_linear_fp8(int tp, int64_t M, int64_t K, int64_t N, const void* X,
                                     int64_t ldx, tp_dtype xdt, const void* const* q_shards,
                                     const float* const* scale_shards,
                                     const float* const* b_shards, tp_act act, void* Y,
                                     int64_t ldy, tp_dtype ydt, tp_stream_t stream) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(M < 0 || K <= 0 || N <= 0, TP_ERR_BAD_SHAPE);
  TP_RET_IF(N % tp, TP_ERR_NOT_DIVISIBLE);
  TP_RET_IF(xdt != TP_BF16 || !valid_io(xdt, ydt), TP_ERR_DTYPE);
  TP_RET_IF(!valid_act(act), TP_ERR_BAD_SHAPE);
  TP_RET_IF(act == TP_ACT_SWIGLU && b_shards, TP_ERR_UNSUPPORTED);
  TP_RET_IF(M > kFp8MaxTokens, TP_ERR_UNSUPPORTED);
  TP_RET_IF(ldx < K || ldy < N, TP_ERR_BAD_SHAPE);
  if (M == 0) return TP_OK;
  tp_status st;
  TP_RET_IF(!X || !Y, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(q_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_bias_array(scale_shards, tp)) != TP_OK, st);
  TP_RET_IF(!scale_shards, TP_ERR_NULL);
  TP_RET_IF((st = check_bias_array(b_shards, tp)) != TP_OK, st);
  TP_RET_IF(!al16(X) || (ldx * 2) % 16 || K % 16, TP_ERR_ALIGNMENT);
  TP_RET_IF(!al_to(Y, esz(ydt)), TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(q_shards, tp)) != TP_OK, st);
  LinearProblem p = column_problem(tp, M, K, N, X, ldx, xdt, q_shards, b_shards, act, Y, ldy, ydt,
                                   N / tp);
  p.fp8 = true;
  for (int i = 0; i < tp; ++i) p.wscale[i] = scale_shards[i];
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

tp_status row_parallel_linear_fp8(int tp, int64_t M, int64_t K, int64_t N, const void* X,
                                  int64_t ldx, tp_dtype xdt, const void* const* q_shards,
                                  const float* const* scale_shards, const float* b, void* Y,
                                  int64_t ldy, tp_dtype ydt, tp_stream_t stream) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(M < 0 || K <= 0 || N <= 0, TP_ERR_BAD_SHAPE);
  TP_RET_IF(K % tp, TP_ERR_NOT_DIVISIBLE);
  TP_RET_IF(xdt != TP_BF16 || !valid_io(xdt, ydt), TP_ERR_DTYPE);
  TP_RET_IF(M > kFp8MaxTokens, TP_ERR_UNSUPPORTED);
  TP_RET_IF(ldx < K || ldy < N, TP_ERR_BAD_SHAPE);
  if (M == 0) return TP_OK;
  tp_status st;
  TP_RET_IF(!X || !Y, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(q_shards, tp)) != TP_OK, st);
  TP_RET_IF(!scale_shards, TP_ERR_NULL);
  TP_RET_IF((st = check_bias_array(scale_shards, tp)) != TP_OK, st);
  TP_RET_IF(!al16(X) || (ldx * 2) % 16 || (K / tp) % 16, TP_ERR_ALIGNMENT);
  TP_RET_IF(!al_to(Y, esz(ydt)) || (b && !al_to(b, 4)), TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(q_shards, tp)) != TP_OK, st);
  LinearProblem p = row_problem(tp, M, K, N, X, ldx, xdt, q_shards, b, Y, ldy, ydt);
  p.fp8 = true;
  for (int i = 0; i < tp; ++i) p.wscale[i] = scale_shards[i];
  return run(p, reinterpret_cast<cudaStream_t>(stream));
}

tp_status tp_mlp_block_fp8(int tp, int64_t M, int64_t d_model, int64_t d_ff, tp_act act,
                           const void* X, const void* const* q1_shards,
                           const float* const* s1_shards, const float* const* b1_shards,
                           const void* const* q2_shards, const float* const* s2_shards,
                           const float* b2, void* h, void* Y, tp_dtype ydt,
                           tp_stream_t stream) {
  TP_RET_IF(!valid_tp(tp), TP_ERR_BAD_SHAPE);
  TP_RET_IF(M < 0 || d_model <= 0 || d_ff <= 0, TP_ERR_BAD_SHAPE);
  TP_RET_IF(d_ff % tp, TP_ERR_NOT_DIVISIBLE);
  TP_RET_IF(!valid_io(TP_BF16, ydt), TP_ERR_DTYPE);
  TP_RET_IF(!valid_act(act), TP_ERR_BAD_SHAPE);
  TP_RET_IF(act == TP_ACT_SWIGLU && b1_shards, TP_ERR_UNSUPPORTED);
  TP_RET_IF(M > kFp8MaxTokens, TP_ERR_UNSUPPORTED);
  if (M == 0) return TP_OK;
  tp_status st;
  TP_RET_IF(!X || !h || !Y, TP_ERR_NULL);
  TP_RET_IF((st = check_ptr_array(q1_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_ptr_array(q2_shards, tp)) != TP_OK, st);
  TP_RET_IF(!s1_shards || !s2_shards, TP_ERR_NULL);
  TP_RET_IF((st = check_bias_array(s1_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_bias_array(s2_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_bias_array(b1_shards, tp)) != TP_OK, st);
  TP_RET_IF(!al16(X) || !al16(h) || d_model % 16 || (d_ff / tp) % 16, TP_ERR_ALIGNMENT);
  TP_RET_IF(!al_to(Y, esz(ydt)) || (b2 && !al_to(b2, 4)), TP_ERR_ALIGNMENT);
  TP_RET_IF((st = check_aligned_array(q1_shards, tp)) != TP_OK, st);
  TP_RET_IF((st = check_aligned_array(q2_shards, tp)) != TP_OK, st);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // h = act(X . W1_i^T + b1_i) in bf16, then Y = sum_i h_i . W2_i^T + b2
  LinearProblem up = column_problem(tp, M, d_model, d_ff, X, d_model, TP_BF16, q1_shards,
                                    b1_shards, act, h, d_ff, TP_BF16, d_ff / tp);
  LinearProblem down = row_problem(tp, M, d_ff, d_model, h, d_ff, TP_BF16, q2_shards, b2, Y,
                                   d_model, ydt);
  up.fp8 = down.fp8 = true;
  for (int i = 0; i < tp; ++i) {
    up.wscale[i] = s1_shards[i];
    down.wscale[i] = s2_shards[i];
  }
  const LinearProblem* seq[2] = {&up, &down};
  return run_seq(seq, 2, s);
}

tp_status tp_mlp_block(int tp, int64_t M, int64_t d_model, int64_t d_ff, tp_act act, tp_dtype xdt,
                       const void* X, const void* const* w1_shards, const float* const* b1_shards,
                       const void* const* w2_shards, const float* b2, void* h, void* Y,
                       tp_dtype ydt, tp_stream_t stream) {
  LinearProblem up, down;
  bool empty = false;
  tp_status st = prepare_mlp(tp, M, d_model, d_ff, act, xdt, X, w1_shards, b1_shards, w2_shards,
                             b2, h, Y, ydt, &up, &down, &empty);
  if (st != TP_OK || empty) return st;
  const LinearProblem* seq[2] = {&up, &down};
  return run_seq(seq, 2, reinterpret_cast<cudaStream_t>(stream));
}

tp_status tp_attn_proj(int tp, int64_t M, int64_t d_model, int n_heads, int n_kv_heads,
                       int head_dim, tp_dtype xdt, const void* X, const void* const* wqkv_shards,
                       const float* const* bqkv_shards, void* qkv_out, tp_dtype qkv_dt,
                       const void* ctx, const void* const* wo_shards, const float* bo, void* Y,
                       tp_dtype ydt, tp_stream_t stream) {
  LinearProblem qkv, o;
  bool empty = false;
  tp_status st = prepare_attn(tp, M, d_model, n_heads, n_kv_heads, head_dim, xdt, X, wqkv_shards,
                              bqkv_shards, qkv_out, qkv_dt, ctx, wo_shards, bo, Y, ydt, &qkv, &o,
                              &empty);
  if (st != TP_OK || empty) return st;
  thread_local Launch launches[2];
  if ((st = prepare_attn_pair(qkv, o, &launches[0], &launches[1])) != TP_OK) return st;
  return fire_all(launches, 2, reinterpret_cast<cudaStream_t>(stream));
}

tp_status tp_layer_forward(const tp_layer_args* a, tp_stream_t stream) {
  TP_RET_IF(!a, TP_ERR_NULL);
  LinearProblem qkv, o, up, down;
  bool empty_attn = false, empty_mlp = false;
  tp_status st = prepare_attn(a->tp, a->M, a->d_model, a->n_heads, a->n_kv_heads, a->head_dim,
                              a->xdt, a->X, a->wqkv_shards, a->bqkv_shards, a->qkv_out, a->qkv_dt,
                              a->ctx, a->wo_shards, a->bo, a->Y_attn, a->attn_ydt, &qkv, &o,
                              &empty_attn);
  if (st != TP_OK) return st;
  st = prepare_mlp(a->tp, a->M, a->d_model, a->d_ff, a->ffn_act, a->xdt, a->X_ffn, a->w1_shards,
                   a->b1_shards, a->w2_shards, a->b2, a->h, a->Y_ffn, a->ffn_ydt, &up, &down,
                   &empty_mlp);
  if (st != TP_OK) return st;
  // The FFN may read the attention block's output directly (X_ffn == Y_attn):
  // then that output must be in the input dtype.
  TP_RET_IF(a->X_ffn == a->Y_attn && a->attn_ydt != a->xdt, TP_ERR_DTYPE);
  if (empty_attn) return TP_OK;
  thread_local Launch launches[4];
  if ((st = prepare_attn_pair(qkv, o, &launches[0], &launches[1])) != TP_OK) return st;
  if ((st = prepare(up, &launches[2])) != TP_OK) return st;
  if ((st = prepare(down, &launches[3])) != TP_OK) return st;
  return fire_all(launches, 4, reinterpret_cast<cudaStream_t>(stream));
}

tp_status tp_device_status(tp_stream_t stream) {
  return read_and_clear_device_error(reinterpret_cast<cudaStream_t>(stream));
}

tp_status tp_selftest_bounded_wait(int64_t limit_ns, tp_stream_t stream) {
  TP_RET_IF(limit_ns < 1 || limit_ns > 10000000000LL, TP_ERR_BAD_SHAPE);
  return launch_bounded_wait_selftest(limit_ns, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
