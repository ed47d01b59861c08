// shard.cu -- tp_shard_weights: cut an unsharded weight into tp contiguous
// shards on the device (a bit-preserving gather).
//
// Shard layouts (unsharded W is [out_f, in_f], row-major):
//   COLUMN     shard i = rows [i*out_f/tp, (i+1)*out_f/tp)                 [out_f/tp, in_f]
//              (ColumnParallelLinear in "Understanding Tensor Parallelism for
//              Multi-GPU LLM Serving"; W[:split], W[split:] in "Tensor parallel
//              serving", "Simulating the split")
//   ROW        shard i = columns [i*in_f/tp, (i+1)*in_f/tp), made contiguous
//              [out_f, in_f/tp] (RowParallelLinear)
//   QKV_HEADS  shard i = its Q heads, then its K heads, then its V heads
//              ("What is tensor parallelism?", "How a layer is split")
//   GATE_UP    shard i = groups of TP_GATE_UP_GROUP gate rows followed by the
//              matching up rows; the last group is zero-padded.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace tpla {
namespace {

struct ShardParams {
  int split, tp, esize;
  const char* W;
  const char* W_up;
  int64_t out_f, in_f;
  int n_heads, n_kv_heads, head_dim;
  int64_t rows, cols;  // one shard
  char* dst[TP_MAX_TP];
};

// Source of destination row r of shard i: the matrix (0 = W, 1 = W_up,
// -1 = zero row), its row index and its first column.
struct Src {
  int which;
  int64_t row;
  int64_t col0;
};

// Row of the unsharded QKV weight that row r of head-group shard i copies.
__device__ __forceinline__ int64_t qkv_source_row(int64_t r, int i, int tp, int H, int Hkv,
                                                  int64_t hd) {
  const int64_t hq = H / tp, hk = Hkv / tp;
  if (r < hq * hd) return (int64_t)i * hq * hd + r;
  if (r < (hq + hk) * hd) return (int64_t)H * hd + (int64_t)i * hk * hd + (r - hq * hd);
  return (int64_t)(H + Hkv) * hd + (int64_t)i * hk * hd + (r - (hq + hk) * hd);
}

__device__ __forceinline__ Src source_row(const ShardParams& p, int i, int64_t r) {
  Src s{0, 0, 0};
  switch (p.split) {
    case TP_SPLIT_COLUMN:
      s.row = (int64_t)i * p.rows + r;
      break;
    case TP_SPLIT_ROW:
      s.row = r;
      s.col0 = (int64_t)i * p.cols;
      break;
    case TP_SPLIT_QKV_HEADS:
      s.row = qkv_source_row(r, i, p.tp, p.n_heads, p.n_kv_heads, p.head_dim);
      break;
    case TP_SPLIT_GATE_UP: {
      const int64_t G = TP_GATE_UP_GROUP;
      const int64_t ns = p.out_f / p.tp;
      const int64_t grp = r / (2 * G);
      const int64_t w = r - grp * 2 * G;
      const int64_t n = grp * G + (w % G);
      if (n >= ns) {
        s.which = -1;
      } else {
        s.which = (w < G) ? 0 : 1;
        s.row = (int64_t)i * ns + n;
      }
      break;
    }
  }
  return s;
}

// One block per destination row (grid-stride); 16-byte copies.
__global__ void __launch_bounds__(256) shard_kernel(const __grid_constant__ ShardParams p) {
  const int64_t total = (int64_t)p.tp * p.rows;
  const int64_t row_bytes = p.cols * p.esize;  // multiple of 16 (validated)
  const int64_t nvec = row_bytes / 16;
  for (int64_t gr = blockIdx.x; gr < total; gr += gridDim.x) {
    const int i = (int)(gr / p.rows);
    const int64_t r = gr - (int64_t)i * p.rows;
    const Src s = source_row(p, i, r);
    uint4* d = reinterpret_cast<uint4*>(p.dst[i] + r * row_bytes);
    if (s.which < 0) {
      for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) d[v] = make_uint4(0, 0, 0, 0);
    } else {
      const char* base = (s.which == 0) ? p.W : p.W_up;
      const uint4* src = reinterpret_cast<const uint4*>(
          base + (s.row * p.in_f + s.col0) * p.esize);
      for (int64_t v = threadIdx.x; v < nvec; v += blockDim.x) d[v] = src[v];
    }
  }
}

struct BiasParams {
  int split, tp;
  const float* b;
  int64_t rows;  // bias entries per shard
  int n_heads, n_kv_heads, head_dim;
  float* dst[TP_MAX_TP];
};

__global__ void shard_bias_kernel(const __grid_constant__ BiasParams p) {
  const int i = blockIdx.y;
  for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < p.rows;
       r += (int64_t)gridDim.x * blockDim.x) {
    const int64_t src = (p.split == TP_SPLIT_QKV_HEADS)
                            ? qkv_source_row(r, i, p.tp, p.n_heads, p.n_kv_heads, p.head_dim)
                            : (int64_t)i * p.rows + r;  // column
    p.dst[i][r] = p.b[src];
  }
}

}  // namespace

tp_status launch_shard(const ShardJob& j, cudaStream_t stream) {
  ShardParams p{};
  p.split = j.split;
  p.tp = j.tp;
  p.esize = j.esize;
  p.W = reinterpret_cast<const char*>(j.W);
  p.W_up = reinterpret_cast<const char*>(j.W_up);
  p.out_f = j.out_f;
  p.in_f = j.in_f;
  p.n_heads = j.n_heads;
  p.n_kv_heads = j.n_kv_heads;
  p.head_dim = j.head_dim;
  p.rows = j.rows;
  p.cols = j.cols;
  for (int i = 0; i < TP_MAX_TP; ++i) p.dst[i] = reinterpret_cast<char*>(j.dst[i]);
  const int64_t total = (int64_t)j.tp * j.rows;
  const int grid = (int)std::min<int64_t>(total, (int64_t)sm_count() * 16);
  if (grid > 0) shard_kernel<<<grid, 256, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return TP_ERR_CUDA;

  if (j.b) {
    BiasParams bp{};
    bp.split = j.split;
    bp.tp = j.tp;
    bp.b = j.b;
    bp.rows = j.rows;
    bp.n_heads = j.n_heads;
    bp.n_kv_heads = j.n_kv_heads;
    bp.head_dim = j.head_dim;
    for (int i = 0; i < TP_MAX_TP; ++i) bp.dst[i] = j.b_dst[i];
    dim3 g((unsigned)std::min<int64_t>((j.rows + 255) / 256, 1024), (unsigned)j.tp);
    shard_bias_kernel<<<g, 256, 0, stream>>>(bp);
    if (cudaGetLastError() != cudaSuccess) return TP_ERR_CUDA;
  }
  return TP_OK;
}

}  // namespace tpla
