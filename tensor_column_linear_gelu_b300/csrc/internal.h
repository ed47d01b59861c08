// internal.h -- host-side declarations shared by the library's translation
// units.  Not part of the public interface (that is include/tpla.h).
#pragma once

#include <cstdint>
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>

#include "tpla.h"

namespace tpla {

// One linear problem of the tensor-parallel path, after validation.
//
// Column-parallel (row == false): output o in [0, n_out) belongs to shard
//   i = o / ns at local column n = o % ns; it is act(X[m,:] . W_i[n,:] + b_i[n])
//   stored at Y + i*y_shard_stride + m*ldy + n.  For SwiGLU, W_i is the packed
//   gate/up shard (groups of TP_GATE_UP_GROUP gate rows, then as many up rows).
// Row-parallel (row == true): output o in [0, n_out) is
//   sum_i X_i[m,:] . W_i[o,:] + bias[0][o], with X_i = X + i*x_shard_off and
//   W_i of shape [n_out, K]; K is the per-shard input width.
struct LinearProblem {
  int tp = 1;
  bool row = false;
  int act = TP_ACT_NONE;
  int xdt = TP_BF16;
  int ydt = TP_BF16;
  int64_t M = 0;
  int64_t K = 0;            // input features per shard (column: all of K)
  int64_t n_out = 0;        // outputs over all shards (column) or N (row)
  int64_t ns = 0;           // outputs per shard (column); n_out (row)
  int64_t w_rows = 0;       // rows of each weight shard buffer
  const void* X = nullptr;
  int64_t ldx = 0;
  int64_t x_shard_off = 0;  // row: element offset of X_i
  const void* W[TP_MAX_TP] = {};
  const float* bias[TP_MAX_TP] = {};
  void* Y = nullptr;
  int64_t ldy = 0;
  int64_t y_shard_stride = 0;  // column: element offset of shard i's output
  // Column side, shard by shard: output features [fo[i], fo[i+1]) belong to
  // shard i, whose buffer has wr[i] rows and whose outputs start at element
  // yoff[i] of Y.  Equal split: fo[i] = i*ns, wr[i] = w_rows,
  // yoff[i] = i*y_shard_stride.  The decode kernel and the GEMV read these
  // tables (so they also run uneven splits); the prefill GEMM needs the
  // equal split.
  int64_t fo[TP_MAX_TP + 1] = {};
  int64_t wr[TP_MAX_TP] = {};
  int64_t yoff[TP_MAX_TP] = {};
  bool uneven = false;
  // FP8 weights: W[i] holds e4m3 codes and wscale[i] the fp32 scale of each
  // of its rows.
  bool fp8 = false;
  const float* wscale[TP_MAX_TP] = {};
};

// Number of elements of Y a problem may write: one past its last output
// element.  Checked builds bound every output store by it.
inline int64_t output_extent(const LinearProblem& p) {
  if (p.M <= 0) return 0;
  if (p.row) return (p.M - 1) * p.ldy + p.n_out;
  int64_t e = 0;
  for (int i = 0; i < p.tp; ++i) {
    const int64_t ei = p.yoff[i] + (p.M - 1) * p.ldy + (p.fo[i + 1] - p.fo[i]);
    if (ei > e) e = ei;
  }
  return e;
}

// A kernel launch prepared in full on the host: the kernel, its parameter
// block (tensor maps already encoded), grid, block, dynamic shared memory and
// cluster size.  Preparing does every host step that can fail except the
// launch itself, so a call that issues several launches prepares all of them
// before the first one starts: an error then leaves every output untouched.
// kernel == nullptr means there is nothing to launch (no tokens).
constexpr size_t kLaunchParamBytes = 8192;
struct Launch {
  const void* kernel = nullptr;
  dim3 grid{1, 1, 1};
  dim3 block{1, 1, 1};
  size_t smem = 0;
  unsigned cluster = 0;  // CTAs per cluster along x; 0: launched without clusters
  // launched with programmatic stream serialization: the kernel signals its
  // dependents early and waits for its predecessors itself (pdl_wait)
  bool pdl = false;
  alignas(64) unsigned char params[kLaunchParamBytes];
  template <class P>
  void set_params(const P& p) {
    static_assert(sizeof(P) <= kLaunchParamBytes, "kernel parameter block too large");
    std::memcpy(params, &p, sizeof(P));
  }
};
// Launch a prepared kernel on `stream` (nothing when L.kernel is null).
tp_status fire(const Launch& L, cudaStream_t stream);

// Each prepare_* fills a Launch for one validated problem.

// Weight-streaming GEMV on CUDA cores (few tokens; also the fp32 path).
tp_status prepare_gemv(const LinearProblem& p, Launch* L);

// tcgen05 / TMEM tensor-core GEMM fed by TMA on CTA pairs (bf16; many
// tokens; 256 x 256 tiles).
tp_status prepare_gemm_pair(const LinearProblem& p, Launch* L);
// Two independent problems in one launch (their tiles share the persistent
// grid); each must be one the prefill GEMM takes, a column problem and a row
// problem at most.
tp_status prepare_gemm_pair2(const LinearProblem& a, const LinearProblem& b, Launch* L);

// tcgen05 decode kernel with the weights as the MMA's N operand (a handful
// of tokens, up to kSkinnyMaxTokens; bf16 weights, or e4m3 weights widened
// to bf16 in shared memory when p.fp8).
constexpr int64_t kSkinnyMaxTokens = 128;
constexpr int kSkinnyMaxCluster = 8;  // CTAs per cluster on its row side
// bf16 calls with at most this many tokens go to the GEMV.
constexpr int64_t kGemvMaxTokens = 2;
tp_status prepare_skinny(const LinearProblem& p, Launch* L);

// 2-D bf16 tensor map for TMA: `rows` rows of `inner` elements, row pitch
// ld_bytes, boxes of 64 elements (one 128-byte swizzle span) x box_rows rows,
// 128-byte swizzle, out-of-range elements read as zero.
bool make_tma_map_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t ld_bytes, uint32_t box_rows);

// 2-D byte tensor map (e4m3 codes): boxes of box_inner bytes (a multiple of
// 16, at most 256; exactly 128 with swizzle128) x box_rows rows, rows landing
// box_inner bytes apart, either plain or with the 128-byte swizzle (16-byte
// chunk c of row r at chunk c ^ (r mod 8)); out-of-range bytes read as zero.
bool make_tma_map_u8(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                     uint64_t ld_bytes, uint32_t box_inner, uint32_t box_rows, bool swizzle128);

// FP8 (e4m3) weights, bf16 activations, at most kFp8MaxTokens tokens: the
// per-row quantizer; the weight-streaming FP8 GEMV (one token, and
// row-parallel calls whose tp exceeds the largest cluster); the e4m3 x e4m3
// kernel (M <= kF8MmaMaxTokens); the FP8 decode kernel with the widened
// weights in tensor memory (M <= kFp8TmemMaxTokens);
// above that the shared-memory decode kernel in its FP8 mode (prepare_skinny
// with p.fp8).
constexpr int64_t kFp8MaxTokens = kSkinnyMaxTokens;
constexpr int64_t kFp8TmemMaxTokens = 64;
// One token takes the FP8 GEMV: measured on the tp=4 SwiGLU FFN (d_model
// 8192, d_ff 28672), 87 + 49 us for the column and row launches against
// 92 + 50 us on the e4m3 x e4m3 kernel.  (At 8 tokens the GEMV took 379 us
// for the column: each token costs it a multiply-add per weight.)
constexpr int64_t kFp8GemvMaxTokens = 1;
// FP8 weights with at most this many tokens take the e4m3 x e4m3
// tensor-core kernel: the codes stream straight into the
// MMA's N operand and each token is split exactly into three e4m3 planes.
constexpr int64_t kF8MmaMaxTokens = 32;
tp_status prepare_f8mma(const LinearProblem& p, Launch* L);
tp_status prepare_decode_fp8(const LinearProblem& p, Launch* L);
tp_status launch_quantize_fp8(const void* W, int64_t rows, int64_t cols, void* Q, float* S,
                              cudaStream_t stream);
tp_status prepare_gemv_fp8(const LinearProblem& p, Launch* L);

// Ring-ordered sum of per-shard partials ([tp][M][N], wire dtype) + bias.
tp_status launch_ring_reduce(int tp, int64_t M, int64_t N, const void* parts, int wire_dt,
                             const float* bias, void* Y, int64_t ldy, int ydt,
                             cudaStream_t stream);

// Shard / pack copies.
struct ShardJob {
  int split = 0;
  int tp = 1;
  int esize = 2;
  const void* W = nullptr;
  const void* W_up = nullptr;
  int64_t out_f = 0, in_f = 0;
  int n_heads = 0, n_kv_heads = 0, head_dim = 0;
  int64_t rows = 0, cols = 0;   // shape of one shard
  void* dst[TP_MAX_TP] = {};
  const float* b = nullptr;
  float* b_dst[TP_MAX_TP] = {};
};
tp_status launch_shard(const ShardJob& j, cudaStream_t stream);

// Device-side error word (bounded waits) and its self-test.
unsigned int* device_error_word();
tp_status read_and_clear_device_error(cudaStream_t stream);
tp_status launch_bounded_wait_selftest(int64_t limit_ns, cudaStream_t stream);

// Number of SMs of the current device (cached per device).
int sm_count();

// How many clusters of cs CTAs of `kernel` (block threads, smem bytes of
// dynamic shared memory, which it sets as the kernel's maximum) the current
// device can hold at once; 0 when the runtime cannot say.  Cached.
int max_active_clusters(const void* kernel, int block, int smem, int cs);

// resident[cs] = max_active_clusters(kernel, block, smem, cs) for the cluster
// sizes cs = unit, 2 unit, ... up to cs_max (the others 0); resident has
// cs_max + 1 entries.
void resident_clusters(const void* kernel, int block, int smem, int cs_max, int unit,
                       int* resident);

}  // namespace tpla
