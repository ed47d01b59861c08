// gemv.cu -- weight-streaming GEMV for few-token (decode-shaped) calls.
//
// Decode reads every weight byte once per call and does a handful of FLOPs
// per byte, so the kernel is bound by HBM bandwidth ("every GPU reads its
// own slice of the weights from its own memory" -- "What is tensor
// parallelism?", "Why it helps when serving").  Design:
//   * one warp owns R outputs (2R weight rows for SwiGLU: the gate row and the
//     up row of each output) and all K of them;
//   * lanes stride over K in 16-byte vectors (8 bf16 or 4 fp32), each lane
//     issuing U vectors per weight row before consuming any, with streaming
//     loads that bypass L1;
//   * activations (MT tokens) are read through the read-only cache, where
//     every warp of the SM reuses them;
//   * fp32 FMA accumulators, then a butterfly warp-shuffle reduction;
//   * the epilogue (bias, GELU / SwiGLU, row-parallel bias after the shard
//     sum) runs in fp32 and rounds once to the output dtype.
//
// Summation order of one output: each lane sums its vectors in increasing k
// (k-vectors lane, lane+32, ...), elements of a vector in order, then the
// butterfly.  It depends on K only -- not on N, tp, M or the template
// configuration -- so column-parallel results are bit-identical to tp = 1.
// Row-parallel: each lane walks shard 0, 1, ..., tp-1 in order with one
// accumulator, so the shard sum happens inside the same fp32 accumulator.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sync.cuh"

namespace tpla {
namespace {

constexpr int kWarps = 8;  // warps per block
constexpr int kThreads = kWarps * 32;

struct GemvParams {
  int tp;
  int act;
  int ydt;
  int64_t M, K, n_out, ns, ldx, x_shard_off, ldy;
  int64_t fo[TP_MAX_TP + 1];  // column: shard i owns outputs [fo[i], fo[i+1])
  int64_t yoff[TP_MAX_TP];    // column: element offset of shard i's outputs in Y
  const void* X;
  const void* W[TP_MAX_TP];
  const float* bias[TP_MAX_TP];
  void* Y;
  int64_t wrows[TP_MAX_TP];   // rows of each weight shard buffer (checked builds)
  unsigned int* err;          // device error word (checked builds)
  int64_t y_extent;           // elements of Y this call may write (checked builds)
};

template <typename T>
struct Vec;
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ static void unpack(const uint4& v, float f[8]) { unpack_bf16x8(v, f); }
};
template <>
struct Vec<float> {
  static constexpr int N = 4;
  __device__ static void unpack(const uint4& v, float f[4]) { unpack_f32x4(v, f); }
};

// Accumulate U k-vectors (starting at vector index c0, stride 32) of NR weight
// rows against MT tokens of X.
template <typename T, int MT, int NR, int U>
__device__ __forceinline__ void accumulate(float (&acc)[MT][NR], const T* const (&wr)[NR],
                                           const T* xbase, int64_t ldx, int64_t M,
                                           int64_t m0, int64_t c0, int64_t nvec) {
  constexpr int E = Vec<T>::N;
  uint4 wv[U][NR];
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t c = c0 + 32 * u;
    if (c < nvec) {
#pragma unroll
      for (int r = 0; r < NR; ++r) wv[u][r] = ld_stream16(wr[r] + c * E);
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u) {
    const int64_t c = c0 + 32 * u;
    if (c < nvec) {
      float wf[NR][E];
#pragma unroll
      for (int r = 0; r < NR; ++r) Vec<T>::unpack(wv[u][r], wf[r]);
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) {
        const int64_t m = m0 + mm;
        uint4 xv = make_uint4(0, 0, 0, 0);
        if (m < M) xv = ld_cached16(xbase + m * ldx + c * E);
        float xf[E];
        Vec<T>::unpack(xv, xf);
#pragma unroll
        for (int r = 0; r < NR; ++r)
#pragma unroll
          for (int e = 0; e < E; ++e) acc[mm][r] = fmaf(xf[e], wf[r][e], acc[mm][r]);
      }
    }
  }
}

template <int MT, int NR>
__device__ __forceinline__ void warp_reduce(float (&acc)[MT][NR]) {
#pragma unroll
  for (int mm = 0; mm < MT; ++mm)
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      float v = acc[mm][r];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      acc[mm][r] = v;
    }
}

template <typename T, int MT, int R, int U, int ACT, bool ROW>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const __grid_constant__ GemvParams p) {
  constexpr bool SW = (ACT == TP_ACT_SWIGLU);
  constexpr int NR = SW ? 2 * R : R;
  constexpr int E = Vec<T>::N;
  constexpr int64_t G = TP_GATE_UP_GROUP;
  static_assert(MT * R <= 32, "one lane stores one output");

  const int lane = threadIdx.x & 31;
  const int64_t warp_global = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int64_t warp_stride = (int64_t)gridDim.x * kWarps;
  const int64_t n_tasks = (p.n_out + R - 1) / R;
  const int64_t nvec = p.K / E;
  const T* X = reinterpret_cast<const T*>(p.X);
  // The next kernel may start now.  (This kernel is launched in plain
  // stream order, so every kernel before it has completed; the wait returns
  // at once and keeps the kernel correct under a programmatic launch too.)
  pdl_launch_dependents();
  pdl_wait();

  for (int64_t t = warp_global; t < n_tasks; t += warp_stride) {
    for (int64_t m0 = 0; m0 < p.M; m0 += MT) {
      float acc[MT][NR];
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
#pragma unroll
        for (int r = 0; r < NR; ++r) acc[mm][r] = 0.0f;

      if constexpr (!ROW) {
        const T* wr[NR];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int64_t o = min(t * R + r, p.n_out - 1);
          int i = 0;
          while (i + 1 < p.tp && p.fo[i + 1] <= o) ++i;
          const int64_t n = o - p.fo[i];
          const T* Wi = reinterpret_cast<const T*>(p.W[i]);
          if constexpr (SW) {
            const int64_t grp = n / G;
            int64_t row = grp * 2 * G + (n - grp * G);
            if (!TP_CHECK(p.err, row + G < p.wrows[i])) row = 0;
            wr[r] = Wi + row * p.K;
            wr[R + r] = Wi + (row + G) * p.K;
          } else {
            wr[r] = Wi + (TP_CHECK(p.err, n < p.wrows[i]) ? n : 0) * p.K;
          }
        }
        for (int64_t c0 = lane; c0 < nvec; c0 += 32 * U)
          accumulate<T, MT, NR, U>(acc, wr, X, p.ldx, p.M, m0, c0, nvec);
      } else {
        for (int i = 0; i < p.tp; ++i) {
          const T* Wi = reinterpret_cast<const T*>(p.W[i]);
          const T* wr[NR];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const int64_t o = min(t * R + r, p.n_out - 1);
            wr[r] = Wi + (TP_CHECK(p.err, o < p.wrows[i]) ? o : 0) * p.K;
          }
          const T* xi = X + i * p.x_shard_off;
          for (int64_t c0 = lane; c0 < nvec; c0 += 32 * U)
            accumulate<T, MT, NR, U>(acc, wr, xi, p.ldx, p.M, m0, c0, nvec);
        }
      }

      warp_reduce<MT, NR>(acc);

      // epilogue: lane (mm*R + r) finishes output (m0+mm, t*R+r)
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (lane != mm * R + r) continue;
          const int64_t m = m0 + mm;
          const int64_t o = t * R + r;
          if (m >= p.M || o >= p.n_out) continue;
          float z = acc[mm][r];
          if constexpr (ROW) {
            if (p.bias[0]) z += p.bias[0][o];
            if (TP_CHECK(p.err, m * p.ldy + o < p.y_extent)) store_out(p.Y, p.ydt, m * p.ldy + o, z);
          } else {
            int i = 0;
            while (i + 1 < p.tp && p.fo[i + 1] <= o) ++i;
            const int64_t n = o - p.fo[i];
            if constexpr (SW) {
              z = act_silu(z) * acc[mm][R + r];
            } else {
              if (p.bias[i]) z += p.bias[i][n];
              if constexpr (ACT == TP_ACT_GELU_ERF) z = act_gelu_erf(z);
            }
            if (TP_CHECK(p.err, p.yoff[i] + m * p.ldy + n < p.y_extent))
              store_out(p.Y, p.ydt, p.yoff[i] + m * p.ldy + n, z);
          }
        }
    }
  }
}

// Prepare one instantiation with a grid capped at (resident blocks x SMs).
template <typename T, int MT, int R, int U, int ACT, bool ROW>
tp_status prepare_one(const GemvParams& gp, Launch* L) {
  auto kern = gemv_kernel<T, MT, R, U, ACT, ROW>;
  static int resident = 0;  // blocks per SM for this instantiation
  static std::once_flag once;
  std::call_once(once, [&] {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kThreads, 0) != cudaSuccess)
      b = 1;
    resident = std::max(b, 1);
  });
  const int64_t n_tasks = (gp.n_out + R - 1) / R;
  const int64_t want = (n_tasks + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)resident * sm_count();
  L->kernel = reinterpret_cast<const void*>(kern);
  L->grid = dim3((unsigned)std::max<int64_t>(1, std::min(want, cap)));
  L->block = dim3(kThreads);
  L->smem = 0;
  L->cluster = 0;
  // Launched in plain stream order (measured: a programmatic launch of the
  // GEMV itself costs it 1-2 %); it still signals its dependents at entry,
  // so a decode kernel after it starts early.
  L->pdl = false;
  L->set_params(gp);
  return TP_OK;
}

// Tokens per pass (MT) and outputs per warp (R): the accumulator array
// acc[MT][R or 2R] stays within ~32 registers.
template <typename T, int ACT, bool ROW>
tp_status dispatch_mt(const GemvParams& gp, Launch* L) {
  constexpr bool SW = (ACT == TP_ACT_SWIGLU);
  if (gp.M <= 1) return prepare_one<T, 1, SW ? 2 : 4, 4, ACT, ROW>(gp, L);
  if (gp.M <= 2) return prepare_one<T, 2, SW ? 2 : 4, 4, ACT, ROW>(gp, L);
  if (gp.M <= 4) return prepare_one<T, 4, SW ? 2 : 4, 2, ACT, ROW>(gp, L);
  return prepare_one<T, 8, SW ? 2 : 4, 2, ACT, ROW>(gp, L);
}

template <typename T>
tp_status dispatch_act(const LinearProblem& p, const GemvParams& gp, Launch* L) {
  if (p.row) return dispatch_mt<T, TP_ACT_NONE, true>(gp, L);
  switch (p.act) {
    case TP_ACT_NONE: return dispatch_mt<T, TP_ACT_NONE, false>(gp, L);
    case TP_ACT_GELU_ERF: return dispatch_mt<T, TP_ACT_GELU_ERF, false>(gp, L);
    case TP_ACT_SWIGLU: return dispatch_mt<T, TP_ACT_SWIGLU, false>(gp, L);
  }
  return TP_ERR_BAD_SHAPE;
}

}  // namespace

tp_status prepare_gemv(const LinearProblem& p, Launch* L) {
  GemvParams gp{};
  gp.tp = p.tp;
  gp.act = p.act;
  gp.ydt = p.ydt;
  gp.M = p.M;
  gp.K = p.K;
  gp.n_out = p.n_out;
  gp.ns = p.ns;
  gp.ldx = p.ldx;
  gp.x_shard_off = p.x_shard_off;
  gp.ldy = p.ldy;
  for (int i = 0; i <= p.tp; ++i) gp.fo[i] = p.fo[i];
  for (int i = 0; i < p.tp; ++i) gp.yoff[i] = p.yoff[i];
  gp.X = p.X;
  gp.Y = p.Y;
  for (int i = 0; i < TP_MAX_TP; ++i) {
    gp.W[i] = p.W[i];
    gp.bias[i] = p.bias[i];
  }
  for (int i = 0; i < p.tp; ++i) gp.wrows[i] = p.row ? p.w_rows : p.wr[i];
  gp.err = device_error_word();
  if (!gp.err) return TP_ERR_CUDA;
  gp.y_extent = output_extent(p);
  if (p.xdt == TP_F32) return dispatch_act<float>(p, gp, L);
  return dispatch_act<__nv_bfloat16>(p, gp, L);
}

}  // namespace tpla
