// fp8.cu -- FP8 (e4m3) weights for decode-shaped calls: the per-row quantizer
// and a weight-streaming GEMV that reads one byte per weight.
//
// "Model Parallelism" (statistical-learning-notes) sizes model weights at
// about one byte per parameter in FP8: for a decode-shaped call, which is
// bound by the weight bytes it streams, that halves the time of bf16 weights.
// The pages fix no format or scaling; the library's reading:
//   * e4m3 codes (4 exponent bits, bias 7, 3 mantissa bits, no infinities,
//     largest finite value 448);
//   * one fp32 scale per weight row, s = max_k |W[r,k]| / 448 (1 for a row of
//     zeros), code = W[r,k] / s rounded to nearest even, saturating at 448 --
//     scale and quotient in fp32, the precision that decides the code;
//   * y = s * (x . q): the dot product runs in fp32 on the e4m3 values and the
//     row's scale multiplies the result.  On the row-parallel side each shard
//     is quantized as its own [N, K/tp] matrix, so each shard's partial is
//     scaled by its own s before the in-kernel shard sum.
// GEMV structure as in gemv.cu: one warp owns R outputs (2R weight rows for
// SwiGLU), lanes stride over K in 16-byte vectors (16 weights, 16 tokens' worth
// of bf16 X in two loads), U vectors in flight per row, streaming loads,
// butterfly reduction, fused epilogue.
#include <cuda_fp8.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "sync.cuh"

namespace tpla {
namespace {

// ---------------------------------------------------------------- quantizer
constexpr int QTHREADS = 256;

__global__ void __launch_bounds__(QTHREADS) quantize_fp8_rows_kernel(
    const __nv_bfloat16* __restrict__ W, int64_t rows, int64_t cols, uint8_t* __restrict__ Q,
    float* __restrict__ S) {
  __shared__ float red[QTHREADS / 32];
  __shared__ float s_scale;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const __nv_bfloat16* w = W + r * cols;
    float amax = 0.0f;
    for (int64_t c = threadIdx.x; c < cols; c += QTHREADS)
      amax = fmaxf(amax, fabsf(__bfloat162float(w[c])));
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x == 0) {
      float m = red[0];
      for (int i = 1; i < QTHREADS / 32; ++i) m = fmaxf(m, red[i]);
      const float sc = m > 0.0f ? __fdiv_rn(m, 448.0f) : 1.0f;
      s_scale = sc;
      S[r] = sc;
    }
    __syncthreads();
    const float sc = s_scale;
    for (int64_t c = threadIdx.x; c < cols; c += QTHREADS) {
      const float v = __fdiv_rn(__bfloat162float(w[c]), sc);
      Q[r * cols + c] = (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
    }
    __syncthreads();  // red / s_scale are reused by the next row
  }
}

// ---------------------------------------------------------------- GEMV
// Warps per block: one for a single token -- 32-thread blocks spread the
// warps evenly over the SMs (one-token SwiGLU FFN, tp 4: column 81 against
// 83 us, step 128 against 130 us; 2- and 4-warp blocks were slower than 8);
// eight for more tokens.  A one-token row split takes two warps per output
// group, each walking half of the shards (RSPLIT below).
template <int MT, bool ROW>
constexpr bool row_halves() { return ROW && MT == 1; }
template <int MT, bool ROW>
constexpr int warps_of() { return row_halves<MT, ROW>() ? 2 : (MT == 1 ? 1 : 8); }
constexpr int E = 16;  // weights per 16-byte vector

struct Fp8Params {
  int tp, act, ydt;
  int64_t M, K, n_out, ldx, x_shard_off, ldy;
  int64_t fo[TP_MAX_TP + 1];   // column: shard i owns outputs [fo[i], fo[i+1])
  int64_t yoff[TP_MAX_TP];     // column: element offset of shard i's outputs in Y
  const __nv_bfloat16* X;
  const uint8_t* W[TP_MAX_TP];
  const float* S[TP_MAX_TP];   // row scales of each shard buffer
  const float* bias[TP_MAX_TP];
  void* Y;
  int64_t wrows[TP_MAX_TP];    // rows of each code buffer (checked builds)
  unsigned int* err;           // device error word (checked builds)
  int64_t y_extent;            // elements of Y this call may write (checked builds)
};

__device__ __forceinline__ void fp8x16_to_float(const uint4& v, float (&f)[16]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    __nv_fp8x4_e4m3 q;
    q.__x = w[j];
    const float4 t = static_cast<float4>(q);
    f[4 * j + 0] = t.x;
    f[4 * j + 1] = t.y;
    f[4 * j + 2] = t.z;
    f[4 * j + 3] = t.w;
  }
}

// Accumulate U k-vectors (vector index c0, stride 32) of NR weight rows.
template <int MT, int NR, int U>
__device__ __forceinline__ void accumulate_fp8(float (&acc)[MT][NR], const uint8_t* const (&wr)[NR],
                                               const __nv_bfloat16* xbase, int64_t ldx, int64_t M,
                                               int64_t m0, int64_t c0, int64_t nvec) {
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
#pragma unroll
      for (int mm = 0; mm < MT; ++mm) {
        const int64_t m = m0 + mm;
        uint4 x0 = make_uint4(0, 0, 0, 0), x1 = make_uint4(0, 0, 0, 0);
        if (m < M) {
          x0 = ld_cached16(xbase + m * ldx + c * E);
          x1 = ld_cached16(xbase + m * ldx + c * E + 8);
        }
        float xf[16];
        unpack_bf16x8(x0, xf);
        unpack_bf16x8(x1, xf + 8);
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          float wf[16];
          fp8x16_to_float(wv[u][r], wf);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[mm][r] = fmaf(xf[e], wf[e], acc[mm][r]);
        }
      }
    }
  }
}

template <int MT, int R, int U, int ACT, bool ROW>
__global__ void __launch_bounds__(warps_of<MT, ROW>() * 32) gemv_fp8_kernel(const __grid_constant__ Fp8Params p) {
  constexpr int kWarps = warps_of<MT, ROW>();
  // RSPLIT (one token, row split): the block's two warps take the same
  // output group, warp h the shards [h*tp/2, (h+1)*tp/2); warp 0 adds warp
  // 1's sums to its own (a fixed order) and stores.  Twice the warps stream
  // the same bytes, so twice the loads are in flight.
  constexpr bool RSPLIT = row_halves<MT, ROW>();
  __shared__ float half_sum[RSPLIT ? 32 : 1];
  constexpr bool SW = (ACT == TP_ACT_SWIGLU);
  constexpr int NR = SW ? 2 * R : R;
  constexpr int64_t G = TP_GATE_UP_GROUP;
  static_assert(MT * R <= 32, "one lane stores one output");

  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;  // warp in block
  const int64_t warp_global = RSPLIT ? blockIdx.x : (int64_t)blockIdx.x * kWarps + wib;
  const int64_t warp_stride = RSPLIT ? gridDim.x : (int64_t)gridDim.x * kWarps;
  const int64_t n_tasks = (p.n_out + R - 1) / R;
  const int64_t nvec = p.K / E;
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
      float sc[NR];  // column side: the row scale of each weight row

      if constexpr (!ROW) {
        const uint8_t* wr[NR];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int64_t o = min(t * R + r, p.n_out - 1);
          int i = 0;
          while (i + 1 < p.tp && p.fo[i + 1] <= o) ++i;
          const int64_t n = o - p.fo[i];
          int64_t row = n;
          if constexpr (SW) row = (n / G) * 2 * G + n % G;
          if (!TP_CHECK(p.err, row + (SW ? G : 0) < p.wrows[i])) row = 0;
          wr[r] = p.W[i] + row * p.K;
          sc[r] = __ldg(p.S[i] + row);
          if constexpr (SW) {
            wr[R + r] = p.W[i] + (row + G) * p.K;
            sc[R + r] = __ldg(p.S[i] + row + G);
          }
        }
        for (int64_t c0 = lane; c0 < nvec; c0 += 32 * U)
          accumulate_fp8<MT, NR, U>(acc, wr, p.X, p.ldx, p.M, m0, c0, nvec);
      } else {
        // each shard's lane partial is scaled by that shard's row scale, then
        // added to the running sum (shard order 0..tp-1; RSPLIT: within each
        // half, then half 1's sum added to half 0's)
        const int i0 = RSPLIT ? wib * p.tp / 2 : 0;
        const int i1 = RSPLIT ? (wib + 1) * p.tp / 2 : p.tp;
        for (int i = i0; i < i1; ++i) {
          const uint8_t* wr[NR];
          float part[MT][NR];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            int64_t o = min(t * R + r, p.n_out - 1);
            if (!TP_CHECK(p.err, o < p.wrows[i])) o = 0;
            wr[r] = p.W[i] + o * p.K;
            sc[r] = __ldg(p.S[i] + o);
          }
#pragma unroll
          for (int mm = 0; mm < MT; ++mm)
#pragma unroll
            for (int r = 0; r < NR; ++r) part[mm][r] = 0.0f;
          const __nv_bfloat16* xi = p.X + i * p.x_shard_off;
          for (int64_t c0 = lane; c0 < nvec; c0 += 32 * U)
            accumulate_fp8<MT, NR, U>(part, wr, xi, p.ldx, p.M, m0, c0, nvec);
#pragma unroll
          for (int mm = 0; mm < MT; ++mm)
#pragma unroll
            for (int r = 0; r < NR; ++r) acc[mm][r] = fmaf(sc[r], part[mm][r], acc[mm][r]);
        }
      }

      // butterfly warp reduction
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
#pragma unroll
        for (int r = 0; r < NR; ++r) {
          float v = acc[mm][r];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          acc[mm][r] = v;
        }

      if constexpr (RSPLIT) {
        if (wib == 1 && lane == 0) {
#pragma unroll
          for (int r = 0; r < R; ++r) half_sum[r] = acc[0][r];
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < R; ++r) acc[0][r] += half_sum[r];
        __syncthreads();  // half_sum is rewritten for the next output group
      }

      // epilogue: lane (mm*R + r) finishes output (m0+mm, t*R+r)
#pragma unroll
      for (int mm = 0; mm < MT; ++mm)
#pragma unroll
        for (int r = 0; r < R; ++r) {
          if (lane != mm * R + r || (RSPLIT && wib != 0)) continue;
          const int64_t m = m0 + mm;
          const int64_t o = t * R + r;
          if (m >= p.M || o >= p.n_out) continue;
          if constexpr (ROW) {
            float z = acc[mm][r];
            if (p.bias[0]) z += p.bias[0][o];
            if (TP_CHECK(p.err, m * p.ldy + o < p.y_extent)) store_out(p.Y, p.ydt, m * p.ldy + o, z);
          } else {
            int i = 0;
            while (i + 1 < p.tp && p.fo[i + 1] <= o) ++i;
            const int64_t n = o - p.fo[i];
            float z = sc[r] * acc[mm][r];
            if constexpr (SW) {
              z = act_silu(z) * (sc[R + r] * acc[mm][R + r]);
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

template <int MT, int R, int U, int ACT, bool ROW>
tp_status prepare_fp8(const Fp8Params& gp, Launch* L) {
  auto kern = gemv_fp8_kernel<MT, R, U, ACT, ROW>;
  constexpr int kWarps = warps_of<MT, ROW>();
  constexpr int kThreads = kWarps * 32;
  static int resident = 0;
  static std::once_flag once;
  std::call_once(once, [&] {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kern, kThreads, 0) != cudaSuccess) b = 1;
    resident = std::max(b, 1);
  });
  const int64_t n_tasks = (gp.n_out + R - 1) / R;
  const int64_t want = row_halves<MT, ROW>() ? n_tasks : (n_tasks + kWarps - 1) / kWarps;
  L->kernel = reinterpret_cast<const void*>(kern);
  L->grid = dim3((unsigned)std::max<int64_t>(1, std::min(want, (int64_t)resident * sm_count())));
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

template <int ACT, bool ROW>
tp_status dispatch_fp8_mt(const Fp8Params& gp, Launch* L) {
  constexpr bool SW = (ACT == TP_ACT_SWIGLU);
  // one token: a SwiGLU column warp takes one output (its gate and up rows)
  // with four 16-byte loads per row in flight -- 81 us against 87 us with two
  // outputs and two loads; the row and the other columns keep four outputs
  // (fewer made the row launch slower: 65 against 47 us)
  if (gp.M <= 1) return prepare_fp8<1, SW ? 1 : 4, 4, ACT, ROW>(gp, L);
  if (gp.M <= 2) return prepare_fp8<2, SW ? 2 : 4, 2, ACT, ROW>(gp, L);
  if (gp.M <= 4) return prepare_fp8<4, SW ? 2 : 4, 1, ACT, ROW>(gp, L);
  return prepare_fp8<8, SW ? 2 : 4, 1, ACT, ROW>(gp, L);
}

}  // namespace

tp_status launch_quantize_fp8(const void* W, int64_t rows, int64_t cols, void* Q, float* S,
                              cudaStream_t stream) {
  if (rows == 0) return TP_OK;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(rows, (int64_t)sm_count() * 16));
  quantize_fp8_rows_kernel<<<grid, QTHREADS, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(W), rows, cols, static_cast<uint8_t*>(Q), S);
  return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

tp_status prepare_gemv_fp8(const LinearProblem& p, Launch* L) {
  Fp8Params gp{};
  gp.tp = p.tp;
  gp.act = p.act;
  gp.ydt = p.ydt;
  gp.M = p.M;
  gp.K = p.K;
  gp.n_out = p.n_out;
  gp.ldx = p.ldx;
  gp.x_shard_off = p.x_shard_off;
  gp.ldy = p.ldy;
  for (int i = 0; i <= p.tp; ++i) gp.fo[i] = p.fo[i];
  for (int i = 0; i < p.tp; ++i) gp.yoff[i] = p.yoff[i];
  gp.X = static_cast<const __nv_bfloat16*>(p.X);
  gp.Y = p.Y;
  for (int i = 0; i < p.tp; ++i) gp.wrows[i] = p.row ? p.w_rows : p.wr[i];
  gp.err = device_error_word();
  if (!gp.err) return TP_ERR_CUDA;
  gp.y_extent = output_extent(p);
  for (int i = 0; i < TP_MAX_TP; ++i) {
    gp.W[i] = static_cast<const uint8_t*>(p.W[i]);
    gp.S[i] = p.wscale[i];
    gp.bias[i] = p.bias[i];
  }
  if (p.row) return dispatch_fp8_mt<TP_ACT_NONE, true>(gp, L);
  switch (p.act) {
    case TP_ACT_NONE: return dispatch_fp8_mt<TP_ACT_NONE, false>(gp, L);
    case TP_ACT_GELU_ERF: return dispatch_fp8_mt<TP_ACT_GELU_ERF, false>(gp, L);
    case TP_ACT_SWIGLU: return dispatch_fp8_mt<TP_ACT_SWIGLU, false>(gp, L);
  }
  return TP_ERR_BAD_SHAPE;
}

}  // namespace tpla
