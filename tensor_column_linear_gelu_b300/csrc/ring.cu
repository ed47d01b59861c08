// ring.cu -- the all-reduce-faithful row-parallel mode: the per-shard partials,
// held in the wire dtype, are added in the order a ring all-reduce adds them.
//
// "Tensor parallel serving" ("Communication cost") describes the ring
// all-reduce: the message is cut into p chunks and, in the reduce-scatter,
// each chunk's running sum travels once around the ring, picking up one rank's
// partial per hop; the all-gather then copies the finished chunks.
// RowParallelLinear ("Understanding Tensor Parallelism for Multi-GPU LLM
// Serving") all-reduces each rank's local partial with SUM and adds the bias
// afterwards.  This kernel does that arithmetic on one GPU:
//   * the flattened [M, N] message of L = M*N elements is cut into p chunks,
//     chunk c = elements [c*L/p, (c+1)*L/p) (integer division);
//   * chunk c's sum starts with rank c's partial and adds ranks c+1, ...,
//     c+p-1 (mod p), one per hop, in fp32, rounded to the wire dtype after
//     every hop (each hop transmits the running sum in that dtype);
//   * the bias is added once at the end in fp32 and the result is rounded
//     once to the output dtype.
// Each partial is read once and Y written once, so the kernel is bound by
// HBM bandwidth: a thread takes 8 consecutive elements (16-byte loads of
// every partial, one 16-byte store) when the shapes allow, else one element.
#include <algorithm>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace tpla {
namespace {

template <typename T>
__device__ __forceinline__ float load_f(const T* p);
template <>
__device__ __forceinline__ float load_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float load_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));
}

template <typename T>
__device__ __forceinline__ float to_wire(float x);
template <>
__device__ __forceinline__ float to_wire<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_wire<__nv_bfloat16>(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

template <typename TW>
__global__ void ring_reduce_kernel(const TW* __restrict__ parts, int64_t L, int64_t N, int tp,
                                   const float* __restrict__ bias, void* Y, int64_t ldy,
                                   int ydt) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < L; e += stride) {
    // chunk of e: the c with c*L/tp <= e < (c+1)*L/tp
    const int c = (int)(((e + 1) * tp - 1) / L);
    float acc = load_f(parts + (int64_t)c * L + e);
    for (int s = 1; s < tp; ++s) {
      int r = c + s;
      if (r >= tp) r -= tp;
      acc = to_wire<TW>(acc + load_f(parts + (int64_t)r * L + e));
    }
    const int64_t m = e / N;
    const int64_t n = e - m * N;
    if (bias) acc += __ldg(bias + n);
    store_out(Y, ydt, m * ldy + n, acc);
  }
}

// Chunk starts c*L/tp for c = 0 .. tp (host-computed).
struct RingBounds {
  int64_t start[TP_MAX_TP + 1];
};

// 8 elements per thread.  Requires N % 8 == 0, ldy % 8 == 0 and 16-byte
// aligned partials and Y, so a vector never leaves its row; a vector that
// straddles a chunk boundary is done element by element.
template <typename TW>
__global__ void ring_reduce_vec8_kernel(const TW* __restrict__ parts, int64_t L, int64_t N, int tp,
                                        const RingBounds bnd, const float* __restrict__ bias,
                                        void* Y, int64_t ldy, int ydt) {
  constexpr int E = 16 / sizeof(TW);  // elements per 16-byte load
  const int64_t nvec = L / 8;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += stride) {
    const int64_t e0 = v * 8;
    int c = 0;
    while (c + 1 < tp && bnd.start[c + 1] <= e0) ++c;
    float acc[8];
    if (e0 + 8 <= bnd.start[c + 1]) {
      // all 8 in chunk c: start at rank c, then c+1, ... (mod tp)
      uint4 pv[TP_MAX_TP][8 / E];
#pragma unroll
      for (int s = 0; s < TP_MAX_TP; ++s) {
        if (s >= tp) break;
        int r = c + s;
        if (r >= tp) r -= tp;
        const uint4* src = reinterpret_cast<const uint4*>(parts + (int64_t)r * L + e0);
#pragma unroll
        for (int j = 0; j < 8 / E; ++j) pv[s][j] = __ldg(src + j);
      }
#pragma unroll
      for (int s = 0; s < TP_MAX_TP; ++s) {
        if (s >= tp) break;
        float f[8];
        if constexpr (E == 8) {
          unpack_bf16x8(pv[s][0], f);
        } else {
          unpack_f32x4(pv[s][0], f);
          unpack_f32x4(pv[s][1], f + 4);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = (s == 0) ? f[j] : to_wire<TW>(acc[j] + f[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t e = e0 + j;
        const int cj = (e >= bnd.start[c + 1]) ? c + 1 : c;
        float a = load_f(parts + (int64_t)cj * L + e);
        for (int s = 1; s < tp; ++s) {
          int r = cj + s;
          if (r >= tp) r -= tp;
          a = to_wire<TW>(a + load_f(parts + (int64_t)r * L + e));
        }
        acc[j] = a;
      }
    }
    const int64_t m = e0 / N;
    const int64_t n = e0 - m * N;
    if (bias) {
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] += __ldg(bias + n + j);
    }
    store_row8(Y, ydt, m * ldy, n, 8, acc);
  }
}

}  // namespace

tp_status launch_ring_reduce(int tp, int64_t M, int64_t N, const void* parts, int wire_dt,
                             const float* bias, void* Y, int64_t ldy, int ydt,
                             cudaStream_t stream) {
  const int64_t L = M * N;
  if (L == 0) return TP_OK;
  const int threads = 256;
  const int64_t ye = ydt == TP_F32 ? 4 : 2;
  const bool vec = N % 8 == 0 && ldy % 8 == 0 && (reinterpret_cast<uintptr_t>(parts) & 15u) == 0 &&
                   (reinterpret_cast<uintptr_t>(Y) & 15u) == 0 && (L * (wire_dt == TP_F32 ? 4 : 2)) % 16 == 0 &&
                   (ldy * ye) % 16 == 0;
  if (vec) {
    RingBounds bnd{};
    for (int c = 0; c <= tp; ++c) bnd.start[c] = (int64_t)c * L / tp;
    const int64_t want = (L / 8 + threads - 1) / threads;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 8));
    if (wire_dt == TP_BF16)
      ring_reduce_vec8_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(parts), L, N, tp, bnd, bias, Y, ldy, ydt);
    else
      ring_reduce_vec8_kernel<float><<<grid, threads, 0, stream>>>(
          static_cast<const float*>(parts), L, N, tp, bnd, bias, Y, ldy, ydt);
    return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
  }
  const int64_t want = (L + threads - 1) / threads;
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)sm_count() * 8));
  if (wire_dt == TP_BF16)
    ring_reduce_kernel<__nv_bfloat16><<<grid, threads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(parts), L, N, tp, bias, Y, ldy, ydt);
  else
    ring_reduce_kernel<float><<<grid, threads, 0, stream>>>(static_cast<const float*>(parts), L,
                                                            N, tp, bias, Y, ldy, ydt);
  return cudaGetLastError() == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}

}  // namespace tpla
