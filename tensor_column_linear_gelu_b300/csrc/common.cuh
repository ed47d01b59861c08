// common.cuh -- small device helpers shared by the library's kernels.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tpla.h"

namespace tpla {

// Programmatic dependent launch.  launch_dependents lets the next kernel of
// the stream (when it was launched with programmatic stream serialization)
// start its prologue while this one runs; wait blocks until every preceding
// kernel of the stream has completed and its memory writes are visible.  A
// kernel calls wait before it touches memory that an earlier kernel may
// write or read (its activations and its outputs); weights are written only
// by set-up kernels, which never signal early, so they may be read before.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- activations
// Applied in fp32 to the fp32 accumulator (plus bias) before the single
// rounding to the output dtype.

// GELU, exact (erf) form: 0.5 z (1 + erf(z / sqrt 2)).
__device__ __forceinline__ float act_gelu_erf(float z) {
  return 0.5f * z * (1.0f + erff(z * 0.70710678118654752440f));
}

// SiLU: z * sigmoid(z) = z / (1 + e^-z).  The quotient uses the
// approximate division (within 2 ulp; a denominator of 2^126 or more, which
// only z < -87 produces, gives the limit 0): the IEEE-rounded division
// branches to a slow path for such denominators, and that branch serialised
// the decode kernel's single epilogue warp.
__device__ __forceinline__ float act_silu(float z) { return __fdividef(z, 1.0f + expf(-z)); }

// ---------------------------------------------------------------- bf16 bits
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// 8 bf16 (one 16-byte vector) -> 8 fp32, element 0 at the lowest address.
__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float f[8]) {
  f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
  f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
  f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
  f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ void unpack_f32x4(const uint4& v, float f[4]) {
  f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}

// Two fp32 -> packed bf16x2 (round to nearest even), lo at the lower address.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------- loads
// Streaming 16-byte load for data read exactly once (weights): read-only
// path, no L1 allocation, 256-byte L2 prefetch.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}

// 16-byte load through the read-only cache (activations, reused by many warps).
__device__ __forceinline__ uint4 ld_cached16(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------- stores
__device__ __forceinline__ void store_out(void* Y, int ydt, int64_t idx, float v) {
  if (ydt == TP_F32)
    reinterpret_cast<float*>(Y)[idx] = v;
  else
    reinterpret_cast<__nv_bfloat16*>(Y)[idx] = __float2bfloat16_rn(v);
}

}  // namespace tpla
