// sync.cuh -- mbarrier helpers with BOUNDED waits.
//
// Every spin-wait in the library's kernels goes through mbar_wait_bounded:
// it polls mbarrier.try_wait and gives up after `limit_ns` nanoseconds of
// %globaltimer (or when a CTA-wide abort flag is raised), returning false.
// The caller then records the failure in the device error word (read by
// tp_device_status) and unwinds: it never traps.
#pragma once

#include <cstdint>

namespace tpla {

// Default limit for pipeline waits: far above any legitimate wait (a whole
// GEMM of the largest supported shape takes milliseconds).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

enum : uint32_t {
  kErrTimeoutProducer = 1u << 0,
  kErrTimeoutMma = 1u << 1,
  kErrTimeoutEpilogue = 1u << 2,
  kErrTimeoutDrain = 1u << 3,
  kErrSelftest = 1u << 4,
  kErrTimeoutConvert = 1u << 5,
  kErrIndexCheck = 1u << 6,  // checked builds: an index check failed
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed, or give up after
// limit_ns, or as soon as *abort (if given) becomes non-zero.  Returns true on
// completion.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs,
                                                  const volatile int* abort = nullptr) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (abort && *abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
}

__device__ __forceinline__ void report_error(unsigned int* err, uint32_t code) {
  if (err) atomicOr(err, code);
}

// Index checks of checked builds (-DTPLA_CHECKED): TP_CHECK(err, cond) is true
// when cond holds; otherwise it records kErrIndexCheck in the device error
// word and is false, and the caller skips the access.  In release builds it
// is the constant true and compiles away.  (No assert or trap: a failed check
// leaves the context usable and surfaces as TP_ERR_DEVICE_CHECK.)
#ifdef TPLA_CHECKED
#define TP_CHECK(err, cond) ((cond) || (::tpla::report_error((err), ::tpla::kErrIndexCheck), false))
#else
#define TP_CHECK(err, cond) true
#endif

}  // namespace tpla
