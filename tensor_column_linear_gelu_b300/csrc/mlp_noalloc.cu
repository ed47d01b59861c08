// mlp_noalloc.cu -- tp_mlp_block_noalloc: the FFN block for callers that cannot
// allocate device memory.
//
// tp_mlp_block needs a [M, d_ff] workspace for the intermediate activation h.
// Some callers cannot provide one: their device memory is owned by another
// allocator (a serving engine that reserves the GPU at start-up, a plugin
// whose host application hands out no device memory), or they run on a path
// where cudaMalloc is not allowed because it can synchronise the device and
// stall unrelated work.  For them the workspace lives here, in a fixed buffer
// that is part of the library image: every GPU that loads the library holds
// it until the process exits.  This call allocates nothing.
#include <cstdint>

#include "internal.h"

namespace tpla {
namespace {

// The shared workspace.  In host code this name is only a stand-in for the
// device object: host code must never hand it to a kernel; it passes the
// device address that scratch_address() looks up instead.
static __device__ __align__(256) unsigned char g_mlp_scratch[TP_NOALLOC_SCRATCH_BYTES];

// Device address of g_mlp_scratch on the current device, looked up on every
// call with that device current (a cheap host query).  Nothing is cached, so
// an address can never outlive the context it belongs to (a device reset, a
// context torn down and re-created).  The very first lookup on a device may
// load the library's device code there; that first call must come before any
// stream capture on the device.
void* scratch_address(tp_status* status) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_mlp_scratch) != cudaSuccess || p == nullptr) {
    *status = TP_ERR_CUDA;
    return nullptr;
  }
  return p;
}

}  // namespace
}  // namespace tpla

extern "C" tp_status tp_mlp_block_noalloc(int tp, int64_t M, int64_t d_model, int64_t d_ff,
                                          tp_act act, tp_dtype xdt, const void* X,
                                          const void* const* w1_shards,
                                          const float* const* b1_shards,
                                          const void* const* w2_shards, const float* b2,
                                          void* Y, tp_dtype ydt, tp_stream_t stream) {
  if (xdt != TP_F32 && xdt != TP_BF16) return TP_ERR_DTYPE;
  if (M < 0 || d_model <= 0 || d_ff <= 0) return TP_ERR_BAD_SHAPE;
  // h is [M, d_ff] in the input dtype; it must fit the fixed buffer.
  const int64_t es = (xdt == TP_F32) ? 4 : 2;
  if (M > (int64_t)TP_NOALLOC_SCRATCH_BYTES / es / d_ff) return TP_ERR_UNSUPPORTED;
  tp_status st = TP_OK;
  void* h = tpla::scratch_address(&st);
  if (!h) return st;
  // The column kernel writes every element of h[0:M, 0:d_ff] before the row
  // kernel (later in stream order) reads it, so nothing left in the buffer by
  // an earlier call is ever read and nothing needs clearing.
  return tp_mlp_block(tp, M, d_model, d_ff, act, xdt, X, w1_shards, b1_shards, w2_shards, b2, h,
                      Y, ydt, stream);
}
