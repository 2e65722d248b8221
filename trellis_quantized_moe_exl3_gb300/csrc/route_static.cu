// Routing without a caller-supplied workspace (exl3_moe_route_static).
//
// The pages have no counterpart: this is a convenience for callers that
// cannot allocate device memory.  It runs the same routing kernels as
// exl3_moe_route; only the source of their scratch differs.  The scratch is
// one file-scope device array of EXL3_ROUTE_STATIC_SCRATCH_BYTES, which every
// device that loads this library keeps until the process exits.
#include <mutex>

#include "internal.h"

namespace exl3 {
namespace {

static __device__ __align__(256) unsigned char g_route_scratch[EXL3_ROUTE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mutex;
void* g_addr[kMaxDevices] = {};

// Device address of g_route_scratch on the current device.  In host code the
// array's name is only a host-side shadow, so the address has to come from
// the runtime, once per device, with that device current.  The address is
// cached by device index, which assumes every call runs in the device's
// primary context (the runtime's default) for the life of the process: after
// cudaDeviceReset, or under a context the caller made current itself, the
// cached address would belong to a module that is gone.
cudaError_t static_scratch(void** out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_addr_mutex);
  if (!g_addr[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess) return err;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace exl3

using namespace exl3;

extern "C" exl3_status exl3_moe_route_static(const float* logits, int T, int E, int top_k,
                                             int32_t* ids, float* w, int32_t* seg_offsets,
                                             int32_t* seg_pairs, void* stream) {
  if (T < 0 || E < 1 || E > kMaxExperts) return EXL3_ERR_SHAPE;
  if (top_k < 1 || top_k > kMaxTopK || top_k > E) return EXL3_ERR_ARG;
  if (!seg_offsets) return EXL3_ERR_ARG;
  if (T > 0 && (!logits || !ids || !w || !seg_pairs)) return EXL3_ERR_ARG;
  if (route_scratch_bytes(T, E, top_k) > (size_t)EXL3_ROUTE_STATIC_SCRATCH_BYTES)
    return EXL3_ERR_SHAPE;
  void* scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) return EXL3_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RouteBuffers rb{};
  route_carve(scratch, T, E, top_k, &rb);
  rb.ids = ids; rb.w = w; rb.seg_offsets = seg_offsets; rb.seg_pairs = seg_pairs;
  // The array keeps the previous call's contents; the routing kernel clears
  // the status word, and every other scratch word is written before it is read.
  if (launch_route(logits, T, E, top_k, rb, st) != cudaSuccess) return EXL3_ERR_CUDA;
  return EXL3_OK;
}
