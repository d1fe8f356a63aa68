// moe_static.cu — moe_forward for callers that cannot allocate device memory.
//
// Some callers can't call cudaMalloc: code that issues the layer while a
// stream is being captured into a CUDA graph in the global capture mode (the
// runtime rejects cudaMalloc there), serving engines that reserve all device
// memory at start-up and forbid allocation afterwards, and plain-C hosts that
// link only this library and have no device allocator of their own.  This
// entry point needs no workspace from them: the intermediates live in one
// file-scope device array of MOE_STATIC_SCRATCH_BYTES, which the CUDA loader
// reserves on every GPU that loads this library and which is held until the
// process exits.
//
// The array is shared by every call: calls whose work overlaps on the GPU
// (two streams, or two host threads) race on it and must be serialised by the
// caller.  Nothing in it has to start at zero — each call writes every
// intermediate before reading it, and the index build clears dev_status.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"

namespace {

__device__ __align__(256) unsigned char g_moe_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_moe_scratch, looked up once per device while that
// device is current (in host code the symbol is only a stand-in).
struct ScratchAddress {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};
ScratchAddress g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" MOE_API moe_status moe_forward_static(const moe_shape* shape, const void* x,
                                                 const void* w13, const void* w2,
                                                 const int32_t* topk_ids, const float* topk_w,
                                                 const moe_scales* scales, void* out,
                                                 int32_t* dev_status, void* stream) {
  moe_workspace_layout layout;
  const moe_status st = moe_plan(shape, nullptr, &layout);
  if (st != MOE_OK) return st;
  if (layout.total_bytes > MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  ScratchAddress& a = g_scratch_addr[dev];
  std::call_once(a.once, [&a] { a.err = cudaGetSymbolAddress(&a.ptr, g_moe_scratch); });
  if (a.err != cudaSuccess || a.ptr == nullptr) return MOE_ERR_CUDA;
  return moe_forward(shape, x, w13, w2, topk_ids, topk_w, scales, out, a.ptr,
                     MOE_STATIC_SCRATCH_BYTES, dev_status, stream);
}
