// moe_static.cu — moe_forward for callers that cannot allocate device memory.
//
// Some callers can't call cudaMalloc: serving engines that reserve all device
// memory at start-up and forbid allocation afterwards, and plain-C hosts that
// link only this library and have no device allocator of their own.  This
// entry point needs no workspace from them: the intermediates live in one
// file-scope device array of MOE_STATIC_SCRATCH_BYTES that every GPU using
// this library holds until the process exits.
//
// When the array is reserved: this translation unit has no kernels, so under
// the CUDA runtime's lazy module loading (the default) its module is loaded,
// and the array reserved on a device, by the address lookup inside the first
// moe_forward_static call on that device.  A caller that reserves device
// memory up front must make that first call before it does so.  A lookup that
// fails (for example for lack of memory) is not remembered: the next call on
// that device tries again.
//
// The array is shared by every call: calls whose work overlaps on the GPU
// (two streams, or two host threads) race on it and must be serialised by the
// caller.  Nothing in it has to start at zero — each call writes every
// intermediate before reading it, and the first kernel of the call clears
// dev_status.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/moe.h"

namespace {

__device__ __align__(256) unsigned char g_moe_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_moe_scratch, looked up while that device is current
// (in host code the symbol is only a stand-in).  Only a successful lookup is
// kept; the mutex orders concurrent first calls on one device.
struct ScratchAddress {
  std::mutex mu;
  void* ptr = nullptr;
};
ScratchAddress g_scratch_addr[kMaxDevices];

void* scratch_address(int dev) {
  ScratchAddress& a = g_scratch_addr[dev];
  std::lock_guard<std::mutex> lock(a.mu);
  if (a.ptr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_scratch) != cudaSuccess) {
      cudaGetLastError();   // do not leave the failure as the thread's sticky error
      return nullptr;
    }
    a.ptr = p;
  }
  return a.ptr;
}

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
  void* scratch = scratch_address(dev);
  if (scratch == nullptr) return MOE_ERR_CUDA;
  return moe_forward(shape, x, w13, w2, topk_ids, topk_w, scales, out, scratch,
                     MOE_STATIC_SCRATCH_BYTES, dev_status, stream);
}
