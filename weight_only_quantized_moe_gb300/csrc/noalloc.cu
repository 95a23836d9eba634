// noalloc.cu - a forward for callers that may not allocate device memory.
//
// qmoe_forward needs a caller-provided workspace.  Some callers cannot
// provide one at call time: an inference engine plugin whose device memory
// plan is fixed before execution and that receives no scratch buffer, or a
// latency-critical serving loop whose allocator must not be entered (cudaMalloc
// can synchronise the device, and pool allocators can grow or fragment).  This
// entry point runs the same forward with its scratch in a fixed-size device
// array that is part of the library image, so the call itself allocates
// nothing.
#include <mutex>

#include "qmoe.h"
#include "qmoe_internal.h"

namespace {

// Largest workspace the static scratch holds: 64 MiB.  Every GPU that loads
// the library keeps this array resident until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(64) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
void* scratch_on_current_device(qmoe_status* st) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *st = QMOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      *st = QMOE_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *st = QMOE_OK;
  return addr[dev];
}

}  // namespace

extern "C" qmoe_status qmoe_forward_noalloc(const qmoe_layer* layer, const void* x, int64_t M,
                                            const int32_t* topk_ids, const float* topk_weights, int32_t top_k,
                                            void* out, void* stream) {
  const size_t need = qmoe_workspace_size(layer, M, top_k);
  if (need == 0) {
    // the layer or the sizes are invalid: the regular forward's validation
    // names the reason (it fails before it looks at the workspace)
    const qmoe_status st = qmoe::forward_into_workspace(layer, x, M, topk_ids, topk_weights, top_k, out, nullptr, 0,
                                                        static_cast<cudaStream_t>(stream));
    return st != QMOE_OK ? st : QMOE_ERR_INVALID_ARG;
  }
  if (need > kNoAllocScratchBytes) return QMOE_ERR_WORKSPACE;
  qmoe_status st;
  void* scratch = scratch_on_current_device(&st);
  if (scratch == nullptr) return st;
  return qmoe::forward_into_workspace(layer, x, M, topk_ids, topk_weights, top_k, out, scratch,
                                      kNoAllocScratchBytes, static_cast<cudaStream_t>(stream));
}

extern "C" qmoe_status qmoe_read_noalloc_status(void* stream) {
  qmoe_status st;
  void* scratch = scratch_on_current_device(&st);
  if (scratch == nullptr) return st;
  // the status word sits at the start of the workspace, where the forward's
  // first kernel clears it
  return qmoe_read_device_status(scratch, stream);
}
