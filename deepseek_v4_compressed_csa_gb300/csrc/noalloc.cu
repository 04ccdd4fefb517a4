// csa_index_topk_static: the decode indexer with its scratch memory in a
// fixed-size array that lives in the library image, for callers that cannot
// allocate device memory (see include/csa.h).  Same kernels and results as
// csa_index_topk; only the origin of the scratch buffer differs.
#include <atomic>

#include "kernels.h"

namespace {

// Scratch shared by every call on a device.  Held by each GPU that loads the
// library until the process exits.
constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB
__device__ __align__(256) unsigned char g_csa_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once per
// device (host code cannot use the array's name as a device pointer).
cudaError_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    e = cudaGetSymbolAddress(&p, g_csa_static_scratch);
    if (e != cudaSuccess || p == nullptr) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" size_t csa_static_scratch_bytes(void) { return kStaticScratchBytes; }

extern "C" csa_status csa_index_topk_static(const csa_layer* layer, const void* iq, const void* iw, int B,
                                            const void* ikeys, int cap, const int32_t* n_rows, const int32_t* pos,
                                            const float* inv_freq, int32_t* sel, int32_t* n_sel, int32_t* err,
                                            void* stream) {
  size_t need = 0;
  csa_status st = csa_workspace_size(layer, CSA_OP_INDEX_TOPK, B, 1, cap, &need);
  if (st != CSA_OK) return st;
  if (need > kStaticScratchBytes) return CSA_ERR_WORKSPACE;
  void* ws = nullptr;
  if (static_scratch(&ws) != cudaSuccess) return CSA_ERR_CUDA;
  return csa_index_topk(layer, iq, iw, B, ikeys, cap, n_rows, pos, inv_freq, sel, n_sel, ws, kStaticScratchBytes,
                        err, stream);
}
