// csa_index_topk_static: the decode indexer with its scratch memory in a
// fixed-size array that lives in the library image, for callers that cannot
// allocate device memory (see include/csa.h).  Same kernels and results as
// csa_index_topk; only the origin of the scratch buffer differs.
#include <cudaTypedefs.h>

#include "kernels.h"
#include "scratch_cache.h"

namespace {

// Scratch shared by every call on a device.  Held by each GPU that loads the
// library until the process exits.
constexpr size_t kStaticScratchBytes = 4u << 20;  // 4 MiB
__device__ __align__(256) unsigned char g_csa_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
csa::ContextAddressCache<kMaxDevices> g_scratch_addr;

// Unique id of the calling thread's current CUDA context, or 0 if there is none (yet) or the driver entry points
// cannot be had.  Taken through the runtime's driver entry-point query, so the library needs no libcuda link.
unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static bool resolved = false;
  if (!resolved) {
    void* f0 = nullptr;
    void* f1 = nullptr;
    cudaDriverEntryPointQueryResult q0, q1;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f0, 4000, cudaEnableDefault, &q0) == cudaSuccess &&
        q0 == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
        q1 == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f0);
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f1);
    }
    resolved = true;
  }
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current device's context.  Host code cannot use the array's name as
// a device pointer, so the address is looked up with cudaGetSymbolAddress and cached per device together with the
// id of the context it belongs to; after a device reset the context id changes and the address is looked up again.
cudaError_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = nullptr;
  if (g_scratch_addr.lookup(dev, current_context_id(), &p)) {
    *out = p;
    return cudaSuccess;
  }
  e = cudaGetSymbolAddress(&p, g_csa_static_scratch);  // makes the device's primary context current if needed
  if (e != cudaSuccess) return e;
  if (p == nullptr) return cudaErrorInvalidSymbol;
  g_scratch_addr.store(dev, current_context_id(), p);
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
