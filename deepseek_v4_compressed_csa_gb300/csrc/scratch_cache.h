// Host-side cache of a device address per (device, CUDA context).
//
// The device address of a file-scope __device__ array is fixed only for the
// lifetime of the context the module was loaded into.  If the context is torn
// down and created again (cudaDeviceReset, then any runtime call), the module
// is loaded again and the array may move; an address cached per device alone
// would then point at unmapped memory.  Entries here therefore record the
// unique id of the context the address was looked up in (cuCtxGetId), and a
// lookup under any other id misses, so the caller resolves the address again.
//
// Plain C++ (no CUDA headers), so its logic is unit-tested on a machine
// without a GPU.  Thread-safe: one mutex around the table.
#pragma once
#include <mutex>

namespace csa {

template <int kMaxDevices>
class ContextAddressCache {
 public:
  // The address cached for `dev` if it was looked up under context `ctx_id`.  ctx_id 0 (no context known)
  // never hits.
  bool lookup(int dev, unsigned long long ctx_id, void** out) {
    if (dev < 0 || dev >= kMaxDevices || ctx_id == 0) return false;
    std::lock_guard<std::mutex> g(mu_);
    const Entry& e = table_[dev];
    if (e.ctx_id != ctx_id || e.addr == nullptr) return false;
    *out = e.addr;
    return true;
  }
  // Record `addr` for `dev` under context `ctx_id`, replacing what an earlier context left.  ctx_id 0 or a null
  // address clears the entry instead (nothing is cached that a later lookup could not validate).
  void store(int dev, unsigned long long ctx_id, void* addr) {
    if (dev < 0 || dev >= kMaxDevices) return;
    std::lock_guard<std::mutex> g(mu_);
    if (ctx_id == 0 || addr == nullptr) {
      table_[dev] = Entry{};
      return;
    }
    table_[dev] = Entry{ctx_id, addr};
  }

 private:
  struct Entry {
    unsigned long long ctx_id = 0;
    void* addr = nullptr;
  };
  std::mutex mu_;
  Entry table_[kMaxDevices];
};

}  // namespace csa
