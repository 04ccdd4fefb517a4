// Host-only check of csa::ContextAddressCache (the per-device, per-context cache of the static scratch array's
// device address).  Built and run by tests/test_scratch_cache.py with g++; no GPU involved.  Exits 0 when every
// check holds, else prints the failed line and exits 1.
#include <cstdio>

#include "../deepseek_v4_compressed_csa_gb300/csrc/scratch_cache.h"

#define CHECK(c)                                     \
  do {                                               \
    if (!(c)) {                                      \
      std::printf("check failed, line %d: %s\n", __LINE__, #c); \
      return 1;                                      \
    }                                                \
  } while (0)

int main() {
  csa::ContextAddressCache<4> cache;
  int a_obj = 0, b_obj = 0;
  void* a = &a_obj;
  void* b = &b_obj;
  void* out = nullptr;
  CHECK(!cache.lookup(0, 11, &out));           // empty
  cache.store(0, 11, a);
  CHECK(cache.lookup(0, 11, &out) && out == a);  // same device, same context: hit
  CHECK(!cache.lookup(1, 11, &out));           // another device has its own entry
  CHECK(!cache.lookup(0, 12, &out));           // the context was re-created (reset): miss
  cache.store(0, 12, b);                        // looked up again in the new context
  CHECK(cache.lookup(0, 12, &out) && out == b);
  CHECK(!cache.lookup(0, 11, &out));           // the old context's address is gone for good
  CHECK(!cache.lookup(0, 0, &out));            // no current context: never a hit
  cache.store(0, 0, a);                         // an address without a known context is not kept
  CHECK(!cache.lookup(0, 12, &out));
  cache.store(2, 5, a);
  cache.store(2, 5, nullptr);                   // a null address clears the entry
  CHECK(!cache.lookup(2, 5, &out));
  cache.store(-1, 5, a);                        // devices outside the table are ignored
  cache.store(4, 5, a);
  CHECK(!cache.lookup(-1, 5, &out) && !cache.lookup(4, 5, &out));
  cache.store(3, 7, b);
  CHECK(cache.lookup(3, 7, &out) && out == b);
  std::printf("ok\n");
  return 0;
}
