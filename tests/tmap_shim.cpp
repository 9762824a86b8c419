// Test shim: the tensor-map cache of tmap_cache.h, compiled here as plain C++
// with a stand-in encoder, so the CPU tests can check hits, misses and the
// replacement order without a GPU.
#include "tmap_cache.h"

namespace {
g10::TmapCache g_cache;
int g_encodes = 0;
int g_fail = 0;
}  // namespace

extern "C" {

void tmap_reset() {
  g_cache = g10::TmapCache();
  g_encodes = 0;
}

void tmap_fail_next(int f) { g_fail = f; }

// Look up the map of a description; the stand-in encoder writes the
// description's base address and a serial number into the map's first bytes.
// Returns 1 on success and writes (base, serial) to out.
int tmap_get(uint64_t base, const uint64_t* dims, const uint64_t* strides, const uint32_t* box, int dtype,
             int swizzle, int promo, uint64_t* out) {
  const g10::TmapDesc d = g10::tmap_desc(reinterpret_cast<const void*>(base), dims, strides, box, dtype, swizzle,
                                         promo);
  CUtensorMap m;
  const bool ok = g_cache.get(d, &m, [](const g10::TmapDesc& k, CUtensorMap* dst) {
    if (g_fail) return false;
    uint64_t words[2] = {k.base, static_cast<uint64_t>(++g_encodes)};
    std::memcpy(dst, words, sizeof(words));
    return true;
  });
  if (!ok) return 0;
  std::memcpy(out, &m, 2 * sizeof(uint64_t));
  return 1;
}

void tmap_stats(uint64_t* hits, uint64_t* misses, int* encodes) {
  *hits = g_cache.hits;
  *misses = g_cache.misses;
  *encodes = g_encodes;
}

}  // extern "C"
