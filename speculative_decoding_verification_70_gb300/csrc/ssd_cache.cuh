// ssd_cache.cuh -- key layout, slot hash and bounded probe of the
// speculation cache (open addressing over a power-of-two table, exact
// 64-bit key compare), shared by the cache kernels and by the draw kernel
// that looks up each row's realised outcome.
#pragma once

#include <stdint.h>

#include "ssd_layout.h"

namespace ssd {

constexpr unsigned long long kEmptyKey = 0xffffffffffffffffull;

__device__ __forceinline__ unsigned long long splitmix64(unsigned long long z) {
  z ^= z >> 30;
  z *= 0xbf58476d1ce4e5b9ull;
  z ^= z >> 27;
  z *= 0x94d049bb133111ebull;
  z ^= z >> 31;
  return z;
}

__device__ __forceinline__ bool make_key(int b, int pos, int tok, unsigned long long& key) {
  if (b < 0 || b >= (1 << 24) || pos < 0 || pos >= 256 || tok < 0) return false;
  key = (static_cast<unsigned long long>(b) << 40) | (static_cast<unsigned long long>(pos) << 32) |
        static_cast<unsigned long long>(static_cast<uint32_t>(tok));
  return true;
}

// Slot holding `key`, or -1 (bounded probe).
__device__ __forceinline__ int find_slot(const CacheView& c, unsigned long long key) {
  const unsigned mask = static_cast<unsigned>(c.capacity - 1);
  unsigned h = static_cast<unsigned>(splitmix64(key)) & mask;
  for (int probe = 0; probe < c.capacity; ++probe) {
    unsigned long long k = c.keys[h];
    if (k == key) return static_cast<int>(h);
    if (k == kEmptyKey) return -1;
    h = (h + 1) & mask;
  }
  return -1;
}

// The realised outcome of batch row b: key (b, pos, tok); hit flag and the
// entry's depth payload tokens (-1 on a miss).
__device__ __forceinline__ void cache_lookup_one(const CacheView& c, int b, int pos, int tok,
                                                 int32_t* hit, int32_t* tok_out) {
  unsigned long long key;
  int s = -1;
  if (make_key(b, pos, tok, key)) s = find_slot(c, key);
  *hit = s >= 0 ? 1 : 0;
  const int32_t* src = c.payload + static_cast<int64_t>(s < 0 ? 0 : s) * c.depth;
  for (int d = 0; d < c.depth; ++d) tok_out[d] = s >= 0 ? src[d] : -1;
}

}  // namespace ssd
