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

// Insert of one entry by one thread: claim a slot for `key` (bounded linear
// probe), record the sequence number call << 32 | input index in the slot's
// winner word and copy the payload.  For callers whose keys are distinct
// within the call (so this entry's number is the largest the slot has
// seen): the forks of one verify call.  A full table drops the entry and
// sets SSD_DEVERR_CACHE_FULL.  The first 8 payload words are loaded before
// the claim, so the two round trips overlap.
__device__ __forceinline__ void cache_insert_unique(const CacheView& c, unsigned long long key,
                                                    unsigned long long seq_idx,
                                                    const int32_t* src) {
  int32_t head[8];
#pragma unroll
  for (int d = 0; d < 8; ++d)
    if (d < c.depth) head[d] = src[d];
  const unsigned mask = static_cast<unsigned>(c.capacity - 1);
  unsigned h = static_cast<unsigned>(splitmix64(key)) & mask;
  for (int probe = 0; probe < c.capacity; ++probe) {
    const unsigned long long prev = atomicCAS(&c.keys[h], kEmptyKey, key);
    if (prev == kEmptyKey || prev == key) {
      atomicMax(&c.winner[h], seq_idx);
      int32_t* dst = c.payload + static_cast<int64_t>(h) * c.depth;
#pragma unroll
      for (int d = 0; d < 8; ++d)
        if (d < c.depth) dst[d] = head[d];
      for (int d = 8; d < c.depth; ++d) dst[d] = src[d];
      return;
    }
    h = (h + 1) & mask;
  }
  atomicOr(c.err, 0x8);
}

// The realised outcome of batch row b: key (b, pos, tok); hit flag and the
// entry's depth payload tokens (-1 on a miss).  The home slot's key and its
// first 8 payload words are loaded together (one round trip when the key
// sits in its home slot, the common case).
__device__ __forceinline__ void cache_lookup_one(const CacheView& c, int b, int pos, int tok,
                                                 int32_t* hit, int32_t* tok_out) {
  unsigned long long key;
  int s = -1;
  int32_t head[8];
  if (make_key(b, pos, tok, key)) {
    const unsigned mask = static_cast<unsigned>(c.capacity - 1);
    unsigned h = static_cast<unsigned>(splitmix64(key)) & mask;
    const int32_t* home = c.payload + static_cast<int64_t>(h) * c.depth;
#pragma unroll
    for (int d = 0; d < 8; ++d)
      if (d < c.depth) head[d] = home[d];
    const unsigned long long k0 = c.keys[h];
    if (k0 == key) {
      s = static_cast<int>(h);
    } else if (k0 != kEmptyKey) {
      s = find_slot(c, key);
      const int32_t* src = c.payload + static_cast<int64_t>(s < 0 ? 0 : s) * c.depth;
#pragma unroll
      for (int d = 0; d < 8; ++d)
        if (d < c.depth) head[d] = src[d];
    }
  }
  *hit = s >= 0 ? 1 : 0;
  const int32_t* src = c.payload + static_cast<int64_t>(s < 0 ? 0 : s) * c.depth;
#pragma unroll
  for (int d = 0; d < 8; ++d)
    if (d < c.depth) tok_out[d] = s >= 0 ? head[d] : -1;
  for (int d = 8; d < c.depth; ++d) tok_out[d] = s >= 0 ? src[d] : -1;
}

}  // namespace ssd
