// ssd_cache.cu -- the speculation cache on the device (kernel K-D).
//
// "SSD: drafting and verification on separate GPUs", "What changes in SSD":
// the drafter speculates for the likely verification outcomes ahead of time
// and a correct guess is returned at once; the roadmap names the speculation
// cache.  "tanishqkumar/ssd" summary, module notes: forked recovery tokens are
// chosen with masking to handle cache hits and misses.
//
// Table: open addressing over `capacity` (a power of two) slots, linear
// probing bounded by the capacity, exact 64-bit key compare.  Key layout:
// b << 40 | position << 32 | token.  Slot choice: the splitmix64 finaliser
// (Steele, Lea & Flood 2014) of the key, masked to the capacity.  An empty
// slot holds all-ones, which no valid key can equal (token < 2^31).
//
// Insert is two kernels so that duplicates resolve deterministically: claim
// (CAS the key into a slot, then atomicMax a 64-bit sequence number
// call << 32 | input index into the slot's winner word) and write (the input
// whose sequence number won copies its payload).  The last duplicate, in
// input order and across calls, wins.  The call number lives on the device:
// both kernels read the count of finished inserts, and the write kernel's
// last CTA (atomic ticket, no waiting) advances it, so an insert captured in
// a CUDA graph draws a fresh call number on every replay.
#include <stdint.h>

#include "ssd_cache.cuh"
#include "ssd_device.cuh"
#include "ssd_layout.h"

namespace ssd {

__device__ __forceinline__ bool insert_key(const InsertArgs& a, int i, unsigned long long& key) {
  int b, pos, tok;
  if (a.b) {
    b = a.b[i];
    pos = a.pos[i];
    tok = a.tok[i];
  } else {
    tok = a.fork_tok[i];
    int bj = i / a.f;
    b = bj / a.P;
    pos = bj % a.P;
  }
  return make_key(b, pos, tok, key);
}

__device__ __forceinline__ unsigned long long call_seq(const CacheView& c) {
  return (__ldcg(c.calls) + 1ull) << 32;
}

__global__ void cache_claim_kernel(CacheView c, InsertArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.n) return;
  const unsigned long long seq = call_seq(c);
  unsigned long long key;
  if (!insert_key(a, i, key)) return;
  const unsigned mask = static_cast<unsigned>(c.capacity - 1);
  unsigned h = static_cast<unsigned>(splitmix64(key)) & mask;
  for (int probe = 0; probe < c.capacity; ++probe) {
    unsigned long long prev = atomicCAS(&c.keys[h], kEmptyKey, key);
    if (prev == kEmptyKey || prev == key) {
      atomicMax(&c.winner[h], seq | static_cast<unsigned long long>(i));
      return;
    }
    h = (h + 1) & mask;
  }
  atomicOr(c.err, 0x8);  // table full: the entry is dropped
}

__global__ void cache_write_kernel(CacheView c, InsertArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  const unsigned long long seq = call_seq(c);  // read before this CTA's ticket
  unsigned long long key;
  if (i < a.n && insert_key(a, i, key)) {
    const int s = find_slot(c, key);
    if (s >= 0 && c.winner[s] == (seq | static_cast<unsigned long long>(i))) {
      const int32_t* src = a.payload + static_cast<int64_t>(i) * c.depth;
      int32_t* dst = c.payload + static_cast<int64_t>(s) * c.depth;
      for (int d = 0; d < c.depth; ++d) dst[d] = src[d];
    }
  }
  // the last CTA to finish advances the call counter (every CTA has read it)
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(c.done, 1u) == gridDim.x - 1) {
      *c.done = 0u;
      *c.calls = seq >> 32;
      __threadfence();
    }
  }
}

__global__ void cache_lookup_kernel(CacheView c, LookupArgs a) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.n) return;
  int b, pos, tok;
  if (a.b) {
    b = a.b[i];
    pos = a.pos[i];
    tok = a.tok[i];
  } else {
    b = i;
    pos = a.accept_len[i];
    tok = (pos >= 0 && pos <= a.k) ? a.out_tok[static_cast<int64_t>(i) * (a.k + 1) + pos] : -1;
  }
  unsigned long long key;
  int s = -1;
  if (make_key(b, pos, tok, key)) s = find_slot(c, key);
  a.hit[i] = s >= 0 ? 1 : 0;
  int32_t* dst = a.tok_out + static_cast<int64_t>(i) * c.depth;
  const int32_t* src = c.payload + static_cast<int64_t>(s < 0 ? 0 : s) * c.depth;
  for (int d = 0; d < c.depth; ++d) dst[d] = s >= 0 ? src[d] : -1;
}

cudaError_t launch_cache_claim(const CacheView& c, const InsertArgs& a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  cache_claim_kernel<<<(a.n + 255) / 256, 256, 0, s>>>(c, a);
  return cudaGetLastError();
}

cudaError_t launch_cache_write(const CacheView& c, const InsertArgs& a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  cache_write_kernel<<<(a.n + 255) / 256, 256, 0, s>>>(c, a);
  return cudaGetLastError();
}

cudaError_t launch_cache_lookup(const CacheView& c, const LookupArgs& a, cudaStream_t s) {
  if (a.n <= 0) return cudaSuccess;
  cache_lookup_kernel<<<(a.n + 255) / 256, 256, 0, s>>>(c, a);
  return cudaGetLastError();
}

}  // namespace ssd
