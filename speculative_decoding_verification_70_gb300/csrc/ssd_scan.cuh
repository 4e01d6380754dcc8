// ssd_scan.cuh -- per-thread streaming statistics (running max, lowest
// argmax, online exponential sum) and small warp helpers shared by the row
// statistics kernels.
#pragma once

#include <math.h>

#include "ssd_device.cuh"
#include "ssd_layout.h"

namespace ssd {

constexpr int kIdxNone = 0x7fffffff;

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// (v1, i1) ranks before (v2, i2): larger value, then lower index.
__device__ __forceinline__ bool ranks_before(float v1, int i1, float v2, int i2) {
  return v1 > v2 || (v1 == v2 && i1 < i2);
}

// Order-preserving map of binary32 to uint32 (for atomicMax on floats).
__device__ __forceinline__ unsigned f2ord(float x) {
  unsigned b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float ord2f(unsigned o) {
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// 64-bit order key of token (z, idx): descending key order is logit
// descending, then index ascending (the order of top-k / top-p filtering and
// of the forked recovery).  -0 and +0 compare equal as logits, so -0 is
// taken as +0.  z must not be NaN.
__device__ __forceinline__ unsigned long long order_key(float z, int idx) {
  const float zc = (z == 0.f) ? 0.f : z;
  return (static_cast<unsigned long long>(f2ord(zc)) << 32) |
         static_cast<unsigned long long>(~static_cast<unsigned>(idx));
}
__device__ __forceinline__ float key_logit(unsigned long long key) {
  return ord2f(static_cast<unsigned>(key >> 32));
}
__device__ __forceinline__ int key_index(unsigned long long key) {
  return static_cast<int>(~static_cast<unsigned>(key & 0xffffffffull));
}

// Per-thread running statistics of the streaming pass.
struct ScanState {
  float m;    // running maximum
  float s;    // running sum of 2^((z - m) c) (with sb: two lanes of a packed pair)
  int idx;    // lowest index attaining m (during the pass: the first index of
              // the first vector attaining m; scan_resolve makes it exact)
  int nan;    // a NaN was seen
  float m2;   // second largest value -- kept only for top-f rows
  float sb;   // second lane of the running sum (pairs of elements)
};

__device__ __forceinline__ void scan_init(ScanState& st) {
  st.m = -INFINITY;
  st.s = 0.f;
  st.idx = kIdxNone;
  st.nan = 0;
  st.m2 = -INFINITY;
  st.sb = 0.f;
}

// The running sum: both lanes.
__device__ __forceinline__ float scan_sum(const ScanState& st) { return st.s + st.sb; }

// Second largest of the first n values of z (n = 1, 4 or 8), branch-free.
__device__ __forceinline__ float second_max(const float (&z)[8], int n) {
  if (n == 1) return -INFINITY;
  const float h01 = fmaxf(z[0], z[1]), l01 = fminf(z[0], z[1]);
  const float h23 = fmaxf(z[2], z[3]), l23 = fminf(z[2], z[3]);
  const float m4 = fmaxf(h01, h23);
  const float s4 = fmaxf(fminf(h01, h23), fmaxf(l01, l23));
  if (n == 4) return s4;
  const float h45 = fmaxf(z[4], z[5]), l45 = fminf(z[4], z[5]);
  const float h67 = fmaxf(z[6], z[7]), l67 = fminf(z[6], z[7]);
  const float n4 = fmaxf(h45, h67);
  const float t4 = fmaxf(fminf(h45, h67), fmaxf(l45, l67));
  return fmaxf(fminf(m4, n4), fmaxf(s4, t4));
}

// The running maximum's update by one vector (maximum vm, first index
// base_idx), without a branch: the warps' lanes meet new maxima at different
// vectors, and a divergent branch would be taken by the whole warp on most
// vectors of a short pass.  The sum is rescaled by f = 2^((m - m') c) only
// when the maximum grows (f = 1 exactly otherwise, so the bits are those of
// a branch around the rescale).  The position inside the vector is found
// once, at the end (scan_resolve).
template <bool DO_EXP>
__device__ __forceinline__ void scan_max(ScanState& st, float vm, int base_idx, float c) {
  const bool take = vm > st.m || st.idx == kIdxNone;
  const float nm = take ? vm : st.m;
  if (DO_EXP) {
    const float f = (st.m == nm) ? 1.f : ex2_fast((st.m - nm) * c);
    const f32x2 s2 = mul2(pk2(st.s, st.sb), pk2(f, f));
    up2(s2, st.s, st.sb);
  }
  st.idx = take ? base_idx : st.idx;
  st.m = nm;
}

// Max / argmax / NaN / (optionally) the online exponential sum over one
// vector of n logits starting at index base_idx.  vm is the vector maximum
// with NaN propagation (NaN iff the vector holds a NaN).  With SECOND the
// thread also keeps m2, the second largest value among its elements
// (m2 <- max(m2, min(vector max, old max), second max of the vector), exact
// for values; without DEFER the vector's second value is formed only when
// the maximum grows, the vector maximum bounding it otherwise).  DEFER: the
// branch-free update of scan_max, the
// index resolved by scan_resolve at the end; otherwise a branch taken when
// the maximum grows finds the index at once (a long pass over fp32 rows,
// where the extra exponential per vector would cost more than the branch).
template <bool DO_EXP, bool SECOND = false, bool DEFER = false>
__device__ __forceinline__ void scan_vector(ScanState& st, const float (&z)[8], int n,
                                            float vm, int base_idx, float c) {
  if (vm != vm) {  // a NaN in the vector: the row is invalid
    st.nan = 1;
    return;
  }
  if (DEFER) {
    if (SECOND) st.m2 = fmaxf(st.m2, fmaxf(fminf(vm, st.m), second_max(z, n)));
    scan_max<DO_EXP>(st, vm, base_idx, c);
  } else if (vm > st.m || st.idx == kIdxNone) {
    // a new maximum: the old one and the vector's second value can be
    // second; on the (common) other path the vector's own maximum bounds
    // all its elements, so the second-largest network runs only here --
    // the same m2 as taking min(vm, m) and the vector's second value always
    if (SECOND) st.m2 = fmaxf(st.m2, fmaxf(st.m, second_max(z, n)));
    int e_star = n - 1;
#pragma unroll
    for (int e = 7; e >= 0; --e)
      if (e < n && z[e] == vm) e_star = e;
    if (DO_EXP) {
      // rescale the running sum to the new maximum
      const float f = (st.m == vm) ? 1.f : ex2_fast((st.m - vm) * c);
      st.s = st.s * f;
      st.sb = st.sb * f;
    }
    st.m = vm;
    st.idx = base_idx + e_star;
  } else if (SECOND) {
    st.m2 = fmaxf(st.m2, vm);  // vm <= m
  }
  if (DO_EXP) {
    float base = (st.m == -INFINITY) ? 0.f : st.m;
    if (n == 1) {
      st.s += ex2_fast((z[0] - base) * c);
    } else {
      // pairs of elements: (z - base) * c and the sum in packed fp32 (the
      // exponent arguments are those of the scalar form, bit for bit)
      const f32x2 b2 = pk2(base, base), c2 = pk2(c, c);
      f32x2 s2 = pk2(st.s, st.sb);
#pragma unroll
      for (int e = 0; e < 8; e += 2)
        if (e + 1 < n) {
          float x0, x1;
          up2(mul2(sub2(pk2(z[e], z[e + 1]), b2), c2), x0, x1);
          s2 = add2(s2, pk2(ex2_fast(x0), ex2_fast(x1)));
        }
      up2(s2, st.s, st.sb);
    }
  }
}

// The end of a thread's pass: st.idx names the first vector attaining st.m
// (n logits z, as loaded again); the lowest element of it equal to st.m
// makes the index exact.
__device__ __forceinline__ void scan_resolve(ScanState& st, const float (&z)[8], int n) {
  int e_star = n - 1;
#pragma unroll
  for (int e = 7; e >= 0; --e)
    if (e < n && z[e] == st.m) e_star = e;
  st.idx += e_star;
}

// ---------------------------------------------------------------------------
// bf16 vectors straight from the loaded words (eight logits in four 32-bit
// words, element 2j in the low half of word j): the vector maximum (and, for
// top-f rows, the second largest value) from bf16x2 maxima and minima --
// exact, as bf16 values compare exactly -- and the exponentials on the
// widened pairs.  Every float result is bit-identical to widening the eight
// logits first and running scan_vector on them: the same operations on the
// same values, the same lanes (even elements to s, odd ones to sb) and the
// same order of the sums.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned bf2_max_nan(unsigned a, unsigned b) {
  unsigned r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ unsigned bf2_max(unsigned a, unsigned b) {
  unsigned r;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ unsigned bf2_min(unsigned a, unsigned b) {
  unsigned r;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float bf_lo(unsigned w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(unsigned w) { return __uint_as_float(w & 0xffff0000u); }
// both halves of w widened to binary32, as one packed pair (low half first)
__device__ __forceinline__ f32x2 bf2_widen(unsigned w) {
  f32x2 r;
  asm("{\n\t.reg .b32 l, h;\n\tshl.b32 l, %1, 16;\n\tand.b32 h, %1, 0xffff0000;\n\t"
      "mov.b64 %0, {l, h};\n\t}"
      : "=l"(r)
      : "r"(w));
  return r;
}

template <bool DO_EXP, bool SECOND = false>
__device__ __forceinline__ void scan_bf16(ScanState& st, const uint4& w, int base_idx, float c) {
  float vm, v2 = -INFINITY;
  if (SECOND) {
    // per lane (even / odd elements) the largest and second largest of four,
    // then the two lanes combined: the second largest of the eight values
    const unsigned h01 = bf2_max_nan(w.x, w.y), l01 = bf2_min(w.x, w.y);
    const unsigned h23 = bf2_max_nan(w.z, w.w), l23 = bf2_min(w.z, w.w);
    const unsigned h = bf2_max_nan(h01, h23);
    const unsigned s = bf2_max(bf2_min(h01, h23), bf2_max(l01, l23));
    const float h0 = bf_lo(h), h1 = bf_hi(h);
    vm = max_nan(h0, h1);
    v2 = fmaxf(fminf(h0, h1), fmaxf(bf_lo(s), bf_hi(s)));
  } else {
    const unsigned h = bf2_max_nan(bf2_max_nan(w.x, w.y), bf2_max_nan(w.z, w.w));
    vm = max_nan(bf_lo(h), bf_hi(h));
  }
  if (vm != vm) {  // a NaN in the vector: the row is invalid
    st.nan = 1;
    return;
  }
  if (SECOND) st.m2 = fmaxf(st.m2, fmaxf(fminf(vm, st.m), v2));
  scan_max<DO_EXP>(st, vm, base_idx, c);
  if (DO_EXP) {
    const float base = (st.m == -INFINITY) ? 0.f : st.m;
    const f32x2 b2 = pk2(base, base), c2 = pk2(c, c);
    f32x2 s2 = pk2(st.s, st.sb);
    const unsigned ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float x0, x1;
      up2(mul2(sub2(bf2_widen(ws[j]), b2), c2), x0, x1);
      s2 = add2(s2, pk2(ex2_fast(x0), ex2_fast(x1)));
    }
    up2(s2, st.s, st.sb);
  }
}

__device__ __forceinline__ void merge_stat(float& m, float& s, int& idx, float m2, float s2,
                                           int i2, float c, bool do_exp) {
  float mm = fmaxf(m, m2);
  if (do_exp) {
    float f1 = (m == mm) ? 1.f : ex2_fast((m - mm) * c);
    float f2 = (m2 == mm) ? 1.f : ex2_fast((m2 - mm) * c);
    s = s * f1 + s2 * f2;
  }
  int ni;
  if (m > m2) ni = idx;
  else if (m2 > m) ni = i2;
  else ni = min(idx, i2);
  m = mm;
  idx = ni;
}

__device__ __forceinline__ bool is_masked(int idx, const int* msk, int M) {
  bool m = false;
  for (int q = 0; q < M; ++q) m |= (msk[q] == idx);
  return m;
}

__device__ __forceinline__ float pick8(const float (&z)[8], int e) {
  float r = z[0];
#pragma unroll
  for (int k = 1; k < 8; ++k) r = (e == k) ? z[k] : r;
  return r;
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(kFull, v, o);
    int oi = __shfl_xor_sync(kFull, i, o);
    if (ranks_before(ov, oi, v, i)) {
      v = ov;
      i = oi;
    }
  }
}

// Block reduction of the per-thread statistics; thread 0 writes the chunk's
// partial record.  Contains a __syncthreads().
__device__ __forceinline__ void block_stats_write(const ScanState& st, float c, bool do_exp,
                                                  float* sm_m, float* sm_s, int* sm_i,
                                                  int* sm_n, PartStat* out_part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float m = st.m, s = scan_sum(st);
  int idx = st.idx, nan = st.nan;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(kFull, m, o);
    float s2 = __shfl_xor_sync(kFull, s, o);
    int i2 = __shfl_xor_sync(kFull, idx, o);
    nan |= __shfl_xor_sync(kFull, nan, o);
    merge_stat(m, s, idx, m2, s2, i2, c, do_exp);
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_s[warp] = s;
    sm_i[warp] = idx;
    sm_n[warp] = nan;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kWarps; ++w) {
      nan |= sm_n[w];
      merge_stat(m, s, idx, sm_m[w], sm_s[w], sm_i[w], c, do_exp);
    }
    PartStat ps;
    ps.m = m;
    ps.s = do_exp ? s : 0.f;
    ps.idx = idx;
    ps.flags = nan;
    *out_part = ps;
  }
}

}  // namespace ssd
