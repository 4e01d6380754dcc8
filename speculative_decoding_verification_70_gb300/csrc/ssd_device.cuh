// ssd_device.cuh -- device helpers shared by the verify-and-recover kernels:
// 16-byte streaming loads of fp32 / bf16 logit rows, the fast MUFU exp2 used
// by the streaming statistics pass, an extended-precision exp2 and
// double-float arithmetic used by the recovery draw, and deterministic
// integer (fixed-point) block scans.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "exp2_table.inc"

namespace ssd {

constexpr int kThreads = 256;           // threads per CTA in every kernel
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;

// Fixed-point scales of the recovery draw.  Probabilities (p - q, p) are at
// most 1 each and sum to at most 1 (+ rounding): 2^60 units.  Unnormalised
// exponentials 2^x, x <= 0, are at most 1 each and sum to at most V < 2^21:
// 2^42 units.
constexpr float kFixResidual = 1152921504606846976.0f;  // 2^60
constexpr float kFixMass = 4398046511104.0f;            // 2^42
constexpr double kInvFixMass = 1.0 / 4398046511104.0;

// ---------------------------------------------------------------------------
// Logit element types.  bf16 is the upper half of a binary32, so widening is
// a 16-bit shift.
// ---------------------------------------------------------------------------
// Loads in flight per thread of the streaming pass (vectors issued before
// the first is used) and the resident CTAs per SM its register budget is
// cut for, per element type.
#ifndef SSD_STATS_UNROLL_F32
#define SSD_STATS_UNROLL_F32 4
#endif
#ifndef SSD_STATS_UNROLL_BF16
#define SSD_STATS_UNROLL_BF16 4
#endif
#ifndef SSD_STATS_BLOCKS_F32
#define SSD_STATS_BLOCKS_F32 6
#endif
#ifndef SSD_STATS_BLOCKS_BF16
#define SSD_STATS_BLOCKS_BF16 6
#endif

struct F32Tag {
  using Elem = float;
  static constexpr int kVec = 4;  // elements per 16-byte vector
  static constexpr int kUnroll = SSD_STATS_UNROLL_F32;
  static constexpr int kBlocks = SSD_STATS_BLOCKS_F32;
  using Raw = float4;
  __device__ __forceinline__ static float load1(const Elem* p) { return __ldg(p); }
  __device__ __forceinline__ static Raw loadraw(const Elem* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
  }
  __device__ __forceinline__ static void unpackraw(const Raw& v, float (&o)[8]) {
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  __device__ __forceinline__ static void loadv(const Elem* p, float (&o)[8]) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  // cached (L1) variant for rows read more than once
  __device__ __forceinline__ static void loadv_cached(const Elem* p, float (&o)[8]) {
    float4 v = __ldg(reinterpret_cast<const float4*>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
};

struct BF16Tag {
  using Elem = uint16_t;
  static constexpr int kVec = 8;
  static constexpr int kUnroll = SSD_STATS_UNROLL_BF16;
  static constexpr int kBlocks = SSD_STATS_BLOCKS_BF16;
  using Raw = uint4;
  __device__ __forceinline__ static Raw loadraw(const Elem* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
  }
  __device__ __forceinline__ static void unpackraw(const Raw& v, float (&o)[8]) {
    unpack(v.x, v.y, v.z, v.w, o);
  }
  __device__ __forceinline__ static float load1(const Elem* p) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
  }
  __device__ __forceinline__ static void unpack(uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                                float (&o)[8]) {
    o[0] = __uint_as_float(a << 16); o[1] = __uint_as_float(a & 0xffff0000u);
    o[2] = __uint_as_float(b << 16); o[3] = __uint_as_float(b & 0xffff0000u);
    o[4] = __uint_as_float(c << 16); o[5] = __uint_as_float(c & 0xffff0000u);
    o[6] = __uint_as_float(d << 16); o[7] = __uint_as_float(d & 0xffff0000u);
  }
  __device__ __forceinline__ static void loadv(const Elem* p, float (&o)[8]) {
    uint32_t a, b, c, d;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(a), "=r"(b), "=r"(c), "=r"(d)
                 : "l"(p));
    unpack(a, b, c, d, o);
  }
  __device__ __forceinline__ static void loadv_cached(const Elem* p, float (&o)[8]) {
    uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    unpack(v.x, v.y, v.z, v.w, o);
  }
};

// ---------------------------------------------------------------------------
// Fast exp2 (one MUFU op).  Used where an error of a few ulp is harmless: the
// streaming row statistics, whose sums feed p(x)/q(x) for acceptance.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Packed fp32 pairs (add / sub / mul / fma .f32x2 of sm_100+): two IEEE
// binary32 operations per instruction, each lane rounded as its scalar
// counterpart.  A pair lives in one 64-bit register (low lane first).
// ---------------------------------------------------------------------------
typedef unsigned long long f32x2;
__device__ __forceinline__ f32x2 pk2(float a, float b) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void up2(f32x2 v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before its predecessor in the stream has
// finished; pdl_wait() blocks until the predecessor has completed and its
// memory is visible (a no-op for an ordinary launch).  pdl_trigger() lets
// the successor's launch begin once every CTA of this grid has called it.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Error-free transformations (Knuth's TwoSum, FMA-based TwoProduct).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Exact argument x = (z - m) * (c_hi + c_lo) as a float pair (xh, xl); the
// product error is kept to ~2^-46 relative.
__device__ __forceinline__ void arg_df(float z, float m, float c_hi, float c_lo, float& xh,
                                       float& xl) {
  float dh, dl;
  two_sum(z, -m, dh, dl);
  xh = __fmul_rn(dh, c_hi);
  xl = __fmaf_rn(dh, c_hi, -xh);
  xl = __fmaf_rn(dh, c_lo, xl);
  xl = __fmaf_rn(dl, c_hi, xl);
}

// 2^(xh + xl) for xh <= 0 as a normalised float pair (hi, lo: |lo| <= half
// an ulp of hi), relative error ~1e-9.  Method: J = round(64 xh) (one add
// of 1.5 * 2^23 gives both the rounded float and the integer), x = J/64 + g
// with |g| <= 1/128 (exact) plus xl; 2^x = 2^(J >> 6) * 2^((J & 63)/64) *
// (1 + P(g)) with the table 2^(j/64) held as float pairs and P the degree-3
// Taylor polynomial of 2^g - 1 (truncation < 4e-11, below the float
// rounding of P).  Results below 2^-125 (relative to the row maximum 1)
// return 0.  `tab` is a shared-memory copy of kExp2Tab.
__device__ __forceinline__ void exp2_df(float xh, float xl, const float2* tab, float& hi,
                                        float& lo) {
  if (!(xh > -125.0f)) {
    hi = 0.f;
    lo = 0.f;
    return;
  }
  const float kMagic = 12582912.0f;  // 1.5 * 2^23: exact rounding for |v| < 2^22
  const float tj = __fmaf_rn(xh, 64.0f, kMagic);
  const float Jf = __fsub_rn(tj, kMagic);
  const int J = __float_as_int(tj) - 0x4B400000;
  float g = __fmaf_rn(Jf, -0.015625f, xh);     // exact, |g| <= 1/128
  g = __fadd_rn(g, xl);
  float P = __fmaf_rn(g, SSD_EXP2_C3, SSD_EXP2_C2);
  P = __fmaf_rn(g, P, SSD_LN2_LO);
  P = __fmul_rn(g, P);
  P = __fmaf_rn(g, SSD_LN2_HI, P);             // 2^g - 1
  const float2 t = tab[J & 63];
  const float l = __fmaf_rn(t.x, P, __fmaf_rn(t.y, P, t.y));
  const float scale = __int_as_float(((J >> 6) + 127) << 23);  // J >> 6 in [-126, 0]
  // renormalise (|l| < 0.6% of t.x: Fast2Sum is exact)
  const float s = __fadd_rn(t.x, l);
  const float e = __fsub_rn(l, __fsub_rn(s, t.x));
  hi = __fmul_rn(s, scale);
  lo = __fmul_rn(e, scale);
}

// ---------------------------------------------------------------------------
// The same operations on two independent lanes at once (packed fp32 pairs):
// each lane computes exactly what the scalar function computes, bit for bit.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void two_sum2(f32x2 a, f32x2 b, f32x2& s, f32x2& e) {
  s = add2(a, b);
  const f32x2 bb = sub2(s, a);
  e = add2(sub2(a, sub2(s, bb)), sub2(b, bb));
}

// arg_df for lanes (z0, m0) and (z1, m1) with one coefficient pair c.
__device__ __forceinline__ void arg_df2(f32x2 z, f32x2 m, f32x2 c_hi, f32x2 c_lo, f32x2& xh,
                                        f32x2& xl) {
  f32x2 dh, dl;
  const f32x2 neg = pk2(-0.0f, -0.0f);
  float m0, m1;
  up2(m, m0, m1);
  two_sum2(z, pk2(-m0, -m1), dh, dl);
  xh = mul2(dh, c_hi);
  xl = fma2(dh, c_hi, sub2(neg, xh));  // dh c_hi - xh, exact
  xl = fma2(dh, c_lo, xl);
  xl = fma2(dl, c_hi, xl);
}

// exp2_df for two lanes; a lane with xh <= -125 (or NaN) gives 0.
__device__ __forceinline__ void exp2_df2(f32x2 xh, f32x2 xl, const float2* tab, f32x2& hi,
                                         f32x2& lo) {
  const float kMagic = 12582912.0f;
  const f32x2 magic = pk2(kMagic, kMagic);
  const f32x2 tj = fma2(xh, pk2(64.0f, 64.0f), magic);
  const f32x2 Jf = sub2(tj, magic);
  float tj0, tj1;
  up2(tj, tj0, tj1);
  const int J0 = __float_as_int(tj0) - 0x4B400000, J1 = __float_as_int(tj1) - 0x4B400000;
  f32x2 g = fma2(Jf, pk2(-0.015625f, -0.015625f), xh);
  g = add2(g, xl);
  f32x2 P = fma2(g, pk2(SSD_EXP2_C3, SSD_EXP2_C3), pk2(SSD_EXP2_C2, SSD_EXP2_C2));
  P = fma2(g, P, pk2(SSD_LN2_LO, SSD_LN2_LO));
  P = mul2(g, P);
  P = fma2(g, pk2(SSD_LN2_HI, SSD_LN2_HI), P);
  const float2 t0 = tab[J0 & 63], t1 = tab[J1 & 63];
  const f32x2 tx = pk2(t0.x, t1.x), ty = pk2(t0.y, t1.y);
  const f32x2 l = fma2(tx, P, fma2(ty, P, ty));
  const f32x2 sc = pk2(__int_as_float(((J0 >> 6) + 127) << 23), __int_as_float(((J1 >> 6) + 127) << 23));
  const f32x2 sm = add2(tx, l);
  const f32x2 e = sub2(l, sub2(sm, tx));
  hi = mul2(sm, sc);
  lo = mul2(e, sc);
  float xh0, xh1, h0, h1, l0, l1;
  up2(xh, xh0, xh1);
  up2(hi, h0, h1);
  up2(lo, l0, l1);
  const bool ok0 = xh0 > -125.0f, ok1 = xh1 > -125.0f;
  hi = pk2(ok0 ? h0 : 0.f, ok1 ? h1 : 0.f);
  lo = pk2(ok0 ? l0 : 0.f, ok1 ? l1 : 0.f);
}

// comp_acc for two lanes, with TwoSum in place of the ordered Fast2Sum: for
// non-negative values both give the exact error of acc + vh, so every lane
// is bit-identical to comp_acc, without the per-lane max / min and the
// repacking they need.
__device__ __forceinline__ void comp_acc2(f32x2& acc, f32x2& comp, f32x2 vh, f32x2 vl) {
  f32x2 t, err;
  two_sum2(acc, vh, t, err);
  comp = add2(comp, add2(err, vl));
  acc = t;
}

// Copy the exp2 table to shared memory (call before the first exp2_df; a
// __syncthreads() must follow).
__device__ __forceinline__ void load_exp2_table(float2* tab) {
  for (int i = threadIdx.x; i < 64; i += blockDim.x) tab[i] = kExp2Tab[i];
}

// double-float helpers
__device__ __forceinline__ void df_mul(float ah, float al, float bh, float bl, float& ph,
                                       float& pl) {
  ph = __fmul_rn(ah, bh);
  pl = __fmaf_rn(ah, bh, -ph);
  pl = __fmaf_rn(ah, bl, pl);
  pl = __fmaf_rn(al, bh, pl);
}

// s = a - b renormalised (|sl| <= ulp(sh)/2)
__device__ __forceinline__ void df_sub(float ah, float al, float bh, float bl, float& sh,
                                       float& sl) {
  float s, e;
  two_sum(ah, -bh, s, e);
  e = __fadd_rn(e, __fsub_rn(al, bl));
  sh = __fadd_rn(s, e);
  sl = __fsub_rn(e, __fsub_rn(sh, s));
}

// Compensated sum of non-negative values: acc += vh with the exact error
// of that add (Fast2Sum after ordering the two) and vl added to comp; the
// pair (acc, comp) carries the sum to O(n u^2).  vh, vl: a normalised pair.
__device__ __forceinline__ void comp_acc(float& acc, float& comp, float vh, float vl) {
  const float big = fmaxf(acc, vh), small = fminf(acc, vh);
  const float t = __fadd_rn(big, small);
  comp = __fadd_rn(comp, __fadd_rn(__fadd_rn(__fsub_rn(big, t), small), vl));
  acc = t;
}

// acc += v (double-float, renormalised)
__device__ __forceinline__ void df_acc(float& ah, float& al, float vh, float vl) {
  float s, e;
  two_sum(ah, vh, s, e);
  e = __fadd_rn(e, __fadd_rn(al, vl));
  ah = __fadd_rn(s, e);
  al = __fsub_rn(e, __fsub_rn(ah, s));
}

// double-float -> fixed point (round to nearest unit of 2^-scale_log2)
__device__ __forceinline__ long long df_to_fix(float h, float l, float scale) {
  return __float2ll_rn(__fmul_rn(h, scale)) + __float2ll_rn(__fmul_rn(l, scale));
}

// An int64 as a float pair (48 significant bits: relative error <= 2^-48).
__device__ __forceinline__ void i64_to_df(long long v, float& h, float& l) {
  h = __ll2float_rn(v);
  l = __ll2float_rn(v - __float2ll_rn(h));
}

// 1 / (h + l) as a normalised float pair: the correctly rounded reciprocal
// of h and one correction from the exact residual 1 - (h + l) r (FMA).
__device__ __forceinline__ void df_recip(float h, float l, float& rh, float& rl) {
  const float r = __frcp_rn(h);
  float e = __fmaf_rn(-h, r, 1.0f);
  e = __fmaf_rn(-l, r, e);
  two_sum(r, __fmul_rn(r, e), rh, rl);
}

// Split a positive double into a float pair.
__device__ __forceinline__ void split_double(double v, float& h, float& l) {
  h = __double2float_rn(v);
  l = __double2float_rn(v - static_cast<double>(h));
}

// c = log2(e) / T as a float pair, clamped so that c stays finite.
__device__ __forceinline__ void temp_coeff(float T, float& c_hi, float& c_lo) {
  double c = SSD_LOG2E / static_cast<double>(T);
  if (c > 1e37) c = 1e37;
  split_double(c, c_hi, c_lo);
}

// The same coefficient computed by thread 0 only and broadcast through
// shared memory: the double division runs once per CTA instead of once per
// thread (the FP64 pipe is narrow).  Every thread must call this (it holds
// a __syncthreads()).
__device__ __forceinline__ float2 cta_temp_coeff(float T, float2* slot) {
  if (threadIdx.x == 0) {
    float h, l;
    temp_coeff(T, h, l);
    *slot = make_float2(h, l);
  }
  __syncthreads();
  return *slot;
}

// ---------------------------------------------------------------------------
// Block-wide inclusive scan of int64 (exact: integer addition is associative,
// so the result does not depend on the order).  Returns the inclusive value;
// *total receives the block total.  `sm` holds kWarps entries.
// ---------------------------------------------------------------------------
__device__ __forceinline__ long long block_scan_i64(long long v, long long* sm,
                                                    long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) sm[warp] = v;
  __syncthreads();
  long long off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    long long s = sm[w];
    if (w < warp) off += s;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return v + off;
}

__device__ __forceinline__ long long block_sum_i64(long long v, long long* sm) {
  long long tot;
  block_scan_i64(v, sm, &tot);
  return tot;
}

}  // namespace ssd
