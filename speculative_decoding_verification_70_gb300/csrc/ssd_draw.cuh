// ssd_draw.cuh -- building blocks of the recovery / bonus draw shared by
// the batched draw kernels (ssd_residual.cu) and the small-batch cluster
// kernel (ssd_chain.cu): the row context, the per-element weights in
// double-float, range sums, the packed pass over an element pair with the
// sign split, the split mass and the exact floor(u W).
#pragma once

#include <math.h>

#include "ssd_device.cuh"
#include "ssd_layout.h"
#include "ssd_scan.cuh"

namespace ssd {

struct RowCtx {
  float mz, md;        // row maxima
  float c_hi, c_lo;    // log2(e)/T
  float iz_hi, iz_lo;  // 1/S_z (filtered rows: 1/P_z, the kept mass)
  float id_hi, id_lo;  // 1/S_d (filtered rows: 1/P_d)
  float rho;           // approximate S_z / S_d from the streaming statistics
  unsigned long long thr_z, thr_d;  // filtered rows: order key of the last kept token
};

constexpr float kSignMargin = 1e-3f;
// 2^48: per-chunk A, B.  a, b <= 1 and a chunk holds at most 2^14
// elements, so a chunk sum stays below 2^62.
constexpr float kFixAcc = 281474976710656.0f;

// Weight of element i in the given quantity:
//   Q_NORM_Z : 2^((z - m_z) c)         (unnormalised, for S_z and the p_k draw)
//   Q_NORM_D : 2^((d - m_d) c)
//   Q_RESID  : max(0, p - q)
//   Q_FILT_TARGET : p_f, the filtered target law (0 outside its kept set)
//   Q_FILT_RESID  : max(0, p_f - q_f) over the filtered laws
enum Quantity { Q_NORM_Z = 0, Q_NORM_D = 1, Q_RESID = 2, Q_FILT_TARGET = 3, Q_FILT_RESID = 4 };

template <int Q>
__device__ __forceinline__ void weight(int i, float z, float d, const RowCtx& cx,
                                       const float2* tab, float& h, float& l) {
  float xh, xl;
  if (Q == Q_FILT_TARGET || Q == Q_FILT_RESID) {
    h = 0.f;
    l = 0.f;
    if (order_key(z, i) < cx.thr_z) return;  // outside the target's kept set: p_f = 0
    float ah, al, ph, pl;
    arg_df(z, cx.mz, cx.c_hi, cx.c_lo, xh, xl);
    exp2_df(xh, xl, tab, ah, al);
    df_mul(ah, al, cx.iz_hi, cx.iz_lo, ph, pl);
    if (Q == Q_FILT_TARGET || order_key(d, i) < cx.thr_d) {
      h = ph;
      l = pl;
      return;
    }
    float bh, bl, qh, ql;
    arg_df(d, cx.md, cx.c_hi, cx.c_lo, xh, xl);
    exp2_df(xh, xl, tab, bh, bl);
    df_mul(bh, bl, cx.id_hi, cx.id_lo, qh, ql);
    df_sub(ph, pl, qh, ql, h, l);
    if (!(h > 0.f)) {
      h = 0.f;
      l = 0.f;
    }
    return;
  }
  if (Q == Q_NORM_Z) {
    arg_df(z, cx.mz, cx.c_hi, cx.c_lo, xh, xl);
    exp2_df(xh, xl, tab, h, l);
  } else if (Q == Q_NORM_D) {
    arg_df(d, cx.md, cx.c_hi, cx.c_lo, xh, xl);
    exp2_df(xh, xl, tab, h, l);
  } else {
    // a = 2^((z - m_z) c) and b = 2^((d - m_d) c) as one packed pair
    float ah, al, bh, bl, ph, pl, qh, ql;
    f32x2 x2h, x2l, e2h, e2l;
    arg_df2(pk2(z, d), pk2(cx.mz, cx.md), pk2(cx.c_hi, cx.c_hi), pk2(cx.c_lo, cx.c_lo), x2h, x2l);
    exp2_df2(x2h, x2l, tab, e2h, e2l);
    up2(e2h, ah, bh);
    up2(e2l, al, bl);
    df_mul(ah, al, cx.iz_hi, cx.iz_lo, ph, pl);
    df_mul(bh, bl, cx.id_hi, cx.id_lo, qh, ql);
    df_sub(ph, pl, qh, ql, h, l);
    if (!(h > 0.f)) {
      h = 0.f;
      l = 0.f;
    }
  }
}

// Double-float sum of the weights over [lo, hi) in index order.  Z and D
// rows start 16-byte aligned when VEC.
template <typename Tag, bool VEC, int Q>
__device__ __forceinline__ void range_sum(const typename Tag::Elem* zr,
                                          const typename Tag::Elem* dr, int lo, int hi,
                                          const RowCtx& cx, const float2* tab, float& sh,
                                          float& sl) {
  sh = 0.f;
  sl = 0.f;
  constexpr int kV = Tag::kVec;
  int i = lo;
  if (VEC) {
    for (; i + kV <= hi; i += kV) {
      float z[8], d[8];
      if (Q != Q_NORM_D) Tag::loadv_cached(zr + i, z);
      if (Q != Q_NORM_Z && Q != Q_FILT_TARGET) Tag::loadv_cached(dr + i, d);
#pragma unroll
      for (int e = 0; e < kV; ++e) {
        float h, l;
        weight<Q>(i + e, z[e], d[e], cx, tab, h, l);
        df_acc(sh, sl, h, l);
      }
    }
  }
  for (; i < hi; ++i) {
    float z = (Q != Q_NORM_D) ? Tag::load1(zr + i) : 0.f;
    float d = (Q != Q_NORM_Z && Q != Q_FILT_TARGET) ? Tag::load1(dr + i) : 0.f;
    float h, l;
    weight<Q>(i, z, d, cx, tab, h, l);
    df_acc(sh, sl, h, l);
  }
}

// Running sums of one thread of the norm pass, as packed pairs (lane 0: the
// target row's a, lane 1: the draft row's b): the normalisers (S_z, S_d)
// and the positive side of the sign split (A, B), each with its
// compensation term.
struct NormAcc {
  f32x2 sh, sl;   // S_z, S_d
  f32x2 ph, pl;   // A, B
};

// One element of the residual pass: a and b (one packed exponential pair)
// added to the normaliser sums, then the sign split against rho~.
__device__ __forceinline__ void pass_pair(float z, float d, int idx, const RowCtx& cx,
                                          const float2* tab, NormAcc& na, int* amb_cnt,
                                          int* amb_idx, int amb_cap) {
  f32x2 xh, xl, eh, el;
  arg_df2(pk2(z, d), pk2(cx.mz, cx.md), pk2(cx.c_hi, cx.c_hi), pk2(cx.c_lo, cx.c_lo), xh, xl);
  exp2_df2(xh, xl, tab, eh, el);
  comp_acc2(na.sh, na.sl, eh, el);
  float a_h, b_h;
  up2(eh, a_h, b_h);
  // the pairs are normalised: hi alone is good to 2^-24 against the margin
  const float rb = cx.rho * b_h;
  const float diff = a_h - rb;
  const float lim = kSignMargin * fmaxf(a_h, rb);
  if (diff > lim) {
    comp_acc2(na.ph, na.pl, eh, el);
  } else if (diff >= -lim && (a_h > 0.f || rb > 0.f)) {
    const int q = atomicAdd(amb_cnt, 1);
    if (q < amb_cap) amb_idx[q] = idx;
  }
}

// (A_t - rho B_t) / S_z in 2^60 units from 2^48 fixed-point A, B (rho and
// 2^12 / S_z as float pairs), clamped at 0: the sign split's residual mass
// of a chunk (or of one thread's range).
__device__ __forceinline__ long long split_mass(long long a, long long b, float2 rho,
                                                float2 inv4096) {
  float ah, al, bh, bl, th, tl, vh, vl;
  i64_to_df(a, ah, al);
  i64_to_df(b, bh, bl);
  df_mul(rho.x, rho.y, bh, bl, th, tl);   // rho B
  df_sub(ah, al, th, tl, vh, vl);         // A - rho B
  df_mul(vh, vl, inv4096.x, inv4096.y, vh, vl);
  const long long w = vh > 0.f ? __float2ll_rn(vh) + __float2ll_rn(vl) : 0;
  return w < 0 ? 0 : w;
}

// floor(total * u) exactly, u a binary32 in [0, 1).
__device__ __forceinline__ unsigned long long scale_by_uniform(unsigned long long total, float u) {
  if (!(u > 0.f)) return 0ull;
  uint32_t bits = __float_as_uint(u);
  uint32_t ex = (bits >> 23) & 0xffu;
  uint64_t mant = bits & 0x7fffffu;
  if (ex != 0) mant |= 0x800000u;
  else ex = 1;
  // u = mant * 2^(ex - 150), shift = 150 - ex >= 24 since u < 1
  int shift = 150 - static_cast<int>(ex);
  unsigned long long lo = total * mant;
  unsigned long long hi = __umul64hi(total, mant);
  if (shift >= 128) return 0ull;
  if (shift >= 64) return hi >> (shift - 64);
  return (lo >> shift) | (shift ? (hi << (64 - shift)) : 0ull);
}

}  // namespace ssd
