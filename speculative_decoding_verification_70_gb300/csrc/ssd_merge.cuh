// ssd_merge.cuh -- merge of a logit row's per-chunk partial records (the
// statistics pass writes one record per chunk: maximum, lowest index
// attaining it, NaN flag and the chunk's sum of 2^((z - m_c) c)).  Shared by
// the finalisation of the chain step and by the token-tree walk.
#pragma once

#include "ssd_device.cuh"
#include "ssd_layout.h"
#include "ssd_scan.cuh"

namespace ssd {

// Merge the C partial records of one row (one warp).  S is accumulated in
// double-float (products s * 2^((m_c - m) c) with extended-precision
// rescaling factors) and returned as the pair (sh, sl) and, in rs.S, as a
// double (one conversion per row: the FP64 pipe is narrow).
inline __device__ void merge_row(const PartStat* parts, int C, float c_hi, float c_lo,
                                 bool do_exp, const float2* tab, RowStat& rs, float& sh,
                                 float& sl) {
  const int lane = threadIdx.x & 31;
  float m = -INFINITY;
  int idx = kIdxNone, nan = 0;
  for (int q = lane; q < C; q += 32) {
    PartStat ps = parts[q];
    nan |= ps.flags & 1;
    if (ps.m > m || (ps.m == m && ps.idx < idx)) {
      m = ps.m;
      idx = ps.idx;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float m2 = __shfl_xor_sync(kFull, m, o);
    int i2 = __shfl_xor_sync(kFull, idx, o);
    nan |= __shfl_xor_sync(kFull, nan, o);
    if (m2 > m || (m2 == m && i2 < idx)) {
      m = m2;
      idx = i2;
    }
  }
  sh = 0.f;
  sl = 0.f;
  if (do_exp) {
    for (int q = lane; q < C; q += 32) {
      PartStat ps = parts[q];
      float fh = 1.f, fl = 0.f;
      if (ps.m != m) {
        float xh, xl;
        arg_df(ps.m, m, c_hi, c_lo, xh, xl);
        exp2_df(xh, xl, tab, fh, fl);
      }
      float ph, pl;
      df_mul(ps.s, 0.f, fh, fl, ph, pl);
      df_acc(sh, sl, ph, pl);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float oh = __shfl_xor_sync(kFull, sh, o);
      const float ol = __shfl_xor_sync(kFull, sl, o);
      df_acc(sh, sl, oh, ol);
    }
  } else {
    sh = 1.f;
  }
  rs.m = m;
  rs.argmax = idx;
  rs.S = static_cast<double>(sh) + static_cast<double>(sl);
  int bad = nan;
  if (do_exp && !(sh > 0.f && sh < INFINITY)) bad = 1;  // +inf, NaN or all -inf at T > 0
  rs.flags = (nan ? 1 : 0) | (bad ? 2 : 0);
}

}  // namespace ssd
