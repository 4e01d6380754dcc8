// ssd_merge.cuh -- merge of a logit row's per-chunk partial records (the
// statistics pass writes one record per chunk: maximum, lowest index
// attaining it, NaN flag and the chunk's sum of 2^((z - m_c) c)) and of its
// per-chunk top-f lists.  Shared by the finalisation of the chain step, the
// small-batch cluster kernel and the token-tree walk.
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

// Top-f of one fork row from its C chunk lists (one warp).  Only the first
// `keep` picks are written; slots keep .. f-1 get (token -1, logit -inf).
inline __device__ void merge_topf_row(const TopEntry* lists, int C, int f, int keep, bool nan,
                               int32_t* tok_out, float* logit_out, int* heads) {
  const int lane = threadIdx.x & 31;
  for (int q = lane; q < C; q += 32) heads[q] = 0;
  __syncwarp();
  for (int r = 0; r < f; ++r) {
    float bv = -INFINITY;
    int bi = kIdxNone, bq = -1;
    for (int q = lane; q < C; q += 32) {
      int h = heads[q];
      if (h < f) {
        TopEntry e = lists[q * f + h];
        if (bq < 0 || ranks_before(e.v, e.i, bv, bi)) {
          bv = e.v; bi = e.i; bq = q;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(kFull, bv, o);
      int oi = __shfl_xor_sync(kFull, bi, o);
      int oq = __shfl_xor_sync(kFull, bq, o);
      bool take = (oq >= 0) && (bq < 0 || ranks_before(ov, oi, bv, bi) ||
                                (ov == bv && oi == bi && oq < bq));
      if (take) { bv = ov; bi = oi; bq = oq; }
    }
    if (bq >= 0 && (bq & 31) == lane) heads[bq] += 1;
    __syncwarp();
    if (lane == 0) {
      if (r >= keep) {
        tok_out[r] = -1;
        logit_out[r] = -INFINITY;
      } else if (nan) {
        tok_out[r] = -1;
        logit_out[r] = NAN;
      } else if (bq < 0 || bi == kIdxNone) {
        tok_out[r] = -1;
        logit_out[r] = -INFINITY;
      } else {
        tok_out[r] = bi;
        logit_out[r] = bv;
      }
    }
  }
}

}  // namespace ssd
