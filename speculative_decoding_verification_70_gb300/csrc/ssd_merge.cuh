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

// Merge the C (<= 256) partial records of one row (one warp).  S is accumulated in
// double-float (products s * 2^((m_c - m) c) with extended-precision
// rescaling factors) and returned as the pair (sh, sl) and, in rs.S, as a
// double (one conversion per row: the FP64 pipe is narrow).
inline __device__ void merge_row(const PartStat* parts, int C, float c_hi, float c_lo,
                                 bool do_exp, const float2* tab, RowStat& rs, float& sh,
                                 float& sl) {
  const int lane = threadIdx.x & 31;
  // the lane's records (q = lane, lane + 32, ...; C <= 256) in one round of loads
  constexpr int kPer = 8;
  PartStat ps[kPer];
#pragma unroll
  for (int t = 0; t < kPer; ++t)
    if (lane + 32 * t < C) ps[t] = parts[lane + 32 * t];
  float m = -INFINITY;
  int idx = kIdxNone, nan = 0;
#pragma unroll
  for (int t = 0; t < kPer; ++t) {
    if (lane + 32 * t >= C) break;
    nan |= ps[t].flags & 1;
    if (ps[t].m > m || (ps[t].m == m && ps[t].idx < idx)) {
      m = ps[t].m;
      idx = ps[t].idx;
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
#pragma unroll
    for (int t = 0; t < kPer; ++t) {
      if (lane + 32 * t >= C) break;
      float fh = 1.f, fl = 0.f;
      if (ps[t].m != m) {
        float xh, xl;
        arg_df(ps[t].m, m, c_hi, c_lo, xh, xl);
        exp2_df(xh, xl, tab, fh, fl);
      }
      float ph, pl;
      df_mul(ps[t].s, 0.f, fh, fl, ph, pl);
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

// Output slot r of a fork row: the pick (bv, bi) or an empty slot.
__device__ __forceinline__ void topf_write(int r, int keep, bool nan, int bq, float bv, int bi,
                                           int32_t* tok_out, float* logit_out) {
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

// Warp-wide best of the lanes' candidates (value descending, index
// ascending, then the lower list on an exact tie).
__device__ __forceinline__ void topf_warp_best(float& bv, int& bi, int& bq) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    float ov = __shfl_xor_sync(kFull, bv, o);
    int oi = __shfl_xor_sync(kFull, bi, o);
    int oq = __shfl_xor_sync(kFull, bq, o);
    bool take = (oq >= 0) && (bq < 0 || ranks_before(ov, oi, bv, bi) ||
                              (ov == bv && oi == bi && oq < bq));
    if (take) { bv = ov; bi = oi; bq = oq; }
  }
}

// merge_topf_row for at most 64 lists of at most 4 entries: every entry in
// registers (lists lane and lane + 32), loaded in one round, so the f rounds
// of the selection read no memory.  The same picks in the same order.
inline __device__ void merge_topf_row_regs(const TopEntry* lists, int C, int f, int keep, bool nan,
                                           int32_t* tok_out, float* logit_out) {
  const int lane = threadIdx.x & 31;
  TopEntry e[2][4];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int q = lane + 32 * t;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      if (q < C && h < f) {
        e[t][h] = lists[q * f + h];
      } else {
        e[t][h].v = -INFINITY;
        e[t][h].i = kIdxNone;
      }
    }
  }
  int hd[2] = {0, 0};
  for (int r = 0; r < f; ++r) {
    float bv = -INFINITY;
    int bi = kIdxNone, bq = -1;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int q = lane + 32 * t;
      const int h = hd[t];
      if (q < C && h < f) {
        const TopEntry x = h == 0 ? e[t][0] : (h == 1 ? e[t][1] : (h == 2 ? e[t][2] : e[t][3]));
        if (bq < 0 || ranks_before(x.v, x.i, bv, bi)) {
          bv = x.v; bi = x.i; bq = q;
        }
      }
    }
    topf_warp_best(bv, bi, bq);
    if (bq == lane) hd[0] += 1;
    else if (bq == lane + 32) hd[1] += 1;
    if (lane == 0) topf_write(r, keep, nan, bq, bv, bi, tok_out, logit_out);
  }
}

// Top-f of one fork row from its C chunk lists (one warp).  Only the first
// `keep` picks are written; slots keep .. f-1 get (token -1, logit -inf).
inline __device__ void merge_topf_row(const TopEntry* lists, int C, int f, int keep, bool nan,
                               int32_t* tok_out, float* logit_out, int* heads) {
  if (C <= 64 && f <= 4) {
    merge_topf_row_regs(lists, C, f, keep, nan, tok_out, logit_out);
    return;
  }
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
    topf_warp_best(bv, bi, bq);
    if (bq >= 0 && (bq & 31) == lane) heads[bq] += 1;
    __syncwarp();
    if (lane == 0) topf_write(r, keep, nan, bq, bv, bi, tok_out, logit_out);
  }
}

// Acceptance of one batch row's k draft tokens (one warp, lane i < k for
// draft position i): x_i is accepted when u_i < p_i(x_i) / q_i(x_i), tested
// as u_i e_d S_z < e_z S_d in double-float (p = e_z / S_z, q = e_d / S_d,
// e = 2^((z - m) c)); greedy rows (T == 0) accept when x_i is the target
// argmax.  Per lane: the token xi, its logits zx = z_i[xi] and dx = d_i[xi]
// (read only when xi is in range), the uniform ux, the merged statistics of
// target row i (maximum, S as a float pair, flags) and of draft row i
// (lanes <= k pass target row flags, lanes < k draft row flags, 0 beyond).
// Returns the first rejected position n (k if none) or the sentinels -1
// (invalid temperature or row) / -2 (token out of range), and each lane's
// p(x_i), q(x_i) (1/0 at T == 0).
struct AcceptOut {
  int n;
  int status;        // 0, -1 or -2
  int err;           // SSD_DEVERR bits of this row
  float pv, qv;
};

inline __device__ AcceptOut accept_warp(int k, int V, bool greedy, bool t_bad, float c_hi,
                                        float c_lo, const float2* tab, int xi, float zx,
                                        float dx, float ux, float mz, float szh, float szl,
                                        int amz, int flz, float md, float sdh, float sdl,
                                        int amd, int fld) {
  const int lane = threadIdx.x & 31;
  const bool tok_bad = lane < k && (xi < 0 || xi >= V);
  const bool any_tok_bad = __any_sync(kFull, tok_bad);
  bool row_bad = false;
  if (lane <= k) row_bad |= (flz & 2) != 0;
  if (lane < k) row_bad |= (fld & 2) != 0;
  const bool any_row_bad = __any_sync(kFull, row_bad);
  AcceptOut o;
  o.status = 0;
  if (t_bad) o.status = -1;
  else if (any_tok_bad) o.status = -2;
  else if (any_row_bad) o.status = -1;
  o.err = t_bad ? 0x1 : (any_tok_bad ? 0x4 : (any_row_bad ? 0x2 : 0));
  o.pv = NAN;
  o.qv = NAN;
  bool acc = false;
  if (o.status == 0 && lane < k) {
    if (greedy) {
      acc = xi == amz;
      o.pv = acc ? 1.f : 0.f;
      o.qv = xi == amd ? 1.f : 0.f;
    } else {
      float xh, xl, ezh, ezl, edh, edl;
      arg_df(zx, mz, c_hi, c_lo, xh, xl);
      exp2_df(xh, xl, tab, ezh, ezl);
      arg_df(dx, md, c_hi, c_lo, xh, xl);
      exp2_df(xh, xl, tab, edh, edl);
      float lh, ll, rh, rl;
      df_mul(edh, edl, szh, szl, lh, ll);
      df_mul(lh, ll, ux, 0.f, lh, ll);
      df_mul(ezh, ezl, sdh, sdl, rh, rl);
      acc = (edh == 0.f) ? (ezh > 0.f) : (lh < rh || (lh == rh && ll < rl));
      o.pv = __fdiv_rn(__fadd_rn(ezh, ezl), __fadd_rn(szh, szl));
      o.qv = __fdiv_rn(__fadd_rn(edh, edl), __fadd_rn(sdh, sdl));
    }
  }
  const unsigned ball = __ballot_sync(kFull, acc);
  const unsigned rej = ~ball & ((1u << k) - 1u);
  o.n = o.status != 0 ? o.status : (rej ? (__ffs(rej) - 1) : k);
  return o;
}

}  // namespace ssd
