// ssd_residual.cu -- the recovery / bonus draw (kernel K-B).
//
// Rule (speculative-sampling summary, "How It Works": regenerate from the
// point of divergence; Leviathan et al. / Chen et al.): after the first
// rejection at position n < k draw from w = max(0, p_n - q_n) (if w is all
// zero, from p_n); after k accepts draw the bonus token from p_k.  The draw
// is the inverse CDF: the smallest j with C_j > u * C_{V-1}.
//
// The draw decides an integer from sums over ~10^5 tiny weights, so fp32
// would move CDF boundaries across the dense tail of the distribution and
// change ~1e-3 of the draws.  Here every weight is evaluated in double-float
// (exp2_df, ~1e-9 relative), each thread sums a contiguous index range with
// compensation (error O(n u^2)), and everything above a thread is exact
// 64-bit fixed point,
// so every level of the three-level select (chunk, thread, element) sees the
// same totals.
//
// Kernels (one CTA per chunk of row n, then one CTA per batch row):
//   residual_norm   one pass over row n of Z and D: S_z = sum a, S_d = sum b
//                   with a = 2^((z - m_z) c), b = 2^((d - m_d) c), and the
//                   residual mass by sign: with rho~ = S_z/S_d taken from the
//                   streaming statistics (relative error ~1e-7), elements with
//                   a - rho~ b clearly positive (margin 1e-3) add to A and B,
//                   so that S_z * W_c = A_c - rho B_c exactly for them once
//                   rho = S_z/S_d is known; clearly negative ones add
//                   nothing; the few ambiguous ones are listed and evaluated
//                   exactly by the select kernel.
//                   Every thread also stores its own fixed-point S_z, A, B,
//                   so that the select finds the thread without
//                   recomputing the chunk.
//   residual_select chunk -> thread -> element select, writes out_tok[b, n];
//                   rows whose ambiguous list overflowed take the direct
//                   W_c = sum max(0, p - q) (computed here, one pass over
//                   the row); in the SSD round step it also looks up the
//                   row's realised outcome in the speculation cache
#include <math.h>

#include "ssd_cache.cuh"
#include "ssd_device.cuh"
#include "ssd_draw.cuh"
#include "ssd_layout.h"
#include "ssd_scan.cuh"

namespace ssd {

__device__ __forceinline__ void norm_inverses(const ResidualParams& p, int b, RowCtx& cx) {
  long long sz = 0, sd = 0;
  for (int q = 0; q < p.C; ++q) {
    sz += p.rnorm[(static_cast<int64_t>(b) * p.C + q) * 2 + 0];
    sd += p.rnorm[(static_cast<int64_t>(b) * p.C + q) * 2 + 1];
  }
  double Sz = static_cast<double>(sz) * kInvFixMass;
  double Sd = static_cast<double>(sd) * kInvFixMass;
  split_double(1.0 / Sz, cx.iz_hi, cx.iz_lo);
  split_double(1.0 / Sd, cx.id_hi, cx.id_lo);
}

// Row context of batch row b, computed by thread 0 (its double divisions run
// once per CTA) and shared through s_cx.  Returns false (uniformly) when the
// row draws nothing.  Holds a __syncthreads() when it returns true.
__device__ __forceinline__ bool load_ctx(const ResidualParams& p, int b, BState& bs, RowCtx& cx,
                                         RowCtx* s_cx, bool with_inverses) {
  bs = p.bstate[b];
  if (bs.mode == kModeNone) return false;
  if (threadIdx.x == 0) {
    RowCtx c;
    c.mz = p.rowstat[static_cast<int64_t>(b) * p.R + bs.n].m;
    c.md = (bs.mode == kModeResidual) ? p.rowstat[static_cast<int64_t>(b) * p.R + p.Pz + bs.n].m
                                      : 0.f;
    c.rho = bs.rho;  // from the streaming statistics, set with the draw state
    c.c_hi = bs.c_hi;
    c.c_lo = bs.c_lo;
    c.iz_hi = c.iz_lo = c.id_hi = c.id_lo = 0.f;
    if (with_inverses) norm_inverses(p, b, c);
    *s_cx = c;
  }
  __syncthreads();
  cx = *s_cx;
  return true;
}

template <typename Tag>
__device__ __forceinline__ void row_ptrs(const ResidualParams& p, int b, int n,
                                         const typename Tag::Elem*& zr,
                                         const typename Tag::Elem*& dr) {
  zr = static_cast<const typename Tag::Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb +
       static_cast<int64_t>(n) * p.V;
  dr = static_cast<const typename Tag::Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
       static_cast<int64_t>(n) * p.V;
}

// grid (C, B)
template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kThreads) residual_norm_kernel(ResidualParams p) {
  __shared__ float2 tab[64];
  __shared__ long long sm[kWarps];
  __shared__ RowCtx s_cx;
  pdl_trigger();  // the mass kernel may be scheduled (it waits for this grid)
  const int c = blockIdx.x, b = blockIdx.y + p.b0;
  BState bs;
  RowCtx cx;
  load_exp2_table(tab);
  if (!load_ctx(p, b, bs, cx, &s_cx, false)) return;
  const typename Tag::Elem *zr, *dr;
  row_ptrs<Tag>(p, b, bs.n, zr, dr);
  const bool resid = bs.mode == kModeResidual;
  const int clo = c * p.CH, chi = min(p.V, clo + p.CH);
  const int lo = min(chi, clo + static_cast<int>(threadIdx.x) * p.E);
  const int hi = min(chi, lo + p.E);
  int* amb_cnt = p.amb_cnt + b;
  int* amb_idx = p.amb_idx + static_cast<int64_t>(b) * p.amb_cap;
  constexpr int kV = Tag::kVec;
  const f32x2 zero = pk2(0.f, 0.f);
  NormAcc na = {zero, zero, zero, zero};
  int i = lo;
  if (resid) {
    if (VEC) {
      for (; i + kV <= hi; i += kV) {
        float z[8], d[8];
        Tag::loadv_cached(zr + i, z);
        Tag::loadv_cached(dr + i, d);
#pragma unroll
        for (int e = 0; e < kV; ++e)
          pass_pair(z[e], d[e], i + e, cx, tab, na, amb_cnt, amb_idx, p.amb_cap);
      }
    }
    for (; i < hi; ++i)
      pass_pair(Tag::load1(zr + i), Tag::load1(dr + i), i, cx, tab, na, amb_cnt, amb_idx,
                p.amb_cap);
  } else {
    // bonus draw: S_z only, two consecutive elements per packed pair (the
    // lanes are summed at the end)
    const f32x2 mz = pk2(cx.mz, cx.mz), ch = pk2(cx.c_hi, cx.c_hi), cl = pk2(cx.c_lo, cx.c_lo);
    if (VEC) {
      for (; i + kV <= hi; i += kV) {
        float z[8];
        Tag::loadv_cached(zr + i, z);
#pragma unroll
        for (int e = 0; e < kV; e += 2) {
          f32x2 xh, xl, eh, el;
          arg_df2(pk2(z[e], z[e + 1]), mz, ch, cl, xh, xl);
          exp2_df2(xh, xl, tab, eh, el);
          comp_acc2(na.sh, na.sl, eh, el);
        }
      }
    }
    for (; i < hi; ++i) {
      float xh, xl, a_h, a_l;
      arg_df(Tag::load1(zr + i), cx.mz, cx.c_hi, cx.c_lo, xh, xl);
      exp2_df(xh, xl, tab, a_h, a_l);
      float s0, s1, c0, c1;
      up2(na.sh, s0, s1);
      up2(na.sl, c0, c1);
      comp_acc(s0, c0, a_h, a_l);
      na.sh = pk2(s0, s1);
      na.sl = pk2(c0, c1);
    }
  }
  float sah, sbh, sal, sbl, ah, bh, al, bl;
  up2(na.sh, sah, sbh);
  up2(na.sl, sal, sbl);
  up2(na.ph, ah, bh);
  up2(na.pl, al, bl);
  long long tz, td = 0, ta = 0, tb = 0;
  long long oz, oa = 0, ob = 0;  // this thread's own S_z, A, B
  if (resid) {
    oz = df_to_fix(sah, sal, kFixMass);
    oa = df_to_fix(ah, al, kFixAcc);
    ob = df_to_fix(bh, bl, kFixAcc);
    tz = block_sum_i64(oz, sm);
    td = block_sum_i64(df_to_fix(sbh, sbl, kFixMass), sm);
    ta = block_sum_i64(oa, sm);
    tb = block_sum_i64(ob, sm);
  } else {  // the two lanes hold the even and odd elements' sums of a
    oz = df_to_fix(sah, sal, kFixMass) + df_to_fix(sbh, sbl, kFixMass);
    tz = block_sum_i64(oz, sm);
  }
  long long* own = p.rthr + (static_cast<int64_t>(b) * p.C + c) * 3 * kDrawThreads + threadIdx.x;
  own[0] = oz;
  own[kDrawThreads] = oa;
  own[2 * kDrawThreads] = ob;
  if (threadIdx.x == 0) {
    const int64_t o = (static_cast<int64_t>(b) * p.C + c) * 2;
    p.rnorm[o + 0] = tz;
    p.rnorm[o + 1] = td;
    p.racc[o + 0] = ta;
    p.racc[o + 1] = tb;
  }
}

// The thread, then the element, holding fixed-point mass `target` of chunk
// [clo, chi): every thread passes `own`, the mass of its range [clo + t E,
// + E) in units of `scale`; warp 0 then walks the picked range with the
// exact per-element weights.
template <typename Tag, bool VEC, int Q>
__device__ int select_from_own(const typename Tag::Elem* zr, const typename Tag::Elem* dr,
                               int clo, int chi, int E, const RowCtx& cx, const float2* tab,
                               float scale, long long target, long long own, long long* sm,
                               int* s_pick) {
  const int tid = threadIdx.x;
  long long tot;
  long long incl = block_scan_i64(own, sm, &tot);
  // a chunk mass taken from the sign split can exceed this chunk's direct
  // total by rounding (~1e-10 relative); such a target picks the chunk's
  // last positive element
  if (target >= tot) target = tot - 1;
  if (tid == 0) *s_pick = kThreads;
  __syncthreads();
  if (incl > target && incl - own <= target) atomicMin(s_pick, tid);
  __syncthreads();
  const int pick = *s_pick;
  int tok = -1;
  if (pick == kThreads) {  // cannot happen: the chunk total exceeds target by construction
    __syncthreads();
    return chi - 1;
  }
  // warp 0 walks the picked thread's range: per-element weights in fixed
  // point, an int64 scan over the lanes, the first element whose cumulative
  // mass passes the target (per-element rounding moves the cumulative by at
  // most a few units of 2^-60 against the thread's own total)
  __shared__ long long s_base;
  if (tid == pick) s_base = incl - own;
  __syncthreads();
  if (tid < 32) {
    const int plo = min(chi, clo + pick * E), phi = min(chi, plo + E);
    const long long base = s_base;
    long long carry = 0;
    int last_pos = -1, found = -1;
    for (int off = plo; off < phi && found < 0; off += 32) {
      const int i = off + tid;
      long long wf = 0;
      if (i < phi) {
        const float z = (Q != Q_NORM_D) ? Tag::load1(zr + i) : 0.f;
        const float d = (Q != Q_NORM_Z && Q != Q_FILT_TARGET) ? Tag::load1(dr + i) : 0.f;
        float wh, wl;
        weight<Q>(i, z, d, cx, tab, wh, wl);
        wf = df_to_fix(wh, wl, scale);
      }
      long long c = wf;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(kFull, c, o);
        if (tid >= o) c += y;
      }
      const unsigned over = __ballot_sync(kFull, i < phi && base + carry + c > target);
      const unsigned posm = __ballot_sync(kFull, i < phi && wf > 0);
      if (posm) last_pos = off + 31 - __clz(posm);
      if (over) found = off + __ffs(over) - 1;
      carry += __shfl_sync(kFull, c, 31);
    }
    if (tid == 0) tok = found >= 0 ? found : (last_pos >= 0 ? last_pos : phi - 1);  // rounding guard
    if (tid == 0) *s_pick = -1 - tok;
  }
  __syncthreads();
  return -1 - *s_pick;
}

// The same with every thread's mass computed here from the exact weights.
template <typename Tag, bool VEC, int Q>
__device__ int select_in_chunk(const typename Tag::Elem* zr, const typename Tag::Elem* dr,
                               int clo, int chi, int E, const RowCtx& cx, const float2* tab,
                               float scale, long long target, long long* sm, int* s_pick) {
  const int lo = min(chi, clo + static_cast<int>(threadIdx.x) * E);
  const int hi = min(chi, lo + E);
  float h, l;
  range_sum<Tag, VEC, Q>(zr, dr, lo, hi, cx, tab, h, l);
  return select_from_own<Tag, VEC, Q>(zr, dr, clo, chi, E, cx, tab, scale, target,
                                      df_to_fix(h, l, scale), sm, s_pick);
}

// The exact residual weights (2^60 fixed point) of the ambiguous-sign
// elements amb[0..n) that lie in [lo, hi), each handed to add(i, w).  A long
// list is taken in batches of K entries per thread, so that a batch's index
// loads, then its logit loads, are in flight together (a row with a few
// thousand entries otherwise pays two dependent global-memory latencies per
// entry and thread); a list of at most one entry per thread takes K = 1.
template <int K, typename Tag, typename Add>
__device__ __forceinline__ void for_ambiguous_k(const int* amb, int n, int lo, int hi,
                                                const typename Tag::Elem* zr,
                                                const typename Tag::Elem* dr, const RowCtx& cx,
                                                const float2* tab, Add&& add) {
  for (int q0 = threadIdx.x; q0 < n; q0 += K * kThreads) {
    int idx[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      const int q = q0 + j * kThreads;
      const int i = q < n ? amb[q] : -1;
      idx[j] = (i >= lo && i < hi) ? i : -1;
    }
    float z[K], d[K];
#pragma unroll
    for (int j = 0; j < K; ++j) {
      z[j] = idx[j] >= 0 ? Tag::load1(zr + idx[j]) : 0.f;
      d[j] = idx[j] >= 0 ? Tag::load1(dr + idx[j]) : 0.f;
    }
#pragma unroll
    for (int j = 0; j < K; ++j) {
      if (idx[j] < 0) continue;
      float wh, wl;
      weight<Q_RESID>(idx[j], z[j], d[j], cx, tab, wh, wl);
      add(idx[j], df_to_fix(wh, wl, kFixResidual));
    }
  }
}

template <typename Tag, typename Add>
__device__ __forceinline__ void for_ambiguous(const int* amb, int n, int lo, int hi,
                                              const typename Tag::Elem* zr,
                                              const typename Tag::Elem* dr, const RowCtx& cx,
                                              const float2* tab, Add&& add) {
  if (n > kThreads) for_ambiguous_k<8, Tag>(amb, n, lo, hi, zr, dr, cx, tab, add);
  else for_ambiguous_k<1, Tag>(amb, n, lo, hi, zr, dr, cx, tab, add);
}

// grid B.  One CTA per batch row; every chunk-level step runs one chunk per
// thread (C <= kThreads): the chunk weights are formed in parallel, an int64
// block scan places the target, and one 128-bit product gives
// floor(u * W).  Within the chunk the thread level reads the norm pass's
// per-thread sums (no exponentials); only the picked thread's range is
// walked element by element.  Only the two normaliser inverses are taken by
// one thread.  Rows whose ambiguous-sign list overflowed evaluate the
// residual directly (chunk masses and the thread level, one pass over the
// row in this CTA).  With p.lookup every row, drawn or not, then looks up
// its realised outcome in the speculation cache.
template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kThreads) residual_select_kernel(ResidualParams p) {
  pdl_wait();  // the norm kernel has completed
  __shared__ float2 tab[64];
  __shared__ long long sm[kWarps];
  __shared__ long long s_amb[kThreads];  // exact mass of the ambiguous elements (2^60) by chunk, then by thread
  __shared__ int s_pick;
  __shared__ int s_chunk;
  __shared__ long long s_target;
  __shared__ RowCtx s_cx;
  __shared__ float2 s_acc[2];            // rho = S_z / S_d and 2^12 / S_z, float pairs
  const int b = blockIdx.x, tid = threadIdx.x;
  const BState bs = p.bstate[b];
  if (bs.mode != kModeNone) {
    load_exp2_table(tab);
    const bool resid_row = bs.mode == kModeResidual;
    const int64_t rb = static_cast<int64_t>(b) * p.C;
    long long cz = 0, cd = 0, ca = 0, cb = 0;
    if (tid < p.C) {
      cz = p.rnorm[(rb + tid) * 2 + 0];
      if (resid_row) {
        cd = p.rnorm[(rb + tid) * 2 + 1];
        ca = p.racc[(rb + tid) * 2 + 0];
        cb = p.racc[(rb + tid) * 2 + 1];
      }
    }
    s_amb[tid] = 0;
    const long long sz = block_sum_i64(cz, sm);
    const long long sd = resid_row ? block_sum_i64(cd, sm) : 1;
    if (tid == 0) {
      RowCtx c;
      c.mz = p.rowstat[static_cast<int64_t>(b) * p.R + bs.n].m;
      c.md = resid_row ? p.rowstat[static_cast<int64_t>(b) * p.R + p.Pz + bs.n].m : 0.f;
      c.rho = 1.f;
      c.c_hi = bs.c_hi;
      c.c_lo = bs.c_lo;
      // normalisers and their inverses in double-float (no FP64 on this
      // thread's chain); the 2^-42 unit scaling is exact
      constexpr float kMass = 2.2737367544323206e-13f;  // 2^-42
      float szh, szl, sdh, sdl;
      i64_to_df(sz, szh, szl);
      i64_to_df(sd, sdh, sdl);
      szh *= kMass; szl *= kMass;
      sdh *= kMass; sdl *= kMass;
      df_recip(szh, szl, c.iz_hi, c.iz_lo);
      df_recip(sdh, sdl, c.id_hi, c.id_lo);
      s_cx = c;
      float rh, rl;
      df_mul(szh, szl, c.id_hi, c.id_lo, rh, rl);
      s_acc[0] = make_float2(rh, rl);
      s_acc[1] = make_float2(c.iz_hi * 4096.f, c.iz_lo * 4096.f);
    }
    __syncthreads();
    const RowCtx cx = s_cx;
    const typename Tag::Elem *zr, *dr;
    row_ptrs<Tag>(p, b, bs.n, zr, dr);
    const int n_amb = resid_row ? p.amb_cnt[b] : 0;
    const bool split = resid_row && n_amb <= p.amb_cap;
    const int* amb = p.amb_idx + static_cast<int64_t>(b) * p.amb_cap;
    if (split) {
      for_ambiguous<Tag>(amb, n_amb, 0, p.V, zr, dr, cx, tab, [&](int i, long long w) {
        atomicAdd(reinterpret_cast<unsigned long long*>(&s_amb[i / p.CH]),
                  static_cast<unsigned long long>(w));
      });
      __syncthreads();
    }
    // chunk weights in the units of the thread level: residual mass in
    // 2^60 (W_c = (A_c - rho B_c) / S_z plus the ambiguous part, or the
    // direct masses when the ambiguous list overflowed), target mass a in
    // 2^42
    long long wq = 0;
    if (split) {
      if (tid < p.C) wq = split_mass(ca, cb, s_acc[0], s_acc[1]) + s_amb[tid];
    } else if (resid_row) {  // direct masses, chunk by chunk
      for (int q = 0; q < p.C; ++q) {
        const int clo = q * p.CH, chi = min(p.V, clo + p.CH);
        const int lo = min(chi, clo + tid * p.E), hi = min(chi, lo + p.E);
        float h, l;
        range_sum<Tag, VEC, Q_RESID>(zr, dr, lo, hi, cx, tab, h, l);
        const long long m = block_sum_i64(df_to_fix(h, l, kFixResidual), sm);
        if (tid == q) wq = m;
      }
    } else {
      wq = cz;
    }
    long long W;
    long long incl = block_scan_i64(wq, sm, &W);
    bool resid = resid_row;
    if (resid && W <= 0) {  // all-zero residual: draw from p_n
      resid = false;
      wq = tid < p.C ? cz : 0;
      incl = block_scan_i64(wq, sm, &W);
    }
    const long long t =
        static_cast<long long>(scale_by_uniform(static_cast<unsigned long long>(W), p.u_smp[b]));
    if (tid == 0) {
      s_chunk = p.C - 1;  // unreachable default: t < W always finds a chunk
      s_target = 0;
    }
    __syncthreads();
    if (wq > 0 && incl > t && incl - wq <= t) {  // exactly one thread
      s_chunk = tid;
      s_target = t - (incl - wq);
    }
    __syncthreads();
    const int q = s_chunk;
    const long long target = s_target;
    const int clo = q * p.CH, chi = min(p.V, clo + p.CH);
    const long long* own = p.rthr + (rb + q) * 3 * kDrawThreads + tid;
    int tok;
    if (!resid) {  // the norm pass's per-thread S_z of this chunk
      tok = select_from_own<Tag, VEC, Q_NORM_Z>(zr, dr, clo, chi, p.E, cx, tab, kFixMass, target,
                                                own[0], sm, &s_pick);
    } else if (split) {
      // per-thread sign-split masses plus each thread's ambiguous elements
      s_amb[tid] = 0;
      __syncthreads();
      for_ambiguous<Tag>(amb, n_amb, clo, chi, zr, dr, cx, tab, [&](int i, long long w) {
        atomicAdd(reinterpret_cast<unsigned long long*>(&s_amb[(i - clo) / p.E]),
                  static_cast<unsigned long long>(w));
      });
      __syncthreads();
      const long long w =
          split_mass(own[kDrawThreads], own[2 * kDrawThreads], s_acc[0], s_acc[1]) + s_amb[tid];
      tok = select_from_own<Tag, VEC, Q_RESID>(zr, dr, clo, chi, p.E, cx, tab, kFixResidual,
                                               target, w, sm, &s_pick);
    } else {
      tok = select_in_chunk<Tag, VEC, Q_RESID>(zr, dr, clo, chi, p.E, cx, tab, kFixResidual,
                                               target, sm, &s_pick);
    }
    if (tid == 0) p.out_tok[static_cast<int64_t>(b) * (p.k + 1) + bs.n] = tok;
  }
  if (p.lookup && tid == 0) {  // the row's outcome: (b, n, out_tok[b][n])
    const int n = bs.n;
    const int tok = (n >= 0 && n <= p.k) ? p.out_tok[static_cast<int64_t>(b) * (p.k + 1) + n] : -1;
    cache_lookup_one(p.cache, b, n, tok, p.hit + b, p.tok_out + static_cast<int64_t>(b) * p.cache.depth);
  }
}

// ---------------------------------------------------------------------------
// The draw over top-k / top-p filtered laws (ssd_verify_topk beyond the
// in-register lists).  Each filtered row is given by the order key of its
// last kept token and its kept mass P (FiltRow), so
// p_f(v) = [key(z_v, v) >= thr_z] 2^((z_v - m_z) c) / P_z, likewise q_f, and
// the weights are max(0, p_f - q_f) after a rejection, p_f for the bonus
// token (p_f also when the residual is all zero).  Same numerics as above:
// double-float weights, per-thread compensated sums, exact fixed point above
// a thread, the chunk -> thread -> element select.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool filt_ctx(const FiltParams& p, int b, BState& bs, RowCtx* s_cx) {
  bs = p.bstate[b];
  if (bs.mode == kModeNone) return false;
  if (threadIdx.x == 0) {
    const FiltRow& fz = p.rows[static_cast<int64_t>(b) * p.R + bs.n];
    RowCtx c;
    c.mz = fz.m;
    c.c_hi = fz.c_hi;
    c.c_lo = fz.c_lo;
    c.rho = 1.f;
    split_double(1.0 / fz.P, c.iz_hi, c.iz_lo);
    c.thr_z = fz.thr;
    c.md = 0.f;
    c.id_hi = c.id_lo = 0.f;
    c.thr_d = ~0ull;
    if (bs.mode == kModeResidual) {
      const FiltRow& fd = p.rows[static_cast<int64_t>(b) * p.R + p.k + 1 + bs.n];
      c.md = fd.m;
      split_double(1.0 / fd.P, c.id_hi, c.id_lo);
      c.thr_d = fd.thr;
    }
    *s_cx = c;
  }
  __syncthreads();
  return true;
}

template <typename Tag>
__device__ __forceinline__ void filt_rows_n(const FiltParams& p, int b, int n,
                                            const typename Tag::Elem*& zr,
                                            const typename Tag::Elem*& dr) {
  zr = static_cast<const typename Tag::Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb +
       static_cast<int64_t>(n) * p.V;
  dr = static_cast<const typename Tag::Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
       static_cast<int64_t>(n < p.k ? n : 0) * p.V;
}

// grid (C, batch rows of this launch): per-chunk masses of the row's weights
// (2^60 units), with the thread ranges of select_in_chunk.
template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kThreads) filt_mass_kernel(FiltParams p) {
  __shared__ float2 tab[64];
  __shared__ long long sm[kWarps];
  __shared__ RowCtx s_cx;
  const int c = blockIdx.x, b = blockIdx.y + p.b0;
  load_exp2_table(tab);
  BState bs;
  if (!filt_ctx(p, b, bs, &s_cx)) return;
  const RowCtx cx = s_cx;
  const typename Tag::Elem *zr, *dr;
  filt_rows_n<Tag>(p, b, bs.n, zr, dr);
  const int clo = c * p.CH, chi = min(p.V, clo + p.CH);
  const int lo = min(chi, clo + static_cast<int>(threadIdx.x) * p.E);
  const int hi = min(chi, lo + p.E);
  float h, l;
  if (bs.mode == kModeResidual)
    range_sum<Tag, VEC, Q_FILT_RESID>(zr, dr, lo, hi, cx, tab, h, l);
  else
    range_sum<Tag, VEC, Q_FILT_TARGET>(zr, dr, lo, hi, cx, tab, h, l);
  const long long t = block_sum_i64(df_to_fix(h, l, kFixResidual), sm);
  if (threadIdx.x == 0) p.rmass[static_cast<int64_t>(b) * p.C + c] = t;
}

// grid B: the chunk, then the token.
template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kThreads) filt_select_kernel(FiltParams p) {
  __shared__ float2 tab[64];
  __shared__ long long sm[kWarps];
  __shared__ long long s_wt[kThreads];
  __shared__ int s_pick, s_chunk;
  __shared__ long long s_target;
  __shared__ RowCtx s_cx;
  const int b = blockIdx.x, tid = threadIdx.x;
  load_exp2_table(tab);
  BState bs;
  if (!filt_ctx(p, b, bs, &s_cx)) return;
  const RowCtx cx = s_cx;
  const typename Tag::Elem *zr, *dr;
  filt_rows_n<Tag>(p, b, bs.n, zr, dr);
  bool resid = bs.mode == kModeResidual;
  long long wq = tid < p.C ? p.rmass[static_cast<int64_t>(b) * p.C + tid] : 0;
  long long W;
  long long incl = block_scan_i64(wq, sm, &W);
  if (resid && W <= 0) {  // all-zero residual: draw from the filtered p_n
    resid = false;
    for (int q = 0; q < p.C; ++q) {
      const int clo = q * p.CH, chi = min(p.V, clo + p.CH);
      const int lo = min(chi, clo + tid * p.E), hi = min(chi, lo + p.E);
      float h, l;
      range_sum<Tag, VEC, Q_FILT_TARGET>(zr, dr, lo, hi, cx, tab, h, l);
      const long long t = block_sum_i64(df_to_fix(h, l, kFixResidual), sm);
      if (tid == 0) s_wt[q] = t;
    }
    __syncthreads();
    wq = tid < p.C ? s_wt[tid] : 0;
    incl = block_scan_i64(wq, sm, &W);
  }
  const long long t =
      static_cast<long long>(scale_by_uniform(static_cast<unsigned long long>(W), p.u_smp[b]));
  if (tid == 0) {
    s_chunk = p.C - 1;
    s_target = 0;
  }
  __syncthreads();
  if (wq > 0 && incl > t && incl - wq <= t) {
    s_chunk = tid;
    s_target = t - (incl - wq);
  }
  __syncthreads();
  const int q = s_chunk;
  const long long target = s_target;
  const int clo = q * p.CH, chi = min(p.V, clo + p.CH);
  int tok;
  if (resid)
    tok = select_in_chunk<Tag, VEC, Q_FILT_RESID>(zr, dr, clo, chi, p.E, cx, tab, kFixResidual,
                                                  target, sm, &s_pick);
  else
    tok = select_in_chunk<Tag, VEC, Q_FILT_TARGET>(zr, dr, clo, chi, p.E, cx, tab, kFixResidual,
                                                   target, sm, &s_pick);
  if (tid == 0) p.out_tok[static_cast<int64_t>(b) * (p.k + 1) + bs.n] = tok;
}

// Prepare the per-row draw state from a caller-supplied accept_len (used by
// the stand-alone residual call).  grid ceil(B / kThreads).

__global__ void residual_prep_kernel(PrepParams p) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  const int n = p.accept_len[b];
  const float T = p.T[b];
  const bool greedy = !(T > 0.f);
  BState bs;
  bs.n = n;
  bs.mode = (n < 0 || n > p.k || greedy || isnan(T)) ? kModeNone
                                                       : (n < p.k ? kModeResidual : kModeTarget);
  bs.c_hi = bs.c_lo = 0.f;
  bs.rho = 1.f;
  if (bs.mode != kModeNone) {
    temp_coeff(T, bs.c_hi, bs.c_lo);
    if (bs.mode == kModeResidual)
      bs.rho = static_cast<float>(p.rowstat[static_cast<int64_t>(b) * p.R + n].S /
                                  p.rowstat[static_cast<int64_t>(b) * p.R + p.k + 1 + n].S);
  }
  bs.pad0 = bs.pad1 = bs.pad2 = 0;
  p.bstate[b] = bs;
  p.amb_cnt[b] = 0;
  int32_t* o = p.out_tok + static_cast<int64_t>(b) * (p.k + 1);
  for (int j = 0; j <= p.k; ++j) {
    int v = -1;
    if (n >= 0 && n <= p.k) {
      if (j < n) v = p.x[static_cast<int64_t>(b) * p.k + j];
      else if (j == n && greedy && !isnan(T)) v = p.rowstat[static_cast<int64_t>(b) * p.R + n].argmax;
    }
    o[j] = v;
  }
}

#define SSD_DISPATCH(KERNEL, GRID)                                                  \
  do {                                                                              \
    if (dtype == 1) {                                                               \
      if (vec) KERNEL<BF16Tag, true><<<GRID, kThreads, 0, s>>>(p);                  \
      else KERNEL<BF16Tag, false><<<GRID, kThreads, 0, s>>>(p);                     \
    } else {                                                                        \
      if (vec) KERNEL<F32Tag, true><<<GRID, kThreads, 0, s>>>(p);                   \
      else KERNEL<F32Tag, false><<<GRID, kThreads, 0, s>>>(p);                      \
    }                                                                               \
  } while (0)

// grids (C, batch rows): at most 65535 batch rows per launch
cudaError_t launch_residual_norm(const ResidualParams& p0, int B, int dtype, bool vec, cudaStream_t s) {
  ResidualParams p = p0;
  for (int b0 = 0; b0 < B; b0 += kMaxGridBatch) {
    p.b0 = b0;
    SSD_DISPATCH(residual_norm_kernel, dim3(p.C, B - b0 < kMaxGridBatch ? B - b0 : kMaxGridBatch));
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
#undef SSD_DISPATCH


// The mass and select kernels follow the norm and mass kernels on the same
// stream with programmatic stream serialization: their launch overlaps the
// predecessor's tail and each waits (griddepcontrol.wait) before touching
// memory.
template <typename Kernel>
static cudaError_t launch_after(Kernel kernel, dim3 grid, cudaStream_t s, const ResidualParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute a[1];
  a[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = a;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

#define SSD_DISPATCH_AFTER(KERNEL, GRID)                                              \
  (dtype == 1 ? (vec ? launch_after(KERNEL<BF16Tag, true>, GRID, s, p)                \
                     : launch_after(KERNEL<BF16Tag, false>, GRID, s, p))              \
              : (vec ? launch_after(KERNEL<F32Tag, true>, GRID, s, p)                 \
                     : launch_after(KERNEL<F32Tag, false>, GRID, s, p)))

cudaError_t launch_residual_select(const ResidualParams& p, int B, int dtype, bool vec, cudaStream_t s) {
  return SSD_DISPATCH_AFTER(residual_select_kernel, dim3(B));
}
#undef SSD_DISPATCH_AFTER

cudaError_t launch_filt_mass(const FiltParams& p0, bool vec, cudaStream_t s) {
  FiltParams p = p0;
  for (int b0 = 0; b0 < p0.B; b0 += kMaxGridBatch) {
    p.b0 = b0;
    const dim3 grid(p.C, p0.B - b0 < kMaxGridBatch ? p0.B - b0 : kMaxGridBatch);
    if (p.dtype == 1) {
      if (vec) filt_mass_kernel<BF16Tag, true><<<grid, kThreads, 0, s>>>(p);
      else filt_mass_kernel<BF16Tag, false><<<grid, kThreads, 0, s>>>(p);
    } else {
      if (vec) filt_mass_kernel<F32Tag, true><<<grid, kThreads, 0, s>>>(p);
      else filt_mass_kernel<F32Tag, false><<<grid, kThreads, 0, s>>>(p);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_filt_select(const FiltParams& p, bool vec, cudaStream_t s) {
  if (p.dtype == 1) {
    if (vec) filt_select_kernel<BF16Tag, true><<<p.B, kThreads, 0, s>>>(p);
    else filt_select_kernel<BF16Tag, false><<<p.B, kThreads, 0, s>>>(p);
  } else {
    if (vec) filt_select_kernel<F32Tag, true><<<p.B, kThreads, 0, s>>>(p);
    else filt_select_kernel<F32Tag, false><<<p.B, kThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_residual_prep(const PrepParams& p, cudaStream_t s) {
  residual_prep_kernel<<<(p.B + 127) / 128, 128, 0, s>>>(p);
  return cudaGetLastError();
}

// Self-test of exp2_df: out[i] = 2^(x_hi + x_lo).
__global__ void selftest_exp2_kernel(const float* xh, const float* xl, double* out, int n) {
  __shared__ float2 tab[64];
  load_exp2_table(tab);
  __syncthreads();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    float h, l;
    exp2_df(xh[i], xl[i], tab, h, l);
    out[i] = static_cast<double>(h) + static_cast<double>(l);
  }
}

cudaError_t launch_selftest_exp2(const float* xh, const float* xl, double* out, int n, cudaStream_t s) {
  int blocks = (n + 255) / 256;
  if (blocks > 1024) blocks = 1024;
  if (blocks < 1) blocks = 1;
  selftest_exp2_kernel<<<blocks, 256, 0, s>>>(xh, xl, out, n);
  return cudaGetLastError();
}

}  // namespace ssd
