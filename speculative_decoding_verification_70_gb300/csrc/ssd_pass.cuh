// ssd_pass.cuh -- one CTA's streaming pass over a chunk of a logit row:
// the online-softmax statistics (maximum, lowest argmax, NaN flag, sum of
// 2^((z - m) c); Milakov & Gimelshein 2018), the certified top-f of the
// chunk for the forked recovery (masked tokens skipped) and, for the
// drafter's own sampling, the best Gumbel-perturbed logit; and one CTA's
// whole unit of the verify statistics (stats_unit).  Shared by the
// statistics kernels (ssd_stats.cu) and the small-batch step kernel
// (ssd_step.cu).
#pragma once

#include <math.h>

#include "ssd_device.cuh"
#include "ssd_layout.h"
#include "ssd_scan.cuh"

namespace ssd {

struct StatsSmem {
  float m[kWarps], s[kWarps];
  int i[kWarps], n[kWarps];
  float gy[kWarps];
  int gi[kWarps];
  int mask[kMaxMask];
};

// ---------------------------------------------------------------------------
// Draft-side sampling: Gumbel-max draws argmax_v (z_v / T - ln(-ln u_v)),
// an exact draw from softmax(z / T) (the Gumbel-max trick), with u_v from
// the counter-based generator Philox4x32-10 (Salmon, Moraes, Dror & Shaw
// 2011): element v of draft row i of batch row b takes word v mod 4 of the
// generator at counter (v / 4, i, b, offset) under key (seed_lo, seed_hi),
// and u = (w >> 9 + 1/2) / 2^23 (23 bits: u and 1 - u are exact floats).
// ---------------------------------------------------------------------------
struct GumbelArgs {
  const uint32_t* rk0;  // round keys: key word 0 of rounds 0..9
  const uint32_t* rk1;  // key word 1
  uint32_t row, b, offset;
  float invT;
};

// Ten rounds of Philox4x32 on counter c with precomputed round keys (the
// seed's key schedule, formed once on the host): per round two 32x32->64
// products, the high halves XORed with the other counter words and the
// round key.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, const uint32_t* rk0,
                                               const uint32_t* rk1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    unsigned long long p0, p1;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c.x), "r"(0xD2511F53u));
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c.z), "r"(0xCD9E8D57u));
    const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
    const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
    c = make_uint4(hi1 ^ c.y ^ rk0[r], lo1, hi0 ^ c.w ^ rk1[r], lo0);
  }
  return c;
}

__device__ __forceinline__ float lg2_fast(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// z / T + G for one element: G = -ln(E), E = -ln u.  E is taken from the
// series v + v^2/2 + ... + v^5/5 of -ln(1 - v), v = 1 - u, when v < 1/16
// (truncation below v^6/6 relative, < 1e-8), else as -ln 2 * log2(u); both
// logarithms use the MUFU log2 (absolute error ~2^-22 in log2), so G is off
// by at most ~2e-6 -- a token can differ from an exact computation only when
// two perturbed logits tie that closely.
__device__ __forceinline__ float gumbel_key(float z, float invT, uint32_t w) {
  const uint32_t m = w >> 9;
  // u = (m + 1/2) 2^-23 and v = 1 - u without an integer-to-float
  // conversion (a quarter-rate instruction): 1 + m 2^-23 is the float with
  // mantissa m, and subtracting 1 - 2^-24 from it is exact (the operands are
  // within a factor 2), as is 1 - u; the values are those of the definition
  constexpr float kLn2 = 0.693147180559945309f;
  const float u = __uint_as_float(0x3f800000u | m) - __uint_as_float(0x3f7fffffu);
  const float v = 1.0f - u;
  float s = fmaf(v, 0.2f, 0.25f);
  s = fmaf(v, s, 0.333333333f);
  s = fmaf(v, s, 0.5f);
  s = fmaf(v, s, 1.0f);
  const float e = v < 0.0625f ? v * s : -kLn2 * lg2_fast(u);
  return fmaf(z, invT, -kLn2 * lg2_fast(e));
}

// Fold the kv elements z[0..kv) starting at index `base` into the thread's
// best (gy, gi); elements arrive in increasing index order, so a strict
// compare keeps the lowest index on ties.
template <int KV>
__device__ __forceinline__ void gumbel_vector(const GumbelArgs& g, const float (&z)[8], int base,
                                              float& gy, int& gi) {
  if (KV == 1) {
    const uint4 w = philox4x32_10(make_uint4(static_cast<uint32_t>(base) >> 2, g.row, g.b, g.offset),
                                  g.rk0, g.rk1);
    const int q = base & 3;
    const uint32_t word = q == 0 ? w.x : (q == 1 ? w.y : (q == 2 ? w.z : w.w));
    const float y = gumbel_key(z[0], g.invT, word);
    if (y > gy) {
      gy = y;
      gi = base;
    }
  } else {
#pragma unroll
    for (int h = 0; h < KV / 4; ++h) {
      const uint4 w = philox4x32_10(
          make_uint4((static_cast<uint32_t>(base) >> 2) + h, g.row, g.b, g.offset), g.rk0, g.rk1);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float y = gumbel_key(z[4 * h + e], g.invT, ws[e]);
        if (y > gy) {
          gy = y;
          gi = base + 4 * h + e;
        }
      }
    }
  }
}

constexpr int kMaxF = 16;

// Top-f scratch: every thread's maximum, the warps' largest second values
// and the selection.
constexpr int kTopfSecond = 256;  // entries of the second-chance buffer

struct TopfScratch {
  float cv[kThreads];
  int ci[kThreads];
  float xv[kTopfSecond];           // second chance: elements of overflowing threads
  int xi[kTopfSecond];
  int nx;
  float w2[kWarps];
  float sv[kMaxF];
  int si[kMaxF];
  float bv[kWarps];
  int bi[kWarps];
};

// Best (value, index) among this thread's elements of [lo, hi) (vectors t,
// t+256, ...) that rank after (pv, pi), skipping masked tokens and NaN.
template <typename Tag, bool VEC>
__device__ __forceinline__ void best_after(const typename Tag::Elem* row, int lo, int hi, float pv,
                                           int pi, const int* msk, int M, float& bv, int& bi) {
  constexpr int kV = VEC ? Tag::kVec : 1;
  bv = -INFINITY;
  bi = kIdxNone;
  const int v0 = lo / kV, v1 = (hi + kV - 1) / kV;
  for (int v = v0 + threadIdx.x; v < v1; v += kThreads) {
    float z[8];
    if (VEC) Tag::loadv_cached(row + static_cast<int64_t>(v) * kV, z);
    else z[0] = Tag::load1(row + v);
#pragma unroll
    for (int e = 0; e < kV; ++e) {
      const int idx = v * kV + e;
      if (z[e] == z[e] && ranks_before(pv, pi, z[e], idx) && ranks_before(z[e], idx, bv, bi) &&
          !is_masked(idx, msk, M)) {
        bv = z[e];
        bi = idx;
      }
    }
  }
}

// First half of the top-f selection, before the block reduction of the
// statistics (whose barrier publishes it): each thread posts its maximum as a
// candidate (none if masked) and each warp the largest "second value" of its
// threads -- m2, every element of a thread except its maximum is at most m2;
// a thread that saw a NaN posts NaN, which sends the CTA to the exact path.
__device__ __forceinline__ void topf_post(const ScanState& st, const int* msk, int M,
                                          TopfScratch& ts) {
  const int tid = threadIdx.x, lane = tid & 31;
  const bool ok = st.idx != kIdxNone && !is_masked(st.idx, msk, M);
  ts.cv[tid] = ok ? st.m : -INFINITY;
  ts.ci[tid] = ok ? st.idx : kIdxNone;
  float w2 = st.nan ? NAN : st.m2;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) w2 = max_nan(w2, __shfl_xor_sync(kFull, w2, o));
  if (lane == 0) ts.w2[tid >> 5] = w2;
}

// Top f of the CTA's elements (logit descending, index ascending, masked
// tokens and NaN skipped).  Warp 0 picks the f best of the 256 posted thread
// maxima.  Certified: with M2 the largest second value of any thread, every
// element that is not a thread maximum is at most M2, so if at least f
// unmasked maxima exceed M2 the picks are exact.  Otherwise (a few percent
// of CTAs; e.g. several top logits in one vector) a second chance: with tau
// the f-th pick, every missing element ranks before tau and sits in a thread
// whose second value is >= tau, so only those threads re-read their own
// elements and add the ones ranking before tau; the f best of the picks and
// these extras are exact.  A NaN, fewer than f picks or an overflowing
// buffer take the last resort: f rounds of a block-wide arg-max.  Needs
// topf_post and a barrier before it.
template <typename Tag, bool VEC>
__device__ void topf_select(const StatsParams& p, const ScanState& st,
                            const typename Tag::Elem* row, int lo, int hi, const int* msk,
                            TopEntry* out_top, int n_slots, TopfScratch& ts) {
  constexpr int kV = VEC ? Tag::kVec : 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int f = p.f, M = p.M;
  float M2 = ts.w2[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M2 = max_nan(M2, ts.w2[w]);
  const bool cand = ts.ci[tid] != kIdxNone && ts.cv[tid] > M2;  // false when M2 is NaN
  if (tid == 0) ts.nx = 0;
  const bool certified = __syncthreads_count(cand) >= f;
  if (warp == 0) {
    float pv = INFINITY;
    int pi = -1;
    for (int r = 0; r < f; ++r) {
      float bv = -INFINITY;
      int bi = kIdxNone;
#pragma unroll
      for (int q = lane; q < kThreads; q += 32) {
        const float v = ts.cv[q];
        const int i = ts.ci[q];
        if (ranks_before(pv, pi, v, i) && ranks_before(v, i, bv, bi)) {
          bv = v;
          bi = i;
        }
      }
      warp_argmax(bv, bi);
      if (lane == 0) {
        ts.sv[r] = bv;
        ts.si[r] = bi;
      }
      pv = bv;
      pi = bi;
    }
  }
  // the group's list goes to its first chunk slot; the other slots of the
  // group get empty entries, which rank last in the merge
  if (certified) {
    if (warp != 0) return;
    __syncwarp();
    for (int q = lane; q < n_slots * f; q += 32) {
      const int slot = q / f, r = q % f;
      out_top[q].v = slot == 0 ? ts.sv[r] : -INFINITY;
      out_top[q].i = slot == 0 ? ts.si[r] : kIdxNone;
    }
    return;
  }
  __syncthreads();
  const float tv = ts.sv[f - 1];
  const int ti = ts.si[f - 1];
  const bool second = ti != kIdxNone && M2 == M2;
  if (second && st.m2 >= tv) {
    const int v0 = lo / kV, v1 = (hi + kV - 1) / kV;
    for (int v = v0 + tid; v < v1; v += kThreads) {
      float z[8];
      if (VEC) Tag::loadv_cached(row + static_cast<int64_t>(v) * kV, z);
      else z[0] = Tag::load1(row + v);
#pragma unroll
      for (int e = 0; e < kV; ++e) {
        const int idx = v * kV + e;
        if (idx != ts.ci[tid] && z[e] == z[e] && ranks_before(z[e], idx, tv, ti) &&
            !is_masked(idx, msk, M)) {
          const int q = atomicAdd(&ts.nx, 1);
          if (q < kTopfSecond) {
            ts.xv[q] = z[e];
            ts.xi[q] = idx;
          }
        }
      }
    }
  }
  __syncthreads();
  const int nx = ts.nx;
  if (second && nx <= kTopfSecond) {
    if (warp != 0) return;
    float pv = INFINITY;
    int pi = -1;
    float keep_v = -INFINITY;
    int keep_i = kIdxNone;
    for (int r = 0; r < f; ++r) {
      float bv = -INFINITY;
      int bi = kIdxNone;
      for (int q = lane; q < f + nx; q += 32) {
        const float v = q < f ? ts.sv[q] : ts.xv[q - f];
        const int i = q < f ? ts.si[q] : ts.xi[q - f];
        if (i != kIdxNone && ranks_before(pv, pi, v, i) && ranks_before(v, i, bv, bi)) {
          bv = v;
          bi = i;
        }
      }
      warp_argmax(bv, bi);
      if (lane == r) {
        keep_v = bv;
        keep_i = bi;
      }
      pv = bv;
      pi = bi;
    }
    __syncwarp();
    if (lane < f) {
      ts.sv[lane] = keep_i == kIdxNone ? -INFINITY : keep_v;
      ts.si[lane] = keep_i;
    }
    __syncwarp();
    for (int q = lane; q < n_slots * f; q += 32) {
      const int slot = q / f, r = q % f;
      out_top[q].v = slot == 0 ? ts.sv[r] : -INFINITY;
      out_top[q].i = slot == 0 ? ts.si[r] : kIdxNone;
    }
    return;
  }
  // last resort: f rounds of a block-wide arg-max over [lo, hi)
  float pv = INFINITY;
  int pi = -1;
  for (int r = 0; r < f; ++r) {
    float bv;
    int bi;
    best_after<Tag, VEC>(row, lo, hi, pv, pi, msk, M, bv, bi);
    warp_argmax(bv, bi);
    if (lane == 0) {
      ts.bv[warp] = bv;
      ts.bi[warp] = bi;
    }
    __syncthreads();
    bv = ts.bv[0];
    bi = ts.bi[0];
    for (int w = 1; w < kWarps; ++w)
      if (ranks_before(ts.bv[w], ts.bi[w], bv, bi)) {
        bv = ts.bv[w];
        bi = ts.bi[w];
      }
    __syncthreads();
    if (tid == 0) {
      ts.sv[r] = bv;
      ts.si[r] = bi;
    }
    pv = bv;
    pi = bi;
  }
  __syncthreads();
  for (int q = tid; q < n_slots * f; q += kThreads) {
    const int slot = q / f, r = q % f;
    out_top[q].v = slot == 0 ? ts.sv[r] : -INFINITY;
    out_top[q].i = slot == 0 ? ts.si[r] : kIdxNone;
  }
}

template <typename Tag, bool VEC, bool DO_EXP, bool TOPF, bool GUMBEL = false>
__device__ void stats_chunk(const StatsParams& p, const typename Tag::Elem* row, int lo, int hi,
                            float c, PartStat* out_part, TopEntry* out_top, int n_slots,
                            StatsSmem& sm, TopfScratch* ts, const GumbelArgs* ga = nullptr,
                            GumbelPart* out_g = nullptr) {
  constexpr int kV = VEC ? Tag::kVec : 1;
  constexpr int U = Tag::kUnroll;
  const int tid = threadIdx.x;
  ScanState st;
  scan_init(st);
  float gy = -INFINITY;
  int gi = kIdxNone;
  const int v0 = lo / kV, v1 = (hi + kV - 1) / kV;
  // the branch-free maximum update (index resolved after the pass) where
  // the per-element work is heavier than a long fp32 stream's: bf16
  // vectors and the Gumbel pass
  constexpr bool kDefer = kV > 1 && (GUMBEL || kV == 8);
  for (int vb = v0 + tid; vb < v1; vb += kThreads * U) {
    typename Tag::Raw raw[U];
    float sc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = vb + u * kThreads;
      if (vi < v1) {
        if (VEC) raw[u] = Tag::loadraw(row + static_cast<int64_t>(vi) * kV);
        else sc[u] = Tag::load1(row + vi);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int vi = vb + u * kThreads;
      if (vi < v1) {
        if constexpr (VEC && !GUMBEL && kV == 8) {
          scan_bf16<DO_EXP, TOPF>(st, raw[u], vi * kV, c);
        } else {
          float z[8];
          if (VEC) Tag::unpackraw(raw[u], z);
          else z[0] = sc[u];
          float m = z[0];
#pragma unroll
          for (int e = 1; e < kV; ++e) m = max_nan(m, z[e]);
          scan_vector<DO_EXP, TOPF, kDefer>(st, z, kV, m, vi * kV, c);
          if constexpr (GUMBEL) gumbel_vector<kV>(*ga, z, vi * kV, gy, gi);
        }
      }
    }
  }
  if constexpr (kDefer) {  // the argmax's place inside its vector (an L2 hit)
    if (st.idx != kIdxNone && !st.nan) {
      float z[8];
      Tag::unpackraw(Tag::loadraw(row + st.idx), z);
      scan_resolve(st, z, kV);
    }
  }
  if constexpr (GUMBEL) {
    warp_argmax(gy, gi);
    if ((tid & 31) == 0) {
      sm.gy[tid >> 5] = gy;
      sm.gi[tid >> 5] = gi;
    }
  }
  if constexpr (TOPF) topf_post(st, sm.mask, p.M, *ts);
  block_stats_write(st, c, DO_EXP, sm.m, sm.s, sm.i, sm.n, out_part);  // holds a barrier
  if constexpr (GUMBEL) {
    if (tid == 0) {
      GumbelPart g;
      g.y = sm.gy[0];
      g.idx = sm.gi[0];
      for (int w = 1; w < kWarps; ++w)
        if (ranks_before(sm.gy[w], sm.gi[w], g.y, g.idx)) {
          g.y = sm.gy[w];
          g.idx = sm.gi[w];
        }
      *out_g = g;
    }
  }
  if constexpr (TOPF) topf_select<Tag, VEC>(p, st, row, lo, hi, sm.mask, out_top, n_slots, *ts);
}

// Statistics of chunks c .. c + G - 1 of logit row r of batch row b (the
// work of one CTA of the statistics kernel; G = p.G): one partial record for
// the group in slot c, identity records in the group's other slots, and for
// a draft row below Pdf its top-f list.  Uniform over the CTA; holds
// barriers.
template <typename Tag, bool VEC>
__device__ __forceinline__ void stats_unit(const StatsParams& p, int b, int r, int c, StatsSmem& sm,
                                           TopfScratch& ts, float2* s_c) {
  using Elem = typename Tag::Elem;
  const int lo = c * p.CH, hi = min(p.V, lo + p.G * p.CH);
  const int n_slots = min(p.G, p.C - c);
  const Elem* row;
  bool need_stats, need_top = false;
  int j = 0;
  if (r < p.Pz) {
    row = static_cast<const Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb + static_cast<int64_t>(r) * p.V;
    need_stats = true;
  } else {
    j = r - p.Pz;
    row = static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db + static_cast<int64_t>(j) * p.V;
    need_stats = j < p.Pds;
    need_top = p.f > 0 && j < p.Pdf;
    if (!need_stats && !need_top) return;
  }
  const float T = p.T ? p.T[b] : 0.f;
  const bool do_exp = need_stats && T > 0.f;  // uniform over the CTA
  float cf = 0.f;
  if (do_exp) cf = cta_temp_coeff(T, s_c).x;
  PartStat* out_part = p.part + (static_cast<int64_t>(b) * p.Rp + r) * p.C + c;
  if (threadIdx.x > 0 && threadIdx.x < n_slots) {
    PartStat id;
    id.m = -INFINITY;
    id.s = 0.f;
    id.idx = kIdxNone;
    id.flags = 0;
    out_part[threadIdx.x] = id;
  }
  if (need_top) {
    if (threadIdx.x < p.M)
      sm.mask[threadIdx.x] = p.mask[(static_cast<int64_t>(b) * p.Pdf + j) * p.M + threadIdx.x];
    __syncthreads();
    TopEntry* out_top = p.topk + ((static_cast<int64_t>(b) * p.Pdf + j) * p.C + c) * p.f;
    if (do_exp)
      stats_chunk<Tag, VEC, true, true>(p, row, lo, hi, cf, out_part, out_top, n_slots, sm, &ts);
    else
      stats_chunk<Tag, VEC, false, true>(p, row, lo, hi, cf, out_part, out_top, n_slots, sm, &ts);
    return;
  }
  if (do_exp)
    stats_chunk<Tag, VEC, true, false>(p, row, lo, hi, cf, out_part, nullptr, 0, sm, nullptr);
  else
    stats_chunk<Tag, VEC, false, false>(p, row, lo, hi, cf, out_part, nullptr, 0, sm, nullptr);
}

}  // namespace ssd

