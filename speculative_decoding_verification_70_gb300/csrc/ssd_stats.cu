// ssd_stats.cu -- the streaming pass over the logit rows (kernel K-A) and the
// per-batch-row finalisation (acceptance, first-reject prefix, greedy token,
// forked top-f merge).
//
// Sources: "tanishqkumar/ssd" summary, module notes (temperature sampler:
// greedy at T = 0; forked recovery: top-k over logits with masking);
// "SSD: drafting and verification on separate GPUs", "What changes in SSD"
// (verify the draft in one pass); speculative-sampling summary, "How It
// Works" (regenerate from the point of divergence); the min(1, p/q)
// acceptance rule of Leviathan et al. / Chen et al.
//
// Layout of the work: one CTA per (chunk, row, batch row).  Each thread reads
// its vectors t, t+256, t+512, ... of the chunk with 16-byte streaming loads,
// keeping a running maximum, the lowest index attaining it and the running
// sum of 2^((z - m) c) (rescaled when the maximum grows: the online-softmax
// recurrence of Milakov & Gimelshein 2018).  For draft rows that feed the
// forked recovery each warp also keeps one shared top-f list.  A CTA writes
// one partial record; a second kernel merges the records of a batch row in
// chunk order.
#include <math.h>

#include "ssd_device.cuh"
#include "ssd_layout.h"
#include "ssd_merge.cuh"
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
  uint32_t k0, k1, row, b, offset;
  float invT;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
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
  const float v = (static_cast<float>(8388607u - m) + 0.5f) * 1.1920928955078125e-7f;  // 1 - u
  constexpr float kLn2 = 0.693147180559945309f;
  const float u = (static_cast<float>(m) + 0.5f) * 1.1920928955078125e-7f;
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
                                  g.k0, g.k1);
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
          make_uint4((static_cast<uint32_t>(base) >> 2) + h, g.row, g.b, g.offset), g.k0, g.k1);
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
  constexpr int U = 4;
  const int tid = threadIdx.x;
  ScanState st;
  scan_init(st);
  float gy = -INFINITY;
  int gi = kIdxNone;
  const int v0 = lo / kV, v1 = (hi + kV - 1) / kV;
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
        float z[8];
        if (VEC) Tag::unpackraw(raw[u], z);
        else z[0] = sc[u];
        float m = z[0];
#pragma unroll
        for (int e = 1; e < kV; ++e) m = max_nan(m, z[e]);
        scan_vector<DO_EXP, TOPF>(st, z, kV, m, vi * kV, c);
        if constexpr (GUMBEL) gumbel_vector<kV>(*ga, z, vi * kV, gy, gi);
      }
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

// grid: (C, rows of this launch, B).  Resident CTAs per SM requested from
// the register allocator: enough 16-byte loads in flight to saturate HBM.
#ifndef SSD_TOPF_MIN_BLOCKS
#define SSD_TOPF_MIN_BLOCKS 6
#endif
template <typename Tag, bool VEC, bool HAS_TOPF>
__global__ void __launch_bounds__(kThreads, HAS_TOPF ? SSD_TOPF_MIN_BLOCKS : 6)
    stats_kernel(StatsParams p) {
  using Elem = typename Tag::Elem;
  // A CTA of the plain variant covers p.G consecutive chunks: one reduction
  // for the group, written to the group's first partial; the others get the
  // identity record (m = -inf, s = 0, no index).
  const int G = p.G;
  const int c = blockIdx.x * G, r = blockIdx.y + p.r0, b = blockIdx.z + p.b0;
  const int lo = c * p.CH;
  const int hi = min(p.V, lo + G * p.CH);
  const int n_slots = min(G, p.C - c);
  __shared__ StatsSmem sm;

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
    need_top = HAS_TOPF && j < p.Pdf;
    if (!need_stats && !need_top) return;
    if (p.tree_parent) {  // a tree leaf's draft row is never used: not read
      const int t = threadIdx.x;
      const bool kid = t > j && t < p.tree_N &&
                       p.tree_parent[static_cast<int64_t>(b) * p.tree_N + t] == j;
      if (!__syncthreads_or(kid)) return;
    }
  }
  float T = p.T ? p.T[b] : 0.f;
  bool do_exp = need_stats && (T > 0.f);  // uniform over the CTA
  float cf = 0.f;
  __shared__ float2 s_c;
  if (do_exp) cf = cta_temp_coeff(T, &s_c).x;
  PartStat* out_part = p.part + (static_cast<int64_t>(b) * p.Rp + r) * p.C + c;
  if (threadIdx.x > 0 && threadIdx.x < n_slots) {
    PartStat id;
    id.m = -INFINITY;
    id.s = 0.f;
    id.idx = kIdxNone;
    id.flags = 0;
    out_part[threadIdx.x] = id;
  }
  if constexpr (HAS_TOPF) {
    if (need_top) {
      __shared__ TopfScratch ts;
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
  }
  if (do_exp)
    stats_chunk<Tag, VEC, true, false>(p, row, lo, hi, cf, out_part, nullptr, 0, sm, nullptr);
  else
    stats_chunk<Tag, VEC, false, false>(p, row, lo, hi, cf, out_part, nullptr, 0, sm, nullptr);
}

// Draft-side sampling pass.  grid: (chunk groups, draft rows of this call,
// batch rows).  Each CTA streams G chunks of draft row i = blockIdx.y + r0
// once and writes, into the verify workspace, the row's partial statistics
// (slot Pz + i, so a later ssd_verify_drafted skips these rows), the best
// Gumbel-perturbed logit (T > 0 rows) and, with HAS_TOPF, a top-(f+1) list
// (the forks with the drafted token masked are taken from it at the merge).
template <typename Tag, bool VEC, bool HAS_TOPF>
__global__ void __launch_bounds__(kThreads, SSD_TOPF_MIN_BLOCKS) draft_kernel(StatsParams p) {
  using Elem = typename Tag::Elem;
  const int G = p.G;
  const int c = blockIdx.x * G, i = blockIdx.y + p.r0, b = blockIdx.z + p.b0;
  const int lo = c * p.CH;
  const int hi = min(p.V, lo + G * p.CH);
  const int n_slots = min(G, p.C - c);
  __shared__ StatsSmem sm;
  __shared__ float2 s_c;
  const Elem* row = static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
                    static_cast<int64_t>(i) * p.V;
  const float T = p.T[b];
  const bool do_exp = T > 0.f;  // NaN and T <= 0: statistics without exponentials
  float cf = 0.f;
  if (do_exp) cf = cta_temp_coeff(T, &s_c).x;
  PartStat* out_part = p.part + (static_cast<int64_t>(b) * p.Rp + p.Pz + i) * p.C + c;
  GumbelPart* out_g = p.gpart + (static_cast<int64_t>(b) * p.Pf + i) * p.C + c;
  if (threadIdx.x < n_slots) {
    GumbelPart none;
    none.y = -INFINITY;
    none.idx = kIdxNone;
    if (threadIdx.x > 0 || !do_exp) out_g[threadIdx.x] = none;
    if (threadIdx.x > 0) {
      PartStat id;
      id.m = -INFINITY;
      id.s = 0.f;
      id.idx = kIdxNone;
      id.flags = 0;
      out_part[threadIdx.x] = id;
    }
  }
  GumbelArgs ga;
  ga.k0 = p.seed_lo;
  ga.k1 = p.seed_hi;
  ga.row = static_cast<uint32_t>(i);
  ga.b = static_cast<uint32_t>(b);
  ga.offset = p.offset;
  ga.invT = do_exp ? 1.0f / T : 0.f;
  if constexpr (HAS_TOPF) {
    __shared__ TopfScratch ts;  // no masked tokens (M == 0)
    TopEntry* out_top = p.topk + ((static_cast<int64_t>(b) * p.Pf + i) * p.C + c) * p.f;
    if (do_exp)
      stats_chunk<Tag, VEC, true, true, true>(p, row, lo, hi, cf, out_part, out_top, n_slots, sm,
                                              &ts, &ga, out_g);
    else
      stats_chunk<Tag, VEC, false, true, false>(p, row, lo, hi, cf, out_part, out_top, n_slots, sm,
                                                &ts);
    return;
  }
  if (do_exp)
    stats_chunk<Tag, VEC, true, false, true>(p, row, lo, hi, cf, out_part, nullptr, 0, sm, nullptr,
                                             &ga, out_g);
  else
    stats_chunk<Tag, VEC, false, false, false>(p, row, lo, hi, cf, out_part, nullptr, 0, sm,
                                               nullptr);
}

// Merge of the draft pass, one warp per (b, draft row): the drafted token
// (T > 0: the best Gumbel-perturbed logit over the chunks; T == 0: the
// argmax; -1 for an invalid temperature or row) and, when f > 0, the f best
// logits of the row other than the drafted token (the SSD forks with the
// drafter's own token masked), from the chunks' top-(f+1) lists.
__global__ void __launch_bounds__(kThreads) draft_finalize_kernel(DraftParams p) {
  __shared__ int heads[kWarps][256];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long w = static_cast<long long>(blockIdx.x) * kWarps + warp;
  if (w >= static_cast<long long>(p.B) * p.rows) return;  // whole warp
  const int b = static_cast<int>(w / p.rows), r = static_cast<int>(w % p.rows), i = p.row0 + r;
  const float T = p.T[b];
  const bool t_bad = isnan(T) || T < 0.f;
  const bool greedy = !(T > 0.f);
  // maximum, lowest argmax and NaN flag of the row
  const PartStat* parts = p.part + (static_cast<int64_t>(b) * p.Rp + p.Pz + i) * p.C;
  float m = -INFINITY;
  int idx = kIdxNone, nan = 0;
  for (int q = lane; q < p.C; q += 32) {
    const PartStat ps = parts[q];
    nan |= ps.flags & 1;
    if (ranks_before(ps.m, ps.idx, m, idx)) {
      m = ps.m;
      idx = ps.idx;
    }
  }
  warp_argmax(m, idx);
  nan = __any_sync(kFull, nan);
  const bool bad = t_bad || nan || (!greedy && (m == INFINITY || m == -INFINITY));
  int x = -1;
  if (!bad && greedy) {
    x = idx == kIdxNone ? -1 : idx;
  } else if (!bad) {
    const GumbelPart* gp = p.gpart + (static_cast<int64_t>(b) * p.Pf + i) * p.C;
    float gy = -INFINITY;
    int gi = kIdxNone;
    for (int q = lane; q < p.C; q += 32) {
      const GumbelPart g = gp[q];
      if (ranks_before(g.y, g.idx, gy, gi)) {
        gy = g.y;
        gi = g.idx;
      }
    }
    warp_argmax(gy, gi);
    x = gi == kIdxNone ? -1 : gi;
  }
  if (lane == 0) {
    p.x_out[static_cast<int64_t>(b) * p.x_bstride + r] = x;
    int e = 0;
    if (t_bad) e |= 0x1;
    else if (bad) e |= 0x2;
    if (e) atomicOr(p.err, e);
  }
  if (p.f <= 0) return;
  // forks: merge the chunks' top-(f+1) lists, skipping the drafted token
  const int F1 = p.f + 1;
  const TopEntry* lists = p.topk + (static_cast<int64_t>(b) * p.Pf + i) * p.C * F1;
  int32_t* tok_out = p.fork_tok + (static_cast<int64_t>(b) * p.rows + r) * p.f;
  float* logit_out = p.fork_logit + (static_cast<int64_t>(b) * p.rows + r) * p.f;
  int* hd = heads[warp];
  for (int q = lane; q < p.C; q += 32) hd[q] = 0;
  __syncwarp();
  int out_n = 0;
  for (int round = 0; round < F1 && out_n < p.f; ++round) {
    float bv = -INFINITY;
    int bi = kIdxNone, bq = -1;
    for (int q = lane; q < p.C; q += 32) {
      const int h = hd[q];
      if (h < F1) {
        const TopEntry e = lists[q * F1 + h];
        if (bq < 0 || ranks_before(e.v, e.i, bv, bi)) {
          bv = e.v;
          bi = e.i;
          bq = q;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, o);
      const int oi = __shfl_xor_sync(kFull, bi, o);
      const int oq = __shfl_xor_sync(kFull, bq, o);
      const bool take = (oq >= 0) && (bq < 0 || ranks_before(ov, oi, bv, bi) ||
                                      (ov == bv && oi == bi && oq < bq));
      if (take) {
        bv = ov;
        bi = oi;
        bq = oq;
      }
    }
    if (bq < 0 || bi == kIdxNone) break;  // lists exhausted
    if (lane == (bq & 31)) hd[bq] += 1;
    __syncwarp();
    if (bi == x) continue;  // the drafted token is masked
    if (lane == 0) {
      tok_out[out_n] = nan ? -1 : bi;
      logit_out[out_n] = nan ? NAN : bv;
    }
    ++out_n;
  }
  if (lane == 0)
    for (int q = out_n; q < p.f; ++q) {
      tok_out[q] = -1;
      logit_out[q] = nan ? NAN : -INFINITY;
    }
}

// ---------------------------------------------------------------------------
// Finalisation.
// ---------------------------------------------------------------------------

__device__ __forceinline__ float logit_at(const void* base, int dtype, int64_t i) {
  if (dtype == 1)
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(base) + i)) << 16);
  return __ldg(static_cast<const float*>(base) + i);
}

// grid: B.  Verification (and, when fork_tok != null, the forked top-f).
// NW warps per CTA: 8 for large batches; 16 at small B, where the CTA's
// row merges are the critical path (one round for 2(k+1) <= 16 rows).
template <int NW>
__global__ void __launch_bounds__(NW * 32) finalize_kernel(FinalizeParams p) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float2 tab[64];
  __shared__ RowStat rs[2 * (32 + 1)];
  __shared__ float2 rsum[2 * (32 + 1)];  // each row's S as a float pair
  __shared__ int heads[NW][256];
  load_exp2_table(tab);
  __syncthreads();

  const float T = p.T ? p.T[b] : 0.f;
  const bool t_bad = p.T ? (isnan(T) || T < 0.f) : false;
  const bool greedy = !(T > 0.f);
  float c_hi = 0.f, c_lo = 0.f;
  __shared__ float2 s_c;
  if (!greedy && !t_bad) {
    const float2 cc = cta_temp_coeff(T, &s_c);
    c_hi = cc.x;
    c_lo = cc.y;
  }

  // 1. merge the row statistics
  const int nstat = p.Pz + p.Pds;
  for (int r = warp; r < p.R; r += NW) {
    bool is_target = r < p.Pz;
    int j = r - p.Pz;
    bool need_stats = is_target || j < p.Pds;
    bool do_exp = need_stats && !greedy && !t_bad;
    RowStat st;
    float sh, sl;
    merge_row(p.part + (static_cast<int64_t>(b) * p.Rp + r) * p.C, p.C, c_hi, c_lo, do_exp, tab, st,
              sh, sl);
    if (lane == 0) {
      rs[r] = st;
      rsum[r] = make_float2(sh, sl);
      p.rowstat[static_cast<int64_t>(b) * p.Rp + r] = st;
    }
    // forked top-f of draft row j
    if (!is_target && j < p.Pdf && p.fork_tok) {
      int64_t o = (static_cast<int64_t>(b) * p.Pdf + j) * p.f;
      // variable fan-out: f_j tokens at position j, clamped to [0, f]
      const int keep = p.fanout ? min(max(__ldg(p.fanout + j), 0), p.f) : p.f;
      merge_topf_row(p.topk + (static_cast<int64_t>(b) * p.Pdf + j) * p.C * p.f, p.C, p.f, keep,
                     (st.flags & 1) != 0, p.fork_tok + o, p.fork_logit + o, heads[warp]);
      if (lane == 0 && (st.flags & 1)) atomicOr(p.err, 0x2);
    }
  }
  __syncthreads();
  if (nstat == 0 || p.k == 0 || warp != 0) return;

  // 2. acceptance at each draft position (lane i), first-reject prefix
  const int k = p.k;
  int xi = -1;
  bool tok_bad = false;
  if (lane < k) {
    xi = p.x[static_cast<int64_t>(b) * k + lane];
    tok_bad = xi < 0 || xi >= p.V;
  }
  bool any_tok_bad = __any_sync(kFull, tok_bad);
  bool row_bad = false;
  if (lane <= k) row_bad |= (rs[lane].flags & 2) != 0;                 // target rows 0..k
  if (lane < k) row_bad |= (rs[p.Pz + lane].flags & 2) != 0;           // draft rows 0..k-1
  bool any_row_bad = __any_sync(kFull, row_bad);

  int status = 0;  // 0 ok, -1 invalid, -2 bad token
  if (t_bad) status = -1;
  else if (any_tok_bad) status = -2;
  else if (any_row_bad) status = -1;

  float pv = NAN, qv = NAN;
  bool acc = false;
  if (status == 0 && lane < k) {
    const RowStat& tz = rs[lane];
    const RowStat& td = rs[p.Pz + lane];
    if (greedy) {
      acc = (xi == tz.argmax);
      pv = acc ? 1.f : 0.f;
      qv = (xi == td.argmax) ? 1.f : 0.f;
    } else {
      float zx = logit_at(p.Z, p.dtype, static_cast<int64_t>(b) * p.zb + static_cast<int64_t>(lane) * p.V + xi);
      float dx = logit_at(p.D, p.dtype, static_cast<int64_t>(b) * p.db + static_cast<int64_t>(lane) * p.V + xi);
      float xh, xl, ezh, ezl, edh, edl;
      arg_df(zx, tz.m, c_hi, c_lo, xh, xl);
      exp2_df(xh, xl, tab, ezh, ezl);
      arg_df(dx, td.m, c_hi, c_lo, xh, xl);
      exp2_df(xh, xl, tab, edh, edl);
      const float2 Sz = rsum[lane], Sd = rsum[p.Pz + lane];
      const float u = p.u_acc[static_cast<int64_t>(b) * k + lane];
      // u < p/q  <=>  u e_d S_z < e_z S_d  (p = e_z / S_z, q = e_d / S_d)
      float lh, ll, rh, rl;
      df_mul(edh, edl, Sz.x, Sz.y, lh, ll);
      df_mul(lh, ll, u, 0.f, lh, ll);
      df_mul(ezh, ezl, Sd.x, Sd.y, rh, rl);
      acc = (edh == 0.f) ? (ezh > 0.f) : (lh < rh || (lh == rh && ll < rl));
      pv = __fdiv_rn(__fadd_rn(ezh, ezl), __fadd_rn(Sz.x, Sz.y));
      qv = __fdiv_rn(__fadd_rn(edh, edl), __fadd_rn(Sd.x, Sd.y));
    }
  }
  unsigned ball = __ballot_sync(kFull, acc);
  unsigned rej = ~ball & ((1u << k) - 1u);
  int n = rej ? (__ffs(rej) - 1) : k;
  if (status != 0) n = status;

  if (lane < k && p.p_at_x) {
    p.p_at_x[static_cast<int64_t>(b) * k + lane] = (status == 0) ? pv : NAN;
    p.q_at_x[static_cast<int64_t>(b) * k + lane] = (status == 0) ? qv : NAN;
  }
  if (p.out_tok && lane <= k) {
    int v = -1;
    if (n >= 0) {
      if (lane < n) v = xi;
      else if (lane == n && greedy) v = rs[n].argmax;
    }
    p.out_tok[static_cast<int64_t>(b) * (k + 1) + lane] = v;
  }
  if (lane == 0) {
    p.accept_len[b] = n;
    BState bs;
    bs.n = n;
    bs.mode = (n < 0 || greedy) ? kModeNone : (n < k ? kModeResidual : kModeTarget);
    bs.c_hi = c_hi;
    bs.c_lo = c_lo;
    bs.rho = (bs.mode == kModeResidual) ? __fdiv_rn(rsum[n].x, rsum[p.Pz + n].x) : 1.f;
    bs.pad0 = bs.pad1 = bs.pad2 = 0;
    p.bstate[b] = bs;
    if (p.amb_cnt) p.amb_cnt[b] = 0;
    int e = 0;
    if (t_bad) e |= 0x1;
    else if (any_tok_bad) e |= 0x4;
    else if (any_row_bad) e |= 0x2;
    if (e) atomicOr(p.err, e);
  }
}

// ---------------------------------------------------------------------------
// Softmax entry: finalise per row and optionally write the probabilities.
// ---------------------------------------------------------------------------

// grid: ceil(rows / kWarps); one warp per row
__global__ void __launch_bounds__(kThreads) softmax_finalize_kernel(SoftmaxParams p) {
  __shared__ float2 tab[64];
  load_exp2_table(tab);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (r >= p.rows) return;
  const float T = p.T[r];
  const bool t_bad = isnan(T) || T < 0.f;
  const bool greedy = !(T > 0.f);
  float c_hi = 0.f, c_lo = 0.f;
  if (!greedy && !t_bad) {  // one double division per warp (row)
    if (lane == 0) temp_coeff(T, c_hi, c_lo);
    c_hi = __shfl_sync(kFull, c_hi, 0);
    c_lo = __shfl_sync(kFull, c_lo, 0);
  }
  RowStat st;
  float sh, sl;
  merge_row(p.part + static_cast<int64_t>(r) * p.C, p.C, c_hi, c_lo, !greedy && !t_bad, tab, st,
            sh, sl);
  bool bad = t_bad || (st.flags & 2) || (st.flags & 1);
  if (lane == 0) {
    if (bad) {
      st.flags |= 2;
      p.row_max[r] = NAN;
      p.row_sum[r] = NAN;
      p.row_argmax[r] = -1;
      atomicOr(p.err, t_bad ? 0x1 : 0x2);
    } else {
      p.row_max[r] = st.m;
      p.row_sum[r] = static_cast<float>(st.S);
      p.row_argmax[r] = st.argmax;
    }
    p.rowstat[r] = st;
  }
}

// grid: (C, rows): p_v = 2^((z_v - m) c) / S, one-hot for greedy rows
template <typename Tag>
__global__ void __launch_bounds__(kThreads) softmax_probs_kernel(SoftmaxParams p) {
  const int c = blockIdx.x, r = blockIdx.y + p.r0;
  const int lo = c * p.CH, hi = min(p.V, lo + p.CH);
  const RowStat st = p.rowstat[r];
  const float T = p.T[r];
  float* out = p.probs + static_cast<int64_t>(r) * p.V;
  const typename Tag::Elem* row = static_cast<const typename Tag::Elem*>(p.L) + static_cast<int64_t>(r) * p.V;
  if (st.flags & 2) {
    for (int i = lo + threadIdx.x; i < hi; i += kThreads) out[i] = NAN;
    return;
  }
  if (!(T > 0.f)) {
    for (int i = lo + threadIdx.x; i < hi; i += kThreads) out[i] = (i == st.argmax) ? 1.f : 0.f;
    return;
  }
  __shared__ float2 s_ci;
  if (threadIdx.x == 0) {
    float h, l;
    temp_coeff(T, h, l);
    s_ci = make_float2(h, static_cast<float>(1.0 / st.S));
  }
  __syncthreads();
  const float cf = s_ci.x;
  const float inv = s_ci.y;
  for (int i = lo + threadIdx.x; i < hi; i += kThreads)
    out[i] = ex2_fast((Tag::load1(row + i) - st.m) * cf) * inv;
}

// ---------------------------------------------------------------------------
// Launchers (host).
// ---------------------------------------------------------------------------
template <typename Tag, bool VEC>
static cudaError_t launch_stats_t(const StatsParams& p0, int B, int rows, bool topf, cudaStream_t s) {
  StatsParams p = p0;
  for (int b0 = 0; b0 < B; b0 += kMaxGridBatch) {
    p.b0 = b0;
    dim3 grid((p.C + p.G - 1) / p.G, rows, B - b0 < kMaxGridBatch ? B - b0 : kMaxGridBatch);
    if (topf) stats_kernel<Tag, VEC, true><<<grid, kThreads, 0, s>>>(p);
    else stats_kernel<Tag, VEC, false><<<grid, kThreads, 0, s>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Rows [r0, r0 + rows) of every batch row; topf selects the variant that
// also keeps the forked top-f lists (draft rows below Pdf).
cudaError_t launch_stats_rows(const StatsParams& p0, int B, int dtype, bool vec, int r0, int rows,
                              bool topf, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  StatsParams p = p0;
  p.r0 = r0;
  if (dtype == 1)
    return vec ? launch_stats_t<BF16Tag, true>(p, B, rows, topf, s)
               : launch_stats_t<BF16Tag, false>(p, B, rows, topf, s);
  return vec ? launch_stats_t<F32Tag, true>(p, B, rows, topf, s)
             : launch_stats_t<F32Tag, false>(p, B, rows, topf, s);
}

template <typename Tag, bool VEC>
static cudaError_t launch_draft_t(const StatsParams& p0, int B, int rows, bool topf, cudaStream_t s) {
  StatsParams p = p0;
  for (int b0 = 0; b0 < B; b0 += kMaxGridBatch) {
    p.b0 = b0;
    dim3 grid((p.C + p.G - 1) / p.G, rows, B - b0 < kMaxGridBatch ? B - b0 : kMaxGridBatch);
    if (topf) draft_kernel<Tag, VEC, true><<<grid, kThreads, 0, s>>>(p);
    else draft_kernel<Tag, VEC, false><<<grid, kThreads, 0, s>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Draft rows [p.r0, p.r0 + rows) of every batch row.
cudaError_t launch_draft(const StatsParams& p, int B, int dtype, bool vec, int rows, bool topf,
                         cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (dtype == 1)
    return vec ? launch_draft_t<BF16Tag, true>(p, B, rows, topf, s)
               : launch_draft_t<BF16Tag, false>(p, B, rows, topf, s);
  return vec ? launch_draft_t<F32Tag, true>(p, B, rows, topf, s)
             : launch_draft_t<F32Tag, false>(p, B, rows, topf, s);
}

cudaError_t launch_draft_finalize(const DraftParams& p, cudaStream_t s) {
  const long long warps = static_cast<long long>(p.B) * p.rows;
  draft_finalize_kernel<<<static_cast<unsigned>((warps + kWarps - 1) / kWarps), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s) {
  if (p.B <= 152) finalize_kernel<16><<<p.B, 16 * 32, 0, s>>>(p);
  else finalize_kernel<kWarps><<<p.B, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_softmax_finalize(const SoftmaxParams& p, cudaStream_t s) {
  softmax_finalize_kernel<<<(p.rows + kWarps - 1) / kWarps, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_softmax_probs(const SoftmaxParams& p0, cudaStream_t s) {
  SoftmaxParams p = p0;
  for (int r0 = 0; r0 < p0.rows; r0 += kMaxGridBatch) {
    p.r0 = r0;
    dim3 grid(p.C, p0.rows - r0 < kMaxGridBatch ? p0.rows - r0 : kMaxGridBatch);
    if (p.dtype == 1) softmax_probs_kernel<BF16Tag><<<grid, kThreads, 0, s>>>(p);
    else softmax_probs_kernel<F32Tag><<<grid, kThreads, 0, s>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ssd
