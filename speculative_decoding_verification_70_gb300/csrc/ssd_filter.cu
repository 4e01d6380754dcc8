// ssd_filter.cu -- verify over top-k / top-p filtered distributions for any
// K (up to V) and for top-p over the whole vocabulary.
//
// The filter (same K and top_p for the target and the draft rows): order
// the tokens by (logit descending, index ascending), keep the first K, then
// the shortest prefix of those holding >= top_p of their probability mass,
// and renormalise ("tanishqkumar/ssd" summary, module notes: the sampler's
// top-k / top-p / temperature surface).  Speculative sampling stays exact
// when both distributions are filtered and the min(1, p/q) rule of
// Leviathan et al. / Chen et al. uses the filtered p and q.
//
// The kept set of a row is every token whose 64-bit order key (logit bits
// << 32 | ~index) is at least the key of the last kept token, so a row is
// described by that threshold key and its kept mass P.  Finding them
// without sorting a row:
//   stats_kernel         row maximum, argmax and NaN flags (no exponentials)
//   filt_rowinit_kernel  merges them per row, log2(e)/T, clears the histogram
//   filt_hist_kernel     per row, tokens binned by x = (m - z) log2(e) / T in
//                        16 bins per unit of x: exact counts and fast masses
//                        (bin-scaled fixed point); with K >= V also the exact
//                        mass of the row (extended-precision exponentials)
//   filt_band_kernel     the bins that must hold the K-th token and the top-p
//                        cut, given a bound on the fast masses' error
//   filt_collect_kernel  exact mass of every token in the bins above the band,
//                        order keys of the band's tokens
//   filt_cut_kernel      sorts the band (bitonic, shared memory) and places
//                        both cuts exactly; a band of more than kFiltCand
//                        tokens (or an inconsistent one) is resolved by
//                        bisection on the order key over the row
//   filt_accept_kernel   acceptance per position from the filtered p(x),
//                        q(x), first-reject prefix, greedy tokens, draw state
// The recovery / bonus draw over the filtered rows is in ssd_residual.cu.
#include <math.h>

#include "ssd_device.cuh"
#include "ssd_layout.h"
#include "ssd_scan.cuh"

namespace ssd {
namespace {

constexpr int kFlagNan = 1;        // a NaN in the row
constexpr int kFlagInvalid = 2;    // +inf or no finite logit (T > 0)
constexpr int kFlagFiltered = 4;   // a T > 0 row that is filtered
constexpr int kFlagResolved = 8;   // threshold and mass known after the band step
constexpr int kDevErrFilter = 0x20;  // a cut fell outside its band (fallback taken)

// Relative error bound of the fast bin masses: each token's mass is rounded
// to a whole unit of its bin's scale 2^(12 + j) (at most 2^-12 relative, its
// value being in (2^11, 2^12] units), on top of ex2.approx (~2^-22) and the
// rounding of x (|x| 2^-23 ln 2 for x < 64); with a margin.
constexpr double kFastMargin = 5e-4;
constexpr float kBinScale = 4096.0f;                   // 2^12
constexpr double kFix42 = 4398046511104.0;             // 2^42
constexpr double kInvFix42 = 1.0 / 4398046511104.0;

// x = (m - z) c_hi with explicit rounding: every kernel bins a token the same
// way, and the bin is non-decreasing in m - z (so in key order).
__device__ __forceinline__ float filt_x(float z, float m, float c_hi) {
  return __fmul_rn(__fsub_rn(m, z), c_hi);
}
__device__ __forceinline__ int filt_bin(float x) {
  constexpr float kTop = static_cast<float>(kFiltBins / kFiltBinsPerUnit);
  return x < kTop ? static_cast<int>(__fmul_rn(x, static_cast<float>(kFiltBinsPerUnit)))
                  : kFiltBins - 1;
}
// A bin's masses are scaled by 2^(12 + j), j = bin / 16 (at most 63): a
// token of bin b then contributes round(2^(j - x) 2^12), in [2^11, 2^12]
// (the tail bin: at most 2^12), so a CTA's 32-bit bin sums cannot overflow
// (a CTA streams at most 2^19 tokens) and a row's 64-bit ones neither.
__device__ __forceinline__ int bin_shift(int bin) {
  const int j = bin / kFiltBinsPerUnit;
  return j < 63 ? j : 63;
}
__device__ __forceinline__ double bin_mass(unsigned long long v, int bin) {
  // 2^-(12 + j) built from its exponent bits (exact)
  const double unit = __longlong_as_double(static_cast<long long>(1023 - 12 - bin_shift(bin)) << 52);
  return static_cast<double>(v) * unit;
}

// Exact (extended-precision) mass 2^((z - m) c) of one token as a double.
__device__ __forceinline__ double exact_mass(float z, float m, float c_hi, float c_lo,
                                             const float2* tab) {
  float xh, xl, h, l;
  arg_df(z, m, c_hi, c_lo, xh, xl);
  exp2_df(xh, xl, tab, h, l);
  return static_cast<double>(h) + static_cast<double>(l);
}

// Block sum of a double (fixed tree: deterministic).  Holds barriers.
__device__ double block_sum_d(double v, double* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  __syncthreads();
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  double t = 0.0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += sm[w];
  return t;
}

__device__ __forceinline__ long long block_sum_ll(long long v, long long* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  __syncthreads();
  if (lane == 0) sm[warp] = v;
  __syncthreads();
  long long t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += sm[w];
  return t;
}

template <typename Tag>
__device__ __forceinline__ const typename Tag::Elem* filt_row_ptr(const FiltParams& p, int b, int r) {
  const int Pz = p.k + 1;
  using Elem = typename Tag::Elem;
  return r < Pz ? static_cast<const Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb + static_cast<int64_t>(r) * p.V
                : static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
                      static_cast<int64_t>(r - Pz) * p.V;
}

// Visit the tokens [lo, hi) of a row, thread-strided 16-byte vectors with
// four in flight (VEC), else single elements: fn(z, index).
template <typename Tag, bool VEC, typename Fn>
__device__ __forceinline__ void for_tokens(const typename Tag::Elem* row, int lo, int hi, Fn&& fn) {
  constexpr int kV = VEC ? Tag::kVec : 1;
  constexpr int U = 4;
  const int v0 = lo / kV, v1 = (hi + kV - 1) / kV;
  for (int vb = v0 + static_cast<int>(threadIdx.x); vb < v1; vb += kThreads * U) {
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
#pragma unroll
        for (int e = 0; e < kV; ++e) fn(z[e], vi * kV + e);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Row set-up: one warp per (b, row).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) filt_rowinit_kernel(FiltParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long w = static_cast<long long>(blockIdx.x) * kWarps + warp;
  if (w >= static_cast<long long>(p.B) * p.R) return;
  const int b = static_cast<int>(w / p.R);
  const PartStat* parts = p.part + w * p.C;
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
  const float T = p.T[b];
  const bool stochastic = T > 0.f;  // false for NaN
  int flags = nan ? kFlagNan : 0;
  if (stochastic && (m == INFINITY || m == -INFINITY)) flags |= kFlagInvalid;
  if (stochastic && !(flags & (kFlagNan | kFlagInvalid))) flags |= kFlagFiltered;
  FiltRow& fr = p.rows[w];
  if (lane == 0) {
    float ch = 0.f, cl = 0.f;
    if (flags & kFlagFiltered) temp_coeff(T, ch, cl);
    fr.thr = 0ull;
    fr.above = 0ull;
    fr.total = 0ull;
    fr.P = 0.0;
    fr.m = m;
    fr.c_hi = ch;
    fr.c_lo = cl;
    fr.argmax = idx == kIdxNone ? 0 : idx;
    fr.flags = flags;
    fr.band_lo = kFiltBins;
    fr.band_hi = kFiltBins - 1;
    fr.cnt_before = 0;
    fr.n_cand = 0;
    fr.keep = 0;
    fr.pad = 0;
  }
  if (flags & kFlagFiltered) {
    unsigned* hc = p.hcnt + w * kFiltBins;
    unsigned long long* hm = p.hmass + w * kFiltBins;
    for (int q = lane; q < kFiltBins; q += 32) {
      hc[q] = 0u;
      hm[q] = 0ull;
    }
  }
}

// ---------------------------------------------------------------------------
// Histogram pass.  grid (chunk groups, R, batch rows of this launch).
// ---------------------------------------------------------------------------
struct HistSmem {
  unsigned mass[kFiltBins];
  unsigned cnt[kFiltBins];
  float2 tab[64];
  double red[kWarps];
};

template <typename Tag, bool VEC, bool TOTAL>
__global__ void __launch_bounds__(kThreads) filt_hist_kernel(FiltParams p) {
  const int c = blockIdx.x * p.G, r = blockIdx.y, b = blockIdx.z + p.b0;
  FiltRow* frp = p.rows + static_cast<int64_t>(b) * p.R + r;
  const int flags = frp->flags;
  if (!(flags & kFlagFiltered)) return;
  const float m = frp->m, c_hi = frp->c_hi, c_lo = frp->c_lo;
  __shared__ HistSmem sm;
  for (int q = threadIdx.x; q < kFiltBins; q += kThreads) {
    sm.mass[q] = 0u;
    sm.cnt[q] = 0u;
  }
  if (TOTAL) load_exp2_table(sm.tab);
  __syncthreads();
  const int lo = c * p.CH, hi = min(p.V, lo + p.G * p.CH);
  float acc = 0.f, comp = 0.f;
  for_tokens<Tag, VEC>(filt_row_ptr<Tag>(p, b, r), lo, hi, [&](float z, int) {
    const float x = filt_x(z, m, c_hi);
    const int bin = filt_bin(x);
    const float y = ex2_fast(__fsub_rn(static_cast<float>(bin_shift(bin)), x));
    atomicAdd(&sm.cnt[bin], 1u);
    atomicAdd(&sm.mass[bin], __float2uint_rn(__fmul_rn(y, kBinScale)));
    if (TOTAL) {
      float xh, xl, h, l;
      arg_df(z, m, c_hi, c_lo, xh, xl);
      exp2_df(xh, xl, sm.tab, h, l);
      comp_acc(acc, comp, h, l);
    }
  });
  __syncthreads();
  const int64_t hrow = (static_cast<int64_t>(b) * p.R + r) * kFiltBins;
  for (int q = threadIdx.x; q < kFiltBins; q += kThreads) {
    const unsigned n = sm.cnt[q];
    if (n) {
      atomicAdd(p.hcnt + hrow + q, n);
      atomicAdd(p.hmass + hrow + q, static_cast<unsigned long long>(sm.mass[q]));
    }
  }
  if (TOTAL) {
    const double s = block_sum_d(static_cast<double>(acc) + static_cast<double>(comp), sm.red);
    if (threadIdx.x == 0)
      atomicAdd(&frp->total, static_cast<unsigned long long>(llrint(s * kFix42)));
  }
}

// ---------------------------------------------------------------------------
// Band selection: one warp per (b, row).  Lane l owns bins [32 l, 32 l + 32).
// ---------------------------------------------------------------------------
// First bin (>= 0) whose cumulative value satisfies pred, from each lane's
// exclusive prefix and its bins; kFiltBins if none.  pred is monotone.
template <typename Pred>
__device__ __forceinline__ int first_bin(const unsigned* hc, const unsigned long long* hm,
                                         long long cnt_ex, double mass_ex, long long cnt_in,
                                         double mass_in, Pred pred) {
  const int lane = threadIdx.x & 31;
  const unsigned hit = __ballot_sync(kFull, pred(cnt_in, mass_in));
  if (!hit) return kFiltBins;
  const int l = __ffs(hit) - 1;
  int found = kFiltBins;
  if (lane == l) {
    long long cn = cnt_ex;
    double ms = mass_ex;
    for (int q = 32 * l; q < 32 * l + 32; ++q) {
      cn += hc[q];
      ms += bin_mass(hm[q], q);
      if (pred(cn, ms)) {
        found = q;
        break;
      }
    }
    if (found == kFiltBins) found = 32 * l + 31;  // rounding: the lane's last bin
  }
  return __shfl_sync(kFull, found, l);
}

// Cumulative count and fast mass of bins [0, bin] (bin < 0: zero).
__device__ __forceinline__ void cum_at(const unsigned* hc, const unsigned long long* hm,
                                       long long cnt_ex, double mass_ex, int bin, long long& cn,
                                       double& ms) {
  const int lane = threadIdx.x & 31;
  const int l = bin < 0 ? 0 : bin / 32;
  long long a = 0;
  double s = 0.0;
  if (lane == l && bin >= 0) {
    a = cnt_ex;
    s = mass_ex;
    for (int q = 32 * l; q <= bin; ++q) {
      a += hc[q];
      s += bin_mass(hm[q], q);
    }
  }
  cn = __shfl_sync(kFull, a, l);
  ms = __shfl_sync(kFull, s, l);
}

__global__ void __launch_bounds__(kThreads) filt_band_kernel(FiltParams p) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long w = static_cast<long long>(blockIdx.x) * kWarps + warp;
  if (w >= static_cast<long long>(p.B) * p.R) return;
  const int b = static_cast<int>(w / p.R);
  FiltRow& fr = p.rows[w];
  if (!(fr.flags & kFlagFiltered)) return;
  const unsigned* hc = p.hcnt + w * kFiltBins;
  const unsigned long long* hm = p.hmass + w * kFiltBins;
  long long cnt = 0;
  double mass = 0.0;
  for (int q = 32 * lane; q < 32 * lane + 32; ++q) {
    cnt += hc[q];
    mass += bin_mass(hm[q], q);
  }
  long long cin = cnt;
  double min_ = mass;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long yc = __shfl_up_sync(kFull, cin, o);
    const double ym = __shfl_up_sync(kFull, min_, o);
    if (lane >= o) {
      cin += yc;
      min_ += ym;
    }
  }
  const long long cex = cin - cnt;
  const double mex = min_ - mass;
  const float tpf = p.top_p ? p.top_p[b] : 1.f;
  const bool pcut = tpf < 1.f;                       // NaN: no cut
  const double tp = static_cast<double>(tpf);
  const long long Keff = p.K < p.V ? p.K : p.V;
  const bool kmode = Keff < p.V;
  int bK = kFiltBins - 1;
  double Mlo, Mhi;
  if (kmode) {
    bK = first_bin(hc, hm, cex, mex, cin, min_,
                   [&](long long cn, double) { return cn >= Keff; });
    if (bK >= kFiltBins) bK = kFiltBins - 1;
    long long c0, c1;
    double m0, m1;
    cum_at(hc, hm, cex, mex, bK - 1, c0, m0);
    cum_at(hc, hm, cex, mex, bK, c1, m1);
    Mlo = m0 * (1.0 - kFastMargin);
    Mhi = m1 * (1.0 + kFastMargin);
  } else {
    Mlo = Mhi = static_cast<double>(fr.total) * kInvFix42;
  }
  int lo, hi;
  if (pcut) {
    const double tlo = tp * Mlo, thi = tp * Mhi;
    lo = first_bin(hc, hm, cex, mex, cin, min_,
                   [&](long long, double ms) { return ms * (1.0 + kFastMargin) >= tlo; });
    hi = first_bin(hc, hm, cex, mex, cin, min_,
                   [&](long long, double ms) { return ms * (1.0 - kFastMargin) >= thi; });
    if (lo >= kFiltBins) lo = kFiltBins - 1;
    if (hi >= kFiltBins) hi = kFiltBins - 1;
    if (kmode) {
      if (lo > bK) lo = bK;
      hi = bK;
    }
  } else if (kmode) {
    lo = hi = bK;
  } else {
    lo = kFiltBins;  // no filter: every token kept, P is the exact row mass
    hi = kFiltBins - 1;
  }
  long long cb;
  double mb;
  cum_at(hc, hm, cex, mex, lo - 1, cb, mb);
  if (lane == 0) {
    fr.band_lo = lo;
    fr.band_hi = hi;
    fr.cnt_before = static_cast<int>(lo >= kFiltBins ? p.V : cb);
    if (!pcut && !kmode) {
      fr.thr = 0ull;
      fr.P = static_cast<double>(fr.total) * kInvFix42;
      fr.keep = p.V;
      fr.flags |= kFlagResolved;
    }
  }
}

// ---------------------------------------------------------------------------
// Collect pass.  grid (chunk groups, R, batch rows of this launch).
// ---------------------------------------------------------------------------
template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kThreads) filt_collect_kernel(FiltParams p) {
  const int c = blockIdx.x * p.G, r = blockIdx.y, b = blockIdx.z + p.b0;
  FiltRow* frp = p.rows + static_cast<int64_t>(b) * p.R + r;
  const int flags = frp->flags;
  if (!(flags & kFlagFiltered) || (flags & kFlagResolved)) return;
  const float m = frp->m, c_hi = frp->c_hi, c_lo = frp->c_lo;
  const int blo = frp->band_lo, bhi = frp->band_hi;
  __shared__ float2 tab[64];
  __shared__ double red[kWarps];
  load_exp2_table(tab);
  __syncthreads();
  unsigned long long* cand = p.cand + (static_cast<int64_t>(b) * p.R + r) * kFiltCand;
  const int lo = c * p.CH, hi = min(p.V, lo + p.G * p.CH);
  const int lane = threadIdx.x & 31;
  float acc = 0.f, comp = 0.f;
  for_tokens<Tag, VEC>(filt_row_ptr<Tag>(p, b, r), lo, hi, [&](float z, int idx) {
    const int bin = filt_bin(filt_x(z, m, c_hi));
    if (bin < blo) {
      float xh, xl, h, l;
      arg_df(z, m, c_hi, c_lo, xh, xl);
      exp2_df(xh, xl, tab, h, l);
      comp_acc(acc, comp, h, l);
    }
    const bool take = bin >= blo && bin <= bhi;
    const unsigned act = __activemask();
    const unsigned want = __ballot_sync(act, take);
    if (want) {
      const int leader = __ffs(want) - 1;
      int base = 0;
      if (lane == leader) base = atomicAdd(&frp->n_cand, __popc(want));
      base = __shfl_sync(act, base, leader);
      if (take) {
        const int pos = base + __popc(want & ((1u << lane) - 1u));
        if (pos < kFiltCand) cand[pos] = order_key(z, idx);
      }
    }
  });
  const double s = block_sum_d(static_cast<double>(acc) + static_cast<double>(comp), red);
  if (threadIdx.x == 0 && s > 0.0)
    atomicAdd(&frp->above, static_cast<unsigned long long>(llrint(s * kFix42)));
}

// ---------------------------------------------------------------------------
// Cut: one CTA per (row, b).
// ---------------------------------------------------------------------------
struct CutSmem {
  unsigned long long key[kFiltCand];
  double pre[kFiltCand];
  float2 tab[64];
  double red[kWarps];
  long long redl[kWarps];
  int pick;
};

// Count of the row's tokens with key >= t and (with_mass) their exact mass.
template <typename Tag, bool VEC>
__device__ void count_mass_ge(const typename Tag::Elem* row, int V, unsigned long long t,
                              bool with_mass, float m, float c_hi, float c_lo, CutSmem& sm,
                              long long& cnt, double& mass) {
  long long n = 0;
  float acc = 0.f, comp = 0.f;
  for_tokens<Tag, VEC>(row, 0, V, [&](float z, int idx) {
    if (order_key(z, idx) >= t) {
      ++n;
      if (with_mass) {
        float xh, xl, h, l;
        arg_df(z, m, c_hi, c_lo, xh, xl);
        exp2_df(xh, xl, sm.tab, h, l);
        comp_acc(acc, comp, h, l);
      }
    }
  });
  cnt = block_sum_ll(n, sm.redl);
  mass = with_mass ? block_sum_d(static_cast<double>(acc) + static_cast<double>(comp), sm.red) : 0.0;
}

// The largest key t with pred(count(key >= t), mass(key >= t)) (pred true at
// t = 0 and monotone): bisection over the 64-bit keys, one row scan per step.
template <typename Tag, bool VEC, typename Pred>
__device__ unsigned long long bisect_key(const typename Tag::Elem* row, int V, bool with_mass,
                                         float m, float c_hi, float c_lo, CutSmem& sm, Pred pred) {
  unsigned long long lo = 0ull, hi = ~0ull;
  while (lo < hi) {
    const unsigned long long mid = lo + (hi - lo) / 2 + 1;
    long long cn;
    double ms;
    count_mass_ge<Tag, VEC>(row, V, mid, with_mass, m, c_hi, c_lo, sm, cn, ms);
    if (pred(cn, ms)) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <typename Tag, bool VEC>
__device__ void cut_by_bisection(const FiltParams& p, int b, int r, FiltRow& fr, CutSmem& sm) {
  const typename Tag::Elem* row = filt_row_ptr<Tag>(p, b, r);
  const float m = fr.m, c_hi = fr.c_hi, c_lo = fr.c_lo;
  const long long Keff = p.K < p.V ? p.K : p.V;
  const float tpf = p.top_p ? p.top_p[b] : 1.f;
  const bool pcut = tpf < 1.f;
  unsigned long long tK = 0ull;
  if (Keff < p.V)
    tK = bisect_key<Tag, VEC>(row, p.V, false, m, c_hi, c_lo, sm,
                              [&](long long cn, double) { return cn >= Keff; });
  long long cn;
  double massK;
  count_mass_ge<Tag, VEC>(row, p.V, tK, true, m, c_hi, c_lo, sm, cn, massK);
  unsigned long long thr = tK;
  if (pcut) {
    const double target = static_cast<double>(tpf) * massK;
    // the cut keeps at least the first token (top_p <= 0 keeps exactly one)
    thr = bisect_key<Tag, VEC>(row, p.V, true, m, c_hi, c_lo, sm,
                               [&](long long cn, double ms) { return cn >= 1 && ms >= target; });
    if (thr < tK) thr = tK;
  }
  double P;
  count_mass_ge<Tag, VEC>(row, p.V, thr, true, m, c_hi, c_lo, sm, cn, P);
  if (threadIdx.x == 0) {
    fr.thr = thr;
    fr.P = P;
    fr.keep = static_cast<int>(cn);
  }
}

template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kThreads) filt_cut_kernel(FiltParams p) {
  const int r = blockIdx.x, b = blockIdx.y + p.b0, tid = threadIdx.x;
  FiltRow& fr = p.rows[static_cast<int64_t>(b) * p.R + r];
  const int flags = fr.flags;
  if (!(flags & kFlagFiltered) || (flags & kFlagResolved)) return;
  __shared__ CutSmem sm;
  load_exp2_table(sm.tab);
  const int n = fr.n_cand;
  const long long Keff = p.K < p.V ? p.K : p.V;
  const bool kmode = Keff < p.V;
  const float tpf = p.top_p ? p.top_p[b] : 1.f;
  const bool pcut = tpf < 1.f;
  const double above = static_cast<double>(fr.above) * kInvFix42;
  const long long before = fr.cnt_before;
  bool ok = n >= 1 && n <= kFiltCand;
  const long long jK = kmode ? Keff - before - 1 : static_cast<long long>(n) - 1;
  if (kmode && (jK < 0 || jK >= n)) ok = false;
  if (!ok) {  // uniform over the CTA: an overflowing band, or an inconsistent one
    if (n <= kFiltCand && tid == 0) atomicOr(p.err, kDevErrFilter);
    __syncthreads();
    cut_by_bisection<Tag, VEC>(p, b, r, fr, sm);
    return;
  }
  // sort the band's keys, descending (bitonic over the next power of two)
  int N2 = 1;
  while (N2 < n) N2 <<= 1;
  const unsigned long long* cand = p.cand + (static_cast<int64_t>(b) * p.R + r) * kFiltCand;
  for (int q = tid; q < N2; q += kThreads) sm.key[q] = q < n ? cand[q] : 0ull;
  __syncthreads();
  for (int kk = 2; kk <= N2; kk <<= 1)
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int pr = tid; pr < N2 / 2; pr += kThreads) {
        const int i = (pr / j) * 2 * j + (pr % j);
        const int l = i + j;
        const bool desc = (i & kk) == 0;
        const unsigned long long a = sm.key[i], c = sm.key[l];
        if (desc ? (c > a) : (a > c)) {
          sm.key[i] = c;
          sm.key[l] = a;
        }
      }
      __syncthreads();
    }
  // exact masses in key order and their inclusive prefix sums: thread t
  // sums entries [8 t, 8 t + 8) serially, then an exclusive scan over threads
  constexpr int kPer = kFiltCand / kThreads;
  double loc[kPer];
  double run = 0.0;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int q = tid * kPer + e;
    double v = 0.0;
    if (q < n) v = exact_mass(key_logit(sm.key[q]), fr.m, fr.c_hi, fr.c_lo, sm.tab);
    run += v;
    loc[e] = run;
  }
  // exclusive scan of the threads' totals (fixed tree)
  const int lane = tid & 31, warp = tid >> 5;
  double incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.red[warp] = incl;
  __syncthreads();
  double off = 0.0;
  for (int w = 0; w < warp; ++w) off += sm.red[w];
  off += incl - run;
#pragma unroll
  for (int e = 0; e < kPer; ++e) {
    const int q = tid * kPer + e;
    if (q < n) sm.pre[q] = off + loc[e];
  }
  if (tid == 0) sm.pick = 0x7fffffff;
  __syncthreads();
  const double massK = kmode ? above + sm.pre[jK] : static_cast<double>(fr.total) * kInvFix42;
  long long jstar = jK;
  bool bad = false;
  if (pcut) {
    // the first position (key order) whose cumulative kept mass reaches
    // top_p of the first K tokens' mass
    const double target = static_cast<double>(tpf) * massK;
    if (above >= target && before > 0) bad = true;  // the cut lies above the band
    for (int q = tid; q <= jK; q += kThreads)
      if (above + sm.pre[q] >= target) {
        atomicMin(&sm.pick, q);
        break;
      }
    __syncthreads();
    const int first = sm.pick;
    if (first == 0x7fffffff) bad = bad || !kmode;  // no cut in the band (K >= V)
    else jstar = first;
  }
  if (bad) {  // uniform: every thread read the same shared values
    if (tid == 0) atomicOr(p.err, kDevErrFilter);
    __syncthreads();
    cut_by_bisection<Tag, VEC>(p, b, r, fr, sm);
    return;
  }
  if (tid == 0) {
    fr.thr = sm.key[jstar];
    fr.P = above + sm.pre[jstar];
    fr.keep = static_cast<int>(before + jstar + 1);
  }
}

// ---------------------------------------------------------------------------
// Acceptance: one warp per batch row.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float logit_of(const void* base, int dtype, int64_t i) {
  if (dtype == 1)
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(base) + i)) << 16);
  return __ldg(static_cast<const float*>(base) + i);
}

__global__ void __launch_bounds__(32) filt_accept_kernel(FiltParams p) {
  __shared__ float2 tab[64];
  const int b = blockIdx.x, lane = threadIdx.x;
  const int k = p.k, Pz = k + 1;
  load_exp2_table(tab);
  __syncwarp();
  const float T = p.T[b];
  const bool t_bad = isnan(T) || T < 0.f;
  const bool greedy = !(T > 0.f);
  const FiltRow* rows = p.rows + static_cast<int64_t>(b) * p.R;
  int xi = -1;
  bool tok_bad = false;
  if (lane < k) {
    xi = p.x[static_cast<int64_t>(b) * k + lane];
    tok_bad = xi < 0 || xi >= p.V;
  }
  const bool any_tok_bad = __any_sync(kFull, tok_bad);
  bool rb = false;
  const int badmask = greedy ? kFlagNan : (kFlagNan | kFlagInvalid);
  if (lane <= k) rb |= (rows[lane].flags & badmask) != 0;
  if (lane < k) rb |= (rows[Pz + lane].flags & badmask) != 0;
  const bool any_row_bad = __any_sync(kFull, rb);
  int status = 0;
  if (t_bad) status = -1;
  else if (any_tok_bad) status = -2;
  else if (any_row_bad) status = -1;
  float pv = NAN, qv = NAN;
  bool acc = false;
  if (status == 0 && lane < k) {
    const FiltRow& rz = rows[lane];
    const FiltRow& rd = rows[Pz + lane];
    if (greedy) {
      acc = xi == rz.argmax;
      pv = acc ? 1.f : 0.f;
      qv = xi == rd.argmax ? 1.f : 0.f;
    } else {
      const float z = logit_of(p.Z, p.dtype, static_cast<int64_t>(b) * p.zb + static_cast<int64_t>(lane) * p.V + xi);
      const float d = logit_of(p.D, p.dtype, static_cast<int64_t>(b) * p.db + static_cast<int64_t>(lane) * p.V + xi);
      const bool in_z = order_key(z, xi) >= rz.thr;
      const bool in_d = order_key(d, xi) >= rd.thr;
      const double pf = in_z ? exact_mass(z, rz.m, rz.c_hi, rz.c_lo, tab) / rz.P : 0.0;
      const double qf = in_d ? exact_mass(d, rd.m, rd.c_hi, rd.c_lo, tab) / rd.P : 0.0;
      const float u = p.u_acc[static_cast<int64_t>(b) * k + lane];
      acc = (qf == 0.0) ? (pf > 0.0) : (static_cast<double>(u) < pf / qf);
      pv = static_cast<float>(pf);
      qv = static_cast<float>(qf);
    }
  }
  const unsigned ball = __ballot_sync(kFull, acc);
  const unsigned rej = ~ball & ((1u << k) - 1u);
  int n = rej ? (__ffs(rej) - 1) : k;
  if (status != 0) n = status;
  if (lane < k && p.p_at_x) {
    p.p_at_x[static_cast<int64_t>(b) * k + lane] = status == 0 ? pv : NAN;
    p.q_at_x[static_cast<int64_t>(b) * k + lane] = status == 0 ? qv : NAN;
  }
  if (p.out_tok && lane <= k) {
    int v = -1;
    if (n >= 0) {
      if (lane < n) v = xi;
      else if (lane == n && greedy) v = rows[n].argmax;
    }
    p.out_tok[static_cast<int64_t>(b) * (k + 1) + lane] = v;
  }
  if (lane == 0) {
    p.accept_len[b] = n;
    BState bs;
    bs.n = n;
    bs.mode = (n < 0 || greedy || !p.u_smp || !p.out_tok) ? kModeNone
                                                          : (n < k ? kModeResidual : kModeTarget);
    bs.c_hi = n >= 0 ? rows[n].c_hi : 0.f;
    bs.c_lo = n >= 0 ? rows[n].c_lo : 0.f;
    bs.rho = 1.f;
    bs.pad0 = bs.pad1 = bs.pad2 = 0;
    p.bstate[b] = bs;
    int e = 0;
    if (t_bad) e |= 0x1;
    else if (any_tok_bad) e |= 0x4;
    else if (any_row_bad) e |= 0x2;
    if (e) atomicOr(p.err, e);
  }
}

}  // namespace

// ---------------------------------------------------------------------------
// Launchers
// ---------------------------------------------------------------------------
cudaError_t launch_filt_rowinit(const FiltParams& p, cudaStream_t s) {
  const long long warps = static_cast<long long>(p.B) * p.R;
  filt_rowinit_kernel<<<static_cast<unsigned>((warps + kWarps - 1) / kWarps), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_filt_band(const FiltParams& p, cudaStream_t s) {
  const long long warps = static_cast<long long>(p.B) * p.R;
  filt_band_kernel<<<static_cast<unsigned>((warps + kWarps - 1) / kWarps), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

// Launches over slices of at most kMaxGridBatch batch rows (grid z / y).
template <typename F>
static cudaError_t over_batch(const FiltParams& p0, F&& launch) {
  FiltParams q = p0;
  for (int b0 = 0; b0 < p0.B; b0 += kMaxGridBatch) {
    q.b0 = b0;
    launch(q, p0.B - b0 < kMaxGridBatch ? p0.B - b0 : kMaxGridBatch);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

template <typename Tag, bool VEC>
static void hist_t(const FiltParams& q, int nb, cudaStream_t s) {
  const dim3 grid((q.C + q.G - 1) / q.G, q.R, nb);
  if (q.total_mode) filt_hist_kernel<Tag, VEC, true><<<grid, kThreads, 0, s>>>(q);
  else filt_hist_kernel<Tag, VEC, false><<<grid, kThreads, 0, s>>>(q);
}

template <typename Tag, bool VEC>
static void collect_t(const FiltParams& q, int nb, cudaStream_t s) {
  const dim3 grid((q.C + q.G - 1) / q.G, q.R, nb);
  filt_collect_kernel<Tag, VEC><<<grid, kThreads, 0, s>>>(q);
}

template <typename Tag, bool VEC>
static void cut_t(const FiltParams& q, int nb, cudaStream_t s) {
  filt_cut_kernel<Tag, VEC><<<dim3(q.R, nb), kThreads, 0, s>>>(q);
}

cudaError_t launch_filt_hist(const FiltParams& p0, bool vec, cudaStream_t s) {
  return over_batch(p0, [&](const FiltParams& q, int nb) {
    if (q.dtype == 1) vec ? hist_t<BF16Tag, true>(q, nb, s) : hist_t<BF16Tag, false>(q, nb, s);
    else vec ? hist_t<F32Tag, true>(q, nb, s) : hist_t<F32Tag, false>(q, nb, s);
  });
}

cudaError_t launch_filt_collect(const FiltParams& p0, bool vec, cudaStream_t s) {
  return over_batch(p0, [&](const FiltParams& q, int nb) {
    if (q.dtype == 1) vec ? collect_t<BF16Tag, true>(q, nb, s) : collect_t<BF16Tag, false>(q, nb, s);
    else vec ? collect_t<F32Tag, true>(q, nb, s) : collect_t<F32Tag, false>(q, nb, s);
  });
}

cudaError_t launch_filt_cut(const FiltParams& p0, bool vec, cudaStream_t s) {
  return over_batch(p0, [&](const FiltParams& q, int nb) {
    if (q.dtype == 1) vec ? cut_t<BF16Tag, true>(q, nb, s) : cut_t<BF16Tag, false>(q, nb, s);
    else vec ? cut_t<F32Tag, true>(q, nb, s) : cut_t<F32Tag, false>(q, nb, s);
  });
}

cudaError_t launch_filt_accept(const FiltParams& p, cudaStream_t s) {
  filt_accept_kernel<<<p.B, 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ssd
