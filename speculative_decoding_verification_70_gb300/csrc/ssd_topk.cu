// ssd_topk.cu -- verify over top-k / top-p filtered distributions.
//
// The sampler surface of the pages' engine ("tanishqkumar/ssd" summary,
// module notes: temperature sampler; SSD project summary, "Highlighted
// Details": optimised kernels) filters the distributions it samples from;
// speculative sampling stays exact when the target and the draft are both
// filtered and verification uses the filtered p and q (the min(1, p/q) rule
// of Leviathan et al. / Chen et al. holds for any pair of distributions).
//
// Filter (same K and top_p for target and draft rows): order the tokens by
// (logit descending, index ascending); keep the first K; keep the shortest
// prefix of those holding >= top_p of their probability mass; renormalise.
// With K <= 32 the filtered distribution lives on at most K tokens, so:
//   topk_pass_kernel      one pass over the 2k+1 rows: per chunk group the K
//                         best (logit, index) pairs plus max / argmax / NaN;
//                         no exponentials.
//   topk_finalize_kernel  per batch row: merge the chunk lists into each
//                         row's top K, the kept masses 2^((z - m) c) in
//                         extended precision (exp2_df) summed in double, the
//                         top-p cut, acceptance (one lane per position,
//                         ballot), and the recovery / bonus draw by inverse
//                         CDF in token order over at most K candidates.
// Nothing after the pass reads a logit row again.
#include <math.h>

#include "ssd_device.cuh"
#include "ssd_layout.h"
#include "ssd_scan.cuh"

namespace ssd {
namespace {

constexpr int kPer = 4;  // candidates kept by each thread

constexpr int kSecond = 256;  // entries of the second-chance buffer

struct PassSmem {
  float sv[kWarps][kThreads / kWarps * 4];  // each warp's 128 candidates (bitonic path)
  int si[kWarps][kThreads / kWarps * 4];
  float lv[kMaxTopK];          // the candidates' top K (sorted)
  int li[kMaxTopK];
  float xv[kSecond];           // second chance: elements of overflowing threads
  int xi[kSecond];
  int nx;
  float wl[kWarps][kMaxTopK];  // each warp's sorted top K
  int wi[kWarps][kMaxTopK];
  float w5[kWarps];
  int cnt;
  float m[kWarps], s[kWarps];
  int i[kWarps], n[kWarps];
  float bv[kWarps];
  int bi[kWarps];
  float tw[2 * kWarps];        // each warp's two largest fourth values
  float tau;
};

// A thread's four best (value, index) pairs, sorted, and b5, the largest
// value among its other elements.  Elements arrive in increasing index
// order, so a strict compare keeps the lower index first on ties.
struct Top4 {
  float t[kPer];
  int i[kPer];
  float b5;
  int nan;
};

__device__ __forceinline__ void top4_push(Top4& s, float z, int idx) {
  if (!(z > s.t[3])) {
    s.b5 = fmaxf(s.b5, z);
    return;
  }
  s.b5 = fmaxf(s.b5, s.t[3]);
  if (z > s.t[2]) {
    s.t[3] = s.t[2];
    s.i[3] = s.i[2];
    if (z > s.t[1]) {
      s.t[2] = s.t[1];
      s.i[2] = s.i[1];
      if (z > s.t[0]) {
        s.t[1] = s.t[0];
        s.i[1] = s.i[0];
        s.t[0] = z;
        s.i[0] = idx;
      } else {
        s.t[1] = z;
        s.i[1] = idx;
      }
    } else {
      s.t[2] = z;
      s.i[2] = idx;
    }
  } else {
    s.t[3] = z;
    s.i[3] = idx;
  }
}

// One compare-exchange of a descending bitonic network on (value, index)
// pairs in shared memory: after it, position i holds the pair that ranks
// first when `desc`, else the one that ranks second.
__device__ __forceinline__ void bitonic_cx(float* v, int* ix, int i, int l, bool desc) {
  const float a = v[i], b = v[l];
  const int ai = ix[i], bi = ix[l];
  const bool swap = desc ? ranks_before(b, bi, a, ai) : ranks_before(a, ai, b, bi);
  if (swap) {
    v[i] = b;
    ix[i] = bi;
    v[l] = a;
    ix[l] = ai;
  }
}

// Warp-synchronous descending bitonic sort of n (a power of two, n / 2 a
// multiple of 32) pairs in shared memory.
__device__ __forceinline__ void warp_bitonic_sort(float* v, int* ix, int n) {
  const int lane = threadIdx.x & 31;
  for (int k = 2; k <= n; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int pr = lane; pr < n / 2; pr += 32) {
        const int i = (pr / j) * 2 * j + (pr % j);
        bitonic_cx(v, ix, i, i + j, (i & k) == 0);
      }
      __syncwarp();
    }
}

// Warp-synchronous: a[0..32) and b[0..32), each sorted descending, become
// their top 32 (descending) in a: a ++ reverse(b) is bitonic, one merge
// sorts it.
__device__ __forceinline__ void warp_merge_top32(float* av, int* ai, const float* bv,
                                                 const int* bi, float* tv, int* ti) {
  const int lane = threadIdx.x & 31;
  tv[lane] = av[lane];
  ti[lane] = ai[lane];
  tv[32 + lane] = bv[31 - lane];
  ti[32 + lane] = bi[31 - lane];
  __syncwarp();
  for (int j = 32; j > 0; j >>= 1) {
    const int i = (lane / j) * 2 * j + (lane % j);
    bitonic_cx(tv, ti, i, i + j, true);
    __syncwarp();
  }
  av[lane] = tv[lane];
  ai[lane] = ti[lane];
  __syncwarp();
}

// A lower bound of the value of the K-th largest element seen so far by
// the CTA: the m-th largest (m = ceil(K/4) <= 2 kWarps) of the warps' two
// largest fourth values, since m threads then hold four elements each at or
// above it.  An element below the bound cannot be among the K largest.
// -inf while fewer than m lists are full.  Every thread must call it (two
// barriers).
__device__ __forceinline__ float topk_lower_bound(float t3, int i3, int m, PassSmem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float v = i3 == kIdxNone ? -INFINITY : t3;
#pragma unroll
  for (int r = 0; r < 2; ++r) {  // this warp's two largest (one instance removed)
    float w = v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) w = fmaxf(w, __shfl_xor_sync(kFull, w, o));
    if (lane == 0) sm.tw[2 * warp + r] = w;
    const unsigned own = __ballot_sync(kFull, v == w);
    if (lane == __ffs(own) - 1) v = -INFINITY;
  }
  __syncthreads();
  if (warp == 0) {  // lane a ranks value a among the 2 kWarps values (ties by position)
    const float x = lane < 2 * kWarps ? sm.tw[lane] : -INFINITY;
    int above = 0;
#pragma unroll
    for (int c = 0; c < 2 * kWarps; ++c) {
      const float y = sm.tw[c];
      above += (y > x || (y == x && c < lane)) ? 1 : 0;
    }
    const unsigned hit = __ballot_sync(kFull, lane < 2 * kWarps && above == m - 1);
    if (lane == __ffs(hit) - 1) sm.tau = x;
  }
  __syncthreads();
  return sm.tau;
}

// Best (value, index) of the elements of [lo, hi) (thread-strided vectors)
// that rank after (pv, pi), -inf and NaN skipped.
template <typename Tag, bool VEC>
__device__ __forceinline__ void next_after(const typename Tag::Elem* row, int lo, int hi,
                                           float pv, int pi, float& bv, int& bi) {
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
      if (z[e] > -INFINITY && ranks_before(pv, pi, z[e], idx) && ranks_before(z[e], idx, bv, bi)) {
        bv = z[e];
        bi = idx;
      }
    }
  }
}

// grid (chunk groups, 2k+1 rows, batch rows).  Row r < k+1 is Z[b, r],
// otherwise D[b, r - k - 1].
template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kThreads, 4) topk_pass_kernel(TopkParams p) {
  using Elem = typename Tag::Elem;
  constexpr int kV = VEC ? Tag::kVec : 1;
  constexpr int U = 4;
  __shared__ PassSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = p.G;
  const int c = blockIdx.x * G, r = blockIdx.y, b = blockIdx.z + p.b0;
  const int lo = c * p.CH, hi = min(p.V, lo + G * p.CH);
  const int n_slots = min(G, p.C - c);
  const int Pz = p.k + 1;
  const Elem* row = (r < Pz)
      ? static_cast<const Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb + static_cast<int64_t>(r) * p.V
      : static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
            static_cast<int64_t>(r - Pz) * p.V;
  PartStat* out_part = p.part + (static_cast<int64_t>(b) * p.R + r) * p.C + c;
  TopEntry* out_list = p.lists + ((static_cast<int64_t>(b) * p.R + r) * p.C + c) * p.K;
  if (tid > 0 && tid < n_slots) {
    PartStat id;
    id.m = -INFINITY;
    id.s = 0.f;
    id.idx = kIdxNone;
    id.flags = 0;
    out_part[tid] = id;
  }
  for (int q = p.K + tid; q < n_slots * p.K; q += kThreads) {  // empty lists of slots 1..
    out_list[q].v = -INFINITY;
    out_list[q].i = kIdxNone;
  }
  if (tid == 0) sm.cnt = 0;

  Top4 st;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    st.t[q] = -INFINITY;
    st.i[q] = kIdxNone;
  }
  st.b5 = -INFINITY;
  st.nan = 0;
  const int v0 = lo / kV, v1 = (hi + kV - 1) / kV;
  // Vectors whose maximum is below tau, a lower bound of the K-th largest
  // value (refreshed after 1, 2, 4, 8, ... rounds), are skipped: at a whole
  // row per CTA this spares most of the divergent list insertions.
  const int m4 = (p.K + kPer - 1) / kPer;
  float tau = -INFINITY;
  int it = 0;
  for (int base = v0; base < v1; base += kThreads * U, ++it) {  // block-uniform trips
    const int vb = base + tid;
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
        float vm = z[0];
#pragma unroll
        for (int e = 1; e < kV; ++e) vm = max_nan(vm, z[e]);
        if (vm != vm) {
          st.nan = 1;
        } else if (vm < tau) {
          // below the bound: none of these is among the K largest
        } else if (!(vm > st.t[3])) {
          st.b5 = fmaxf(st.b5, vm);  // the whole vector stays below the list
        } else {
#pragma unroll
          for (int e = 0; e < kV; ++e) top4_push(st, z[e], vi * kV + e);
        }
      }
    }
    if (((it + 1) & it) == 0 && base + kThreads * U < v1)
      tau = topk_lower_bound(st.t[kPer - 1], st.i[kPer - 1], m4, sm);
  }
  // the warps' largest "fifth" values
  float w5 = st.nan ? NAN : st.b5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) w5 = max_nan(w5, __shfl_xor_sync(kFull, w5, o));
  if (lane == 0) sm.w5[warp] = w5;
  ScanState ss;
  scan_init(ss);
  ss.m = st.t[0];
  ss.idx = st.i[0];
  ss.nan = st.nan;
  block_stats_write(ss, 0.f, false, sm.m, sm.s, sm.i, sm.n, out_part);  // holds a barrier
  float M5 = sm.w5[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M5 = max_nan(M5, sm.w5[w]);
  if (M5 != M5) {  // a NaN: the row is invalid, its list is not used
    for (int q = tid; q < p.K; q += kThreads) {
      out_list[q].v = -INFINITY;
      out_list[q].i = kIdxNone;
    }
    return;
  }
  int mine = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) mine += (st.i[q] != kIdxNone && st.t[q] > M5) ? 1 : 0;
  if (mine) atomicAdd(&sm.cnt, mine);
  __syncthreads();
  // certified: every element outside the candidates is <= M5, and at least K
  // candidates exceed it (or nothing finite lies outside the candidates)
  const bool certified = sm.cnt >= p.K || M5 == -INFINITY;
  // the K best candidates.  K <= 16: each warp ranks its 128 (four per
  // lane, in registers) by K arg-max rounds and warp 0 merges the eight
  // lists by K rounds.  K > 16: each warp bitonic-sorts its 128 in shared
  // memory, then the eight sorted top-32 lists merge pairwise (three levels
  // of bitonic merges); its cost does not grow with K and is below that of
  // 2K rounds from K ~ 20 on (measured at V = 151936).
  if (p.K > 16) {
    float* v = sm.sv[warp];
    int* ix = sm.si[warp];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      v[lane * kPer + q] = st.t[q];
      ix[lane * kPer + q] = st.i[q];
    }
    __syncwarp();
    warp_bitonic_sort(v, ix, 32 * kPer);
    if (tid == 0) sm.nx = 0;
    __syncthreads();
    for (int step = 1; step < kWarps; step <<= 1) {  // lists in sv[w][0..32)
      if ((warp & (2 * step - 1)) == 0)
        warp_merge_top32(sm.sv[warp], sm.si[warp], sm.sv[warp + step], sm.si[warp + step],
                         sm.sv[warp] + 32, sm.si[warp] + 32);
      __syncthreads();
    }
    if (tid < p.K) {
      sm.lv[tid] = sm.si[0][tid] == kIdxNone ? -INFINITY : sm.sv[0][tid];
      sm.li[tid] = sm.si[0][tid];
    }
  } else {
    float t[kPer];
    int ix[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      t[q] = st.t[q];
      ix[q] = st.i[q];
    }
    for (int rr = 0; rr < p.K; ++rr) {
      float bv = t[0];
      int bi = ix[0], bq = 0;
#pragma unroll
      for (int q = 1; q < kPer; ++q)
        if (ranks_before(t[q], ix[q], bv, bi)) {
          bv = t[q];
          bi = ix[q];
          bq = q;
        }
      float wv = bv;
      int wi = bi;
      warp_argmax(wv, wi);
      if (lane == 0) {
        sm.wl[warp][rr] = (wi == kIdxNone) ? -INFINITY : wv;
        sm.wi[warp][rr] = wi;
      }
      if (wi != kIdxNone && wi == bi) {  // this lane held the pick
#pragma unroll
        for (int q = 0; q < kPer; ++q)
          if (q == bq) {
            t[q] = -INFINITY;
            ix[q] = kIdxNone;
          }
      }
    }
    if (tid == 0) sm.nx = 0;
    __syncthreads();
    if (warp == 0) {
      int head = 0;
      for (int rr = 0; rr < p.K; ++rr) {
        float hv = -INFINITY;
        int hi2 = kIdxNone;
        if (lane < kWarps && head < p.K) {
          hv = sm.wl[lane][head];
          hi2 = sm.wi[lane][head];
        }
        float wv = hv;
        int wi = hi2;
        warp_argmax(wv, wi);
        if (wi != kIdxNone && wi == hi2) ++head;
        if (lane == 0) {
          sm.lv[rr] = wv;
          sm.li[rr] = wi;
        }
      }
    }
  }
  __syncthreads();
  if (certified) {
    for (int q = tid; q < p.K; q += kThreads) {
      out_list[q].v = sm.lv[q];
      out_list[q].i = sm.li[q];
    }
    return;
  }
  // Second chance (rare; e.g. several of a row's top logits in one vector).
  // With tau the candidates' K-th best, every element of the true top K
  // that is not a candidate ranks before tau and lies in a thread whose
  // fifth value b5 is >= tau: those threads re-read their own elements and
  // add the ones ranking before tau; the top K of the candidates' list and
  // these extras is exact.
  const float tv = sm.lv[p.K - 1];
  const int ti = sm.li[p.K - 1];
  bool second = ti != kIdxNone;
  if (second && st.b5 >= tv) {
    for (int v = v0 + tid; v < v1; v += kThreads) {
      float z[8];
      if (VEC) Tag::loadv_cached(row + static_cast<int64_t>(v) * kV, z);
      else z[0] = Tag::load1(row + v);
#pragma unroll
      for (int e = 0; e < kV; ++e) {
        const int idx = v * kV + e;
        const bool own = idx == st.i[0] || idx == st.i[1] || idx == st.i[2] || idx == st.i[3];
        if (!own && z[e] > -INFINITY && ranks_before(z[e], idx, tv, ti)) {
          const int q = atomicAdd(&sm.nx, 1);
          if (q < kSecond) {
            sm.xv[q] = z[e];
            sm.xi[q] = idx;
          }
        }
      }
    }
  }
  __syncthreads();
  const int nx = sm.nx;
  if (second && nx <= kSecond) {
    if (warp != 0) return;
    float pv = INFINITY;
    int pi = -1;
    for (int rr = 0; rr < p.K; ++rr) {
      float bv = -INFINITY;
      int bi = kIdxNone;
      for (int q = lane; q < p.K + nx; q += 32) {
        const float ev = q < p.K ? sm.lv[q] : sm.xv[q - p.K];
        const int ei = q < p.K ? sm.li[q] : sm.xi[q - p.K];
        if (ei != kIdxNone && ranks_before(pv, pi, ev, ei) && ranks_before(ev, ei, bv, bi)) {
          bv = ev;
          bi = ei;
        }
      }
      warp_argmax(bv, bi);
      if (lane == 0) {
        out_list[rr].v = bi == kIdxNone ? -INFINITY : bv;
        out_list[rr].i = bi;
      }
      pv = bv;
      pi = bi;
    }
    return;
  }
  // last resort (the list was short or the buffer overflowed): K rounds of
  // a block-wide arg-max over the group's elements
  float pv = INFINITY;
  int pi = -1;
  for (int rr = 0; rr < p.K; ++rr) {
    float bv;
    int bi;
    next_after<Tag, VEC>(row, lo, hi, pv, pi, bv, bi);
    warp_argmax(bv, bi);
    if (lane == 0) {
      sm.bv[warp] = bv;
      sm.bi[warp] = bi;
    }
    __syncthreads();
    bv = sm.bv[0];
    bi = sm.bi[0];
    for (int w = 1; w < kWarps; ++w)
      if (ranks_before(sm.bv[w], sm.bi[w], bv, bi)) {
        bv = sm.bv[w];
        bi = sm.bi[w];
      }
    __syncthreads();
    if (tid == 0) {
      out_list[rr].v = bv;
      out_list[rr].i = bi;
    }
    pv = bv;
    pi = bi;
  }
}

// Finalize shared memory: every row's merged top-K and its kept masses.
struct FinSmem {
  float v[2 * 31 + 1][kMaxTopK];
  int i[2 * 31 + 1][kMaxTopK];
  double a[2 * 31 + 1][kMaxTopK];  // 2^((z - m) c) of the kept entries, 0 beyond the cut
  double S[2 * 31 + 1];            // kept mass
  int len[2 * 31 + 1];             // entries after the top-p cut
  int amax[2 * 31 + 1];            // argmax (lowest index; 0 when every logit is -inf)
  int bad[2 * 31 + 1];             // NaN seen, or (T > 0) +inf / no finite entry
  int heads[kWarps][256];
  double wbuf[kMaxTopK];
  int tbuf[kMaxTopK];
};

// Inclusive warp scan of a double (lane order).
__device__ __forceinline__ double warp_scan_d(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  return v;
}

// p_f of token t in row r (0 when t is not kept); searched by one lane.
__device__ __forceinline__ double kept_prob(const FinSmem& f, int r, int t) {
  for (int j = 0; j < f.len[r]; ++j)
    if (f.i[r][j] == t) return f.a[r][j] / f.S[r];
  return 0.0;
}

// grid: B.  One CTA per batch row.
__global__ void __launch_bounds__(kThreads) topk_finalize_kernel(TopkParams p) {
  __shared__ float2 tab[64];
  __shared__ FinSmem f;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = p.k, K = p.K, Pz = k + 1;
  load_exp2_table(tab);
  const float T = p.T[b];
  const bool t_bad = isnan(T) || T < 0.f;
  const bool greedy = !(T > 0.f);
  const float P = p.top_p ? p.top_p[b] : 1.f;
  float c_hi = 0.f, c_lo = 0.f;
  if (!greedy && !t_bad) temp_coeff(T, c_hi, c_lo);
  __syncthreads();

  // 1. each row's top K: merge its C sorted chunk lists (one warp per row)
  for (int r = warp; r < p.R; r += kWarps) {
    const PartStat* parts = p.part + (static_cast<int64_t>(b) * p.R + r) * p.C;
    const TopEntry* lists = p.lists + (static_cast<int64_t>(b) * p.R + r) * p.C * K;
    int nan = 0;
    float mx = -INFINITY;
    for (int q = lane; q < p.C; q += 32) {
      nan |= parts[q].flags & 1;
      mx = fmaxf(mx, parts[q].m);
    }
    nan = __any_sync(kFull, nan);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
    int* hd = f.heads[warp];
    for (int q = lane; q < p.C; q += 32) hd[q] = 0;
    __syncwarp();
    int n = 0;
    for (; n < K; ++n) {
      float bv = -INFINITY;
      int bi = kIdxNone, bq = -1;
      for (int q = lane; q < p.C; q += 32) {
        const int h = hd[q];
        if (h < K) {
          const TopEntry e = lists[q * K + h];
          if (e.i != kIdxNone && (bq < 0 || ranks_before(e.v, e.i, bv, bi))) {
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
        if (oq >= 0 && (bq < 0 || ranks_before(ov, oi, bv, bi))) {
          bv = ov;
          bi = oi;
          bq = oq;
        }
      }
      if (bq < 0) break;
      if (lane == (bq & 31)) hd[bq] += 1;
      __syncwarp();
      if (lane == 0) {
        f.v[r][n] = bv;
        f.i[r][n] = bi;
      }
    }
    __syncwarp();
    // 2. kept masses, the top-p cut (lane j holds entry j)
    const bool row_bad = nan || (!greedy && (mx == INFINITY || n == 0));
    double a = 0.0;
    if (!greedy && !row_bad && lane < n) {
      float xh, xl, eh, el;
      arg_df(f.v[r][lane], f.v[r][0], c_hi, c_lo, xh, xl);
      exp2_df(xh, xl, tab, eh, el);
      a = static_cast<double>(eh) + static_cast<double>(el);
    }
    const double cum = warp_scan_d(a);
    const double mass = __shfl_sync(kFull, cum, 31);
    int keep = n;
    if (!greedy && P < 1.f) {
      const unsigned hit = __ballot_sync(kFull, lane < n && cum >= static_cast<double>(P) * mass);
      if (hit) keep = __ffs(hit);
    }
    const double S = (keep > 0) ? __shfl_sync(kFull, cum, keep - 1) : 0.0;
    if (lane < kMaxTopK) f.a[r][lane] = (lane < keep) ? a : 0.0;
    if (lane == 0) {
      f.S[r] = S;
      f.len[r] = greedy ? n : keep;
      f.bad[r] = row_bad ? 1 : 0;
      f.amax[r] = n > 0 ? f.i[r][0] : 0;
    }
  }
  __syncthreads();
  if (warp != 0) return;

  // 3. acceptance at each draft position (lane i), first-reject prefix
  int xi = -1;
  bool tok_bad = false;
  if (lane < k) {
    xi = p.x[static_cast<int64_t>(b) * k + lane];
    tok_bad = xi < 0 || xi >= p.V;
  }
  const bool any_tok_bad = __any_sync(kFull, tok_bad);
  bool rb = false;
  if (lane <= k) rb |= f.bad[lane] != 0;
  if (lane < k) rb |= f.bad[Pz + lane] != 0;
  const bool any_row_bad = __any_sync(kFull, rb);
  int status = 0;
  if (t_bad) status = -1;
  else if (any_tok_bad) status = -2;
  else if (any_row_bad) status = -1;
  float pv = NAN, qv = NAN;
  bool acc = false;
  if (status == 0 && lane < k) {
    if (greedy) {
      acc = (xi == f.amax[lane]);
      pv = acc ? 1.f : 0.f;
      qv = (xi == f.amax[Pz + lane]) ? 1.f : 0.f;
    } else {
      const double pd = kept_prob(f, lane, xi);
      const double qd = kept_prob(f, Pz + lane, xi);
      const float u = p.u_acc[static_cast<int64_t>(b) * k + lane];
      acc = (qd == 0.0) ? (pd > 0.0) : (static_cast<double>(u) < pd / qd);
      pv = static_cast<float>(pd);
      qv = static_cast<float>(qd);
    }
  }
  const unsigned ball = __ballot_sync(kFull, acc);
  const unsigned rej = ~ball & ((1u << k) - 1u);
  int n = rej ? (__ffs(rej) - 1) : k;
  if (status != 0) n = status;
  if (lane < k && p.p_at_x) {
    p.p_at_x[static_cast<int64_t>(b) * k + lane] = (status == 0) ? pv : NAN;
    p.q_at_x[static_cast<int64_t>(b) * k + lane] = (status == 0) ? qv : NAN;
  }

  // 4. the recovery / bonus token over the kept candidates of Z[b, n], in
  // token order (the inverse CDF runs over the vocabulary in index order)
  int tok = -1;
  if (n >= 0 && p.out_tok) {
    if (greedy) {
      tok = f.amax[n];
    } else if (p.u_smp) {
      const int L = f.len[n];
      double w = 0.0;
      int t = kIdxNone;
      if (lane < L) {
        t = f.i[n][lane];
        const double pf = f.a[n][lane] / f.S[n];
        w = pf;
        if (n < k) {
          const double d = pf - kept_prob(f, Pz + n, t);
          w = d > 0.0 ? d : 0.0;
        }
      }
      double W = w;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(kFull, W, o);
      if (n < k && W == 0.0 && lane < L) w = f.a[n][lane] / f.S[n];  // all-zero residual
      // rank by token index, then scan in that order
      int rank = 0;
      for (int j = 0; j < L; ++j) rank += (f.i[n][j] < t) ? 1 : 0;
      if (lane < L) {
        f.wbuf[rank] = w;
        f.tbuf[rank] = t;
      }
      __syncwarp();
      const double ws = lane < L ? f.wbuf[lane] : 0.0;
      const int ts = lane < L ? f.tbuf[lane] : -1;
      const double C = warp_scan_d(ws);
      const double total = __shfl_sync(kFull, C, 31);
      const double target = static_cast<double>(p.u_smp[b]) * total;
      const unsigned over = __ballot_sync(kFull, lane < L && C > target);
      const unsigned pos = __ballot_sync(kFull, lane < L && ws > 0.0);
      int pick = over ? (__ffs(over) - 1) : (pos ? (31 - __clz(pos)) : L - 1);
      tok = __shfl_sync(kFull, ts, pick < 0 ? 0 : pick);
    }
  }
  if (p.out_tok && lane <= k) {
    int v = -1;
    if (n >= 0) {
      if (lane < n) v = xi;
      else if (lane == n) v = tok;
    }
    p.out_tok[static_cast<int64_t>(b) * (k + 1) + lane] = v;
  }
  if (lane == 0) {
    p.accept_len[b] = n;
    int e = 0;
    if (t_bad) e |= 0x1;
    else if (any_tok_bad) e |= 0x4;
    else if (any_row_bad) e |= 0x2;
    if (e) atomicOr(p.err, e);
  }
}

}  // namespace

cudaError_t launch_topk_verify(const TopkParams& p0, int dtype, bool vec, cudaStream_t s) {
  TopkParams p = p0;
  for (int b0 = 0; b0 < p0.B; b0 += kMaxGridBatch) {
    p.b0 = b0;
    dim3 grid((p.C + p.G - 1) / p.G, p.R, p0.B - b0 < kMaxGridBatch ? p0.B - b0 : kMaxGridBatch);
    if (dtype == 1) {
      if (vec) topk_pass_kernel<BF16Tag, true><<<grid, kThreads, 0, s>>>(p);
      else topk_pass_kernel<BF16Tag, false><<<grid, kThreads, 0, s>>>(p);
    } else {
      if (vec) topk_pass_kernel<F32Tag, true><<<grid, kThreads, 0, s>>>(p);
      else topk_pass_kernel<F32Tag, false><<<grid, kThreads, 0, s>>>(p);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_topk_finalize(const TopkParams& p, cudaStream_t s) {
  topk_finalize_kernel<<<p.B, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ssd
