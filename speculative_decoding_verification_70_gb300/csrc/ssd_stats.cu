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
#include "ssd_scan.cuh"


namespace ssd {

struct StatsSmem {
  float m[kWarps], s[kWarps];
  int i[kWarps], n[kWarps];
  int mask[kMaxMask];
};

constexpr int kMaxF = 16;

// Top-f scratch: every thread's maximum, the warps' largest second values
// and the selection.
struct TopfScratch {
  float cv[kThreads];
  int ci[kThreads];
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
// tokens and NaN skipped), certified: with M2 the largest second value of
// any thread, every element that is not a thread maximum is at most M2, so
// if at least f unmasked thread maxima exceed M2 the top f are thread
// maxima and warp 0 picks them from the 256 posted candidates while the
// other warps leave.  Otherwise (rare; ties included) the exact selection is
// redone over [lo, hi) by f rounds of a block-wide arg-max.  Needs
// topf_post and a barrier before it.
template <typename Tag, bool VEC>
__device__ void topf_select(const StatsParams& p, const ScanState& st,
                            const typename Tag::Elem* row, int lo, int hi, const int* msk,
                            TopEntry* out_top, int n_slots, TopfScratch& ts) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int f = p.f, M = p.M;
  float M2 = ts.w2[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M2 = max_nan(M2, ts.w2[w]);
  const bool cand = ts.ci[tid] != kIdxNone && ts.cv[tid] > M2;  // false when M2 is NaN
  if (__syncthreads_count(cand) >= f) {
    if (warp != 0) return;
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
    __syncwarp();
    // the group's list goes to its first chunk slot; the other slots of the
    // group get empty entries, which rank last in the merge
    for (int q = lane; q < n_slots * f; q += 32) {
      const int slot = q / f, r = q % f;
      out_top[q].v = slot == 0 ? ts.sv[r] : -INFINITY;
      out_top[q].i = slot == 0 ? ts.si[r] : kIdxNone;
    }
    return;
  }
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

template <typename Tag, bool VEC, bool DO_EXP, bool TOPF>
__device__ void stats_chunk(const StatsParams& p, const typename Tag::Elem* row, int lo, int hi,
                            float c, PartStat* out_part, TopEntry* out_top, int n_slots,
                            StatsSmem& sm, TopfScratch* ts) {
  constexpr int kV = VEC ? Tag::kVec : 1;
  constexpr int U = 4;
  const int tid = threadIdx.x;
  ScanState st;
  scan_init(st);
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
      }
    }
  }
  if constexpr (TOPF) topf_post(st, sm.mask, p.M, *ts);
  block_stats_write(st, c, DO_EXP, sm.m, sm.s, sm.i, sm.n, out_part);
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

// ---------------------------------------------------------------------------
// Finalisation.
// ---------------------------------------------------------------------------

// Merge the C partial records of one row (one warp).  S is accumulated in
// double with extended-precision rescaling factors.
__device__ void merge_row(const PartStat* parts, int C, float c_hi, float c_lo, bool do_exp,
                          const float2* tab, RowStat& rs) {
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
  double S = 0.0;
  if (do_exp) {
    for (int q = lane; q < C; q += 32) {
      PartStat ps = parts[q];
      double fct;
      if (ps.m == m) {
        fct = 1.0;
      } else {
        float xh, xl, eh, el;
        arg_df(ps.m, m, c_hi, c_lo, xh, xl);
        exp2_df(xh, xl, tab, eh, el);
        fct = static_cast<double>(eh) + static_cast<double>(el);
      }
      S += static_cast<double>(ps.s) * fct;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(kFull, S, o);
  }
  rs.m = m;
  rs.argmax = idx;
  rs.S = do_exp ? S : 1.0;
  int bad = nan;
  if (do_exp && !(S > 0.0 && S < INFINITY)) bad = 1;  // +inf, NaN or all -inf at T > 0
  rs.flags = (nan ? 1 : 0) | (bad ? 2 : 0);
}

// Top-f of one fork row from its C chunk lists (one warp).  Only the first
// `keep` picks are written; slots keep .. f-1 get (token -1, logit -inf).
__device__ void merge_topf_row(const TopEntry* lists, int C, int f, int keep, bool nan,
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

__device__ __forceinline__ float logit_at(const void* base, int dtype, int64_t i) {
  if (dtype == 1)
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(base) + i)) << 16);
  return __ldg(static_cast<const float*>(base) + i);
}

// grid: B.  Verification (and, when fork_tok != null, the forked top-f).
__global__ void __launch_bounds__(kThreads) finalize_kernel(FinalizeParams p) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ float2 tab[64];
  __shared__ RowStat rs[2 * (32 + 1)];
  __shared__ int heads[kWarps][256];
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
  for (int r = warp; r < p.R; r += kWarps) {
    bool is_target = r < p.Pz;
    int j = r - p.Pz;
    bool need_stats = is_target || j < p.Pds;
    bool do_exp = need_stats && !greedy && !t_bad;
    RowStat st;
    merge_row(p.part + (static_cast<int64_t>(b) * p.Rp + r) * p.C, p.C, c_hi, c_lo, do_exp, tab, st);
    if (lane == 0) {
      rs[r] = st;
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
      float xh, xl, eh, el;
      arg_df(zx, tz.m, c_hi, c_lo, xh, xl);
      exp2_df(xh, xl, tab, eh, el);
      double pd = (static_cast<double>(eh) + static_cast<double>(el)) / tz.S;
      arg_df(dx, td.m, c_hi, c_lo, xh, xl);
      exp2_df(xh, xl, tab, eh, el);
      double qd = (static_cast<double>(eh) + static_cast<double>(el)) / td.S;
      float u = p.u_acc[static_cast<int64_t>(b) * k + lane];
      acc = (qd == 0.0) ? (pd > 0.0) : (static_cast<double>(u) < pd / qd);
      pv = static_cast<float>(pd);
      qv = static_cast<float>(qd);
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
    bs.pad0 = bs.pad1 = 0;
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
  merge_row(p.part + static_cast<int64_t>(r) * p.C, p.C, c_hi, c_lo, !greedy && !t_bad, tab, st);
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

cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s) {
  finalize_kernel<<<p.B, kThreads, 0, s>>>(p);
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
