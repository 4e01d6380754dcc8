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
#include "ssd_pass.cuh"
#include "ssd_scan.cuh"


namespace ssd {

// grid: (C, rows of this launch, B).  Resident CTAs per SM requested from
// the register allocator: enough 16-byte loads in flight to saturate HBM.
#ifndef SSD_TOPF_MIN_BLOCKS
#define SSD_TOPF_MIN_BLOCKS Tag::kBlocks
#endif
template <typename Tag, bool VEC, bool HAS_TOPF>
__global__ void __launch_bounds__(kThreads, HAS_TOPF ? SSD_TOPF_MIN_BLOCKS : Tag::kBlocks)
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
  pdl_trigger();  // a dependent kernel launched with programmatic serialization may start
  if (p.clr_n > 0) {  // the speculation cache's clear, spread over the grid
    const long long cta = blockIdx.x + static_cast<long long>(gridDim.x) *
                                           (blockIdx.y + static_cast<long long>(gridDim.y) * blockIdx.z);
    const long long nt = static_cast<long long>(gridDim.x) * gridDim.y * gridDim.z * kThreads;
    for (long long i = cta * kThreads + threadIdx.x; i < p.clr_n; i += nt) {
      p.clr_keys[i] = 0xffffffffffffffffull;
      p.clr_winner[i] = 0ull;
    }
  }

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
__global__ void __launch_bounds__(kThreads, SSD_TOPF_MIN_BLOCKS) draft_kernel(const __grid_constant__ StatsParams p) {
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
  ga.rk0 = p.rk0;
  ga.rk1 = p.rk1;
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
// row merges are the critical path (one round for 2(k+1) <= 16 rows).  With
// 8 warps (B > 152) four CTAs fit an SM (64 registers), so 512 rows take one
// wave (measured at B = 512: 18.2 against 22.1 us per launch with the
// unconstrained 112 registers and two CTAs per SM).
template <int NW>
__global__ void __launch_bounds__(NW * 32, NW == 8 ? 4 : 1) finalize_kernel(FinalizeParams p) {
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
  float zx = 0.f, dx = 0.f, ux = 0.f;
  if (lane < k) {
    xi = p.x[static_cast<int64_t>(b) * k + lane];
    ux = p.u_acc[static_cast<int64_t>(b) * k + lane];
    if (!greedy && xi >= 0 && xi < p.V) {
      zx = logit_at(p.Z, p.dtype, static_cast<int64_t>(b) * p.zb + static_cast<int64_t>(lane) * p.V + xi);
      dx = logit_at(p.D, p.dtype, static_cast<int64_t>(b) * p.db + static_cast<int64_t>(lane) * p.V + xi);
    }
  }
  float mz = 0.f, md = 0.f;
  float2 sz = make_float2(0.f, 0.f), sd = make_float2(0.f, 0.f);
  int amz = 0, flz = 0, amd = 0, fld = 0;
  if (lane <= k) {
    mz = rs[lane].m; amz = rs[lane].argmax; flz = rs[lane].flags; sz = rsum[lane];
  }
  if (lane < k) {
    md = rs[p.Pz + lane].m; amd = rs[p.Pz + lane].argmax; fld = rs[p.Pz + lane].flags;
    sd = rsum[p.Pz + lane];
  }
  const AcceptOut ao = accept_warp(k, p.V, greedy, t_bad, c_hi, c_lo, tab, xi, zx, dx, ux, mz,
                                   sz.x, sz.y, amz, flz, md, sd.x, sd.y, amd, fld);
  const int status = ao.status, n = ao.n;
  const float pv = ao.pv, qv = ao.qv;

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
    if (ao.err) atomicOr(p.err, ao.err);
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
