// ssd_chain.cu -- the verify step of a small batch in one kernel after the
// statistics pass: one thread-block cluster per batch row does the
// finalisation (row merges, acceptance, first-reject prefix, forked top-f),
// the recovery / bonus draw and, in the SSD round step, the cache insert of
// its forks and the lookup of its realised outcome.
//
// Rule: speculative-sampling summary, "How It Works" (accept, regenerate from
// the point of divergence); Leviathan et al. / Chen et al.: accept x_i with
// probability min(1, p_i(x_i) / q_i(x_i)); at the first rejection n draw from
// norm(max(0, p_n - q_n)) (p_n if that is all zero), after k accepts from
// p_k; the inverse CDF takes the smallest j with C_j > u C_{V-1}.  "SSD:
// drafting and verification on separate GPUs", "What changes in SSD": the
// speculation cache returns a guessed outcome at once.
//
// At B = 1 the step moves a few MB and is bound by the chain of dependent
// launches (finalisation, norm pass, select, lookup).  Here the chain is one
// launch: the cluster's 8 x 16 warps merge the rows (one warp per row, the
// results written into every CTA's shared memory), every CTA takes the same
// acceptance decisions from the same data (so the cluster's control flow
// and its barriers stay uniform), the draw's pass over row n is split over
// the cluster's threads (the same double-float exponentials and sign split
// as the batched norm pass), the CTAs exchange their fixed-point totals
// through distributed shared memory, and the thread holding floor(u W)
// walks its range.  Hardware cluster barriers only: nothing waits on
// another cluster or kernel.
#include <cooperative_groups.h>
#include <math.h>

#include "ssd_cache.cuh"
#include "ssd_device.cuh"
#include "ssd_draw.cuh"
#include "ssd_layout.h"
#include "ssd_merge.cuh"
#include "ssd_scan.cuh"

namespace ssd {
namespace {

namespace cg = cooperative_groups;

constexpr int kChainThreads = 512;
constexpr int kChainWarps = kChainThreads / 32;
constexpr int kChainAmbCap = 1024;   // ambiguous-sign elements kept per CTA
constexpr int kChainRows = 64;       // 2 (k + 1) <= 64 logit rows per batch row
constexpr int kAccWarp = 1;          // the warp that takes the acceptance decisions

struct ChainSmem {
  float2 tab[64];
  float2 c2;
  // every row's merged statistics (written by its merging warp into every
  // CTA of the cluster)
  float m[kChainRows];
  float sh[kChainRows], sl[kChainRows];
  int am[kChainRows];
  int fl[kChainRows];
  int heads[kChainWarps][256];       // top-f merges
  long long red[kChainWarps];        // block sums and scans
  // every CTA's S_z, S_d, ambiguous overflow and draw mass, pushed by its
  // warp 0 into every CTA of the cluster before a cluster barrier (remote
  // stores: no round trip on the pushing side, local reads after it)
  long long tot[kChainMaxCluster][4];
  int amb_n;
  int amb[kChainAmbCap];
  long long amb_w[kChainThreads];    // exact residual mass of each thread's ambiguous elements
  int res;                           // rank 0: the drawn token
  int pick;
  long long base;
  float2 acc[2];                     // rho = S_z / S_d and 2^12 / S_z, float pairs
  RowCtx cx;
  int dec[2];                        // accepted length (or sentinel), draw mode
};

__device__ __forceinline__ float chain_logit(const void* base, int dtype, int64_t i) {
  if (dtype == 1)
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(base) + i)) << 16);
  return __ldg(static_cast<const float*>(base) + i);
}

// Inclusive block scan of int64 over the 16 warps; *total = the CTA total.
__device__ __forceinline__ long long chain_scan(long long v, long long* red, long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) red[warp] = v;
  __syncthreads();
  long long off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kChainWarps; ++w) {
    const long long s = red[w];
    if (w < warp) off += s;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return v + off;
}

// The forks of batch row b into the cache, spread over the threads of the
// cluster that are not in warp 0: key (b, j, fork_tok[b][j][r]) -> payload
// row (b (k+1) + j) f + r.  A row's forks are distinct tokens per position
// and keys carry b, so no key occurs twice in one call; the claim records
// the call's sequence number in the slot's winner word as the batched
// insert does, so that later calls of either path resolve duplicates by
// call order.
__device__ void chain_insert(const ChainParams& cp, int b, int rank, int cs) {
  const FinalizeParams& p = cp.f;
  const CacheView& c = cp.cache;
  // the call's sequence number: no cluster advances the counter before
  // every cluster has inserted and looked up (the ticket at the end)
  const unsigned long long seq = (__ldcg(c.calls) + 1ull) << 32;
  const int P = p.k + 1, f = p.f;
  const int per_cta = kChainThreads - 32;
  for (int e = rank * per_cta + (static_cast<int>(threadIdx.x) - 32); e < P * f; e += cs * per_cta) {
    const int j = e / f;
    const int64_t idx = static_cast<int64_t>(b) * P * f + e;
    unsigned long long key;
    if (!make_key(b, j, p.fork_tok[idx], key)) continue;
    cache_insert_unique(c, key, seq | static_cast<unsigned long long>(idx),
                        cp.payload + idx * c.depth);
  }
  __threadfence();
}

// Push v into slot `slot` of this CTA's row of every CTA's tot table (lanes
// 0 .. cs-1 of warp 0; every lane must hold v).  A cluster barrier follows.
__device__ __forceinline__ void push_total(cg::cluster_group& cl, ChainSmem& sm, int cs, int rank,
                                           int slot, long long v) {
  const int lane = threadIdx.x & 31;
  if (threadIdx.x < 32 && lane < cs) cl.map_shared_rank(&sm.tot[rank][slot], lane)[0] = v;
}

// The cluster's total of slot `slot` and the part of the CTAs ranked before
// this one, from the local copies.
__device__ __forceinline__ void cluster_prefix(const ChainSmem& sm, int cs, int rank, int slot,
                                               long long& W, long long& before) {
  W = 0;
  before = 0;
#pragma unroll
  for (int r = 0; r < kChainMaxCluster; ++r) {
    const long long v = r < cs ? sm.tot[r][slot] : 0;
    W += v;
    if (r < rank) before += v;
  }
}

// The cluster's totals of slots 0..2 (S_z, S_d, ambiguous overflow).
__device__ __forceinline__ void cluster_sums3(const ChainSmem& sm, int cs, long long& a,
                                              long long& d, long long& o) {
  a = d = o = 0;
#pragma unroll
  for (int r = 0; r < kChainMaxCluster; ++r) {
    if (r < cs) {
      a += sm.tot[r][0];
      d += sm.tot[r][1];
      o += sm.tot[r][2];
    }
  }
}

template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kChainThreads, 1) chain_kernel(ChainParams cp) {
  using Elem = typename Tag::Elem;
  const FinalizeParams& p = cp.f;
  __shared__ ChainSmem sm;
  cg::cluster_group cl = cg::this_cluster();
  const int cs = static_cast<int>(cl.num_blocks()), rank = static_cast<int>(cl.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / cs;
  const int k = p.k, Pz = p.Pz;

  // the cluster barrier's first phase: arrive now, wait before the first
  // access to another CTA's shared memory (every CTA of the cluster has
  // then started)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

  // inputs the statistics pass does not write, fetched before waiting for
  // it: the temperature (thread 0 turns it into log2(e)/T while the rest
  // loads the exp2 table) and what acceptance reads besides the statistics
  // (warp kAccWarp, lane i < k)
  const float T = p.T[b];
  int xi = -1;
  float zx = 0.f, dx = 0.f, ux = 0.f;
  if (warp == kAccWarp && lane < k) {
    xi = p.x[static_cast<int64_t>(b) * k + lane];
    ux = p.u_acc[static_cast<int64_t>(b) * k + lane];
    if (xi >= 0 && xi < p.V) {
      zx = chain_logit(p.Z, p.dtype, static_cast<int64_t>(b) * p.zb + static_cast<int64_t>(lane) * p.V + xi);
      dx = chain_logit(p.D, p.dtype, static_cast<int64_t>(b) * p.db + static_cast<int64_t>(lane) * p.V + xi);
    }
  }
  load_exp2_table(sm.tab);
  if (tid == 0) {
    sm.amb_n = 0;
    sm.res = -1;
  }
  const bool t_bad = isnan(T) || T < 0.f;
  const bool greedy = !(T > 0.f);
  float c_hi = 0.f, c_lo = 0.f;
  if (greedy || t_bad) {  // no exponentials: no coefficient (uniform over the cluster)
    __syncthreads();
  } else {
    const float2 c2 = cta_temp_coeff(T, &sm.c2);  // holds a barrier
    c_hi = c2.x;
    c_lo = c2.y;
  }
  pdl_wait();  // the statistics pass has completed and its partials are visible
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");

  // 1. row merges: cluster-wide warp u < R merges row u; warp R + j merges
  // the top-f lists of fork row j (in parallel with that row's own merge:
  // it needs only the row's NaN flag, an OR over the partial records)
  const int gw = rank * kChainWarps + warp;
  const int n_fork = p.fork_tok ? p.Pdf : 0;
  for (int u = gw; u < p.R + n_fork; u += cs * kChainWarps) {
    if (u < p.R) {
      const int r = u;
      const bool is_target = r < Pz;
      const int j = r - Pz;
      const bool need_stats = is_target || j < p.Pds;
      RowStat st;
      float h, l;
      merge_row(p.part + (static_cast<int64_t>(b) * p.Rp + r) * p.C, p.C, c_hi, c_lo,
                need_stats && !greedy && !t_bad, sm.tab, st, h, l);
      // lane 0's values into every CTA: the CTAs take their decisions from
      // these copies, so they must be the same bits
      st.m = __shfl_sync(kFull, st.m, 0);
      st.argmax = __shfl_sync(kFull, st.argmax, 0);
      st.flags = __shfl_sync(kFull, st.flags, 0);
      h = __shfl_sync(kFull, h, 0);
      l = __shfl_sync(kFull, l, 0);
      if (lane < cs) {
        ChainSmem* dst = cl.map_shared_rank(&sm, lane);
        dst->m[r] = st.m;
        dst->sh[r] = h;
        dst->sl[r] = l;
        dst->am[r] = st.argmax;
        dst->fl[r] = st.flags;
      }
      if (lane == 0) p.rowstat[static_cast<int64_t>(b) * p.Rp + r] = st;
      continue;
    }
    const int j = u - p.R;
    const PartStat* parts = p.part + (static_cast<int64_t>(b) * p.Rp + Pz + j) * p.C;
    int nan = 0;
    for (int q = lane; q < p.C; q += 32) nan |= parts[q].flags & 1;
    nan = __any_sync(kFull, nan != 0);
    const int64_t o = (static_cast<int64_t>(b) * p.Pdf + j) * p.f;
    const int keep = p.fanout ? min(max(__ldg(p.fanout + j), 0), p.f) : p.f;
    merge_topf_row(p.topk + (static_cast<int64_t>(b) * p.Pdf + j) * p.C * p.f, p.C, p.f, keep,
                   nan != 0, p.fork_tok + o, p.fork_logit + o, sm.heads[warp]);
    if (lane == 0 && nan) atomicOr(p.err, 0x2);
    if (cp.cache_on && greedy) {
      // a greedy row draws nothing for the insert to hide behind: its
      // forks go into the cache now, by the warp that merged them
      __syncwarp();
      const unsigned long long seq = (__ldcg(cp.cache.calls) + 1ull) << 32;
      unsigned long long key;
      if (lane < p.f && make_key(b, j, p.fork_tok[o + lane], key))
        cache_insert_unique(cp.cache, key, seq | static_cast<unsigned long long>(o + lane),
                            cp.payload + (o + lane) * cp.cache.depth);
      __threadfence();
    } else if (lane == 0 && cp.cache_on) {
      __threadfence();  // the forks, before the cluster's insert reads them
    }
  }
  cl.sync();  // every row's statistics in every CTA; the forks (greedy: in the cache) in global memory


  // 2. acceptance at each draft position (lane i of warp kAccWarp, in every CTA)
  if (warp == kAccWarp) {
    float mz = 0.f, szh = 0.f, szl = 0.f, md = 0.f, sdh = 0.f, sdl = 0.f;
    int amz = 0, flz = 0, amd = 0, fld = 0;
    if (lane <= k) {
      mz = sm.m[lane]; szh = sm.sh[lane]; szl = sm.sl[lane]; amz = sm.am[lane]; flz = sm.fl[lane];
    }
    if (lane < k) {
      md = sm.m[Pz + lane]; sdh = sm.sh[Pz + lane]; sdl = sm.sl[Pz + lane];
      amd = sm.am[Pz + lane]; fld = sm.fl[Pz + lane];
    }
    const AcceptOut ao = accept_warp(k, p.V, greedy, t_bad, c_hi, c_lo, sm.tab, xi, zx, dx, ux,
                                     mz, szh, szl, amz, flz, md, sdh, sdl, amd, fld);
    const int status = ao.status, n = ao.n;
    const float pv = ao.pv, qv = ao.qv;
    const int mode = (n < 0 || greedy || !cp.u_smp || !p.out_tok)
                         ? kModeNone : (n < k ? kModeResidual : kModeTarget);
    if (rank == 0) {
      if (lane < k && p.p_at_x) {
        p.p_at_x[static_cast<int64_t>(b) * k + lane] = status == 0 ? pv : NAN;
        p.q_at_x[static_cast<int64_t>(b) * k + lane] = status == 0 ? qv : NAN;
      }
      if (p.out_tok && lane <= k) {
        int v = -1;
        if (n >= 0) {
          if (lane < n) v = xi;
          else if (lane == n && greedy) v = sm.am[n];
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
        bs.rho = bs.mode == kModeResidual ? __fdiv_rn(sm.sh[n], sm.sh[Pz + n]) : 1.f;
        bs.pad0 = bs.pad1 = bs.pad2 = 0;
        p.bstate[b] = bs;
        if (p.amb_cnt) p.amb_cnt[b] = 0;
        if (ao.err) atomicOr(p.err, ao.err);
      }
    }
    if (lane == 0) {
      sm.dec[0] = n;
      sm.dec[1] = mode;
    }
  }
  __syncthreads();
  const int n = sm.dec[0], mode = sm.dec[1];

  // 3. the draw: the cluster's threads split row n (and D's row n)
  if (mode != kModeNone) {
    const bool resid_row = mode == kModeResidual;
    const Elem* zr = static_cast<const Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb +
                     static_cast<int64_t>(n) * p.V;
    const Elem* dr = static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
                     static_cast<int64_t>(resid_row ? n : 0) * p.V;
    RowCtx cx;
    cx.mz = sm.m[n];
    cx.md = resid_row ? sm.m[Pz + n] : 0.f;
    cx.c_hi = c_hi;
    cx.c_lo = c_lo;
    cx.rho = resid_row ? __fdiv_rn(sm.sh[n], sm.sh[Pz + n]) : 1.f;
    cx.iz_hi = cx.iz_lo = cx.id_hi = cx.id_lo = 0.f;
    cx.thr_z = cx.thr_d = 0ull;
    const int E = cp.E;
    const int g = rank * kChainThreads + tid;
    const int lo = static_cast<int>(min(static_cast<long long>(p.V), static_cast<long long>(g) * E));
    const int hi = min(p.V, lo + E);
    constexpr int kV = Tag::kVec;
    const f32x2 zero = pk2(0.f, 0.f);
    NormAcc na = {zero, zero, zero, zero};
    int i = lo;
    if (resid_row) {
      if (VEC) {
        for (; i + kV <= hi; i += kV) {
          float z[8], d[8];
          Tag::loadv_cached(zr + i, z);
          Tag::loadv_cached(dr + i, d);
#pragma unroll
          for (int e = 0; e < kV; ++e)
            pass_pair(z[e], d[e], i + e, cx, sm.tab, na, &sm.amb_n, sm.amb, kChainAmbCap);
        }
      }
      for (; i < hi; ++i)
        pass_pair(Tag::load1(zr + i), Tag::load1(dr + i), i, cx, sm.tab, na, &sm.amb_n, sm.amb,
                  kChainAmbCap);
    } else {
      const f32x2 mz = pk2(cx.mz, cx.mz), ch = pk2(c_hi, c_hi), cl2 = pk2(c_lo, c_lo);
      if (VEC) {
        for (; i + kV <= hi; i += kV) {
          float z[8];
          Tag::loadv_cached(zr + i, z);
#pragma unroll
          for (int e = 0; e < kV; e += 2) {
            f32x2 xh, xl, eh, el;
            arg_df2(pk2(z[e], z[e + 1]), mz, ch, cl2, xh, xl);
            exp2_df2(xh, xl, sm.tab, eh, el);
            comp_acc2(na.sh, na.sl, eh, el);
          }
        }
      }
      for (; i < hi; ++i) {
        float xh, xl, a_h, a_l;
        arg_df(Tag::load1(zr + i), cx.mz, c_hi, c_lo, xh, xl);
        exp2_df(xh, xl, sm.tab, a_h, a_l);
        float s0, s1, q0, q1;
        up2(na.sh, s0, s1);
        up2(na.sl, q0, q1);
        comp_acc(s0, q0, a_h, a_l);
        na.sh = pk2(s0, s1);
        na.sl = pk2(q0, q1);
      }
    }
    float sah, sbh, sal, sbl, ah, bh, al, bl;
    up2(na.sh, sah, sbh);
    up2(na.sl, sal, sbl);
    up2(na.ph, ah, bh);
    up2(na.pl, al, bl);
    long long oz, od = 0, oa = 0, ob = 0;  // this thread's S_z, S_d, A, B
    if (resid_row) {
      oz = df_to_fix(sah, sal, kFixMass);
      od = df_to_fix(sbh, sbl, kFixMass);
      oa = df_to_fix(ah, al, kFixAcc);
      ob = df_to_fix(bh, bl, kFixAcc);
    } else {
      oz = df_to_fix(sah, sal, kFixMass) + df_to_fix(sbh, sbl, kFixMass);
    }
    long long tz, td = 0;
    chain_scan(oz, sm.red, &tz);
    if (resid_row) chain_scan(od, sm.red, &td);
    push_total(cl, sm, cs, rank, 0, tz);
    push_total(cl, sm, cs, rank, 1, td);
    push_total(cl, sm, cs, rank, 2, sm.amb_n > kChainAmbCap ? 1 : 0);
    cl.sync();  // the CTAs' normaliser totals
    long long Sz, Sd, ovf;
    cluster_sums3(sm, cs, Sz, Sd, ovf);
    const bool overflow = ovf != 0;
    if (tid == 0) {
      // normalisers and their inverses in double-float; the 2^-42 unit
      // scaling is exact
      constexpr float kMass = 2.2737367544323206e-13f;  // 2^-42
      RowCtx c = cx;
      float szh, szl, sdh, sdl;
      i64_to_df(Sz, szh, szl);
      i64_to_df(resid_row ? Sd : 1, sdh, sdl);
      szh *= kMass; szl *= kMass;
      sdh *= kMass; sdl *= kMass;
      df_recip(szh, szl, c.iz_hi, c.iz_lo);
      df_recip(sdh, sdl, c.id_hi, c.id_lo);
      sm.cx = c;
      float rh, rl;
      df_mul(szh, szl, c.id_hi, c.id_lo, rh, rl);
      sm.acc[0] = make_float2(rh, rl);
      sm.acc[1] = make_float2(c.iz_hi * 4096.f, c.iz_lo * 4096.f);
    }
    sm.amb_w[tid] = 0;
    __syncthreads();
    cx = sm.cx;
    // this thread's residual mass (2^60 units) or target mass (2^42)
    bool resid = resid_row;
    long long own;
    if (!resid) {
      own = oz;
    } else if (!overflow) {
      const int na2 = min(sm.amb_n, kChainAmbCap);
      for (int q = tid; q < na2; q += kChainThreads) {
        const int e = sm.amb[q];
        float wh, wl;
        weight<Q_RESID>(e, Tag::load1(zr + e), Tag::load1(dr + e), cx, sm.tab, wh, wl);
        atomicAdd(reinterpret_cast<unsigned long long*>(&sm.amb_w[e / E - rank * kChainThreads]),
                  static_cast<unsigned long long>(df_to_fix(wh, wl, kFixResidual)));
      }
      __syncthreads();
      own = split_mass(oa, ob, sm.acc[0], sm.acc[1]) + sm.amb_w[tid];
    } else {  // direct exact weights over the thread's range
      float h, l;
      range_sum<Tag, VEC, Q_RESID>(zr, dr, lo, hi, cx, sm.tab, h, l);
      own = df_to_fix(h, l, kFixResidual);
    }
    long long ctot;
    long long incl = chain_scan(own, sm.red, &ctot);
    push_total(cl, sm, cs, rank, 3, ctot);
    cl.sync();  // the CTAs' masses
    long long W, before;
    cluster_prefix(sm, cs, rank, 3, W, before);
    if (resid && W <= 0) {  // all-zero residual: draw from p_n (uniform over the cluster)
      resid = false;
      own = oz;
      incl = chain_scan(own, sm.red, &ctot);
      cl.sync();  // every CTA has read the residual masses
      push_total(cl, sm, cs, rank, 3, ctot);
      cl.sync();
      cluster_prefix(sm, cs, rank, 3, W, before);
    }
    long long t =
        static_cast<long long>(scale_by_uniform(static_cast<unsigned long long>(W), cp.u_smp[b]));
    if (t >= W) t = W - 1;  // u >= 1 (outside the documented range): the last positive element
    // the thread whose range holds the target (exactly one in the cluster)
    if (tid == 0) sm.pick = -1;
    __syncthreads();
    const long long gincl = before + incl;
    if (own > 0 && gincl > t && gincl - own <= t) {
      sm.pick = tid;
      sm.base = gincl - own;
    }
    __syncthreads();
    // the forks into the cache (every warp but warp 0, beside the walk)
    if (cp.cache_on && warp > 0) chain_insert(cp, b, rank, cs);
    if (sm.pick >= 0 && warp == 0) {  // walk the picked range, one lane per element
      const float scale = resid ? kFixResidual : kFixMass;
      const int gp = rank * kChainThreads + sm.pick;
      const int plo = static_cast<int>(min(static_cast<long long>(p.V), static_cast<long long>(gp) * E));
      const int phi = min(p.V, plo + E);
      long long carry = 0;
      int last_pos = -1, found = -1;
      for (int off = plo; off < phi && found < 0; off += 32) {
        const int e = off + lane;
        long long wf = 0;
        if (e < phi) {
          float wh, wl;
          if (resid) weight<Q_RESID>(e, Tag::load1(zr + e), Tag::load1(dr + e), cx, sm.tab, wh, wl);
          else weight<Q_NORM_Z>(e, Tag::load1(zr + e), 0.f, cx, sm.tab, wh, wl);
          wf = df_to_fix(wh, wl, scale);
        }
        long long cc = wf;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long y = __shfl_up_sync(kFull, cc, o);
          if (lane >= o) cc += y;
        }
        const unsigned over = __ballot_sync(kFull, e < phi && sm.base + carry + cc > t);
        const unsigned posm = __ballot_sync(kFull, e < phi && wf > 0);
        if (posm) last_pos = off + 31 - __clz(posm);
        if (over) found = off + __ffs(over) - 1;
        carry += __shfl_sync(kFull, cc, 31);
      }
      // per-element rounding can leave the target just past the range's
      // cumulative mass: the range's last positive element then
      if (lane == 0)
        *cl.map_shared_rank(&sm.res, 0) = found >= 0 ? found : (last_pos >= 0 ? last_pos : phi - 1);
    }
    cl.sync();  // the token is in rank 0's shared memory
    if (rank == 0 && tid == 0) p.out_tok[static_cast<int64_t>(b) * (k + 1) + n] = sm.res;
  } else if (!greedy) {  // (a greedy row's forks went in with the merges)
    if (cp.cache_on && warp > 0) chain_insert(cp, b, rank, cs);
    cl.sync();  // the insert precedes the lookup (rank 0)
  }

  // 4. the realised outcome (b, n, out_tok[b][n]) in the cache; the last
  // cluster to get here advances the cache's insert-call counter
  if (cp.cache_on && rank == 0 && tid == 0) {
    const int tok = (p.out_tok && n >= 0 && n <= k)
                        ? p.out_tok[static_cast<int64_t>(b) * (k + 1) + n] : -1;
    cache_lookup_one(cp.cache, b, n, tok, cp.hit + b,
                     cp.tok_out + static_cast<int64_t>(b) * cp.cache.depth);
    __threadfence();
    if (atomicAdd(cp.cache.done, 1u) == static_cast<unsigned>(p.B) - 1u) {
      *cp.cache.done = 0u;
      *cp.cache.calls = __ldcg(cp.cache.calls) + 1ull;
      __threadfence();
    }
  }
  cl.sync();  // no CTA leaves while another may still touch its shared memory
}

template <typename Tag, bool VEC>
cudaError_t launch_chain_t(const ChainParams& p, int cs, cudaStream_t s) {
  static const bool attrs_ok =
      cudaFuncSetAttribute(chain_kernel<Tag, VEC>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                           1) == cudaSuccess;
  if (!attrs_ok && cs > 8) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.f.B) * cs, 1, 1);
  cfg.blockDim = dim3(kChainThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the launch overlaps the statistics kernel's tail; the kernel waits
  // (griddepcontrol.wait) before it reads the partials
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, chain_kernel<Tag, VEC>, p);
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
      n = v;
  }
  return n;
}

}  // namespace

// Elements per thread of the cluster's draw pass: ceil(V / (cs * 512)),
// rounded up to a multiple of 8 (16-byte aligned ranges).
int chain_elems_per_thread(int V, int cs) {
  const long long nt = static_cast<long long>(cs) * kChainThreads;
  long long E = (V + nt - 1) / nt;
  E = (E + 7) / 8 * 8;
  return static_cast<int>(E);
}

// One cluster per batch row: 16 CTAs while the clusters of the batch fit the
// GPU at one CTA per SM (the kernel's register budget allows no second), else
// 8 (a smaller cluster again when a size cannot be placed).
cudaError_t launch_chain(ChainParams p, int dtype, bool vec, cudaStream_t s) {
  if (p.f.B <= 0) return cudaSuccess;
  const long long sms = sm_count();
  int cs = kChainMaxCluster;
  while (cs > 8 && static_cast<long long>(p.f.B) * cs > sms) cs /= 2;
  for (;; cs /= 2) {
    p.E = chain_elems_per_thread(p.f.V, cs);
    cudaError_t e;
    if (dtype == 1)
      e = vec ? launch_chain_t<BF16Tag, true>(p, cs, s) : launch_chain_t<BF16Tag, false>(p, cs, s);
    else
      e = vec ? launch_chain_t<F32Tag, true>(p, cs, s) : launch_chain_t<F32Tag, false>(p, cs, s);
    if (e == cudaSuccess || cs == 1) return e;
    (void)cudaGetLastError();
  }
}

}  // namespace ssd
