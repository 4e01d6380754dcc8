// ssd_step.cu -- the whole verify call of a small batch as one cooperative
// kernel: statistics pass, row merges and forks, acceptance, the draw and
// (SSD round step) the cache clear, insert and outcome lookup.
//
// Rule: speculative-sampling summary, "How It Works" (accept, regenerate
// from the point of divergence); Leviathan et al. / Chen et al.: accept x_i
// with probability min(1, p_i(x_i) / q_i(x_i)); at the first rejection n
// draw from norm(max(0, p_n - q_n)) (p_n if that is all zero), after k
// accepts from p_k; the inverse CDF takes the smallest j with C_j > u C_{V-1}.
// "tanishqkumar/ssd" summary, module notes: forked recovery tokens by top-k
// over the logits with masking.  "SSD: drafting and verification on separate
// GPUs", "What changes in SSD": the speculation cache returns a guessed
// outcome at once.
//
// A batch of a few rows moves a few MB per call, so the call is bound by
// its chain of dependent launches (statistics, finalisation, norm pass,
// select, cache kernels), each a few microseconds of launch and drain.
// Here the chain is one launch of as many CTAs as the GPU holds at once
// (a cooperative launch guarantees they are all resident), and the steps
// are separated by grid-wide barriers:
//   1. statistics: one CTA per (row, chunk) unit, the same per-chunk pass as
//      the statistics kernel (and the cache clear);
//   2. merges: one warp per logit row -- maximum, S as a float pair, argmax,
//      flags; the fork rows' top-f and their cache inserts;
//   3. acceptance (every CTA, warp b for batch row b, from the merged rows),
//      then the exact normalisers of rows n: every thread sums
//      a = 2^((z - m_z) c) and b = 2^((d - m_d) c) over its range in
//      double-float, 2^42 fixed point per CTA;
//   4. the exact residual mass max(0, a / S_z - b / S_d) of each thread's
//      range (2^60 fixed point), per CTA;
//   5. floor(u W) among the CTA masses, then the threads of the CTA that
//      holds it, then the elements of the thread that holds it.
// Every decision taken in more than one CTA is taken from the same bits by
// the same code, so control flow around the barriers is uniform.  Barriers
// and the exit are bounded: a wait that outlasts its limit sets
// SSD_DEVERR_TIMEOUT and the kernel skips to its exit.
#include <math.h>

#include "ssd_cache.cuh"
#include "ssd_device.cuh"
#include "ssd_draw.cuh"
#include "ssd_layout.h"
#include "ssd_merge.cuh"
#include "ssd_pass.cuh"
#include "ssd_scan.cuh"

namespace ssd {
namespace {

constexpr unsigned long long kStepWaitNs = 1000000000ull;  // a barrier wait gives up after 1 s
constexpr long long kStepSpin = 1ll << 24;                   // and after this many polls
constexpr int kStepMinBlocks = 4;           // resident CTAs per SM requested from the allocator

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void st_release(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier.  Arrival in two levels (CTA g counts on sub-counter
// g mod 8, the last of each group on the top counter) so that no single
// address takes every CTA's atomic; the last arrival resets the counters and
// advances the generation word, which the others poll.  A wait gives up
// after 1 s (global timer) or 2^24 polls: it sets SSD_DEVERR_TIMEOUT and the
// abort word.  Returns false (and the caller goes to its exit) once any CTA
// gave up waiting.
__device__ bool grid_barrier(StepBar* bar, int* err, int* s_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    if (ld_acquire(&bar->abort_[0]) != 0) {
      ok = 0;
    } else {
      const unsigned G = gridDim.x;
      const unsigned s = blockIdx.x % kStepSubBars;
      const unsigned share = (G - s + kStepSubBars - 1) / kStepSubBars;
      const unsigned groups = G < static_cast<unsigned>(kStepSubBars) ? G : kStepSubBars;
      const unsigned g = ld_acquire(&bar->gen[0]);  // before arriving
      __threadfence();
      bool last = false;
      if (atomicAdd(&bar->sub[s][0], 1u) == share - 1) {
        atomicExch(&bar->sub[s][0], 0u);
        __threadfence();
        if (atomicAdd(&bar->top[0], 1u) == groups - 1) {
          atomicExch(&bar->top[0], 0u);
          __threadfence();
          st_release(&bar->gen[0], g + 1);
          last = true;
        }
      }
      if (!last) {
        long long it = 0;
        const unsigned long long t0 = global_ns();
        while (ld_acquire(&bar->gen[0]) == g) {
          if (++it > kStepSpin || global_ns() - t0 > kStepWaitNs ||
              ld_acquire(&bar->abort_[0]) != 0) {
            ok = 0;
            atomicOr(err, 0x10);
            atomicExch(&bar->abort_[0], 1u);
            break;
          }
          __nanosleep(64);
        }
      }
    }
    *s_flag = ok;
  }
  __syncthreads();
  return *s_flag != 0;
}

struct StepSmem {
  union {
    struct {
      StatsSmem st;
      TopfScratch ts;
    } p1;                                  // statistics units
    int heads[kWarps][256];                // top-f merges
  } u;
  float2 tab[64];
  float2 c2;
  long long red[kWarps];
  long long own_a[kStepMaxB][kThreads];    // each thread's S_z of row n (2^42)
  long long own_w[kStepMaxB][kThreads];    // each thread's draw mass of row n
  long long cta_w[kStepMaxB];
  RowCtx cx[kStepMaxB];
  int dec_n[kStepMaxB], dec_mode[kStepMaxB];
  int flag;
};

__device__ __forceinline__ float step_logit(const void* base, int dtype, int64_t i) {
  if (dtype == 1)
    return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const unsigned short*>(base) + i)) << 16);
  return __ldg(static_cast<const float*>(base) + i);
}

__device__ __forceinline__ long long& cta_slot(const StepParams& q, int w, int b) {
  return q.cta[(static_cast<int64_t>(w) * q.f.B + b) * kStepMaxGrid + blockIdx.x];
}

// Sum over the grid's CTAs of cta[w][b][*] (every thread of the CTA gets
// it) and, in *before, the part of CTAs 0 .. blockIdx.x - 1.
__device__ __forceinline__ long long grid_total(const StepParams& q, int w, int b, long long* red,
                                                long long* before) {
  const long long* v = q.cta + (static_cast<int64_t>(w) * q.f.B + b) * kStepMaxGrid;
  long long all = 0, pre = 0;
  for (int g = threadIdx.x; g < static_cast<int>(gridDim.x); g += kThreads) {
    const long long x = __ldcg(v + g);
    all += x;
    if (g < static_cast<int>(blockIdx.x)) pre += x;
  }
  all = block_sum_i64(all, red);
  if (before) *before = block_sum_i64(pre, red);
  return all;
}

template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kThreads, kStepMinBlocks) step_kernel(StepParams q) {
  using Elem = typename Tag::Elem;
  const StatsParams& sp = q.sp;
  const FinalizeParams& p = q.f;
  __shared__ StepSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  const int B = p.B, k = p.k, Pz = p.Pz, V = p.V, R = p.R;

  // what acceptance reads besides the merged rows (warp b, lane i < k),
  // fetched now so that the loads overlap the statistics
  int xi = -1;
  float zx = 0.f, dx = 0.f, ux = 0.f;
  if (warp < B && lane < k) {
    const int b = warp;
    xi = p.x[static_cast<int64_t>(b) * k + lane];
    ux = p.u_acc[static_cast<int64_t>(b) * k + lane];
    if (xi >= 0 && xi < V) {
      zx = step_logit(p.Z, p.dtype, static_cast<int64_t>(b) * p.zb + static_cast<int64_t>(lane) * V + xi);
      dx = step_logit(p.D, p.dtype, static_cast<int64_t>(b) * p.db + static_cast<int64_t>(lane) * V + xi);
    }
  }
  const unsigned long long seq = q.cache_on ? ((__ldcg(q.cache.calls) + 1ull) << 32) : 0ull;
  load_exp2_table(sm.tab);
  if (q.cache_on && q.cache_clear)
    for (int i = blockIdx.x * kThreads + tid; i < q.cache.capacity; i += G * kThreads) {
      q.cache.keys[i] = kEmptyKey;
      q.cache.winner[i] = 0ull;
    }

  // 1. statistics (units: groups of sp.G chunks)
  const int ngroups = (sp.C + sp.G - 1) / sp.G;
  for (int u = blockIdx.x; u < q.units; u += G) {
    const int c = (u % ngroups) * sp.G, rr = u / ngroups;
    __syncthreads();  // the previous unit's scratch
    stats_unit<Tag, VEC>(sp, rr / sp.R, rr % sp.R, c, sm.u.p1.st, sm.u.p1.ts, &sm.c2);
  }
  bool ok = grid_barrier(q.bar, p.err, &sm.flag);

  // 2. row merges (one warp per row) and forks
  if (ok) {
    for (int u = blockIdx.x * kWarps + warp; u < B * R; u += G * kWarps) {
      const int b = u / R, r = u % R;
      const float T = p.T[b];
      const bool t_bad = isnan(T) || T < 0.f;
      const bool greedy = !(T > 0.f);
      float c_hi = 0.f, c_lo = 0.f;
      if (!greedy && !t_bad) {
        if (lane == 0) temp_coeff(T, c_hi, c_lo);
        c_hi = __shfl_sync(kFull, c_hi, 0);
        c_lo = __shfl_sync(kFull, c_lo, 0);
      }
      const bool is_target = r < Pz;
      const int j = r - Pz;
      const bool need_stats = is_target || j < p.Pds;
      RowStat st;
      float h, l;
      merge_row(p.part + (static_cast<int64_t>(b) * p.Rp + r) * p.C, p.C, c_hi, c_lo,
                need_stats && !greedy && !t_bad, sm.tab, st, h, l);
      if (lane == 0) {
        p.rowstat[static_cast<int64_t>(b) * p.Rp + r] = st;
        StepRow sr;
        sr.m = st.m;
        sr.sh = h;
        sr.sl = l;
        sr.argmax = st.argmax;
        sr.flags = st.flags;
        sr.pad[0] = sr.pad[1] = sr.pad[2] = 0;
        q.rows[static_cast<int64_t>(b) * R + r] = sr;
      }
      if (!is_target && j < p.Pdf && p.fork_tok) {
        const int64_t o = (static_cast<int64_t>(b) * p.Pdf + j) * p.f;
        const int keep = p.fanout ? min(max(__ldg(p.fanout + j), 0), p.f) : p.f;
        merge_topf_row(p.topk + (static_cast<int64_t>(b) * p.Pdf + j) * p.C * p.f, p.C, p.f, keep,
                       (st.flags & 1) != 0, p.fork_tok + o, p.fork_logit + o, sm.u.heads[warp]);
        if (lane == 0 && (st.flags & 1)) atomicOr(p.err, 0x2);
        if (q.cache_on) {  // key (b, j, token) -> payload row o + r
          __syncwarp();
          unsigned long long key;
          if (lane < p.f && make_key(b, j, p.fork_tok[o + lane], key))
            cache_insert_unique(q.cache, key, seq | static_cast<unsigned long long>(o + lane),
                                q.payload + (o + lane) * q.cache.depth);
        }
      }
    }
    ok = grid_barrier(q.bar, p.err, &sm.flag);
  }

  // 3. acceptance (warp b of every CTA), then the normalisers of rows n
  if (ok) {
    if (warp < B) {
      const int b = warp;
      const float T = p.T[b];
      const bool t_bad = isnan(T) || T < 0.f;
      const bool greedy = !(T > 0.f);
      float c_hi = 0.f, c_lo = 0.f;
      if (!greedy && !t_bad) {
        if (lane == 0) temp_coeff(T, c_hi, c_lo);
        c_hi = __shfl_sync(kFull, c_hi, 0);
        c_lo = __shfl_sync(kFull, c_lo, 0);
      }
      StepRow tz, td;
      tz.m = td.m = 0.f;
      tz.sh = tz.sl = td.sh = td.sl = 0.f;
      tz.argmax = td.argmax = 0;
      tz.flags = td.flags = 0;
      if (lane <= k) tz = q.rows[static_cast<int64_t>(b) * R + lane];
      if (lane < k) td = q.rows[static_cast<int64_t>(b) * R + Pz + lane];
      const AcceptOut ao = accept_warp(k, V, greedy, t_bad, c_hi, c_lo, sm.tab, xi, zx, dx, ux,
                                       tz.m, tz.sh, tz.sl, tz.argmax, tz.flags, td.m, td.sh,
                                       td.sl, td.argmax, td.flags);
      const int n = ao.n;
      const int src = n < 0 ? 0 : n;
      const float mzn = __shfl_sync(kFull, tz.m, src);
      const float shn = __shfl_sync(kFull, tz.sh, src);
      const int amn = __shfl_sync(kFull, tz.argmax, src);
      const float mdn = __shfl_sync(kFull, td.m, src < k ? src : 0);
      const float sdn = __shfl_sync(kFull, td.sh, src < k ? src : 0);
      const int bmode = (n < 0 || greedy) ? kModeNone : (n < k ? kModeResidual : kModeTarget);
      const int mode = (!q.u_smp || !p.out_tok) ? kModeNone : bmode;
      if (lane == 0) {
        sm.dec_n[b] = n;
        sm.dec_mode[b] = mode;
        RowCtx cx;
        cx.mz = mzn;
        cx.md = mode == kModeResidual ? mdn : 0.f;
        cx.c_hi = c_hi;
        cx.c_lo = c_lo;
        cx.iz_hi = cx.iz_lo = cx.id_hi = cx.id_lo = 0.f;
        cx.rho = 1.f;
        cx.thr_z = cx.thr_d = 0ull;
        sm.cx[b] = cx;
      }
      if (blockIdx.x == 0) {
        if (lane < k && p.p_at_x) {
          p.p_at_x[static_cast<int64_t>(b) * k + lane] = ao.status == 0 ? ao.pv : NAN;
          p.q_at_x[static_cast<int64_t>(b) * k + lane] = ao.status == 0 ? ao.qv : NAN;
        }
        if (p.out_tok && lane <= k) {
          int v = -1;
          if (n >= 0) {
            if (lane < n) v = xi;
            else if (lane == n && greedy) v = amn;
          }
          p.out_tok[static_cast<int64_t>(b) * (k + 1) + lane] = v;
        }
        if (lane == 0) {
          p.accept_len[b] = n;
          BState bs;
          bs.n = n;
          bs.mode = bmode;
          bs.c_hi = c_hi;
          bs.c_lo = c_lo;
          bs.rho = bmode == kModeResidual ? __fdiv_rn(shn, sdn) : 1.f;
          bs.pad0 = bs.pad1 = bs.pad2 = 0;
          p.bstate[b] = bs;
          if (p.amb_cnt) p.amb_cnt[b] = 0;
          if (ao.err) atomicOr(p.err, ao.err);
        }
      }
    }
    __syncthreads();
    const int gt = blockIdx.x * kThreads + tid;
    const int lo = static_cast<int>(min(static_cast<long long>(V), static_cast<long long>(gt) * q.E));
    const int hi = min(V, lo + q.E);
    constexpr int kV = Tag::kVec;
    for (int b = 0; b < B; ++b) {
      const int mode = sm.dec_mode[b];
      if (mode == kModeNone) continue;  // uniform over the grid
      const int n = sm.dec_n[b];
      const RowCtx cx = sm.cx[b];
      const Elem* zr = static_cast<const Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb +
                       static_cast<int64_t>(n) * V;
      const f32x2 zero = pk2(0.f, 0.f);
      f32x2 sh = zero, sl = zero;
      int i = lo;
      long long oa, od = 0;
      if (mode == kModeResidual) {
        // a and b of one element as one packed exponential pair
        const Elem* dr = static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
                         static_cast<int64_t>(n) * V;
        const f32x2 m2 = pk2(cx.mz, cx.md), ch = pk2(cx.c_hi, cx.c_hi), cl = pk2(cx.c_lo, cx.c_lo);
        if (VEC) {
          for (; i + kV <= hi; i += kV) {
            float z[8], d[8];
            Tag::loadv_cached(zr + i, z);
            Tag::loadv_cached(dr + i, d);
#pragma unroll
            for (int e = 0; e < kV; ++e) {
              f32x2 xh, xl, eh, el;
              arg_df2(pk2(z[e], d[e]), m2, ch, cl, xh, xl);
              exp2_df2(xh, xl, sm.tab, eh, el);
              comp_acc2(sh, sl, eh, el);
            }
          }
        }
        for (; i < hi; ++i) {
          f32x2 xh, xl, eh, el;
          arg_df2(pk2(Tag::load1(zr + i), Tag::load1(dr + i)), m2, ch, cl, xh, xl);
          exp2_df2(xh, xl, sm.tab, eh, el);
          comp_acc2(sh, sl, eh, el);
        }
        float ah, bh, al, bl;
        up2(sh, ah, bh);
        up2(sl, al, bl);
        oa = df_to_fix(ah, al, kFixMass);
        od = df_to_fix(bh, bl, kFixMass);
      } else {
        // bonus draw: two consecutive elements per packed pair
        const f32x2 mz = pk2(cx.mz, cx.mz), ch = pk2(cx.c_hi, cx.c_hi), cl = pk2(cx.c_lo, cx.c_lo);
        if (VEC) {
          for (; i + kV <= hi; i += kV) {
            float z[8];
            Tag::loadv_cached(zr + i, z);
#pragma unroll
            for (int e = 0; e < kV; e += 2) {
              f32x2 xh, xl, eh, el;
              arg_df2(pk2(z[e], z[e + 1]), mz, ch, cl, xh, xl);
              exp2_df2(xh, xl, sm.tab, eh, el);
              comp_acc2(sh, sl, eh, el);
            }
          }
        }
        for (; i < hi; ++i) {
          float xh, xl, a_h, a_l;
          arg_df(Tag::load1(zr + i), cx.mz, cx.c_hi, cx.c_lo, xh, xl);
          exp2_df(xh, xl, sm.tab, a_h, a_l);
          float s0, s1, c0, c1;
          up2(sh, s0, s1);
          up2(sl, c0, c1);
          comp_acc(s0, c0, a_h, a_l);
          sh = pk2(s0, s1);
          sl = pk2(c0, c1);
        }
        float s0, s1, c0, c1;
        up2(sh, s0, s1);
        up2(sl, c0, c1);
        oa = df_to_fix(s0, c0, kFixMass) + df_to_fix(s1, c1, kFixMass);
      }
      sm.own_a[b][tid] = oa;
      const long long ta = block_sum_i64(oa, sm.red);
      const long long td = mode == kModeResidual ? block_sum_i64(od, sm.red) : 0;
      if (tid == 0) {
        cta_slot(q, 0, b) = ta;
        cta_slot(q, 1, b) = td;
      }
    }
    ok = grid_barrier(q.bar, p.err, &sm.flag);
  }

  // 4. each thread's draw mass of row n
  if (ok) {
    const int gt = blockIdx.x * kThreads + tid;
    const int lo = static_cast<int>(min(static_cast<long long>(V), static_cast<long long>(gt) * q.E));
    const int hi = min(V, lo + q.E);
    for (int b = 0; b < B; ++b) {
      const int mode = sm.dec_mode[b];
      if (mode == kModeNone) continue;
      long long w;
      if (mode == kModeResidual) {
        const long long Sz = grid_total(q, 0, b, sm.red, nullptr);
        const long long Sd = grid_total(q, 1, b, sm.red, nullptr);
        if (tid == 0) {
          // normalisers and their inverses in double-float; the 2^-42 unit
          // scaling is exact
          constexpr float kMass = 2.2737367544323206e-13f;  // 2^-42
          RowCtx c = sm.cx[b];
          float szh, szl, sdh, sdl;
          i64_to_df(Sz, szh, szl);
          i64_to_df(Sd, sdh, sdl);
          szh *= kMass; szl *= kMass;
          sdh *= kMass; sdl *= kMass;
          df_recip(szh, szl, c.iz_hi, c.iz_lo);
          df_recip(sdh, sdl, c.id_hi, c.id_lo);
          sm.cx[b] = c;
        }
        __syncthreads();
        const RowCtx cx = sm.cx[b];
        const int n = sm.dec_n[b];
        const Elem* zr = static_cast<const Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb +
                         static_cast<int64_t>(n) * V;
        const Elem* dr = static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
                         static_cast<int64_t>(n) * V;
        float h, l;
        range_sum<Tag, VEC, Q_RESID>(zr, dr, lo, hi, cx, sm.tab, h, l);
        w = df_to_fix(h, l, kFixResidual);
      } else {
        w = sm.own_a[b][tid];
      }
      sm.own_w[b][tid] = w;
      const long long tw = block_sum_i64(w, sm.red);
      if (tid == 0) {
        cta_slot(q, 2, b) = tw;
        sm.cta_w[b] = tw;
      }
    }
    ok = grid_barrier(q.bar, p.err, &sm.flag);
  }

  // 5. the draw: the CTA, the thread, the element holding floor(u W)
  if (ok) {
    const int gt = blockIdx.x * kThreads + tid;
    const int lo = static_cast<int>(min(static_cast<long long>(V), static_cast<long long>(gt) * q.E));
    const int hi = min(V, lo + q.E);
    for (int b = 0; b < B; ++b) {
      const int mode = sm.dec_mode[b];
      if (mode == kModeNone) continue;
      const int n = sm.dec_n[b];
      bool resid = mode == kModeResidual;
      long long before, W = grid_total(q, 2, b, sm.red, &before);
      long long mine = sm.cta_w[b], own = sm.own_w[b][tid];
      if (resid && W <= 0) {  // all-zero residual: draw from p_n
        resid = false;
        W = grid_total(q, 0, b, sm.red, &before);
        own = sm.own_a[b][tid];
        mine = block_sum_i64(own, sm.red);
      }
      long long t =
          static_cast<long long>(scale_by_uniform(static_cast<unsigned long long>(W), q.u_smp[b]));
      if (t >= W) t = W - 1;  // u >= 1 (outside the documented range)
      if (t >= before && t < before + mine) {  // this CTA (uniform within it)
        long long tot;
        const long long incl = block_scan_i64(own, sm.red, &tot);
        const long long target = t - before;
        if (own > 0 && incl > target && incl - own <= target) {  // exactly one thread
          const RowCtx cx = sm.cx[b];
          const Elem* zr = static_cast<const Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb +
                           static_cast<int64_t>(n) * V;
          const Elem* dr = static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
                           static_cast<int64_t>(resid ? n : 0) * V;
          const float scale = resid ? kFixResidual : kFixMass;
          long long cum = incl - own;
          int found = -1, last_pos = -1;
          for (int e = lo; e < hi; ++e) {
            float wh, wl;
            if (resid) weight<Q_RESID>(e, Tag::load1(zr + e), Tag::load1(dr + e), cx, sm.tab, wh, wl);
            else weight<Q_NORM_Z>(e, Tag::load1(zr + e), 0.f, cx, sm.tab, wh, wl);
            const long long wf = df_to_fix(wh, wl, scale);
            if (wf > 0) last_pos = e;
            cum += wf;
            if (cum > target) {
              found = e;
              break;
            }
          }
          // per-element rounding can leave the target just past the
          // range's cumulative mass: the range's last positive element then
          const int tok = found >= 0 ? found : (last_pos >= 0 ? last_pos : hi - 1);
          p.out_tok[static_cast<int64_t>(b) * (k + 1) + n] = tok;
          if (q.cache_on)
            cache_lookup_one(q.cache, b, n, tok, q.hit + b,
                             q.tok_out + static_cast<int64_t>(b) * q.cache.depth);
        }
      }
    }
    // rows without a draw look up their outcome in CTA 0 (whose acceptance
    // warps wrote their tokens)
    if (q.cache_on && blockIdx.x == 0 && tid < B && sm.dec_mode[tid] == kModeNone) {
      const int b = tid, n = sm.dec_n[b];
      const int tok = (p.out_tok && n >= 0 && n <= k)
                          ? p.out_tok[static_cast<int64_t>(b) * (k + 1) + n] : -1;
      cache_lookup_one(q.cache, b, n, tok, q.hit + b,
                       q.tok_out + static_cast<int64_t>(b) * q.cache.depth);
    }
  }

  // exit: the last CTA out resets the barrier words (they are zero between
  // calls, also after an abort) and advances the cache's insert counter
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&q.bar->exit_[0], 1u) == static_cast<unsigned>(G) - 1u) {
      for (int s = 0; s < kStepSubBars; ++s) atomicExch(&q.bar->sub[s][0], 0u);
      atomicExch(&q.bar->top[0], 0u);
      atomicExch(&q.bar->abort_[0], 0u);
      atomicExch(&q.bar->exit_[0], 0u);
      if (q.cache_on) *q.cache.calls = seq >> 32;
      __threadfence();
    }
  }
}

template <typename Tag, bool VEC>
int resident_grid() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] > 0) return cached[dev];
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, step_kernel<Tag, VEC>, kThreads, 0) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  int g = per_sm * sms;
  if (g > kStepMaxGrid) g = kStepMaxGrid;
  cached[dev] = g;
  return g;
}

template <typename Tag, bool VEC>
cudaError_t launch_step_t(StepParams q, int max_grid, cudaStream_t s) {
  int G = resident_grid<Tag, VEC>();
  if (G <= 0) return cudaErrorInvalidConfiguration;
  if (max_grid > 0 && G > max_grid) G = max_grid;
  const long long nt = static_cast<long long>(G) * kThreads;
  long long E = (q.f.V + nt - 1) / nt;
  q.E = static_cast<int>((E + 7) / 8 * 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(G), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_kernel<Tag, VEC>, q);
}

}  // namespace

// The whole verify call of B <= kStepMaxB batch rows as one cooperative
// launch of every CTA the GPU holds at once (at most max_grid when > 0).
cudaError_t launch_step(const StepParams& q, int dtype, bool vec, int max_grid, cudaStream_t s) {
  if (q.f.B <= 0 || q.f.B > kStepMaxB) return cudaErrorInvalidValue;
  if (dtype == 1)
    return vec ? launch_step_t<BF16Tag, true>(q, max_grid, s) : launch_step_t<BF16Tag, false>(q, max_grid, s);
  return vec ? launch_step_t<F32Tag, true>(q, max_grid, s) : launch_step_t<F32Tag, false>(q, max_grid, s);
}

}  // namespace ssd
