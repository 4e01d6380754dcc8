// ssd_topf.cu -- the streaming pass over the draft rows that feed SSD's
// forked recovery: softmax statistics plus the top-f tokens of each chunk.
//
// Sources: "tanishqkumar/ssd" summary, module notes: forked recovery tokens
// are picked by top-k over the logits with masking for cache hits.
//
// Each CTA stages its chunk (at most 32 KB) into shared memory with bulk
// asynchronous copies (TMA, completion on an mbarrier; the wait is bounded)
// and then reads it twice from shared memory:
//   pass 1: running max / lowest argmax / online exponential sum per thread
//           (as for the target rows), which also gives each thread's maximum;
//   bound:  in every warp the (f+M)-th best of the 32 lane maxima is a lower
//           bound on the chunk's f-th best unmasked logit (those f+M lane
//           maxima are distinct elements at or above it and at most M of
//           them are masked); the CTA keeps the largest warp bound tau;
//   pass 2: only elements >= tau can be in the chunk's top f; they are
//           gathered into a small candidate buffer and warp 0 selects the
//           top f (logit descending, index ascending) among them.
// If pathological ties overflow the buffer, an exact fallback selects the top
// f by f rounds of a block-wide arg-max over the staged chunk.
#include "ssd_device.cuh"
#include "ssd_layout.h"
#include "ssd_scan.cuh"

namespace ssd {

constexpr int kCandCap = 256;
constexpr int kWaitPolls = 1 << 22;

struct TopfSmem {
  uint64_t mbar;
  float m[kWarps], s[kWarps];
  int i[kWarps], n[kWarps];
  int mask[kMaxMask];
  unsigned tau;
  int cnt;
  float cv[kCandCap];
  int ci[kCandCap];
  float bv[kWarps];
  int bi[kWarps];
  float cf;
};

// Best (value, index) of this thread's elements that rank after (pv, pi),
// skipping masked tokens and NaN.
template <typename Tag>
__device__ __forceinline__ void best_after(const typename Tag::Raw* vec, int nvec, int lo, float pv,
                                           int pi, const int* msk, int M, float& bv, int& bi) {
  constexpr int kV = Tag::kVec;
  bv = -INFINITY;
  bi = kIdxNone;
  for (int v = threadIdx.x; v < nvec; v += kThreads) {
    float z[8];
    Tag::unpackraw(vec[v], z);
#pragma unroll
    for (int e = 0; e < kV; ++e) {
      const int idx = lo + v * kV + e;
      if (z[e] == z[e] && ranks_before(pv, pi, z[e], idx) && ranks_before(z[e], idx, bv, bi) &&
          !is_masked(idx, msk, M)) {
        bv = z[e];
        bi = idx;
      }
    }
  }
}

template <typename Tag, bool DO_EXP>
__device__ void topf_chunk(const StatsParams& p, const typename Tag::Elem* /*row*/,
                           const typename Tag::Raw* vec, int nvec, int lo, float c, bool need_stats,
                           PartStat* out_part, TopEntry* out_top, TopfSmem& sm) {
  constexpr int kV = Tag::kVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int M = p.M, f = p.f;
  // pass 1
  ScanState st;
  st.m = -INFINITY;
  st.s = 0.f;
  st.idx = kIdxNone;
  st.nan = 0;
#pragma unroll 4
  for (int v = tid; v < nvec; v += kThreads) {
    float z[8];
    Tag::unpackraw(vec[v], z);
    float vm = z[0];
#pragma unroll
    for (int e = 1; e < kV; ++e) vm = max_nan(vm, z[e]);
    scan_vector<DO_EXP>(st, z, kV, vm, lo + v * kV, c);
  }
  // Lower bound on the chunk's f-th best unmasked logit.  If f + M <= 8: the
  // (f+M)-th largest of the 8 warp maxima (8 distinct elements).  Otherwise,
  // per warp, the (f+M)-th largest of its 32 lane maxima.
  const int need = f + M;
  float tw = -INFINITY;
  if (need <= kWarps) {
    float wm = st.m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(kFull, wm, o));
    if (lane == 0) sm.bv[warp] = wm;
    __syncthreads();
    if (tid == 0) {
      // (need)-th largest of the 8 values: count, for each value, how many
      // rank strictly above it (ties broken by warp number)
      float best = -INFINITY;
      for (int a = 0; a < kWarps; ++a) {
        int above = 0;
        for (int q = 0; q < kWarps; ++q)
          above += (sm.bv[q] > sm.bv[a]) || (sm.bv[q] == sm.bv[a] && q < a);
        if (above == need - 1) best = sm.bv[a];
      }
      sm.tau = f2ord(best);
    }
  } else if (need <= 32) {
    float cv = st.m;
    int ci = st.idx;
    for (int r = 0; r < need; ++r) {
      float mv = cv;
      int mi = ci;
      warp_argmax(mv, mi);
      if (mi != kIdxNone && ci == mi) {
        cv = -INFINITY;
        ci = kIdxNone;
      }
      if (r == need - 1) tw = (mi == kIdxNone) ? -INFINITY : mv;
    }
    if (lane == 0) atomicMax(&sm.tau, f2ord(tw));
  }
  // statistics of the chunk (its __syncthreads also publishes tau)
  if (need_stats) {
    block_stats_write(st, c, DO_EXP, sm.m, sm.s, sm.i, sm.n, out_part);
  } else {
    // fork-only row: still report max / argmax / NaN (no exponentials)
    block_stats_write(st, c, false, sm.m, sm.s, sm.i, sm.n, out_part);
  }
  const float tau = ord2f(sm.tau);
  // pass 2: candidates at or above the bound
  for (int v = tid; v < nvec; v += kThreads) {
    float z[8];
    Tag::unpackraw(vec[v], z);
    float vm = z[0];
#pragma unroll
    for (int e = 1; e < kV; ++e) vm = max_nan(vm, z[e]);
    if (vm >= tau) {  // false for vectors holding a NaN (the row is invalid then)
#pragma unroll
      for (int e = 0; e < kV; ++e) {
        const int idx = lo + v * kV + e;
        if (z[e] >= tau && !is_masked(idx, sm.mask, M)) {
          const int k = atomicAdd(&sm.cnt, 1);
          if (k < kCandCap) {
            sm.cv[k] = z[e];
            sm.ci[k] = idx;
          }
        }
      }
    }
  }
  __syncthreads();
  const int cnt = sm.cnt;
  if (cnt <= kCandCap) {
    if (warp == 0) {
      float pv = INFINITY;
      int pi = -1;  // ranks before everything
      for (int r = 0; r < f; ++r) {
        float bv = -INFINITY;
        int bi = kIdxNone;
        for (int q = lane; q < cnt; q += 32) {
          const float v = sm.cv[q];
          const int i = sm.ci[q];
          if (ranks_before(pv, pi, v, i) && ranks_before(v, i, bv, bi)) {
            bv = v;
            bi = i;
          }
        }
        warp_argmax(bv, bi);
        if (lane == 0) {
          out_top[r].v = bv;
          out_top[r].i = bi;
        }
        pv = bv;
        pi = bi;
      }
    }
    return;
  }
  // exact fallback: f rounds of a block-wide arg-max over the staged chunk
  float pv = INFINITY;
  int pi = -1;
  for (int r = 0; r < f; ++r) {
    float bv;
    int bi;
    best_after<Tag>(vec, nvec, lo, pv, pi, sm.mask, M, bv, bi);
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
      out_top[r].v = bv;
      out_top[r].i = bi;
    }
    pv = bv;
    pi = bi;
  }
}

// grid: (C, Pdf, B); rows r0 .. r0+Pdf-1 are draft rows 0 .. Pdf-1.
// Dynamic shared memory: CH * sizeof(element) bytes (at most 32 KB).
template <typename Tag>
__global__ void __launch_bounds__(kThreads, 6) stats_topf_kernel(StatsParams p) {
  using Elem = typename Tag::Elem;
  extern __shared__ __align__(128) unsigned char dyn[];
  __shared__ TopfSmem sm;
  const int c = blockIdx.x, j = blockIdx.y, b = blockIdx.z;
  const int r = p.r0 + j;
  const int tid = threadIdx.x;
  const int lo = c * p.CH;
  const int hi = min(p.V, lo + p.CH);
  const int nvec = (hi - lo) / Tag::kVec;
  const unsigned nbytes = static_cast<unsigned>(hi - lo) * sizeof(Elem);
  const Elem* src = static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
                    static_cast<int64_t>(j) * p.V + lo;
  const bool need_stats = j < p.Pds;
  const float T = p.T ? p.T[b] : 0.f;
  const bool do_exp = need_stats && (T > 0.f);
  if (tid == 0) {
    mbar_init(&sm.mbar, 1);
    sm.tau = f2ord(-INFINITY);
    sm.cnt = 0;
    float h = 0.f, l = 0.f;
    if (do_exp) temp_coeff(T, h, l);  // one double division per CTA
    sm.cf = h;
  }
  if (tid < p.M) sm.mask[tid] = p.mask[(static_cast<int64_t>(b) * p.Pdf + j) * p.M + tid];
  __syncthreads();
  if (tid == 0) {
    mbar_expect_tx(&sm.mbar, nbytes);
    for (unsigned off = 0; off < nbytes; off += 16384u)
      bulk_g2s(dyn + off, reinterpret_cast<const unsigned char*>(src) + off,
               min(16384u, nbytes - off), &sm.mbar);
  }
  const float cf = sm.cf;
  PartStat* out_part = p.part + (static_cast<int64_t>(b) * p.Rp + r) * p.C + c;
  TopEntry* out_top = p.topk + ((static_cast<int64_t>(b) * p.Pdf + j) * p.C + c) * p.f;
  // one thread waits (bounded) so the others do not spin; the barrier then
  // orders the staged data for every thread
  const bool ok = (tid == 0) ? mbar_wait_bounded(&sm.mbar, 0, kWaitPolls) : true;
  if (!__syncthreads_and(ok)) {
    // the copy did not complete in time: report, let our own copy finish,
    // and leave a NaN-flagged partial so the row reads as invalid
    if (tid == 0) {
      atomicOr(p.err, 0x10);
      mbar_wait_bounded(&sm.mbar, 0, kWaitPolls);
      PartStat ps;
      ps.m = -INFINITY;
      ps.s = 0.f;
      ps.idx = kIdxNone;
      ps.flags = 1;
      *out_part = ps;
      for (int q = 0; q < p.f; ++q) {
        out_top[q].v = -INFINITY;
        out_top[q].i = kIdxNone;
      }
    }
    return;
  }
  const typename Tag::Raw* vec = reinterpret_cast<const typename Tag::Raw*>(dyn);
  if (do_exp)
    topf_chunk<Tag, true>(p, src, vec, nvec, lo, cf, need_stats, out_part, out_top, sm);
  else
    topf_chunk<Tag, false>(p, src, vec, nvec, lo, cf, need_stats, out_part, out_top, sm);
}

cudaError_t launch_stats_topf(const StatsParams& p, int B, int dtype, cudaStream_t s) {
  dim3 grid(p.C, p.Pdf, B);
  const size_t dyn = static_cast<size_t>(p.CH) * (dtype == 1 ? 2 : 4);
  if (dyn > 32768) return cudaErrorInvalidValue;
  if (dtype == 1) stats_topf_kernel<BF16Tag><<<grid, kThreads, dyn, s>>>(p);
  else stats_topf_kernel<F32Tag><<<grid, kThreads, dyn, s>>>(p);
  return cudaGetLastError();
}

}  // namespace ssd
