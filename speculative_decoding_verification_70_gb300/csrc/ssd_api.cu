// ssd_api.cu -- the C-ABI entry points (include/ssd.h): host-side argument
// checks, workspace layout and kernel launches.  No entry point allocates
// memory except ssd_spec_cache_create.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <new>
#include <vector>

#ifndef SSD_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

#include "../../include/ssd.h"
#include "ssd_layout.h"


namespace ssd {
cudaError_t launch_stats_rows(const StatsParams& p, int B, int dtype, bool vec, int r0, int rows,
                              bool topf, cudaStream_t s);
cudaError_t launch_finalize(const FinalizeParams& p, cudaStream_t s);
cudaError_t launch_draft(const StatsParams& p, int B, int dtype, bool vec, int rows, bool topf,
                         cudaStream_t s);
cudaError_t launch_draft_finalize(const DraftParams& p, cudaStream_t s);
cudaError_t launch_topk_verify(const TopkParams& p, int dtype, bool vec, cudaStream_t s);
#ifndef SSD_TOPK_MAX_GROUP
#define SSD_TOPK_MAX_GROUP 32
#endif
cudaError_t launch_topk_finalize(const TopkParams& p, cudaStream_t s);
cudaError_t launch_tree_walk(const TreeParams& p, int dtype, bool vec, cudaStream_t s);
cudaError_t launch_softmax_finalize(const SoftmaxParams& p, cudaStream_t s);
cudaError_t launch_softmax_probs(const SoftmaxParams& p, cudaStream_t s);
cudaError_t launch_residual_norm(const ResidualParams& p, int B, int dtype, bool vec, cudaStream_t s);
cudaError_t launch_residual_select(const ResidualParams& p, int B, int dtype, bool vec, cudaStream_t s);
cudaError_t launch_residual_prep(const PrepParams& p, cudaStream_t s);
cudaError_t launch_selftest_exp2(const float* xh, const float* xl, double* out, int n, cudaStream_t s);

cudaError_t launch_filt_rowinit(const FiltParams& p, cudaStream_t s);
cudaError_t launch_filt_hist(const FiltParams& p, bool vec, cudaStream_t s);
cudaError_t launch_filt_band(const FiltParams& p, cudaStream_t s);
cudaError_t launch_filt_collect(const FiltParams& p, bool vec, cudaStream_t s);
cudaError_t launch_filt_cut(const FiltParams& p, bool vec, cudaStream_t s);
cudaError_t launch_filt_accept(const FiltParams& p, cudaStream_t s);
cudaError_t launch_filt_mass(const FiltParams& p, bool vec, cudaStream_t s);
cudaError_t launch_filt_select(const FiltParams& p, bool vec, cudaStream_t s);

cudaError_t launch_cache_claim(const CacheView& c, const InsertArgs& a, cudaStream_t s);
cudaError_t launch_cache_write(const CacheView& c, const InsertArgs& a, cudaStream_t s);
cudaError_t launch_cache_lookup(const CacheView& c, const LookupArgs& a, cudaStream_t s);
cudaError_t launch_chain(ChainParams p, int dtype, bool vec, cudaStream_t s);
cudaError_t launch_step(const StepParams& q, int dtype, bool vec, int max_grid, cudaStream_t s);
}  // namespace ssd

using namespace ssd;

struct ssd_spec_cache {
  CacheView view;
  int device;
};

namespace {

// ---------------------------------------------------------------------------
// launch profiler
// ---------------------------------------------------------------------------
struct ProfRecord {
  int kernel;
  cudaEvent_t a, b;
};
struct Profiler {
  std::mutex mu;
  bool on = false;
  int cap = 0;
  std::vector<cudaEvent_t> pool;
  std::vector<ProfRecord> recs;
  std::vector<const char*> names;
  std::vector<int> counts;
  int kernel_id(const char* n) {
    for (size_t i = 0; i < names.size(); ++i)
      if (strcmp(names[i], n) == 0) return static_cast<int>(i);
    names.push_back(n);
    counts.push_back(0);
    return static_cast<int>(names.size() - 1);
  }
};
Profiler g_prof;

// Brackets one kernel launch when profiling is on.  A phase scope
// (launch = false) brackets several launches, possibly on other streams
// joined back by events, and adds no launch to the count.
struct ProfScope {
  cudaStream_t s = nullptr;
  int rec = -1;
  ProfScope() = default;
  ProfScope(const char* name, cudaStream_t st, bool launch = true) { begin(name, st, launch); }
  void begin(const char* name, cudaStream_t st, bool launch = true) {
    s = st;
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    int id = g_prof.kernel_id(name);
    if (launch) g_prof.counts[id] += 1;
    size_t used = g_prof.recs.size();
    if (static_cast<int>(used) >= g_prof.cap) return;
    ProfRecord r;
    r.kernel = id;
    r.a = g_prof.pool[2 * used];
    r.b = g_prof.pool[2 * used + 1];
    if (cudaEventRecord(r.a, s) != cudaSuccess) return;
    g_prof.recs.push_back(r);
    rec = static_cast<int>(used);
  }
  void end() {
    if (rec < 0) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    cudaEventRecord(g_prof.recs[rec].b, s);
    rec = -1;
  }
  ~ProfScope() { end(); }
  ProfScope(const ProfScope&) = delete;
  ProfScope& operator=(const ProfScope&) = delete;
};

// One NVTX range per library call (header-only NVTX3: a no-op unless a
// profiler such as Nsight Systems or Nsight Compute injects itself).
struct CallRange {
#ifndef SSD_NO_NVTX
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
#else
  explicit CallRange(const char*) {}
#endif
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};

inline cudaStream_t S(ssd_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline ssd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline size_t esize(ssd_dtype dt) { return dt == SSD_BF16 ? 2 : 4; }

inline bool dtype_ok(ssd_dtype dt) { return dt == SSD_F32 || dt == SSD_BF16; }

// 16-byte vector loads are legal when every row start is 16-byte aligned.
inline bool vec_ok(const void* base, int64_t bstride, int V, ssd_dtype dt) {
  const size_t s = esize(dt);
  return aligned(base, 16) && (static_cast<size_t>(bstride) * s) % 16 == 0 &&
         (static_cast<size_t>(V) * s) % 16 == 0;
}

inline char* wsp(void* ws, size_t off) { return static_cast<char*>(ws) + off; }

struct VerifyCall {
  const void* Z; int64_t zb;
  const void* D; int64_t db;
  ssd_dtype dt;
  int B, k, V;
  const int32_t* x; const float* T; const float* u_acc;
  int32_t* accept_len; float* p_at_x; float* q_at_x;
  const float* u_smp; int32_t* out_tok;
  int f; const int32_t* mask; int M; int32_t* fork_tok; float* fork_logit;
  const int32_t* fanout;  // [k+1] device, or null (f at every position)
  bool drafted;           // draft rows' statistics already in ws (ssd_draft_sample)
  // SSD round step (ssd_verify_fork_cache): clear + insert the forks, then
  // look up each row's realised outcome
  const CacheView* cache; bool cache_clear; const int32_t* payload;
  int32_t* hit; int32_t* tok_out;
  void* ws; size_t ws_bytes;
  cudaStream_t stream;
  bool single_stream;  // no internal streams (the no-allocation entry point)
};

ssd_status check_common(const VerifyCall& c, bool fork) {
  if (!dtype_ok(c.dt)) return SSD_ERR_UNSUPPORTED_DTYPE;
  if (!c.Z || !c.D || !c.x || !c.T || !c.u_acc || !c.accept_len || !c.ws) return SSD_ERR_INVALID_ARG;
  if (c.B < 1 || c.k < 1 || c.k > SSD_MAX_K || c.V < 2) return SSD_ERR_INVALID_ARG;
  if ((c.p_at_x == nullptr) != (c.q_at_x == nullptr)) return SSD_ERR_INVALID_ARG;
  if (c.u_smp && !c.out_tok) return SSD_ERR_INVALID_ARG;
  const int64_t rowz = static_cast<int64_t>(c.k + 1) * c.V;
  const int64_t rowd = static_cast<int64_t>(fork ? c.k + 1 : c.k) * c.V;
  if (c.zb < rowz || c.db < rowd) return SSD_ERR_INVALID_ARG;
  if (!aligned(c.Z, esize(c.dt)) || !aligned(c.D, esize(c.dt))) return SSD_ERR_INVALID_ARG;
  if (fork) {
    if (c.f < 1 || c.f > SSD_MAX_F || c.f >= c.V) return SSD_ERR_INVALID_ARG;
    if (c.M < 0 || c.M > SSD_MAX_M || (c.M > 0 && !c.mask)) return SSD_ERR_INVALID_ARG;
    if (!c.fork_tok || !c.fork_logit) return SSD_ERR_INVALID_ARG;
  }
  // the kernels index rows with int for element offsets within a row and
  // int64 across rows; V must fit chunk arithmetic
  if (c.V > (1 << 28)) return SSD_ERR_INVALID_ARG;
  return SSD_OK;
}

// The streaming pass: rows without forked top-f in one kernel ("stats"),
// the draft rows that feed the forked recovery in another ("stats_topf").
// When s_plain != s_topf, the target rows and the draft rows go to the two
// streams and run concurrently.
// Chunks per statistics CTA: the largest power of two (a whole row at most)
// that still leaves two waves of CTAs (2 x 6 resident x 152 SMs).  Longer
// CTAs pay their set-up, block reduction and (top-f) selection once per
// more bytes: measured at B = 512, k = 7, V = 151936 fp32 the pass took
// 743 us with 4 chunks per CTA and 700 us with a whole row; at B = 64,
// k = 5 bf16, 87 us with 1 chunk and 78 us with 2.
inline int stats_group(long long rows, int C) {
  int G = 1;
  while (G < C && rows * ((C + 2 * G - 1) / (2 * G)) >= 1824) G *= 2;
  return G;
}

// group > 0 fixes the chunks per CTA of both launches.
cudaError_t run_stats2(const StatsParams& sp0, int B, int dtype, bool vec, cudaStream_t s_plain,
                       cudaStream_t s_topf, int group = 0) {
  StatsParams sp = sp0;
  const bool topf = sp.Pdf > 0 && sp.f > 0;
  const bool split = s_plain != s_topf;
  const int rows_plain = topf ? sp.Pz : (split ? sp.Pz : sp.R);
  sp.G = group > 0 ? group
                   : split_group(stats_group(static_cast<long long>(B) * rows_plain, sp.C), sp.C);
  cudaError_t e = cudaSuccess;
  // the top-f rows first: their CTAs run longer, and the plain rows' CTAs
  // then fill the last wave (measured at B = 64, k = 5, bf16: statistics
  // phase 70 against 78 us; at B = 512 fp32: 907 against 908 us per step)
  if (topf && split) {
    ProfScope ps("stats_topf", s_topf);
    StatsParams pt = sp;
    pt.G = group > 0 ? group
                     : split_group(stats_group(static_cast<long long>(B) * sp.Pdf, sp.C), sp.C);
    e = launch_stats_rows(pt, B, dtype, vec, sp.Pz, sp.Pdf, true, s_topf);
    if (e != cudaSuccess) return e;
    ProfScope ps2("stats", s_plain);
    return launch_stats_rows(sp, B, dtype, vec, 0, rows_plain, false, s_plain);
  }
  if (rows_plain > 0) {
    ProfScope ps("stats", s_plain);
    e = launch_stats_rows(sp, B, dtype, vec, 0, rows_plain, false, s_plain);
  }
  if (e != cudaSuccess) return e;
  if (!topf) {
    if (split && sp.R > sp.Pz) {  // draft statistics rows on the second stream
      ProfScope ps("stats", s_topf);
      e = launch_stats_rows(sp, B, dtype, vec, sp.Pz, sp.R - sp.Pz, false, s_topf);
    }
    return e;
  }
  ProfScope ps("stats_topf", s_topf);
  StatsParams pt = sp;
  pt.G = group > 0 ? group
                   : split_group(stats_group(static_cast<long long>(B) * sp.Pdf, sp.C), sp.C);
  return launch_stats_rows(pt, B, dtype, vec, sp.Pz, sp.Pdf, true, s_topf);
}

cudaError_t run_stats(const StatsParams& sp, int B, int dtype, bool vec, cudaStream_t s,
                      int group = 0) {
  return run_stats2(sp, B, dtype, vec, s, s, group);
}

// Chunks per statistics CTA of a verify call: the policy for the target
// rows' launch of the two-stream schedule (whose draft-row launch uses the
// same value), so that every schedule streams the same chunk groups and the
// partial sums, hence p(x) and q(x), are the same bits.
inline int verify_group(const StatsParams& sp, int B) {
  return split_group(stats_group(static_cast<long long>(B) * sp.Pz, sp.C), sp.C);
}

// Every row in one launch (the top-f variant, whose target and
// statistics-only rows take the plain path): small batches, where a second
// launch costs more than the rows it would run concurrently.
cudaError_t run_stats_one(const StatsParams& sp0, int B, int dtype, bool vec, cudaStream_t s) {
  StatsParams sp = sp0;
  sp.G = verify_group(sp, B);
  const bool topf = sp.Pdf > 0 && sp.f > 0;
  ProfScope ps(topf ? "stats_topf" : "stats", s);
  return launch_stats_rows(sp, B, dtype, vec, 0, sp.R, topf, s);
}

cudaError_t cache_insert(const CacheView& v, const InsertArgs& a, cudaStream_t s) {
  cudaError_t e;
  {
    ProfScope ps("cache_claim", s);
    e = launch_cache_claim(v, a, s);
  }
  if (e != cudaSuccess) return e;
  ProfScope ps("cache_write", s);
  return launch_cache_write(v, a, s);
}

// The draw: the norm pass, then (after `between`, if given: work that must
// precede the select) the select.
template <typename Between>
cudaError_t run_residual(const ResidualParams& rp, int B, int dtype, bool vec, cudaStream_t s,
                         Between&& between) {
  cudaError_t e;
  {
    ProfScope ps("residual_norm", s);
    e = launch_residual_norm(rp, B, dtype, vec, s);
  }
  if (e != cudaSuccess) return e;
  e = between();
  if (e != cudaSuccess) return e;
  ProfScope ps("residual_select", s);
  return launch_residual_select(rp, B, dtype, vec, s);
}

cudaError_t run_residual(const ResidualParams& rp, int B, int dtype, bool vec, cudaStream_t s) {
  return run_residual(rp, B, dtype, vec, s, [] { return cudaSuccess; });
}

// ---------------------------------------------------------------------------
// Per-device internal streams for the pipelined verify schedule.
// ---------------------------------------------------------------------------
constexpr int kMaxSlices = 8;
constexpr int kMaxDevs = 64;

struct DevStreams {
  std::mutex mu;
  bool ready = false;
  bool failed = false;
  // s1: target-row statistics; s2: draft-row (top-f) statistics, at the
  // device's greatest priority so that its CTAs are dispatched first when
  // both streams wait on the same fork event (the longer top-f CTAs first,
  // the plain ones filling the last wave: at B = 512 the pass took 693 us
  // in that order and 758 us in the other, which equal priorities left to
  // chance from one call to the next)
  cudaStream_t s1 = nullptr, s2 = nullptr;
  // the cache insert beside the draw, at the device's greatest priority: the
  // norm pass fills every SM, and a side stream of equal priority got its
  // CTAs only as the norm pass drained, so the select (which waits for the
  // insert) started ~25 us after the norm pass at B = 512
  cudaStream_t s3 = nullptr;
  cudaEvent_t ev[3 + 2 * kMaxSlices] = {};  // fork, per-slice joins, cache step
};
DevStreams g_streams[kMaxDevs];

// Streams and events of the current device, created on first use (no
// device memory is allocated).  Returns null if they cannot be created.
DevStreams* device_streams() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevs) return nullptr;
  DevStreams& d = g_streams[dev];
  std::lock_guard<std::mutex> lk(d.mu);
  if (d.ready) return &d;
  if (d.failed) return nullptr;
  int least = 0, greatest = 0;
  bool ok = cudaDeviceGetStreamPriorityRange(&least, &greatest) == cudaSuccess &&
            cudaStreamCreateWithFlags(&d.s1, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithPriority(&d.s2, cudaStreamNonBlocking, greatest) == cudaSuccess &&
            cudaStreamCreateWithPriority(&d.s3, cudaStreamNonBlocking, greatest) == cudaSuccess;
  for (auto& e : d.ev) ok = ok && cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    d.failed = true;
    return nullptr;
  }
  d.ready = true;
  return &d;
}

// Number of batch slices of the pipelined schedule (0: the plain
// single-stream schedule).  Measured on mixed512 (B=512): one slice with the
// target-row and draft-row statistics on two concurrent streams beats 2, 4
// or 8 slices, whose per-slice draw launches put their latency on the
// critical path.
#ifndef SSD_SLICE_ROWS
#define SSD_SLICE_ROWS 1024
#endif
// Smallest batch that uses the two internal streams (target-row and
// draft-row statistics concurrently, the cache insert beside the draw).
// Measured at B = 1 (ssd_fork step with the cache): 67 / 53 us eager / as a
// graph on one stream, 49 / 43 us on two.
// Smallest batch whose cache lookup runs inside the draw's select kernel.
#ifndef SSD_FUSE_LOOKUP_MIN_B
#define SSD_FUSE_LOOKUP_MIN_B 16
#endif
#ifndef SSD_MIN_STREAMED_B
#define SSD_MIN_STREAMED_B 1
#endif
int verify_slices(int B) {
  if (B < SSD_MIN_STREAMED_B) return 0;
  int S = B / SSD_SLICE_ROWS;
  if (S < 1) S = 1;
  return S > kMaxSlices ? kMaxSlices : S;
}

struct SliceParams {
  StatsParams sp;
  FinalizeParams fp;
  ResidualParams rp;
};

// Parameter blocks of batch rows [b0, b0 + Bs): every per-row pointer and
// workspace region is offset by b0 rows.
SliceParams slice_params(const VerifyCall& c, bool fork, const WsLayout& L, int b0, int Bs) {
  SliceParams q;
  const size_t es = esize(c.dt);
  const char* Zb = static_cast<const char*>(c.Z) + static_cast<size_t>(b0) * c.zb * es;
  const char* Db = static_cast<const char*>(c.D) + static_cast<size_t>(b0) * c.db * es;
  const int Pf = c.k + 1;
  const size_t C = static_cast<size_t>(L.ch.C);
  PartStat* part = reinterpret_cast<PartStat*>(wsp(c.ws, L.part)) + static_cast<size_t>(b0) * L.R * C;
  TopEntry* topk = reinterpret_cast<TopEntry*>(wsp(c.ws, L.topk)) +
                   static_cast<size_t>(b0) * Pf * C * (fork ? c.f : 0);
  RowStat* rowstat = reinterpret_cast<RowStat*>(wsp(c.ws, L.rowstat)) + static_cast<size_t>(b0) * L.R;
  BState* bstate = reinterpret_cast<BState*>(wsp(c.ws, L.bstate)) + b0;
  int* err = reinterpret_cast<int*>(wsp(c.ws, L.err));

  StatsParams& sp = q.sp;
  memset(&sp, 0, sizeof sp);
  sp.Z = Zb; sp.zb = c.zb; sp.Pz = c.k + 1;
  sp.D = Db; sp.db = c.db; sp.Pds = c.drafted ? 0 : c.k; sp.Pdf = fork ? Pf : 0;
  sp.T = c.T + b0;
  sp.mask = fork && c.M > 0 ? c.mask + static_cast<size_t>(b0) * Pf * c.M : nullptr;
  sp.M = fork ? c.M : 0; sp.f = fork ? c.f : 0;
  sp.V = c.V; sp.C = L.ch.C; sp.CH = L.ch.CH;
  sp.R = sp.Pz + (sp.Pdf > sp.Pds ? sp.Pdf : sp.Pds);
  sp.Rp = L.R;
  sp.part = part; sp.topk = topk; sp.err = err;

  FinalizeParams& fp = q.fp;
  memset(&fp, 0, sizeof fp);
  fp.Z = Zb; fp.zb = c.zb; fp.Pz = sp.Pz;
  fp.D = Db; fp.db = c.db; fp.Pds = c.k; fp.Pdf = sp.Pdf;
  fp.dtype = c.dt == SSD_BF16 ? 1 : 0;
  fp.B = Bs; fp.k = c.k; fp.V = c.V; fp.C = L.ch.C; fp.Rp = L.R; fp.f = sp.f;
  fp.R = sp.Pz + (sp.Pdf > c.k ? sp.Pdf : c.k);
  fp.T = c.T + b0; fp.x = c.x + static_cast<size_t>(b0) * c.k;
  fp.u_acc = c.u_acc + static_cast<size_t>(b0) * c.k;
  fp.accept_len = c.accept_len + b0;
  fp.p_at_x = c.p_at_x ? c.p_at_x + static_cast<size_t>(b0) * c.k : nullptr;
  fp.q_at_x = c.q_at_x ? c.q_at_x + static_cast<size_t>(b0) * c.k : nullptr;
  fp.out_tok = c.out_tok ? c.out_tok + static_cast<size_t>(b0) * (c.k + 1) : nullptr;
  fp.fork_tok = fork ? c.fork_tok + static_cast<size_t>(b0) * Pf * c.f : nullptr;
  fp.fork_logit = fork ? c.fork_logit + static_cast<size_t>(b0) * Pf * c.f : nullptr;
  fp.fanout = fork ? c.fanout : nullptr;
  fp.part = part; fp.topk = topk;
  fp.rowstat = rowstat; fp.bstate = bstate; fp.err = err;

  ResidualParams& rp = q.rp;
  memset(&rp, 0, sizeof rp);
  rp.Z = Zb; rp.zb = c.zb; rp.Pz = sp.Pz;
  rp.D = Db; rp.db = c.db;
  rp.V = c.V; rp.C = L.dch.C; rp.CH = L.dch.CH; rp.E = L.dch.E; rp.R = L.R; rp.k = c.k;
  rp.T = c.T + b0; rp.u_smp = c.u_smp ? c.u_smp + b0 : nullptr;
  rp.rowstat = rowstat; rp.bstate = bstate;
  const size_t Cd = static_cast<size_t>(L.dch.C);
  rp.rnorm = reinterpret_cast<long long*>(wsp(c.ws, L.rnorm)) + static_cast<size_t>(b0) * Cd * 2;
  rp.rthr = reinterpret_cast<long long*>(wsp(c.ws, L.rthr)) + static_cast<size_t>(b0) * Cd * 3 * kDrawThreads;
  rp.racc = reinterpret_cast<long long*>(wsp(c.ws, L.racc)) + static_cast<size_t>(b0) * Cd * 2;
  rp.amb_cnt = reinterpret_cast<int*>(wsp(c.ws, L.amb_cnt)) + b0;
  rp.amb_cap = amb_cap(c.V);
  rp.amb_idx = reinterpret_cast<int*>(wsp(c.ws, L.amb_idx)) + static_cast<size_t>(b0) * rp.amb_cap;
  rp.out_tok = fp.out_tok;
  fp.amb_cnt = rp.amb_cnt;
  return q;
}

// finalize + (optional) draw of one slice on stream s
// The cache step of an SSD round: (clear,) insert the forks of all B rows.
cudaError_t cache_forks(const VerifyCall& c, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if (c.cache_clear) {
    const size_t kb = sizeof(unsigned long long) * c.cache->capacity;
    e = cudaMemsetAsync(c.cache->keys, 0xff, kb, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(c.cache->winner, 0, kb, s);
  }
  if (e != cudaSuccess) return e;
  InsertArgs a;
  memset(&a, 0, sizeof a);
  a.fork_tok = c.fork_tok; a.P = c.k + 1; a.f = c.f; a.payload = c.payload;
  a.n = c.B * (c.k + 1) * c.f;
  return cache_insert(*c.cache, a, s);
}

cudaError_t cache_lookup_outcome(const VerifyCall& c, cudaStream_t s) {
  LookupArgs a;
  memset(&a, 0, sizeof a);
  a.accept_len = c.accept_len; a.out_tok = c.out_tok; a.k = c.k; a.n = c.B;
  a.hit = c.hit; a.tok_out = c.tok_out;
  ProfScope ps("cache_lookup", s);
  return launch_cache_lookup(*c.cache, a, s);
}

// Largest batch whose verify after the statistics pass runs as the one
// cluster kernel (finalisation, draw and the SSD round step's cache work in
// one launch, ssd_chain.cu); larger batches take the batched kernels, whose
// grids spread the draw's passes over the whole GPU.  ssd_set_chain_batch
// overrides it.
#ifndef SSD_CHAIN_MAX_B
#define SSD_CHAIN_MAX_B 16
#endif
std::atomic<int> g_chain_max_b{-1};

bool use_chain(int B) {
  const int ov = g_chain_max_b.load(std::memory_order_relaxed);
  return B <= (ov >= 0 ? ov : SSD_CHAIN_MAX_B);
}

// The whole tail of a one-slice call as the cluster kernel (the cache, if
// any, already cleared when the call asks for it).
cudaError_t enqueue_chain(const VerifyCall& c, const SliceParams& q, bool vec, cudaStream_t s) {
  ChainParams cp;
  memset(&cp, 0, sizeof cp);
  cp.f = q.fp;
  cp.u_smp = q.rp.u_smp;
  if (c.cache) {
    cp.cache_on = 1;
    cp.cache = *c.cache;
    cp.payload = c.payload;
    cp.hit = c.hit;
    cp.tok_out = c.tok_out;
  }
  ProfScope ps("chain", s);
  return launch_chain(cp, q.fp.dtype, vec, s);
}

// finalize + (optional) draw of one slice on stream s.  With a cache step
// and a side stream, the last slice's forks go into the cache on the side
// stream while the draw runs (side waits on the finalize, s on the insert
// before the lookup).  A small batch in one slice takes the cluster kernel.
cudaError_t enqueue_tail(const VerifyCall& c, const SliceParams& q, int Bs, bool vec,
                         cudaStream_t s, bool last = true, cudaStream_t side = nullptr,
                         cudaEvent_t ev_fin = nullptr, cudaEvent_t ev_ins = nullptr) {
  cudaError_t e;
  {
    ProfScope ps("finalize", s);
    e = launch_finalize(q.fp, s);
  }
  if (e != cudaSuccess) return e;
  const bool cache = c.cache && last;
  const bool overlap = cache && side && ev_fin && ev_ins;
  if (overlap) {
    e = cudaEventRecord(ev_fin, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, ev_fin, 0);
    if (e == cudaSuccess) e = cache_forks(c, side);
    if (e == cudaSuccess) e = cudaEventRecord(ev_ins, side);
    if (e != cudaSuccess) return e;
  }
  // the forks must be in the cache before any row's outcome is looked up
  auto inserted = [&]() -> cudaError_t {
    if (!cache) return cudaSuccess;
    return overlap ? cudaStreamWaitEvent(s, ev_ins, 0) : cache_forks(c, s);
  };
  if (c.u_smp) {
    // one slice holding every row: the select kernel looks up each row's
    // outcome as soon as its token is final (no separate lookup launch);
    // it then waits for the insert instead of overlapping the norm pass's
    // tail, so small batches, whose insert outlasts the norm pass, keep
    // the separate lookup
    const bool fuse = cache && Bs == c.B && c.B >= SSD_FUSE_LOOKUP_MIN_B;
    ResidualParams rp = q.rp;
    if (fuse) {
      rp.lookup = 1;
      rp.cache = *c.cache;
      rp.hit = c.hit;
      rp.tok_out = c.tok_out;
    }
    e = run_residual(rp, Bs, q.fp.dtype, vec, s, inserted);
    if (e != cudaSuccess || !cache || fuse) return e;
    return cache_lookup_outcome(c, s);
  }
  if (!cache) return e;
  e = inserted();
  if (e == cudaSuccess) e = cache_lookup_outcome(c, s);
  return e;
}

// Largest batch whose whole call runs as the one cooperative kernel
// (ssd_step.cu; at most kStepMaxB); ssd_set_step_schedule overrides it and
// can cap the kernel's grid.
#ifndef SSD_STEP_MAX_B
#define SSD_STEP_MAX_B 0
#endif
std::atomic<int> g_step_max_b{-1};
std::atomic<int> g_step_grid{0};

bool use_step(int B) {
  const int ov = g_step_max_b.load(std::memory_order_relaxed);
  const int lim = ov >= 0 ? ov : SSD_STEP_MAX_B;
  return B <= lim && B <= kStepMaxB;
}

// The call as the cooperative kernel.  Returns false (nothing enqueued) if
// the launch was refused, e.g. because the grid cannot be made resident;
// the caller then takes the launch-by-launch schedule.
bool enqueue_step(const VerifyCall& c, bool fork, const WsLayout& L, bool vec, int dtype) {
  const SliceParams sl = slice_params(c, fork, L, 0, c.B);
  StepParams q;
  memset(&q, 0, sizeof q);
  q.sp = sl.sp;
  q.sp.G = verify_group(sl.sp, c.B);
  q.f = sl.fp;
  q.u_smp = sl.rp.u_smp;
  q.units = c.B * sl.sp.R * ((sl.sp.C + q.sp.G - 1) / q.sp.G);
  q.rows = reinterpret_cast<StepRow*>(wsp(c.ws, L.srows));
  q.cta = reinterpret_cast<long long*>(wsp(c.ws, L.scta));
  q.bar = reinterpret_cast<StepBar*>(wsp(c.ws, L.sbar));
  if (c.cache) {
    q.cache_on = 1;
    q.cache_clear = c.cache_clear ? 1 : 0;
    q.cache = *c.cache;
    q.payload = c.payload;
    q.hit = c.hit;
    q.tok_out = c.tok_out;
  }
  ProfScope ps("step", c.stream);
  if (launch_step(q, dtype, vec, g_step_grid.load(std::memory_order_relaxed), c.stream) ==
      cudaSuccess)
    return true;
  (void)cudaGetLastError();
  return false;
}

// Schedule: for B >= SSD_MIN_STREAMED_B (every batch by default) the batch
// is cut into S = max(1, B / SSD_SLICE_ROWS) slices (one slice up to 2047
// rows).  The target-row and draft-row statistics of each slice run on two
// internal streams; the slice's finalisation and draw run on the caller's
// stream after both (events), overlapping the next slice's statistics.  The
// caller's stream waits for everything before its next work, so stream order
// is kept.
ssd_status run_verify(const VerifyCall& c, bool fork) {
  ssd_status st = check_common(c, fork);
  if (st != SSD_OK) return st;
  const WsLayout L = make_layout(c.B, c.k, c.V, fork ? c.f : 0, static_cast<int>(esize(c.dt)));
  if (c.ws_bytes < L.total) return SSD_ERR_WORKSPACE;
  if (!aligned(c.ws, 256)) return SSD_ERR_INVALID_ARG;
  const bool vec = vec_ok(c.Z, c.zb, c.V, c.dt) && vec_ok(c.D, c.db, c.V, c.dt);
  const int dtype = c.dt == SSD_BF16 ? 1 : 0;
  if (use_step(c.B) && enqueue_step(c, fork, L, vec, dtype)) return SSD_OK;
  if (use_chain(c.B)) {
    // one statistics launch over every row (and the cache clear), then the
    // cluster kernel: two launches on the caller's stream
    const SliceParams q = slice_params(c, fork, L, 0, c.B);
    StatsParams sp = q.sp;
    if (c.cache && c.cache_clear) {
      sp.clr_keys = c.cache->keys;
      sp.clr_winner = c.cache->winner;
      sp.clr_n = c.cache->capacity;
    }
    cudaError_t e = run_stats_one(sp, c.B, dtype, vec, c.stream);
    if (e == cudaSuccess) e = enqueue_chain(c, q, vec, c.stream);
    return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  }
  const int S = c.single_stream ? 0 : verify_slices(c.B);
  DevStreams* ds = S > 0 ? device_streams() : nullptr;
  if (!ds) {
    const SliceParams q = slice_params(c, fork, L, 0, c.B);
    if (run_stats(q.sp, c.B, dtype, vec, c.stream, verify_group(q.sp, c.B)) != cudaSuccess)
      return SSD_ERR_CUDA;
    return enqueue_tail(c, q, c.B, vec, c.stream) == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lk(ds->mu);
  ProfScope pass;  // the concurrent statistics pass as one phase (one slice)
  if (S == 1) pass.begin("stats_pass", c.stream, false);
  cudaError_t e = cudaEventRecord(ds->ev[0], c.stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->s1, ds->ev[0], 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(ds->s2, ds->ev[0], 0);
  for (int i = 0; i < S && e == cudaSuccess; ++i) {
    const int b0 = static_cast<int>(static_cast<long long>(c.B) * i / S);
    const int b1 = static_cast<int>(static_cast<long long>(c.B) * (i + 1) / S);
    const SliceParams q = slice_params(c, fork, L, b0, b1 - b0);
    e = run_stats2(q.sp, b1 - b0, dtype, vec, ds->s1, ds->s2, verify_group(q.sp, b1 - b0));
    if (e == cudaSuccess) e = cudaEventRecord(ds->ev[1 + 2 * i], ds->s1);
    if (e == cudaSuccess) e = cudaEventRecord(ds->ev[2 + 2 * i], ds->s2);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c.stream, ds->ev[1 + 2 * i], 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c.stream, ds->ev[2 + 2 * i], 0);
    pass.end();
    if (e == cudaSuccess)
      e = enqueue_tail(c, q, b1 - b0, vec, c.stream, i == S - 1, ds->s3, ds->ev[1 + 2 * kMaxSlices],
                       ds->ev[2 + 2 * kMaxSlices]);
  }
  return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* ssd_status_string(ssd_status s) {
  switch (s) {
    case SSD_OK: return "ok";
    case SSD_ERR_INVALID_ARG: return "invalid argument";
    case SSD_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
    case SSD_ERR_CUDA: return "CUDA error";
    case SSD_ERR_CACHE_FULL: return "speculation cache full";
    case SSD_ERR_TIMEOUT: return "timeout";
    case SSD_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

int ssd_version(void) { return 100; }

size_t ssd_workspace_bytes(int B, int k, int V, int f) {
  if (B < 1 || k < 0 || k > SSD_MAX_K || V < 2 || f < 0 || f > SSD_MAX_F) return 0;
  return make_layout(B, k, V, f).total;
}

size_t ssd_softmax_workspace_bytes(int rows, int V) {
  if (rows < 1 || V < 1) return 0;
  return make_softmax_layout(rows, V).total;
}

ssd_status ssd_workspace_init(void* ws, size_t bytes, ssd_stream_t stream) {
  if (!ws) return SSD_ERR_INVALID_ARG;
  return cuda_status(cudaMemsetAsync(ws, 0, bytes, S(stream)));
}

ssd_status ssd_get_device_error(void* ws, ssd_stream_t stream, int32_t* out, int clear) {
  if (!ws || !out) return SSD_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, S(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(S(stream));
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  *out = v;
  if (clear) {
    e = cudaMemsetAsync(ws, 0, sizeof v, S(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(S(stream));
  }
  return cuda_status(e);
}

ssd_status ssd_softmax_temp(const void* logits, ssd_dtype dtype, int rows, int V, const float* T,
                            float* probs, float* row_max, float* row_sum, int32_t* row_argmax,
                            void* ws, size_t ws_bytes, ssd_stream_t stream) {
  CallRange nvtx_range("ssd_softmax_temp");
  if (!dtype_ok(dtype)) return SSD_ERR_UNSUPPORTED_DTYPE;
  if (!logits || !T || !row_max || !row_sum || !row_argmax || !ws) return SSD_ERR_INVALID_ARG;
  if (rows < 1 || V < 1 || V > (1 << 28)) return SSD_ERR_INVALID_ARG;
  if (!aligned(logits, esize(dtype)) || !aligned(ws, 256)) return SSD_ERR_INVALID_ARG;
  const WsLayout L = make_softmax_layout(rows, V, static_cast<int>(esize(dtype)));
  if (ws_bytes < L.total) return SSD_ERR_WORKSPACE;
  const bool vec = vec_ok(logits, V, V, dtype);
  StatsParams sp;
  memset(&sp, 0, sizeof sp);
  sp.Z = logits; sp.zb = V; sp.Pz = 1;
  sp.D = logits; sp.db = V;
  sp.T = T;
  sp.V = V; sp.C = L.ch.C; sp.CH = L.ch.CH; sp.R = 1; sp.Rp = 1;
  sp.part = reinterpret_cast<PartStat*>(wsp(ws, L.part));
  sp.err = reinterpret_cast<int*>(wsp(ws, L.err));
  cudaError_t e = run_stats(sp, rows, dtype == SSD_BF16 ? 1 : 0, vec, S(stream));
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  SoftmaxParams p;
  memset(&p, 0, sizeof p);
  p.L = logits; p.dtype = dtype == SSD_BF16 ? 1 : 0; p.rows = rows; p.V = V;
  p.C = L.ch.C; p.CH = L.ch.CH; p.T = T; p.part = sp.part;
  p.rowstat = reinterpret_cast<RowStat*>(wsp(ws, L.rowstat));
  p.probs = probs; p.row_max = row_max; p.row_sum = row_sum; p.row_argmax = row_argmax;
  p.err = reinterpret_cast<int*>(wsp(ws, L.err));
  {
    ProfScope ps("softmax_finalize", S(stream));
    e = launch_softmax_finalize(p, S(stream));
  }
  if (e == cudaSuccess && probs) {
    ProfScope ps("softmax_probs", S(stream));
    e = launch_softmax_probs(p, S(stream));
  }
  return cuda_status(e);
}

ssd_status ssd_verify(const void* Z, int64_t z_bstride, const void* D, int64_t d_bstride,
                      ssd_dtype dtype, int B, int k, int V, const int32_t* x, const float* T,
                      const float* u_acc, int32_t* accept_len, float* p_at_x, float* q_at_x,
                      const float* u_smp, int32_t* out_tok, void* ws, size_t ws_bytes,
                      ssd_stream_t stream) {
  CallRange nvtx_range("ssd_verify");
  VerifyCall c;
  memset(&c, 0, sizeof c);
  c.Z = Z; c.zb = z_bstride; c.D = D; c.db = d_bstride; c.dt = dtype;
  c.B = B; c.k = k; c.V = V; c.x = x; c.T = T; c.u_acc = u_acc;
  c.accept_len = accept_len; c.p_at_x = p_at_x; c.q_at_x = q_at_x;
  c.u_smp = u_smp; c.out_tok = out_tok; c.ws = ws; c.ws_bytes = ws_bytes; c.stream = S(stream);
  return run_verify(c, false);
}

ssd_status ssd_verify_drafted(const void* Z, int64_t z_bstride, const void* D, int64_t d_bstride,
                              ssd_dtype dtype, int B, int k, int V, const int32_t* x,
                              const float* T, const float* u_acc, int32_t* accept_len,
                              float* p_at_x, float* q_at_x, const float* u_smp, int32_t* out_tok,
                              void* ws, size_t ws_bytes, ssd_stream_t stream) {
  CallRange nvtx_range("ssd_verify_drafted");
  VerifyCall c;
  memset(&c, 0, sizeof c);
  c.Z = Z; c.zb = z_bstride; c.D = D; c.db = d_bstride; c.dt = dtype;
  c.B = B; c.k = k; c.V = V; c.x = x; c.T = T; c.u_acc = u_acc;
  c.accept_len = accept_len; c.p_at_x = p_at_x; c.q_at_x = q_at_x;
  c.u_smp = u_smp; c.out_tok = out_tok; c.drafted = true;
  c.ws = ws; c.ws_bytes = ws_bytes; c.stream = S(stream);
  return run_verify(c, false);
}

ssd_status ssd_draft_sample(const void* D, int64_t d_bstride, ssd_dtype dtype, int B, int k,
                            int V, int row0, int rows, const float* T, uint64_t seed,
                            uint32_t offset, int32_t* x_out, int64_t x_bstride, int f,
                            int32_t* fork_tok, float* fork_logit, void* ws, size_t ws_bytes,
                            ssd_stream_t stream) {
  CallRange nvtx_range("ssd_draft_sample");
  if (!dtype_ok(dtype)) return SSD_ERR_UNSUPPORTED_DTYPE;
  if (!D || !T || !x_out || !ws) return SSD_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || k > SSD_MAX_K || V < 2 || V > (1 << 28)) return SSD_ERR_INVALID_ARG;
  if (row0 < 0 || rows < 1 || row0 + rows > k + 1) return SSD_ERR_INVALID_ARG;
  if (d_bstride < static_cast<int64_t>(row0 + rows) * V) return SSD_ERR_INVALID_ARG;
  if (B > 1 && x_bstride < rows) return SSD_ERR_INVALID_ARG;
  if (f < 0 || f + 1 > SSD_MAX_F || f + 1 >= V) return SSD_ERR_INVALID_ARG;
  if (f > 0 && (!fork_tok || !fork_logit)) return SSD_ERR_INVALID_ARG;
  if (!aligned(D, esize(dtype)) || !aligned(ws, 256)) return SSD_ERR_INVALID_ARG;
  const WsLayout L = make_layout(B, k, V, f > 0 ? f + 1 : 0, static_cast<int>(esize(dtype)));
  if (ws_bytes < L.total) return SSD_ERR_WORKSPACE;
  const bool vec = vec_ok(D, d_bstride, V, dtype);
  StatsParams sp;
  memset(&sp, 0, sizeof sp);
  sp.D = D; sp.db = d_bstride;
  sp.Pz = k + 1;  // draft row i's partials sit at row Pz + i of the verify layout
  sp.T = T;
  sp.f = f > 0 ? f + 1 : 0;
  sp.V = V; sp.C = L.ch.C; sp.CH = L.ch.CH; sp.R = L.R; sp.Rp = L.R; sp.r0 = row0;
  sp.part = reinterpret_cast<PartStat*>(wsp(ws, L.part));
  sp.topk = reinterpret_cast<TopEntry*>(wsp(ws, L.topk));
  sp.gpart = reinterpret_cast<GumbelPart*>(wsp(ws, L.gpart));
  sp.err = reinterpret_cast<int*>(wsp(ws, L.err));
  sp.seed_lo = static_cast<uint32_t>(seed);
  sp.seed_hi = static_cast<uint32_t>(seed >> 32);
  for (int r = 0; r < 10; ++r) {  // Philox4x32's key schedule: the Weyl increments
    sp.rk0[r] = sp.seed_lo + static_cast<uint32_t>(r) * 0x9E3779B9u;
    sp.rk1[r] = sp.seed_hi + static_cast<uint32_t>(r) * 0xBB67AE85u;
  }
  sp.offset = offset;
  sp.Pf = L.Pf;
  sp.G = 1;
  while (sp.G < 4 && static_cast<long long>(B) * rows * ((sp.C + 2 * sp.G - 1) / (2 * sp.G)) >= 2432)
    sp.G *= 2;
  sp.G = split_group(sp.G, sp.C);
  const int dt = dtype == SSD_BF16 ? 1 : 0;
  cudaError_t e;
  {
    ProfScope ps("draft_stats", S(stream));
    e = launch_draft(sp, B, dt, vec, rows, f > 0, S(stream));
  }
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  DraftParams dp;
  memset(&dp, 0, sizeof dp);
  dp.B = B; dp.V = V; dp.C = L.ch.C; dp.Rp = L.R; dp.Pz = k + 1; dp.Pf = L.Pf;
  dp.row0 = row0; dp.rows = rows; dp.T = T;
  dp.part = sp.part; dp.gpart = sp.gpart; dp.topk = sp.topk; dp.f = f;
  dp.x_out = x_out; dp.x_bstride = x_bstride; dp.fork_tok = fork_tok; dp.fork_logit = fork_logit;
  dp.err = sp.err;
  ProfScope ps("draft_finalize", S(stream));
  return cuda_status(launch_draft_finalize(dp, S(stream)));
}

size_t ssd_tree_workspace_bytes(int B, int N, int V) {
  if (B < 1 || N < 1 || N > kMaxTreeNodes || V < 2) return 0;
  return make_tree_layout(B, N, V).total;
}

ssd_status ssd_verify_tree(const void* Z, int64_t z_bstride, const void* D, int64_t d_bstride,
                           ssd_dtype dtype, int B, int N, int V, const int32_t* parent,
                           const int32_t* tok, const float* T, const float* u_acc,
                           const float* u_smp, int32_t* accept_len, int32_t* out_tok,
                           int32_t* out_node, void* ws, size_t ws_bytes, ssd_stream_t stream) {
  CallRange nvtx_range("ssd_verify_tree");
  if (!dtype_ok(dtype)) return SSD_ERR_UNSUPPORTED_DTYPE;
  if (!Z || !D || !parent || !tok || !T || !u_acc || !u_smp || !accept_len || !out_tok || !ws)
    return SSD_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || N > kMaxTreeNodes || V < 2 || V > (1 << 28)) return SSD_ERR_INVALID_ARG;
  if (z_bstride < static_cast<int64_t>(N) * V || d_bstride < static_cast<int64_t>(N) * V)
    return SSD_ERR_INVALID_ARG;
  if (!aligned(Z, esize(dtype)) || !aligned(D, esize(dtype)) || !aligned(ws, 256))
    return SSD_ERR_INVALID_ARG;
  const TreeLayout L = make_tree_layout(B, N, V, static_cast<int>(esize(dtype)));
  if (ws_bytes < L.total) return SSD_ERR_WORKSPACE;
  const bool vec = vec_ok(Z, z_bstride, V, dtype) && vec_ok(D, d_bstride, V, dtype);
  const int dt = dtype == SSD_BF16 ? 1 : 0;
  StatsParams sp;
  memset(&sp, 0, sizeof sp);
  sp.Z = Z; sp.zb = z_bstride; sp.Pz = N;
  sp.D = D; sp.db = d_bstride; sp.Pds = N; sp.Pdf = 0;
  sp.T = T; sp.V = V; sp.C = L.ch.C; sp.CH = L.ch.CH; sp.R = L.R; sp.Rp = L.R;
  sp.part = reinterpret_cast<PartStat*>(wsp(ws, L.part));
  sp.err = reinterpret_cast<int*>(wsp(ws, L.err));
  sp.tree_parent = parent;  // leaves' draft rows are skipped
  sp.tree_N = N;
  cudaError_t e = run_stats(sp, B, dt, vec, S(stream));  // the 2N rows, one launch
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  TreeParams tp;
  memset(&tp, 0, sizeof tp);
  tp.Z = Z; tp.zb = z_bstride; tp.D = D; tp.db = d_bstride;
  tp.B = B; tp.N = N; tp.V = V; tp.C = L.ch.C; tp.Rp = L.R;
  tp.parent = parent; tp.tok = tok; tp.T = T; tp.u_acc = u_acc; tp.u_smp = u_smp;
  tp.part = sp.part; tp.accept_len = accept_len; tp.out_tok = out_tok; tp.out_node = out_node;
  tp.err = sp.err;
  tp.cache = reinterpret_cast<float4*>(wsp(ws, L.cache));
  tp.cache_stride = static_cast<int64_t>(L.cache_stride);
  ProfScope ps("tree_walk", S(stream));
  return cuda_status(launch_tree_walk(tp, dt, vec, S(stream)));
}

size_t ssd_topk_workspace_bytes(int B, int k, int V, int K) {
  if (B < 1 || k < 1 || k > SSD_MAX_K || V < 2 || K < 1) return 0;
  const int Ke = K < V ? K : V;
  if (Ke <= kMaxTopK) return make_topk_layout(B, k, V, Ke).total;
  if (V > kFiltMaxV) return 0;
  return make_filt_layout(B, k, V).total;
}

namespace {

// ssd_verify_topk beyond the in-register lists (K > kMaxTopK, top-p over
// the whole vocabulary): threshold keys per row found from histograms, see
// ssd_filter.cu.
ssd_status run_verify_filtered(const void* Z, int64_t zb, const void* D, int64_t db,
                               ssd_dtype dtype, int B, int k, int V, const int32_t* x,
                               const float* T, int K, const float* top_p, const float* u_acc,
                               int32_t* accept_len, float* p_at_x, float* q_at_x,
                               const float* u_smp, int32_t* out_tok, void* ws, size_t ws_bytes,
                               cudaStream_t st) {
  if (V > kFiltMaxV) return SSD_ERR_INVALID_ARG;
  const FiltLayout L = make_filt_layout(B, k, V, static_cast<int>(esize(dtype)));
  if (ws_bytes < L.total) return SSD_ERR_WORKSPACE;
  const bool vec = vec_ok(Z, zb, V, dtype) && vec_ok(D, db, V, dtype);
  const int dt = dtype == SSD_BF16 ? 1 : 0;
  // 1. row maxima, argmax and NaN flags of the 2k+1 rows (no exponentials)
  StatsParams sp;
  memset(&sp, 0, sizeof sp);
  sp.Z = Z; sp.zb = zb; sp.Pz = k + 1;
  sp.D = D; sp.db = db; sp.Pds = k; sp.Pdf = 0;
  sp.T = nullptr;
  sp.V = V; sp.C = L.ch.C; sp.CH = L.ch.CH; sp.R = L.R; sp.Rp = L.R;
  sp.part = reinterpret_cast<PartStat*>(wsp(ws, L.part));
  sp.err = reinterpret_cast<int*>(wsp(ws, L.err));
  cudaError_t e = run_stats(sp, B, dt, vec, st);
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  FiltParams fp;
  memset(&fp, 0, sizeof fp);
  fp.Z = Z; fp.zb = zb; fp.D = D; fp.db = db; fp.dtype = dt;
  fp.B = B; fp.k = k; fp.V = V; fp.C = L.ch.C; fp.CH = L.ch.CH; fp.E = L.ch.E; fp.R = L.R;
  fp.K = K;
  fp.total_mode = K >= V ? 1 : 0;
  fp.G = 1;
  while (fp.G < fp.C &&
         static_cast<long long>(B) * L.R * ((fp.C + 2 * fp.G - 1) / (2 * fp.G)) >= 2432)
    fp.G *= 2;
  fp.G = split_group(fp.G, fp.C);
  if (static_cast<long long>(fp.G) * fp.CH > (1 << 19)) fp.G = (1 << 19) / fp.CH;  // 32-bit bin sums
  fp.T = T; fp.top_p = top_p; fp.x = x; fp.u_acc = u_acc; fp.u_smp = u_smp;
  fp.accept_len = accept_len; fp.p_at_x = p_at_x; fp.q_at_x = q_at_x; fp.out_tok = out_tok;
  fp.part = sp.part;
  fp.rows = reinterpret_cast<FiltRow*>(wsp(ws, L.rows));
  fp.hcnt = reinterpret_cast<unsigned*>(wsp(ws, L.hcnt));
  fp.hmass = reinterpret_cast<unsigned long long*>(wsp(ws, L.hmass));
  fp.cand = reinterpret_cast<unsigned long long*>(wsp(ws, L.cand));
  fp.bstate = reinterpret_cast<BState*>(wsp(ws, L.bstate));
  fp.rmass = reinterpret_cast<long long*>(wsp(ws, L.rmass));
  fp.err = sp.err;
  {
    ProfScope ps("filt_rowinit", st);
    e = launch_filt_rowinit(fp, st);
  }
  if (e == cudaSuccess) {
    ProfScope ps("filt_hist", st);
    e = launch_filt_hist(fp, vec, st);
  }
  if (e == cudaSuccess) {
    ProfScope ps("filt_band", st);
    e = launch_filt_band(fp, st);
  }
  if (e == cudaSuccess) {
    ProfScope ps("filt_collect", st);
    e = launch_filt_collect(fp, vec, st);
  }
  if (e == cudaSuccess) {
    ProfScope ps("filt_cut", st);
    e = launch_filt_cut(fp, vec, st);
  }
  if (e == cudaSuccess) {
    ProfScope ps("filt_accept", st);
    e = launch_filt_accept(fp, st);
  }
  if (e == cudaSuccess && u_smp && out_tok) {
    {
      ProfScope ps("filt_mass", st);
      e = launch_filt_mass(fp, vec, st);
    }
    if (e == cudaSuccess) {
      ProfScope ps("filt_select", st);
      e = launch_filt_select(fp, vec, st);
    }
  }
  return cuda_status(e);
}

}  // namespace

ssd_status ssd_verify_topk(const void* Z, int64_t z_bstride, const void* D, int64_t d_bstride,
                           ssd_dtype dtype, int B, int k, int V, const int32_t* x, const float* T,
                           int K, const float* top_p, const float* u_acc, int32_t* accept_len,
                           float* p_at_x, float* q_at_x, const float* u_smp, int32_t* out_tok,
                           void* ws, size_t ws_bytes, ssd_stream_t stream) {
  CallRange nvtx_range("ssd_verify_topk");
  if (!dtype_ok(dtype)) return SSD_ERR_UNSUPPORTED_DTYPE;
  if (!Z || !D || !x || !T || !u_acc || !accept_len || !ws) return SSD_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || k > SSD_MAX_K || V < 2 || V > (1 << 28)) return SSD_ERR_INVALID_ARG;
  if (K < 1) return SSD_ERR_INVALID_ARG;
  if ((p_at_x == nullptr) != (q_at_x == nullptr)) return SSD_ERR_INVALID_ARG;
  if (u_smp && !out_tok) return SSD_ERR_INVALID_ARG;
  if (z_bstride < static_cast<int64_t>(k + 1) * V || d_bstride < static_cast<int64_t>(k) * V)
    return SSD_ERR_INVALID_ARG;
  if (!aligned(Z, esize(dtype)) || !aligned(D, esize(dtype)) || !aligned(ws, 256))
    return SSD_ERR_INVALID_ARG;
  const int Ke = K < V ? K : V;  // more than V tokens: all of them
  if (Ke > kMaxTopK)
    return run_verify_filtered(Z, z_bstride, D, d_bstride, dtype, B, k, V, x, T, K, top_p,
                               u_acc, accept_len, p_at_x, q_at_x, u_smp, out_tok, ws, ws_bytes,
                               S(stream));
  const TopkLayout L = make_topk_layout(B, k, V, Ke, static_cast<int>(esize(dtype)));
  if (ws_bytes < L.total) return SSD_ERR_WORKSPACE;
  const bool vec = vec_ok(Z, z_bstride, V, dtype) && vec_ok(D, d_bstride, V, dtype);
  TopkParams tp;
  memset(&tp, 0, sizeof tp);
  tp.Z = Z; tp.zb = z_bstride; tp.D = D; tp.db = d_bstride;
  tp.dtype = dtype == SSD_BF16 ? 1 : 0;
  tp.B = B; tp.k = k; tp.V = V; tp.C = L.ch.C; tp.CH = L.ch.CH; tp.R = L.R; tp.K = Ke;
  // chunk groups up to a whole row per CTA while the grid keeps ~16 CTAs per
  // SM: the end-of-CTA selection (K rounds) is then paid once per row
  tp.G = 1;
  while (tp.G < SSD_TOPK_MAX_GROUP && tp.G < tp.C &&
         static_cast<long long>(B) * L.R * ((tp.C + 2 * tp.G - 1) / (2 * tp.G)) >= 2432)
    tp.G *= 2;
  tp.G = split_group(tp.G, tp.C);
  tp.T = T; tp.top_p = top_p; tp.x = x; tp.u_acc = u_acc; tp.u_smp = u_smp;
  tp.accept_len = accept_len; tp.p_at_x = p_at_x; tp.q_at_x = q_at_x; tp.out_tok = out_tok;
  tp.part = reinterpret_cast<PartStat*>(wsp(ws, L.part));
  tp.lists = reinterpret_cast<TopEntry*>(wsp(ws, L.lists));
  tp.err = reinterpret_cast<int*>(wsp(ws, L.err));
  cudaError_t e;
  {
    ProfScope ps("topk_pass", S(stream));
    e = launch_topk_verify(tp, tp.dtype, vec, S(stream));
  }
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  ProfScope ps("topk_finalize", S(stream));
  return cuda_status(launch_topk_finalize(tp, S(stream)));
}

ssd_status ssd_verify_fork_fanout(const void* Z, int64_t z_bstride, const void* D,
                                  int64_t d_bstride, ssd_dtype dtype, int B, int k, int V,
                                  const int32_t* x, const float* T, const float* u_acc,
                                  int32_t* accept_len, float* p_at_x, float* q_at_x,
                                  const float* u_smp, int32_t* out_tok, int F,
                                  const int32_t* fanout, const int32_t* mask, int M,
                                  int32_t* fork_tok, float* fork_logit, void* ws, size_t ws_bytes,
                                  ssd_stream_t stream) {
  CallRange nvtx_range("ssd_verify_fork_fanout");
  VerifyCall c;
  memset(&c, 0, sizeof c);
  c.Z = Z; c.zb = z_bstride; c.D = D; c.db = d_bstride; c.dt = dtype;
  c.B = B; c.k = k; c.V = V; c.x = x; c.T = T; c.u_acc = u_acc;
  c.accept_len = accept_len; c.p_at_x = p_at_x; c.q_at_x = q_at_x;
  c.u_smp = u_smp; c.out_tok = out_tok;
  c.f = F; c.mask = mask; c.M = M; c.fork_tok = fork_tok; c.fork_logit = fork_logit;
  c.fanout = fanout;
  c.ws = ws; c.ws_bytes = ws_bytes; c.stream = S(stream);
  return run_verify(c, true);
}

ssd_status ssd_verify_fork_cache(const void* Z, int64_t z_bstride, const void* D,
                                 int64_t d_bstride, ssd_dtype dtype, int B, int k, int V,
                                 const int32_t* x, const float* T, const float* u_acc,
                                 int32_t* accept_len, float* p_at_x, float* q_at_x,
                                 const float* u_smp, int32_t* out_tok, int f, const int32_t* mask,
                                 int M, int32_t* fork_tok, float* fork_logit,
                                 ssd_spec_cache* cache, int clear, const int32_t* payload,
                                 int32_t* hit, int32_t* tok_out, void* ws, size_t ws_bytes,
                                 ssd_stream_t stream) {
  CallRange nvtx_range("ssd_verify_fork_cache");
  if (!cache || !payload || !hit || !tok_out || !out_tok) return SSD_ERR_INVALID_ARG;
  if (k + 1 > 256 || static_cast<int64_t>(B) * (k + 1) * f > 0x7fffffff) return SSD_ERR_INVALID_ARG;
  VerifyCall c;
  memset(&c, 0, sizeof c);
  c.Z = Z; c.zb = z_bstride; c.D = D; c.db = d_bstride; c.dt = dtype;
  c.B = B; c.k = k; c.V = V; c.x = x; c.T = T; c.u_acc = u_acc;
  c.accept_len = accept_len; c.p_at_x = p_at_x; c.q_at_x = q_at_x;
  c.u_smp = u_smp; c.out_tok = out_tok;
  c.f = f; c.mask = mask; c.M = M; c.fork_tok = fork_tok; c.fork_logit = fork_logit;
  c.cache = &cache->view; c.cache_clear = clear != 0; c.payload = payload;
  c.hit = hit; c.tok_out = tok_out;
  c.ws = ws; c.ws_bytes = ws_bytes; c.stream = S(stream);
  return run_verify(c, true);
}

ssd_status ssd_verify_fork(const void* Z, int64_t z_bstride, const void* D, int64_t d_bstride,
                           ssd_dtype dtype, int B, int k, int V, const int32_t* x, const float* T,
                           const float* u_acc, int32_t* accept_len, float* p_at_x, float* q_at_x,
                           const float* u_smp, int32_t* out_tok, int f, const int32_t* mask, int M,
                           int32_t* fork_tok, float* fork_logit, void* ws, size_t ws_bytes,
                           ssd_stream_t stream) {
  return ssd_verify_fork_fanout(Z, z_bstride, D, d_bstride, dtype, B, k, V, x, T, u_acc,
                                accept_len, p_at_x, q_at_x, u_smp, out_tok, f, nullptr, mask, M,
                                fork_tok, fork_logit, ws, ws_bytes, stream);
}

ssd_status ssd_sample_residual(const void* Z, int64_t z_bstride, const void* D, int64_t d_bstride,
                               ssd_dtype dtype, int B, int k, int V, const int32_t* x,
                               const float* T, const int32_t* accept_len, const float* u_smp,
                               int32_t* out_tok, void* ws, size_t ws_bytes, ssd_stream_t stream) {
  CallRange nvtx_range("ssd_sample_residual");
  if (!dtype_ok(dtype)) return SSD_ERR_UNSUPPORTED_DTYPE;
  if (!Z || !D || !x || !T || !accept_len || !u_smp || !out_tok || !ws) return SSD_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || k > SSD_MAX_K || V < 2 || V > (1 << 28)) return SSD_ERR_INVALID_ARG;
  if (z_bstride < static_cast<int64_t>(k + 1) * V || d_bstride < static_cast<int64_t>(k) * V)
    return SSD_ERR_INVALID_ARG;
  if (!aligned(Z, esize(dtype)) || !aligned(D, esize(dtype)) || !aligned(ws, 256))
    return SSD_ERR_INVALID_ARG;
  // the row statistics of the verify call sit at f-independent offsets
  const WsLayout L = make_layout(B, k, V, 0, static_cast<int>(esize(dtype)));
  if (ws_bytes < L.total) return SSD_ERR_WORKSPACE;
  const bool vec = vec_ok(Z, z_bstride, V, dtype) && vec_ok(D, d_bstride, V, dtype);
  PrepParams pp;
  pp.B = B; pp.k = k; pp.T = T; pp.x = x; pp.accept_len = accept_len;
  pp.rowstat = reinterpret_cast<RowStat*>(wsp(ws, L.rowstat));
  pp.R = L.R;
  pp.bstate = reinterpret_cast<BState*>(wsp(ws, L.bstate));
  pp.out_tok = out_tok;
  pp.amb_cnt = reinterpret_cast<int*>(wsp(ws, L.amb_cnt));
  cudaError_t e;
  {
    ProfScope ps("residual_prep", S(stream));
    e = launch_residual_prep(pp, S(stream));
  }
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  ResidualParams rp;
  memset(&rp, 0, sizeof rp);
  rp.Z = Z; rp.zb = z_bstride; rp.Pz = k + 1;
  rp.D = D; rp.db = d_bstride;
  rp.V = V; rp.C = L.dch.C; rp.CH = L.dch.CH; rp.E = L.dch.E; rp.R = L.R; rp.k = k;
  rp.T = T; rp.u_smp = u_smp;
  rp.rowstat = pp.rowstat; rp.bstate = pp.bstate;
  rp.rnorm = reinterpret_cast<long long*>(wsp(ws, L.rnorm));
  rp.rthr = reinterpret_cast<long long*>(wsp(ws, L.rthr));
  rp.racc = reinterpret_cast<long long*>(wsp(ws, L.racc));
  rp.amb_cnt = reinterpret_cast<int*>(wsp(ws, L.amb_cnt));
  rp.amb_idx = reinterpret_cast<int*>(wsp(ws, L.amb_idx));
  rp.amb_cap = amb_cap(V);
  rp.out_tok = out_tok;
  return cuda_status(run_residual(rp, B, dtype == SSD_BF16 ? 1 : 0, vec, S(stream)));
}

ssd_status ssd_forked_recovery(const void* L_, int64_t l_bstride, ssd_dtype dtype, int B, int P,
                               int V, int f, const int32_t* mask, int M, int32_t* fork_tok,
                               float* fork_logit, void* ws, size_t ws_bytes, ssd_stream_t stream) {
  return ssd_forked_recovery_fanout(L_, l_bstride, dtype, B, P, V, f, nullptr, mask, M, fork_tok,
                                    fork_logit, ws, ws_bytes, stream);
}

ssd_status ssd_forked_recovery_fanout(const void* L_, int64_t l_bstride, ssd_dtype dtype, int B,
                                      int P, int V, int f, const int32_t* fanout,
                                      const int32_t* mask, int M, int32_t* fork_tok,
                                      float* fork_logit, void* ws, size_t ws_bytes,
                                      ssd_stream_t stream) {
  CallRange nvtx_range("ssd_forked_recovery_fanout");
  if (!dtype_ok(dtype)) return SSD_ERR_UNSUPPORTED_DTYPE;
  if (!L_ || !fork_tok || !fork_logit || !ws) return SSD_ERR_INVALID_ARG;
  if (B < 1 || P < 1 || P > SSD_MAX_K + 1 || V < 2 || V > (1 << 28)) return SSD_ERR_INVALID_ARG;
  if (f < 1 || f > SSD_MAX_F || f >= V) return SSD_ERR_INVALID_ARG;
  if (M < 0 || M > SSD_MAX_M || (M > 0 && !mask)) return SSD_ERR_INVALID_ARG;
  if (l_bstride < static_cast<int64_t>(P) * V) return SSD_ERR_INVALID_ARG;
  if (!aligned(L_, esize(dtype)) || !aligned(ws, 256)) return SSD_ERR_INVALID_ARG;
  const WsLayout L = make_layout(B, P - 1, V, f, static_cast<int>(esize(dtype)));
  if (ws_bytes < L.total) return SSD_ERR_WORKSPACE;
  const bool vec = vec_ok(L_, l_bstride, V, dtype);
  StatsParams sp;
  memset(&sp, 0, sizeof sp);
  sp.Z = nullptr; sp.zb = 0; sp.Pz = 0;
  sp.D = L_; sp.db = l_bstride; sp.Pds = 0; sp.Pdf = P;
  sp.T = nullptr;
  sp.mask = mask; sp.M = M; sp.f = f;
  sp.V = V; sp.C = L.ch.C; sp.CH = L.ch.CH; sp.R = P; sp.Rp = L.R;
  sp.part = reinterpret_cast<PartStat*>(wsp(ws, L.part));
  sp.topk = reinterpret_cast<TopEntry*>(wsp(ws, L.topk));
  sp.err = reinterpret_cast<int*>(wsp(ws, L.err));
  cudaError_t e = run_stats(sp, B, dtype == SSD_BF16 ? 1 : 0, vec, S(stream));
  if (e != cudaSuccess) return SSD_ERR_CUDA;
  FinalizeParams fp;
  memset(&fp, 0, sizeof fp);
  fp.Z = nullptr; fp.Pz = 0;
  fp.D = L_; fp.db = l_bstride; fp.Pds = 0; fp.Pdf = P;
  fp.dtype = dtype == SSD_BF16 ? 1 : 0;
  fp.B = B; fp.k = 0; fp.V = V; fp.C = L.ch.C; fp.R = P; fp.Rp = L.R; fp.f = f;
  fp.fork_tok = fork_tok; fp.fork_logit = fork_logit; fp.fanout = fanout;
  fp.part = sp.part; fp.topk = sp.topk;
  fp.rowstat = reinterpret_cast<RowStat*>(wsp(ws, L.rowstat));
  fp.bstate = reinterpret_cast<BState*>(wsp(ws, L.bstate));
  fp.err = reinterpret_cast<int*>(wsp(ws, L.err));
  ProfScope ps("finalize", S(stream));
  return cuda_status(launch_finalize(fp, S(stream)));
}

// ---------------------------------------------------------------------------
// Speculation cache
// ---------------------------------------------------------------------------
ssd_status ssd_spec_cache_create(int capacity, int depth, ssd_spec_cache** out) {
  if (!out) return SSD_ERR_INVALID_ARG;
  *out = nullptr;
  if (capacity < 2 || (capacity & (capacity - 1)) != 0 || capacity > (1 << 28) || depth < 1 ||
      depth > 4096)
    return SSD_ERR_INVALID_ARG;
  ssd_spec_cache* c = new (std::nothrow) ssd_spec_cache;
  if (!c) return SSD_ERR_INVALID_ARG;
  memset(c, 0, sizeof *c);
  c->view.capacity = capacity;
  c->view.depth = depth;
  cudaGetDevice(&c->device);
  const size_t kb = sizeof(unsigned long long) * capacity;
  const size_t pb = sizeof(int32_t) * static_cast<size_t>(capacity) * depth;
  cudaError_t e = cudaMalloc(&c->view.keys, kb);
  if (e == cudaSuccess) e = cudaMalloc(&c->view.winner, kb);
  if (e == cudaSuccess) e = cudaMalloc(&c->view.payload, pb);
  // one small block: the error word, the write kernel's ticket, the call counter
  void* misc = nullptr;
  if (e == cudaSuccess) e = cudaMalloc(&misc, 64);
  if (e == cudaSuccess) {
    c->view.err = static_cast<int*>(misc);
    c->view.done = reinterpret_cast<unsigned*>(static_cast<char*>(misc) + 16);
    c->view.calls = reinterpret_cast<unsigned long long*>(static_cast<char*>(misc) + 32);
  }
  if (e == cudaSuccess) e = cudaMemset(c->view.keys, 0xff, kb);
  if (e == cudaSuccess) e = cudaMemset(c->view.winner, 0, kb);
  if (e == cudaSuccess) e = cudaMemset(c->view.payload, 0xff, pb);
  if (e == cudaSuccess) e = cudaMemset(misc, 0, 64);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    ssd_spec_cache_destroy(c);
    return SSD_ERR_CUDA;
  }
  *out = c;
  return SSD_OK;
}

void ssd_spec_cache_destroy(ssd_spec_cache* c) {
  if (!c) return;
  if (c->view.keys) cudaFree(c->view.keys);
  if (c->view.winner) cudaFree(c->view.winner);
  if (c->view.payload) cudaFree(c->view.payload);
  if (c->view.err) cudaFree(c->view.err);
  delete c;
}

ssd_status ssd_spec_cache_clear(ssd_spec_cache* c, ssd_stream_t stream) {
  CallRange nvtx_range("ssd_spec_cache_clear");
  if (!c) return SSD_ERR_INVALID_ARG;
  const size_t kb = sizeof(unsigned long long) * c->view.capacity;
  cudaError_t e = cudaMemsetAsync(c->view.keys, 0xff, kb, S(stream));
  if (e == cudaSuccess) e = cudaMemsetAsync(c->view.winner, 0, kb, S(stream));
  return cuda_status(e);
}

ssd_status ssd_spec_cache_insert(ssd_spec_cache* c, const int32_t* b, const int32_t* pos,
                                 const int32_t* tok, const int32_t* payload, int n,
                                 ssd_stream_t stream) {
  CallRange nvtx_range("ssd_spec_cache_insert");
  if (!c || n < 0) return SSD_ERR_INVALID_ARG;
  if (n == 0) return SSD_OK;
  if (!b || !pos || !tok || !payload) return SSD_ERR_INVALID_ARG;
  InsertArgs a;
  memset(&a, 0, sizeof a);
  a.b = b; a.pos = pos; a.tok = tok; a.payload = payload; a.n = n;
  return cuda_status(cache_insert(c->view, a, S(stream)));
}

ssd_status ssd_spec_cache_insert_forks(ssd_spec_cache* c, const int32_t* fork_tok, int B, int P,
                                       int f, const int32_t* payload, ssd_stream_t stream) {
  CallRange nvtx_range("ssd_spec_cache_insert_forks");
  if (!c || !fork_tok || !payload || B < 1 || P < 1 || P > 256 || f < 1) return SSD_ERR_INVALID_ARG;
  if (static_cast<int64_t>(B) * P * f > 0x7fffffff) return SSD_ERR_INVALID_ARG;
  InsertArgs a;
  memset(&a, 0, sizeof a);
  a.fork_tok = fork_tok; a.P = P; a.f = f; a.payload = payload; a.n = B * P * f;
  return cuda_status(cache_insert(c->view, a, S(stream)));
}

ssd_status ssd_spec_cache_lookup(const ssd_spec_cache* c, const int32_t* b, const int32_t* pos,
                                 const int32_t* tok, int n, int32_t* hit, int32_t* tok_out,
                                 ssd_stream_t stream) {
  CallRange nvtx_range("ssd_spec_cache_lookup");
  if (!c || n < 0) return SSD_ERR_INVALID_ARG;
  if (n == 0) return SSD_OK;
  if (!b || !pos || !tok || !hit || !tok_out) return SSD_ERR_INVALID_ARG;
  LookupArgs a;
  memset(&a, 0, sizeof a);
  a.b = b; a.pos = pos; a.tok = tok; a.n = n; a.hit = hit; a.tok_out = tok_out;
  ProfScope ps("cache_lookup", S(stream));
  return cuda_status(launch_cache_lookup(c->view, a, S(stream)));
}

ssd_status ssd_spec_cache_lookup_outcome(const ssd_spec_cache* c, const int32_t* accept_len,
                                         const int32_t* out_tok, int B, int k, int32_t* hit,
                                         int32_t* tok_out, ssd_stream_t stream) {
  CallRange nvtx_range("ssd_spec_cache_lookup_outcome");
  if (!c || !accept_len || !out_tok || !hit || !tok_out || B < 1 || k < 1 || k > SSD_MAX_K)
    return SSD_ERR_INVALID_ARG;
  LookupArgs a;
  memset(&a, 0, sizeof a);
  a.accept_len = accept_len; a.out_tok = out_tok; a.k = k; a.n = B; a.hit = hit; a.tok_out = tok_out;
  ProfScope ps("cache_lookup", S(stream));
  return cuda_status(launch_cache_lookup(c->view, a, S(stream)));
}

ssd_status ssd_spec_cache_get_error(ssd_spec_cache* c, ssd_stream_t stream, int32_t* out,
                                    int clear) {
  if (!c || !out) return SSD_ERR_INVALID_ARG;
  return ssd_get_device_error(c->view.err, stream, out, clear);
}

int ssd_spec_cache_capacity(const ssd_spec_cache* c) { return c ? c->view.capacity : 0; }
int ssd_spec_cache_depth(const ssd_spec_cache* c) { return c ? c->view.depth : 0; }

ssd_status ssd_selftest_exp2(const float* x_hi, const float* x_lo, double* out, int n,
                             ssd_stream_t stream) {
  if (n < 0 || (n > 0 && (!x_hi || !x_lo || !out))) return SSD_ERR_INVALID_ARG;
  if (n == 0) return SSD_OK;
  return cuda_status(launch_selftest_exp2(x_hi, x_lo, out, n, S(stream)));
}

// ---------------------------------------------------------------------------
// ssd_verify_noalloc: the verify path with its scratch in a static array.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace {
// Scratch of ssd_verify_noalloc.  In host code this name is only a stand-in:
// the kernels get the device address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once per
// device, with that device current).
ssd_status noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return SSD_OK;
}
}  // namespace

extern "C" {

ssd_status ssd_verify_noalloc(const void* Z, int64_t z_bstride, const void* D, int64_t d_bstride,
                              ssd_dtype dtype, int B, int k, int V, const int32_t* x,
                              const float* T, const float* u_acc, int32_t* accept_len,
                              float* p_at_x, float* q_at_x, const float* u_smp, int32_t* out_tok,
                              ssd_stream_t stream) {
  CallRange nvtx_range("ssd_verify_noalloc");
  VerifyCall c;
  memset(&c, 0, sizeof c);
  c.Z = Z; c.zb = z_bstride; c.D = D; c.db = d_bstride; c.dt = dtype;
  c.B = B; c.k = k; c.V = V; c.x = x; c.T = T; c.u_acc = u_acc;
  c.accept_len = accept_len; c.p_at_x = p_at_x; c.q_at_x = q_at_x;
  c.u_smp = u_smp; c.out_tok = out_tok; c.stream = S(stream);
  // sizes first (ssd_workspace_bytes is 0 for invalid ones), then the size
  // limit, then every pointer: nothing reaches the scratch lookup or a
  // launch unless all of them pass
  if (!dtype_ok(dtype)) return SSD_ERR_UNSUPPORTED_DTYPE;
  if (B < 1 || k < 1 || k > SSD_MAX_K || V < 2 || V > (1 << 28)) return SSD_ERR_INVALID_ARG;
  if (ssd_workspace_bytes(B, k, V, 0) > SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_WORKSPACE;
  c.ws = &c;  // stands in for the scratch pointer in the argument check only
  ssd_status st = check_common(c, false);
  if (st != SSD_OK) return st;
  st = noalloc_scratch(&c.ws);
  if (st != SSD_OK) return st;
  c.ws_bytes = SSD_NOALLOC_SCRATCH_BYTES;
  c.single_stream = true;
  return run_verify(c, false);
}

ssd_status ssd_set_split(int chunk_elems, int chunks_per_cta) {
  if (chunk_elems < 0 || chunks_per_cta < 0) return SSD_ERR_INVALID_ARG;
  g_split.chunk.store(chunk_elems, std::memory_order_relaxed);
  g_split.group.store(chunks_per_cta, std::memory_order_relaxed);
  return SSD_OK;
}

ssd_status ssd_set_step_schedule(int max_b, int max_grid) {
  if (max_grid < 0) return SSD_ERR_INVALID_ARG;
  g_step_max_b.store(max_b < 0 ? -1 : max_b, std::memory_order_relaxed);
  g_step_grid.store(max_grid, std::memory_order_relaxed);
  return SSD_OK;
}

ssd_status ssd_set_chain_batch(int max_b) {
  g_chain_max_b.store(max_b < 0 ? -1 : max_b, std::memory_order_relaxed);
  return SSD_OK;
}

ssd_status ssd_profile_begin(int max_launches) {
  if (max_launches < 0 || max_launches > (1 << 20)) return SSD_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (g_prof.on) return SSD_ERR_INVALID_ARG;
  g_prof.recs.clear();
  g_prof.names.clear();
  g_prof.counts.clear();
  g_prof.pool.assign(2 * static_cast<size_t>(max_launches), nullptr);
  for (auto& ev : g_prof.pool) {
    if (cudaEventCreate(&ev) != cudaSuccess) {
      for (auto& e2 : g_prof.pool)
        if (e2) cudaEventDestroy(e2);
      g_prof.pool.clear();
      return SSD_ERR_CUDA;
    }
  }
  g_prof.cap = max_launches;
  g_prof.recs.reserve(max_launches);
  g_prof.on = true;
  return SSD_OK;
}

ssd_status ssd_profile_end(ssd_profile_entry* out, int cap, int* n_out) {
  std::lock_guard<std::mutex> lk(g_prof.mu);
  if (!g_prof.on) return SSD_ERR_INVALID_ARG;
  g_prof.on = false;
  ssd_status st = SSD_OK;
  std::vector<double> ms(g_prof.names.size(), 0.0);
  std::vector<int> timed(g_prof.names.size(), 0);
  for (const ProfRecord& r : g_prof.recs) {
    if (cudaEventSynchronize(r.b) != cudaSuccess) {
      st = SSD_ERR_CUDA;
      continue;
    }
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess) {
      st = SSD_ERR_CUDA;
      continue;
    }
    ms[r.kernel] += t;
    timed[r.kernel] += 1;
  }
  // "stats_span": for each statistics-pass phase (fork to join on the
  // caller's stream), the span of its two launches on the internal streams,
  // from the earlier of their begin events to the later of their end events
  // (the kernels' own time, without the fork and join)
  auto find_id = [&](const char* nm) {
    for (size_t i = 0; i < g_prof.names.size(); ++i)
      if (strcmp(g_prof.names[i], nm) == 0) return static_cast<int>(i);
    return -1;
  };
  const int id_pass = find_id("stats_pass"), id_t = find_id("stats_topf"), id_p = find_id("stats");
  if (id_pass >= 0 && id_t >= 0 && id_p >= 0) {
    const int id_span = g_prof.kernel_id("stats_span");
    ms.resize(g_prof.names.size(), 0.0);
    timed.resize(g_prof.names.size(), 0);
    const size_t nr = g_prof.recs.size();
    for (size_t i = 0; i < nr; ++i) {
      if (g_prof.recs[i].kernel != id_pass) continue;
      const ProfRecord* rt = nullptr;
      const ProfRecord* rp = nullptr;
      for (size_t j = i + 1; j < nr && g_prof.recs[j].kernel != id_pass; ++j) {
        if (g_prof.recs[j].kernel == id_t && !rt) rt = &g_prof.recs[j];
        if (g_prof.recs[j].kernel == id_p && !rp) rp = &g_prof.recs[j];
      }
      if (!rt || !rp) continue;
      const cudaEvent_t ref = g_prof.recs[i].a;
      float bt = 0.f, bp = 0.f, et = 0.f, ep = 0.f;
      if (cudaEventElapsedTime(&bt, ref, rt->a) != cudaSuccess ||
          cudaEventElapsedTime(&bp, ref, rp->a) != cudaSuccess ||
          cudaEventElapsedTime(&et, ref, rt->b) != cudaSuccess ||
          cudaEventElapsedTime(&ep, ref, rp->b) != cudaSuccess)
        continue;
      ms[id_span] += static_cast<double>(et > ep ? et : ep) - (bt < bp ? bt : bp);
      timed[id_span] += 1;
    }
  }
  int n = 0;
  for (size_t i = 0; i < g_prof.names.size() && out && n < cap; ++i, ++n) {
    memset(&out[n], 0, sizeof out[n]);
    strncpy(out[n].name, g_prof.names[i], sizeof out[n].name - 1);
    out[n].launches = g_prof.counts[i];
    out[n].timed = timed[i];
    out[n].total_ms = ms[i];
  }
  if (n_out) *n_out = n;
  for (auto& ev : g_prof.pool) cudaEventDestroy(ev);
  g_prof.pool.clear();
  g_prof.recs.clear();
  return st;
}

}  // extern "C"
