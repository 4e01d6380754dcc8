// ssd_tree.cu -- token-tree verification: the walk over a draft tree of N
// nodes per batch row after the statistics pass over its 2N logit rows.
//
// Sources: "tanishqkumar/ssd" summary, module notes (tree decoding in
// asynchronous speculative decoding; the temperature sampler: greedy at
// T = 0); "SSD: drafting and verification on separate GPUs", "What changes
// in SSD" (verification keeps the target's output law); the verification
// rule for a tree whose children were drawn from the draft's q at their
// parent is the multi-step speculative sampling of SpecInfer (Miao et al.
// 2024): at the current node with target law r (initially its p) the
// children are tried in index order, a child x is accepted when
// u < r(x)/q(x), a rejection replaces r by norm(max(0, r - q)), and when the
// children run out the token is drawn from r.
//
// Closed form used here (instead of materialising r): after j rejections at
// a node, r_j = max(0, p - c_j q) / W(c_j) with W(c) = sum_v max(0, p - c q),
// c_0 = 0 and c_{j+1} = c_j + W(c_j).  In the row's own units (e_z = 2^((z -
// m_z) c2), e_d likewise, S_z, S_d their sums) that is the weight
// w(v) = max(0, e_z(v) - rho_j e_d(v)) with rho_j = c_j S_z / S_d and the
// scaled mass Wsc_j = sum_v w(v) = W(c_j) S_z; rho_{j+1} = rho_j + Wsc_j / S_d.
// The acceptance test u < r_j(x)/q(x) becomes u Wsc_j e_d(x) < S_d w(x), and
// each rejection costs one pass over the node's two rows for the next Wsc.
//
// Layout of the work: one thread-block cluster of cs CTAs (1..8, chosen so
// that the grid fills the GPU) per batch row.  Every CTA merges the row
// statistics and takes the walk's decisions itself (thread 0, the same
// deterministic arithmetic on the same data in every CTA, so the cluster's
// control flow stays uniform); a pass splits the row's elements over the
// cluster's threads, each owning a contiguous range of E elements (so that
// the draw's inverse CDF is a scan of per-thread sums followed by a walk of
// one range).  Pass totals are exchanged through distributed shared memory
// (each CTA publishes its sum, a cluster barrier, every CTA adds the cs
// sums in rank order).  Element weights are double-float with compensated
// sums; a node's first residual pass keeps each element's two exponentials
// in the workspace (rows of at least 32768 elements) for the later passes
// at that node and the draw.  The draw converts the per-thread sums to
// exact 2^-48 fixed point for an order-independent scan.  Rank 0 writes the
// outputs.
#include <cooperative_groups.h>
#include <math.h>

#include "ssd_device.cuh"
#include "ssd_layout.h"
#include "ssd_merge.cuh"
#include "ssd_scan.cuh"

namespace ssd {
namespace {

constexpr int kTreeWarps = kTreeThreads / 32;
constexpr float kFix = 281474976710656.0f;  // 2^48

namespace cg = cooperative_groups;

struct TreeSmem {
  float2 tab[64];
  float2 c2;
  // every CTA's pass sum (by pass parity), fixed-point total and last
  // positive index (the draw), pushed by that CTA into every CTA of the
  // cluster before a cluster barrier: remote stores, then local reads
  float2 slot[2][SSD_TREE_MAX_CLUSTER];
  long long ctot[SSD_TREE_MAX_CLUSTER];
  int clast_all[SSD_TREE_MAX_CLUSTER];
  int clast;                                 // this CTA's last positive index
  int res;                                   // rank 0: the drawn token (-1: none)
  int par[kMaxTreeNodes], tok[kMaxTreeNodes];
  float m[2 * kMaxTreeNodes];                // row maxima: target rows, then draft rows
  float sh[2 * kMaxTreeNodes], sl[2 * kMaxTreeNodes];  // row sums (float pairs)
  int am[2 * kMaxTreeNodes];                 // lowest index of the maximum
  int flags, bad;
  float rh[kTreeWarps], rl[kTreeWarps];      // block sums
  long long scan[kTreeWarps];
  int accept;                                // thread 0's decision
  float2 ez[kMaxTreeNodes], ed[kMaxTreeNodes];  // node j's e_z, e_d at its parent's rows
  float u[kMaxTreeNodes];                    // node j's acceptance uniform
};

// Block-wide inclusive scan of int64 (exact).  *total gets the block total.
__device__ __forceinline__ long long tree_scan_i64(long long v, long long* sm, long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) sm[warp] = v;
  __syncthreads();
  long long off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kTreeWarps; ++w) {
    const long long s = sm[w];
    if (w < warp) off += s;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return v + off;
}

// Block sum of float pairs (every thread gets the total).
__device__ __forceinline__ void tree_sum_df(float h, float l, TreeSmem& sm, float& th,
                                            float& tl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float oh = __shfl_xor_sync(kFull, h, o);
    const float ol = __shfl_xor_sync(kFull, l, o);
    df_acc(h, l, oh, ol);
  }
  if (lane == 0) {
    sm.rh[warp] = h;
    sm.rl[warp] = l;
  }
  __syncthreads();
  th = 0.f;
  tl = 0.f;
  for (int w = 0; w < kTreeWarps; ++w) df_acc(th, tl, sm.rh[w], sm.rl[w]);
  __syncthreads();
}

// max(0, e_z - rho e_d) from the two exponentials (float pairs); false when
// the weight is zero.
__device__ __forceinline__ bool tree_w(float ah, float al, float bh, float bl, float rho_h,
                                       float rho_l, float& wh, float& wl) {
  float rbh, rbl;
  df_mul(rho_h, rho_l, bh, bl, rbh, rbl);
  df_sub(ah, al, rbh, rbl, wh, wl);
  return wh > 0.f;
}

// The two exponentials of one element: e_z = 2^((z - m_z) c2), e_d likewise.
__device__ __forceinline__ void tree_exps(float z, float d, float mz, float md, float2 c2,
                                          const float2* tab, float4& e) {
  float xh, xl;
  arg_df(z, mz, c2.x, c2.y, xh, xl);
  exp2_df(xh, xl, tab, e.x, e.y);
  arg_df(d, md, c2.x, c2.y, xh, xl);
  exp2_df(xh, xl, tab, e.z, e.w);
}

// The draw weight of one element: max(0, e_z - rho e_d) as a float pair
// (e_z alone when rho == 0).  Returns false when the weight is zero.
__device__ __forceinline__ bool tree_weight(float z, float d, float mz, float md, float2 c2,
                                            float rho_h, float rho_l, const float2* tab,
                                            float& wh, float& wl) {
  if (rho_h == 0.f) {
    float xh, xl;
    arg_df(z, mz, c2.x, c2.y, xh, xl);
    exp2_df(xh, xl, tab, wh, wl);
    return wh > 0.f;
  }
  float4 e;
  tree_exps(z, d, mz, md, c2, tab, e);
  return tree_w(e.x, e.y, e.z, e.w, rho_h, rho_l, wh, wl);
}

// Passes over a node's rows.  kCompute: weights from the logits (rho == 0:
// e_z alone); kStore: the same with rho != 0, keeping each element's two
// exponentials in the tree's cache row; kCached: later passes at the same
// node read them back (a load and a few double-float operations instead of
// two exponentials).  Every thread reads back only what it wrote; element
// lo + i of thread g sits at cache[i * nt + g] (nt threads per tree), so a
// warp's accesses are 512 contiguous bytes.
constexpr int kCompute = 0, kStore = 1, kCached = 2;

// One pass over the node's rows: this thread's compensated sum of the
// weights of its range and the last index with a positive weight (-1).
template <typename Tag, bool VEC>
__device__ __forceinline__ void tree_pass(const typename Tag::Elem* zr,
                                          const typename Tag::Elem* dr, int lo, int hi, float mz,
                                          float md, float2 c2, float rho_h, float rho_l,
                                          const float2* tab, float4* cache, int nt, int mode,
                                          float& acc, float& comp, int& last) {
  acc = 0.f;
  comp = 0.f;
  last = -1;
  if (mode == kCached) {
    for (int v = lo; v < hi; ++v) {
      const float4 e = cache[static_cast<int64_t>(v - lo) * nt];
      float wh, wl;
      if (tree_w(e.x, e.y, e.z, e.w, rho_h, rho_l, wh, wl)) {
        comp_acc(acc, comp, wh, wl);
        last = v;
      }
    }
    return;
  }
  if (mode == kStore) {
    if (VEC) {
      constexpr int kV = Tag::kVec;
      for (int v = lo; v < hi; v += kV) {
        float z[8], d[8];
        Tag::loadv_cached(zr + v, z);
        Tag::loadv_cached(dr + v, d);
#pragma unroll
        for (int e = 0; e < kV; ++e) {
          float4 x;
          tree_exps(z[e], d[e], mz, md, c2, tab, x);
          cache[static_cast<int64_t>(v + e - lo) * nt] = x;
          float wh, wl;
          if (tree_w(x.x, x.y, x.z, x.w, rho_h, rho_l, wh, wl)) {
            comp_acc(acc, comp, wh, wl);
            last = v + e;
          }
        }
      }
    } else {
      for (int v = lo; v < hi; ++v) {
        float4 x;
        tree_exps(Tag::load1(zr + v), Tag::load1(dr + v), mz, md, c2, tab, x);
        cache[static_cast<int64_t>(v - lo) * nt] = x;
        float wh, wl;
        if (tree_w(x.x, x.y, x.z, x.w, rho_h, rho_l, wh, wl)) {
          comp_acc(acc, comp, wh, wl);
          last = v;
        }
      }
    }
    return;
  }
  const bool use_d = rho_h != 0.f;
  if (VEC) {
    constexpr int kV = Tag::kVec;
    for (int v = lo; v < hi; v += kV) {
      float z[8], d[8];
      Tag::loadv_cached(zr + v, z);
      if (use_d) Tag::loadv_cached(dr + v, d);
#pragma unroll
      for (int e = 0; e < kV; ++e) {
        float wh, wl;
        if (tree_weight(z[e], use_d ? d[e] : 0.f, mz, md, c2, rho_h, rho_l, tab, wh, wl)) {
          comp_acc(acc, comp, wh, wl);
          last = v + e;
        }
      }
    }
  } else {
    for (int v = lo; v < hi; ++v) {
      float wh, wl;
      const float d = use_d ? Tag::load1(dr + v) : 0.f;
      if (tree_weight(Tag::load1(zr + v), d, mz, md, c2, rho_h, rho_l, tab, wh, wl)) {
        comp_acc(acc, comp, wh, wl);
        last = v;
      }
    }
  }
}

// Cluster total of the CTAs' sums (h, l; every thread holds its CTA's):
// threads 0 .. cs-1 push the sum into slot [parity][rank] of every CTA,
// cluster barrier, then every CTA adds the cs local copies in rank order
// (the same bits everywhere).  Slots alternate by pass parity, so a CTA
// rewrites another's slot only after the barrier that follows that CTA's
// reads.
__device__ __forceinline__ void cluster_total(cg::cluster_group& cl, TreeSmem& sm, int& parity,
                                              float h, float l, float& th, float& tl) {
  const int cs = static_cast<int>(cl.num_blocks());
  const int rank = static_cast<int>(cl.block_rank());
  if (static_cast<int>(threadIdx.x) < cs)
    *cl.map_shared_rank(&sm.slot[parity][rank], static_cast<int>(threadIdx.x)) = make_float2(h, l);
  cl.sync();
  th = 0.f;
  tl = 0.f;
  for (int r = 0; r < cs; ++r) {
    const float2 v = sm.slot[parity][r];
    df_acc(th, tl, v.x, v.y);
  }
  parity ^= 1;
}

template <typename Tag, bool VEC>
__global__ void __launch_bounds__(kTreeThreads) tree_walk_kernel(TreeParams p) {
  using Elem = typename Tag::Elem;
  __shared__ TreeSmem sm;
  cg::cluster_group cl = cg::this_cluster();
  const int cs = static_cast<int>(cl.num_blocks()), rank = static_cast<int>(cl.block_rank());
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x / cs, N = p.N;
  const bool lead = rank == 0 && tid == 0;   // writes the outputs
  // the cluster barrier's first phase: arrive now, wait before the first
  // store into another CTA's shared memory (every CTA has then started)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  load_exp2_table(sm.tab);
  if (tid < N) {
    sm.par[tid] = p.parent[static_cast<int64_t>(b) * N + tid];
    sm.tok[tid] = p.tok[static_cast<int64_t>(b) * N + tid];
  }
  if (tid == 0) {
    sm.flags = 0;
    sm.bad = 0;
    sm.res = -1;
  }
  const float T = p.T[b];
  const bool t_bad = !(T >= 0.f);  // NaN or negative
  const bool greedy = T == 0.f;
  const float2 c2 = cta_temp_coeff(greedy || t_bad ? 1.f : T, &sm.c2);  // holds a barrier
  if (tid < N) {
    const int pj = sm.par[tid], tj = sm.tok[tid];
    const bool ok = tid == 0 ? pj == -1 : (pj >= 0 && pj < tid && tj >= 0 && tj < p.V);
    if (!ok) atomicOr(&sm.bad, 1);
  }
  // merged statistics of the N target rows and of the draft rows of nodes
  // with children (one warp per row, in every CTA); a leaf's draft row was
  // not read
  const bool do_exp = !greedy && !t_bad;
  for (int r = warp; r < 2 * N; r += kTreeWarps) {
    if (r >= N) {
      bool kid = false;
      for (int c = r - N + 1 + lane; c < N; c += 32) kid |= sm.par[c] == r - N;
      if (!__any_sync(kFull, kid)) {
        if (lane == 0) {
          sm.m[r] = -INFINITY;
          sm.am[r] = kIdxNone;
          sm.sh[r] = 0.f;
          sm.sl[r] = 0.f;
        }
        continue;
      }
    }
    RowStat rs;
    float h, l;
    merge_row(p.part + (static_cast<int64_t>(b) * p.Rp + r) * p.C, p.C, c2.x, c2.y, do_exp,
              sm.tab, rs, h, l);
    if (lane == 0) {
      sm.m[r] = rs.m;
      sm.am[r] = rs.argmax;
      sm.sh[r] = h;
      sm.sl[r] = l;
      if (rs.flags) atomicOr(&sm.flags, rs.flags);
    }
  }
  int32_t* out_tok = p.out_tok + static_cast<int64_t>(b) * N;
  int32_t* out_node = p.out_node ? p.out_node + static_cast<int64_t>(b) * N : nullptr;
  if (rank == 0)
    for (int i = tid; i < N; i += kTreeThreads) {
      out_tok[i] = -1;
      if (out_node) out_node[i] = -1;
    }
  __syncthreads();
  if (t_bad || sm.bad || sm.flags) {  // sentinels, in the order of the oracle's checks
    if (lead) {
      p.accept_len[b] = (!t_bad && sm.bad) ? -2 : -1;
      atomicOr(p.err, t_bad ? 0x1 : (sm.bad ? 0x4 : 0x2));
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    return;  // every CTA of the cluster leaves here (same data, same test)
  }
  if (greedy) {  // first child carrying the argmax, then the argmax
    if (lead) {
      int cur = 0, depth = 0;
      for (;;) {
        const int a = sm.am[cur];
        int nxt = 0;
        for (int c = cur + 1; c < N; ++c)
          if (sm.par[c] == cur && sm.tok[c] == a) {
            nxt = c;
            break;
          }
        out_tok[depth] = a;
        if (!nxt) break;
        if (out_node) out_node[depth] = nxt;
        ++depth;
        cur = nxt;
      }
      p.accept_len[b] = depth;
    }
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    return;  // every CTA of the cluster leaves here (T is the row's)
  }

  // every child's e_z(x) and e_d(x) at its parent's rows, gathered in
  // parallel (one thread per node) so that each decision is a few
  // double-float operations of thread 0
  if (tid > 0 && tid < N) {
    const int pj = sm.par[tid], x = sm.tok[tid];
    const Elem* zr = static_cast<const Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb +
                     static_cast<int64_t>(pj) * p.V;
    const Elem* dr = static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db +
                     static_cast<int64_t>(pj) * p.V;
    float xh, xl, h, l;
    arg_df(Tag::load1(zr + x), sm.m[pj], c2.x, c2.y, xh, xl);
    exp2_df(xh, xl, sm.tab, h, l);
    sm.ez[tid] = make_float2(h, l);
    arg_df(Tag::load1(dr + x), sm.m[N + pj], c2.x, c2.y, xh, xl);
    exp2_df(xh, xl, sm.tab, h, l);
    sm.ed[tid] = make_float2(h, l);
    sm.u[tid] = p.u_acc[static_cast<int64_t>(b) * N + tid];
  }
  __syncthreads();

  const int V = p.V;
  int E = (V + cs * kTreeThreads - 1) / (cs * kTreeThreads);
  E = (E + 7) / 8 * 8;
  const int g = rank * kTreeThreads + tid;
  const int lo = static_cast<int>(min(static_cast<long long>(V), static_cast<long long>(g) * E));
  const int hi = min(V, lo + E);
  const Elem* Zb = static_cast<const Elem*>(p.Z) + static_cast<int64_t>(b) * p.zb;
  const Elem* Db = static_cast<const Elem*>(p.D) + static_cast<int64_t>(b) * p.db;
  int cur = 0, depth = 0, c = 1, parity = 0;
  float rho_h = 0.f, rho_l = 0.f;           // rho of the current residual
  float W_h = sm.sh[0], W_l = sm.sl[0];     // its scaled mass (S_z at a fresh node)
  bool ready = false;                       // acc/comp/last hold a pass for (rho, W)
  float acc = 0.f, comp = 0.f;
  int last = -1;
  const int nt = cs * kTreeThreads;         // E * nt <= V + 8 nt <= V + kTreeCachePad
  const bool use_cache = p.cache_stride > 0;
  float4* cache = use_cache ? p.cache + static_cast<int64_t>(b) * p.cache_stride + g : nullptr;
  int cached = -1;                          // the node whose exponentials the cache holds
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  for (;;) {
    while (c < N && sm.par[c] != cur) ++c;
    if (c >= N) break;  // the children of cur are exhausted
    const Elem* zr = Zb + static_cast<int64_t>(cur) * V;
    const Elem* dr = Db + static_cast<int64_t>(cur) * V;
    const float mz = sm.m[cur], md = sm.m[N + cur];
    if (tid == 0) {
      const float ezh = sm.ez[c].x, ezl = sm.ez[c].y, edh = sm.ed[c].x, edl = sm.ed[c].y;
      float wh, wl, th, tl, lh, ll, rh, rl, dh, dl;
      df_mul(rho_h, rho_l, edh, edl, th, tl);
      df_sub(ezh, ezl, th, tl, wh, wl);          // w(x) = e_z - rho e_d
      int ok = 0;
      if (wh > 0.f) {
        df_mul(W_h, W_l, edh, edl, th, tl);
        df_mul(sm.u[c], 0.f, th, tl, lh, ll);                                   // u Wsc e_d
        df_mul(sm.sh[N + cur], sm.sl[N + cur], wh, wl, rh, rl);                 // S_d w(x)
        df_sub(rh, rl, lh, ll, dh, dl);
        ok = dh > 0.f;
      }
      sm.accept = ok;
    }
    __syncthreads();
    const bool accepted = sm.accept != 0;
    __syncthreads();
    if (accepted) {
      if (lead) {
        out_tok[depth] = sm.tok[c];
        if (out_node) out_node[depth] = c;
      }
      ++depth;
      cur = c;
      c = cur + 1;
      rho_h = rho_l = 0.f;
      W_h = sm.sh[cur];
      W_l = sm.sl[cur];
      ready = false;
      continue;
    }
    // rejected: rho' = rho + Wsc / S_d, Wsc' = sum_v max(0, e_z - rho' e_d)
    float ih, il, qh, ql, nh, nl;
    df_recip(sm.sh[N + cur], sm.sl[N + cur], ih, il);
    df_mul(W_h, W_l, ih, il, qh, ql);
    nh = rho_h;
    nl = rho_l;
    df_acc(nh, nl, qh, ql);
    float a2, c2p;
    int l2;
    tree_pass<Tag, VEC>(zr, dr, lo, hi, mz, md, c2, nh, nl, sm.tab, cache, nt,
                        !use_cache ? kCompute : (cached == cur ? kCached : kStore), a2, c2p,
                        l2);
    cached = cur;
    float sh2, sl2, Bh, Bl, Th, Tl;
    two_sum(a2, c2p, sh2, sl2);
    tree_sum_df(sh2, sl2, sm, Bh, Bl);
    cluster_total(cl, sm, parity, Bh, Bl, Th, Tl);
    if (Th > 0.f) {
      rho_h = nh;
      rho_l = nl;
      W_h = Th;
      W_l = Tl;
      acc = a2;
      comp = c2p;
      last = l2;
      ready = true;
    }  // else: an all-zero residual leaves r unchanged
    ++c;
  }
  // the final token: inverse CDF of the weights max(0, e_z - rho e_d)
  const Elem* zr = Zb + static_cast<int64_t>(cur) * V;
  const Elem* dr = Db + static_cast<int64_t>(cur) * V;
  const float mz = sm.m[cur], md = sm.m[N + cur];
  const bool from_cache = use_cache && rho_h != 0.f && cached == cur;
  if (!ready) {
    tree_pass<Tag, VEC>(zr, dr, lo, hi, mz, md, c2, rho_h, rho_l, sm.tab, cache, nt,
                        from_cache ? kCached : kCompute, acc, comp, last);
    float sh2, sl2, Bh, Bl;
    two_sum(acc, comp, sh2, sl2);
    tree_sum_df(sh2, sl2, sm, Bh, Bl);
    cluster_total(cl, sm, parity, Bh, Bl, W_h, W_l);
  }
  // per-thread sums in units of 2^-48 of the total
  float rwh, rwl, fh, fl;
  df_recip(W_h, W_l, rwh, rwl);
  {
    float h, l;
    two_sum(acc, comp, h, l);
    df_mul(h, l, rwh, rwl, fh, fl);
  }
  const long long mine = df_to_fix(fh, fl, kFix);
  long long cta_total;
  const long long incl_cta = tree_scan_i64(mine, sm.scan, &cta_total);
  if (tid == 0) sm.clast = -1;
  __syncthreads();
  if (last >= 0) atomicMax(&sm.clast, last);
  __syncthreads();
  if (tid < cs) {  // this CTA's total and last positive index into every CTA
    TreeSmem* dst = cl.map_shared_rank(&sm, tid);
    dst->ctot[rank] = cta_total;
    dst->clast_all[rank] = sm.clast;
  }
  cl.sync();
  long long before = 0;                     // the fixed-point totals of lower ranks
  int clast = -1;
  for (int r = 0; r < cs; ++r) {
    if (r < rank) before += sm.ctot[r];
    clast = max(clast, sm.clast_all[r]);
  }
  const long long incl = before + incl_cta;
  const float u = p.u_smp[b];
  const long long target = __float2ll_rd(__fmul_rn(u, kFix));
  if (incl > target && incl - mine <= target) {  // one thread of the cluster
    long long cum = incl - mine;
    int tok = last;
    for (int v = lo; v < hi; ++v) {  // walk the range in the order of the pass
      float wh, wl;
      bool pos;
      if (from_cache) {
        const float4 e = cache[static_cast<int64_t>(v - lo) * nt];
        pos = tree_w(e.x, e.y, e.z, e.w, rho_h, rho_l, wh, wl);
      } else {
        const float d = rho_h != 0.f ? Tag::load1(dr + v) : 0.f;
        pos = tree_weight(Tag::load1(zr + v), d, mz, md, c2, rho_h, rho_l, sm.tab, wh, wl);
      }
      if (pos) {
        float ph, pl;
        df_mul(wh, wl, rwh, rwl, ph, pl);
        cum += df_to_fix(ph, pl, kFix);
        if (cum > target) {
          tok = v;
          break;
        }
      }
    }
    *cl.map_shared_rank(&sm.res, 0) = tok;
  }
  cl.sync();  // the token is in rank 0's shared memory; no remote access follows
  if (lead) {
    out_tok[depth] = sm.res >= 0 ? sm.res : clast;  // rounding left no crossing: last positive
    p.accept_len[b] = depth;
  }
}

}  // namespace

// Cluster size per batch row: about SSD_TREE_CTAS_PER_SM 512-thread CTAs
// per SM over the grid (two are resident at a time), at most
// SSD_TREE_MAX_CLUSTER.  Oversubscribing balances the trees' unequal pass
// counts: measured walk times at B = 64 / 128 / 512 were 0.218 / 0.403 /
// 1.107 ms with 2 per SM, 0.177 / 0.332 / 0.923 ms with 8.
static_assert(8 * SSD_TREE_MAX_CLUSTER * kTreeThreads <= kTreeCachePad,
              "the tree cache rows must cover the largest cluster's thread ranges");
#ifndef SSD_TREE_CTAS_PER_SM
#define SSD_TREE_CTAS_PER_SM 8
#endif

template <typename Tag, bool VEC>
static cudaError_t launch_tree_t(const TreeParams& p, int cs, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.B) * cs, 1, 1);
  cfg.blockDim = dim3(kTreeThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tree_walk_kernel<Tag, VEC>, p);
}

cudaError_t launch_tree_walk(const TreeParams& p, int dtype, bool vec, cudaStream_t s) {
  if (p.B <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 1;
  int cs = 1;
  while (cs < SSD_TREE_MAX_CLUSTER &&
         static_cast<long long>(p.B) * cs * 2 <= static_cast<long long>(SSD_TREE_CTAS_PER_SM) * sms)
    cs *= 2;
  for (;;) {
    cudaError_t e;
    if (dtype == 1)
      e = vec ? launch_tree_t<BF16Tag, true>(p, cs, s) : launch_tree_t<BF16Tag, false>(p, cs, s);
    else
      e = vec ? launch_tree_t<F32Tag, true>(p, cs, s) : launch_tree_t<F32Tag, false>(p, cs, s);
    if (e == cudaSuccess || cs == 1) return e;
    (void)cudaGetLastError();  // a cluster this size cannot be placed: halve it
    cs /= 2;
  }
}

}  // namespace ssd
