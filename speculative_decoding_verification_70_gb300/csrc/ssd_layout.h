// ssd_layout.h -- workspace layout and kernel parameter blocks shared by the
// host entry points and the kernels of the verify-and-recover library.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace ssd {

constexpr int kMaxMask = 64;        // masked tokens per (b, position)
constexpr int kAmbCap = 8192;       // ambiguous-sign elements kept per row (draw), at most
                                    // V (amb_cap(V) below)
constexpr int kMaxGridBatch = 65535;  // batch rows per launch (grid y / z limit)
constexpr int kMaxChunkBytes = 32768;  // a chunk fits one shared-memory stage
constexpr int kDrawThreads = 256;      // threads per CTA of the draw kernels

// Partial statistics of one chunk of one logit row.
struct PartStat {
  float m;    // chunk maximum (NaN-free; -inf if the chunk is all -inf/NaN)
  float s;    // sum over the chunk of 2^((z - m) * c), 0 for greedy rows
  int idx;    // lowest index attaining m
  int flags;  // bit 0: a NaN was seen
};

struct TopEntry {
  float v;
  int i;  // 0x7fffffff marks an empty slot
};

// Best Gumbel-perturbed logit of a chunk (draft-side sampling).
struct GumbelPart {
  float y;    // max over the chunk of z / T - ln(-ln u)
  int idx;    // lowest index attaining it (0x7fffffff: none)
};

// Merged statistics of one logit row.
struct RowStat {
  double S;    // sum over the row of 2^((z - m) * c)
  float m;
  int argmax;
  int flags;   // bit 0: NaN seen; bit 1: row invalid for its use
  int pad;
};

enum ResidualMode : int { kModeNone = 0, kModeResidual = 1, kModeTarget = 2 };

struct BState {
  int n;        // accepted prefix length (or sentinel)
  int mode;     // ResidualMode
  float c_hi;   // log2(e) / T as a float pair (0 for greedy rows)
  float c_lo;
  float rho;    // S_z / S_d of rows n from the streaming statistics (residual mode)
  int pad0, pad1, pad2;
};

struct Chunking {
  int C;   // chunks per row
  int CH;  // elements per chunk (multiple of 8), last chunk ragged
  int E;   // elements per thread in the recovery kernels (multiple of 8)
};

// The whole verify call of a small batch as one cooperative kernel
// (ssd_step.cu): the statistics pass, the row merges and forks, acceptance,
// the two exact passes of the draw over rows n and the select, separated by
// grid-wide barriers.  At most kStepMaxB batch rows (one warp of a CTA per
// row at acceptance) and kStepMaxGrid CTAs.
constexpr int kStepMaxB = 8;
constexpr int kStepMaxGrid = 2048;
constexpr int kStepSubBars = 8;

// Merged statistics of one row as the step kernel's acceptance reads them.
struct StepRow {
  float m, sh, sl;   // maximum, S as a float pair
  int argmax, flags;
  int pad[3];
};

// Grid barrier words (each on its own 128-byte line): eight arrival
// sub-counters, the top counter, the generation the waiters poll, the exit
// ticket and the abort word.  All zero between calls.
struct StepBar {
  unsigned sub[kStepSubBars][32];
  unsigned top[32];
  unsigned gen[32];
  unsigned exit_[32];
  unsigned abort_[32];
};

// Workspace of the verify / fork / residual calls.
struct WsLayout {
  size_t err, part, topk, rowstat, bstate, rnorm, rthr, racc, amb_cnt, amb_idx, gpart, total;
  size_t srows, scta, sbar;   // the step kernel (batches of at most kStepMaxB rows)
  int B, R, Pf, f;
  Chunking ch;    // the statistics pass
  Chunking dch;   // the draw's passes
};

struct StatsParams {
  const void* Z;       // target logits (may be null when Pz == 0)
  int64_t zb;          // batch stride (elements)
  int Pz;              // target rows per batch row
  const void* D;       // draft logits
  int64_t db;
  int Pds;             // draft rows needing softmax statistics
  int Pdf;             // draft rows needing top-f
  const float* T;      // [B] temperatures (null: no exponentials)
  const int32_t* mask; // [B, Pdf, M]
  int M, f;
  int V, C, CH, R;     // R: rows per batch row
  int Rp;              // row pitch of part[] (>= R)
  int r0;              // first row of this launch
  int b0;              // first batch row of this launch (grids hold <= 65535)
  int G;               // chunks per CTA in the plain statistics kernel
  PartStat* part;      // [B][Rp][C]
  TopEntry* topk;      // [B][Pdf][C][f]
  int* err;            // device error word
  // draft-side sampling (draft_kernel only)
  GumbelPart* gpart;   // [B][Pf][C]
  uint32_t seed_lo, seed_hi, offset;
  uint32_t rk0[10], rk1[10];  // the generator's round keys (key schedule of the seed)
  int Pf;              // row pitch of gpart[] and topk[] (k + 1)
  // token trees: draft row j is read only if node j has a child (null: all)
  const int32_t* tree_parent;  // [B][tree_N]
  int tree_N;
  // the SSD round step's cache clear, done by the statistics kernel's CTAs
  // (the insert runs in a later kernel): clr_n slots of keys / winner words
  unsigned long long* clr_keys;
  unsigned long long* clr_winner;
  int clr_n;
};

struct FinalizeParams {
  const void* Z; int64_t zb; int Pz;
  const void* D; int64_t db; int Pds; int Pdf;
  int dtype;           // 0 f32, 1 bf16
  int B, k, V, C, R, f;
  int Rp;              // row pitch of part[] and rowstat[]
  const float* T;
  const int32_t* x;
  const float* u_acc;
  int32_t* accept_len;
  float* p_at_x;
  float* q_at_x;
  int32_t* out_tok;    // may be null
  int32_t* fork_tok;   // may be null
  float* fork_logit;
  const int32_t* fanout;  // [Pdf] tokens kept per position (null: f everywhere)
  const PartStat* part;
  const TopEntry* topk;
  RowStat* rowstat;    // [B][Rp]
  BState* bstate;      // [B]
  int* err;
  int* amb_cnt;        // [B], zeroed here for the draw
};

struct CacheView {
  unsigned long long* keys;
  unsigned long long* winner;
  int32_t* payload;
  int* err;                  // device error word
  unsigned long long* calls; // inserts completed so far (device counter)
  unsigned* done;            // finished CTAs of the running insert's write kernel
  int capacity;
  int depth;
};

struct ResidualParams {
  const void* Z; int64_t zb; int Pz;
  const void* D; int64_t db;
  int V, C, CH, E, R, k;  // R: row pitch of rowstat[]
  const float* T;
  const float* u_smp;
  const RowStat* rowstat;
  const BState* bstate;
  long long* rnorm;    // [B][C][2]
  long long* rthr;     // [B][C][3][kThreads]: each norm-pass thread's S_z, A, B
  long long* racc;     // [B][C][2]
  int* amb_cnt;        // [B]
  int* amb_idx;        // [B][amb_cap]
  int amb_cap;         // ambiguous elements kept per row
  int b0;              // first batch row of this launch (grids hold <= 65535)
  int B;               // batch rows of this call (row-strided kernels)
  int32_t* out_tok;    // [B][k+1]
  // the SSD round step: the select kernel looks up each row's realised
  // outcome (b, n, out_tok[b][n]) once its token is final
  int lookup;
  CacheView cache;
  int32_t* hit;        // [B]
  int32_t* tok_out;    // [B][depth]
};

// The verify step of a small batch after the statistics pass in one kernel
// (ssd_chain.cu): one cluster of up to kChainMaxCluster CTAs per batch row
// does the finalisation, the draw and, in the SSD round step, the cache
// insert of the row's forks and the lookup of its outcome.
constexpr int kChainMaxCluster = 16;

struct ChainParams {
  FinalizeParams f;
  const float* u_smp;      // [B] or null (no draw)
  int E;                   // elements per thread of the cluster's draw pass (multiple of 8)
  int cache_on;            // SSD round step
  CacheView cache;
  const int32_t* payload;  // [B][k+1][f][depth]
  int32_t* hit;            // [B]
  int32_t* tok_out;        // [B][depth]
};

struct StepParams {
  StatsParams sp;          // the statistics pass (one chunk per unit)
  FinalizeParams f;        // merges, acceptance, forks, outputs
  const float* u_smp;      // [B] or null (no draw)
  int E;                   // elements per thread of the draw passes (multiple of 8)
  int units;               // statistics units B * sp.R * C, chunk fastest
  StepRow* rows;           // [B][f.R]
  long long* cta;          // [3][B][kStepMaxGrid]: per-CTA S_z, S_d and draw mass
  StepBar* bar;
  int cache_on;            // SSD round step
  int cache_clear;         // clear the cache first
  CacheView cache;
  const int32_t* payload;  // [B][k+1][f][depth]
  int32_t* hit;            // [B]
  int32_t* tok_out;        // [B][depth]
};

// Token-tree verification (ssd_verify_tree).
constexpr int kMaxTreeNodes = 64;

constexpr int kTreeCacheMinV = 32768;

// The tree walk runs kTreeThreads threads per CTA in clusters of at most
// SSD_TREE_MAX_CLUSTER CTAs.  A pass gives each of the cluster's nt threads a
// range of E = ceil(V / nt) elements rounded up to a multiple of 8, so the
// ranges cover at most V + 8 nt slots of a tree's cache row: kTreeCachePad is
// that padding for the largest cluster.
constexpr int kTreeThreads = 512;
#ifndef SSD_TREE_MAX_CLUSTER
#define SSD_TREE_MAX_CLUSTER 8
#endif
constexpr int kTreeCachePad = 8 * SSD_TREE_MAX_CLUSTER * kTreeThreads;

struct TreeLayout {
  size_t err, part, cache, cache_stride, total;
  int R;          // rows per batch row: N target, N draft
  Chunking ch;
};

struct TreeParams {
  const void* Z; int64_t zb;
  const void* D; int64_t db;
  int B, N, V, C, Rp;
  const int32_t* parent;   // [B][N]
  const int32_t* tok;      // [B][N]
  const float* T;
  const float* u_acc;      // [B][N]
  const float* u_smp;      // [B]
  const PartStat* part;    // [B][Rp][C]: target rows 0..N-1, draft rows N..2N-1
  int32_t* accept_len;
  int32_t* out_tok;        // [B][N]
  int32_t* out_node;       // [B][N] or null
  int* err;
  float4* cache;           // [B][cache_stride]: e_z, e_d (float pairs) at the node being walked
  int64_t cache_stride;    // 0: no cache (short rows)
};

// Top-k / top-p filtered verify (ssd_verify_topk).
constexpr int kMaxTopK = 32;

struct TopkLayout {
  size_t err, part, lists, total;
  int R;          // rows per batch row: k+1 target, k draft
  Chunking ch;
};

struct TopkParams {
  const void* Z; int64_t zb;
  const void* D; int64_t db;
  int dtype;           // 0 f32, 1 bf16
  int B, k, V, C, CH, R, K, G;
  int b0;              // first batch row of this launch
  const float* T;
  const float* top_p;  // [B] or null (1)
  const int32_t* x;
  const float* u_acc;
  const float* u_smp;  // may be null (no draw)
  int32_t* accept_len;
  float* p_at_x;
  float* q_at_x;
  int32_t* out_tok;
  PartStat* part;      // [B][R][C]
  TopEntry* lists;     // [B][R][C][K]
  int* err;
};

inline TopkLayout make_topk_layout(int B, int k, int V, int K, int esize = 4);

// Filtered verify beyond the in-register lists: K > kMaxTopK (any K up to V)
// and top-p over the whole vocabulary.  Each logit row of a T > 0 batch row
// gets a histogram of x = (m - z) log2(e) / T in kFiltBinsPerUnit bins per
// unit (x >= kFiltBins / kFiltBinsPerUnit in the last bin), a band of bins
// that must hold the cut, and the order keys of the band's tokens.
constexpr int kFiltBins = 1024;
constexpr int kFiltBinsPerUnit = 16;
constexpr int kFiltCand = 2048;       // band tokens kept per row (more: bisection fallback)
constexpr int kFiltMaxV = 1 << 21;    // fixed-point sums of 2^42 units stay below 2^63

// One filtered logit row.  Tokens are ordered by the 64-bit key
// (order-preserving bits of z) << 32 | ~index: key descending is logit
// descending, then index ascending.  Kept tokens are those with key >= thr.
struct FiltRow {
  unsigned long long thr;    // key of the last kept token (0 keeps every token)
  unsigned long long above;  // 2^42 fixed point: exact mass of the tokens in bins < band_lo
  unsigned long long total;  // 2^42 fixed point: exact mass of the row (K >= V only)
  double P;                  // kept mass, sum of 2^((z - m) c) over kept tokens
  float m;                   // row maximum
  float c_hi, c_lo;          // log2(e) / T as a float pair
  int argmax;                // lowest index attaining m
  int flags;                 // bit 0: NaN; bit 1: invalid at T > 0; bit 2: T > 0 (filtered)
  int band_lo, band_hi;      // bins whose tokens are collected
  int cnt_before;            // tokens in bins < band_lo
  int n_cand;                // band tokens seen (above kFiltCand: overflow)
  int keep;                  // kept tokens
  int pad;
};

struct FiltLayout {
  size_t err, part, rows, hcnt, hmass, cand, bstate, rmass, total;
  int R;          // rows per batch row: k+1 target, k draft
  Chunking ch;
};

struct FiltParams {
  const void* Z; int64_t zb;
  const void* D; int64_t db;
  int dtype;           // 0 f32, 1 bf16
  int B, k, V, C, CH, E, R, K, G;
  int b0;              // first batch row of this launch
  int total_mode;      // K >= V: the histogram pass also sums each row's exact mass
  const float* T;
  const float* top_p;  // [B] or null (1)
  const int32_t* x;
  const float* u_acc;
  const float* u_smp;  // may be null (no draw)
  int32_t* accept_len;
  float* p_at_x;
  float* q_at_x;
  int32_t* out_tok;
  PartStat* part;                 // [B][R][C]
  FiltRow* rows;                  // [B][R]
  unsigned* hcnt;                 // [B][R][kFiltBins]
  unsigned long long* hmass;      // [B][R][kFiltBins] bin-scaled fixed point
  unsigned long long* cand;       // [B][R][kFiltCand] order keys
  BState* bstate;                 // [B]
  long long* rmass;               // [B][C]: the draw's chunk masses (2^60 units)
  int* err;
};

// Merge of the draft-side sampling pass: one warp per (b, draft row).
struct DraftParams {
  int B, V, C, Rp, Pz, Pf, row0, rows;
  const float* T;
  const PartStat* part;      // [B][Rp][C], draft row i at Pz + i
  const GumbelPart* gpart;   // [B][Pf][C]
  const TopEntry* topk;      // [B][Pf][C][F1], F1 = f + 1
  int f;                     // forks kept per row (0: none)
  int32_t* x_out;            // [b * x_bstride + (i - row0)]
  int64_t x_bstride;
  int32_t* fork_tok;         // [B][rows][f]
  float* fork_logit;
  int* err;
};

struct SoftmaxParams {
  const void* L;
  int dtype, rows, V, C, CH;
  int r0;              // first row of this launch (grids hold <= 65535 rows)
  const float* T;
  const PartStat* part;
  RowStat* rowstat;
  float* probs;
  float* row_max;
  float* row_sum;
  int32_t* row_argmax;
  int* err;
};

struct PrepParams {
  int B, k;
  const float* T;
  const int32_t* x;
  const int32_t* accept_len;
  const RowStat* rowstat;
  int R;
  BState* bstate;
  int32_t* out_tok;
  int* amb_cnt;
};


struct InsertArgs {
  const int32_t* b;
  const int32_t* pos;
  const int32_t* tok;
  const int32_t* payload;
  const int32_t* fork_tok;
  int P, f;
  int n;
};

struct LookupArgs {
  const int32_t* b;
  const int32_t* pos;
  const int32_t* tok;
  const int32_t* accept_len;
  const int32_t* out_tok;
  int k;
  int n;
  int32_t* hit;
  int32_t* tok_out;
};

// Host-side override of the vocabulary split (ssd_set_split): elements per
// chunk and chunks per statistics CTA, 0 for the policy.  Read when a call
// lays out its workspace and sizes its grids.
struct SplitOverride {
  std::atomic<int> chunk{0};
  std::atomic<int> group{0};
};
inline SplitOverride g_split;

// Chunks per CTA of a streaming pass: the override if set (at most C), else
// the policy's choice.
inline int split_group(int policy, int C) {
  const int g = g_split.group.load(std::memory_order_relaxed);
  if (g <= 0) return policy;
  return g < C ? g : C;
}

// Chunking policy: chunks of at most 32 KB (so that one chunk fits a
// shared-memory stage); for small batches more chunks, enough for about one
// wave of the statistics kernel (912 CTAs: 6 per SM on 152 SMs), but no
// chunk below 2048 elements.  Aiming at 2432 CTAs (16 per SM) gave small
// CTAs whose fixed costs set the time: the verify + fork + cache step with
// one-wave chunks takes 36.8 / 40.8 / 62.9 us at B = 2 / 4 / 8 (ssd_fork
// rows) against 41.0 / 45.3 / 65.7, and 41.1 / 74.0 us at B = 4 / 16
// (qwen_b64 rows) against 46.3 / 76.3.  esize is the logit element size; sizing with esize = 4 gives
// the most chunks, which is what the workspace is sized for.  An override
// of the chunk length is clamped to [ceil(V / 256), 32 KB of elements] (at
// most 256 chunks: the draw's select runs one chunk per thread; at most
// 2^14 elements: its per-chunk fixed-point sums stay below 2^62).
inline Chunking make_chunking(int B, int rows_per_b, int V, int esize) {
  Chunking c;
  long long rows = static_cast<long long>(B) * (rows_per_b > 0 ? rows_per_b : 1);
  const long long max_ch = kMaxChunkBytes / esize;
  long long c0 = (V + max_ch - 1) / max_ch;
  long long want = (912 + rows - 1) / rows;
  long long cap = (V + 2047) / 2048;
  long long C = want < cap ? want : cap;
  if (C < c0) C = c0;
  if (C > 256) C = 256;
  if (C < 1) C = 1;
  // a grid below two waves of the statistics kernel (6 CTAs per SM on 152
  // SMs) is cut to half a wave, three CTAs per SM: there the CTAs' fixed
  // costs (set-up, block reduction, top-f selection) and the sharing of an
  // SM by six CTAs set the pass's time (B = 1, ssd_fork's 16 rows: 28
  // chunks per row, 448 CTAs; the step as a graph 17.9 / 32.3 us at T = 0 /
  // 1 against 18.0 / 32.6 us with the one-wave cut's 57 chunks; llama_sd
  // 22.3 against 22.9 us at T = 1)
  if (rows * C < 1824 && 456 / rows >= c0) C = 456 / rows;
  long long CH = (V + C - 1) / C;
  const int ov = g_split.chunk.load(std::memory_order_relaxed);
  if (ov > 0) {
    const long long lo = (V + 255) / 256;
    CH = ov;
    if (CH < lo) CH = lo;
    if (CH > max_ch) CH = max_ch;
  }
  CH = (CH + 7) / 8 * 8;
  C = (V + CH - 1) / CH;
  c.C = static_cast<int>(C);
  c.CH = static_cast<int>(CH);
  long long E = (CH + 255) / 256;
  E = (E + 7) / 8 * 8;
  c.E = static_cast<int>(E);
  return c;
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Chunking of the draw's passes (norm pass, select): the statistics' chunks,
// or more when B batch rows would give the norm pass too few CTAs to fill
// the GPU (it aims at ~2432 CTAs, 16 per SM, like the statistics policy);
// chunks of at least 2048 elements and at most 256 per row (the select runs
// one chunk per thread).  At B = 64, V = 151936: 38 chunks of 4000 instead of
// the statistics' 10 of 15200.  The per-thread sums of the norm pass take
// 24 bytes per E elements of every row.
inline Chunking make_draw_chunking(int B, int V, const Chunking& st) {
  // batches of at most 16 rows draw in the cluster kernel by default; their
  // batched draw (when selected) keeps the statistics' chunks, and so does
  // their workspace
  if (B <= 16) return st;
  long long want = (2432 + (B > 0 ? B : 1) - 1) / (B > 0 ? B : 1);
  const long long cap = (V + 2047) / 2048;
  if (want > cap) want = cap;
  if (want > 256) want = 256;
  if (want <= st.C) return st;
  Chunking d;
  long long CH = (V + want - 1) / want;
  CH = (CH + 7) / 8 * 8;
  d.C = static_cast<int>((V + CH - 1) / CH);
  d.CH = static_cast<int>(CH);
  long long E = (CH + 255) / 256;
  d.E = static_cast<int>((E + 7) / 8 * 8);
  return d;
}

// Every workspace layout starts with the same header: the device error word
// at offset 0 and the step kernel's barrier words at kWsStepBar.  No other
// region of any layout overlaps the header, so the barrier words, zero when
// the workspace is first zero-filled and left zero by every step kernel,
// stay zero whatever other calls (other shapes, other entry points) use the
// same workspace in between.
constexpr size_t kWsStepBar = 256;
constexpr size_t kWsHeader = (kWsStepBar + sizeof(StepBar) + 255) & ~static_cast<size_t>(255);

// Ambiguous-sign elements kept per row of the draw: a row holds at most V.
inline int amb_cap(int V) { return V < kAmbCap ? V : kAmbCap; }

inline WsLayout make_layout(int B, int k, int V, int f, int esize = 4) {
  WsLayout L;
  L.B = B;
  L.R = 2 * (k + 1);
  L.Pf = k + 1;
  L.f = f;
  L.ch = make_chunking(B, L.R, V, esize);
  const size_t C = static_cast<size_t>(L.ch.C);
  size_t off = 0;
  L.err = off;                      off = kWsHeader;
  // every region but the forked top-f lists is independent of f, so a
  // workspace sized for (B, k, V, f) serves the f = 0 calls too
  L.part = off;                     off = align256(off + sizeof(PartStat) * B * L.R * C);
  L.rowstat = off;                  off = align256(off + sizeof(RowStat) * B * L.R);
  L.bstate = off;                   off = align256(off + sizeof(BState) * B);
  L.dch = make_draw_chunking(B, V, L.ch);
  const size_t Cd = static_cast<size_t>(L.dch.C);
  L.rnorm = off;                    off = align256(off + sizeof(long long) * 2 * B * Cd);
  L.rthr = off;                     off = align256(off + sizeof(long long) * 3 * kDrawThreads * B * Cd);
  L.racc = off;                     off = align256(off + sizeof(long long) * 2 * B * Cd);
  L.amb_cnt = off;                  off = align256(off + sizeof(int) * B);
  L.amb_idx = off;                  off = align256(off + sizeof(int) * B * amb_cap(V));
  L.gpart = off;                    off = align256(off + sizeof(GumbelPart) * B * L.Pf * C);
  const size_t sb = static_cast<size_t>(B < kStepMaxB ? B : kStepMaxB);
  L.sbar = kWsStepBar;
  L.srows = off;                    off = align256(off + sizeof(StepRow) * sb * L.R);
  L.scta = off;                     off = align256(off + sizeof(long long) * 3 * sb * kStepMaxGrid);
  L.topk = off;                     off = align256(off + sizeof(TopEntry) * B * L.Pf * C * (f > 0 ? f : 0));
  L.total = off;
  return L;
}

inline TreeLayout make_tree_layout(int B, int N, int V, int esize = 4) {
  TreeLayout L;
  L.R = 2 * N;
  L.ch = make_chunking(B, L.R, V, esize);
  size_t off = 0;
  L.err = off;                      off = kWsHeader;
  L.part = off;                     off = align256(off + sizeof(PartStat) * B * L.R * L.ch.C);
  // per tree V + kTreeCachePad slots (the walk's thread ranges, padded)
  // when rows are long enough for the cache to pay; none otherwise
  L.cache_stride = V >= kTreeCacheMinV ? static_cast<size_t>(V) + kTreeCachePad : 0;
  L.cache = off;                    off = align256(off + sizeof(float) * 4 * B * L.cache_stride);
  L.total = off;
  return L;
}

inline TopkLayout make_topk_layout(int B, int k, int V, int K, int esize) {
  TopkLayout L;
  L.R = 2 * k + 1;
  L.ch = make_chunking(B, 2 * (k + 1), V, esize);
  const size_t C = static_cast<size_t>(L.ch.C);
  size_t off = 0;
  L.err = off;                      off = kWsHeader;
  L.part = off;                     off = align256(off + sizeof(PartStat) * B * L.R * C);
  L.lists = off;                    off = align256(off + sizeof(TopEntry) * B * L.R * C * K);
  L.total = off;
  return L;
}

inline FiltLayout make_filt_layout(int B, int k, int V, int esize = 4) {
  FiltLayout L;
  L.R = 2 * k + 1;
  L.ch = make_chunking(B, 2 * (k + 1), V, esize);
  const size_t C = static_cast<size_t>(L.ch.C);
  const size_t rows = static_cast<size_t>(B) * L.R;
  size_t off = 0;
  L.err = off;                      off = kWsHeader;
  L.part = off;                     off = align256(off + sizeof(PartStat) * rows * C);
  L.rows = off;                     off = align256(off + sizeof(FiltRow) * rows);
  L.hcnt = off;                     off = align256(off + sizeof(unsigned) * rows * kFiltBins);
  L.hmass = off;                    off = align256(off + sizeof(unsigned long long) * rows * kFiltBins);
  L.cand = off;                     off = align256(off + sizeof(unsigned long long) * rows * kFiltCand);
  L.bstate = off;                   off = align256(off + sizeof(BState) * B);
  L.rmass = off;                    off = align256(off + sizeof(long long) * B * C);
  L.total = off;
  return L;
}

// Workspace of ssd_softmax_temp: rows are "batch rows" with one target row.
inline WsLayout make_softmax_layout(int rows, int V, int esize = 4) {
  WsLayout L;
  L.B = rows;
  L.R = 1;
  L.Pf = 0;
  L.f = 0;
  L.ch = make_chunking(rows, 1, V, esize);
  L.dch = L.ch;
  const size_t C = static_cast<size_t>(L.ch.C);
  size_t off = 0;
  L.err = off;                      off = kWsHeader;
  L.part = off;                     off = align256(off + sizeof(PartStat) * rows * C);
  L.topk = off;
  L.rowstat = off;                  off = align256(off + sizeof(RowStat) * rows);
  L.bstate = off; L.rnorm = off; L.rthr = off; L.racc = off; L.amb_cnt = off; L.amb_idx = off;
  L.gpart = off; L.srows = off; L.scta = off;
  L.sbar = kWsStepBar;
  L.total = off;
  return L;
}

}  // namespace ssd
