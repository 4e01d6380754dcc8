/*
 * ssd.h -- C ABI of the GB300 verify-and-recover library for speculative
 * decoding (SD) and Speculative Speculative Decoding (SSD).
 *
 * Sources (page title, section):
 *   [SUM]  "tanishqkumar/ssd" repository summary (thehardwarestore.ai),
 *          module notes: the sampler mixes greedy and stochastic sampling by
 *          temperature; get_forked_recovery_tokens_from_logits picks tokens by
 *          top-k over logits with masking for cache hits and misses.
 *   [SSD]  "SSD: drafting and verification on separate GPUs, in parallel"
 *          (hysenlabs.com), "What changes in SSD": the target verifies the
 *          draft in one forward pass; the method is exact; the drafter
 *          pre-speculates likely outcomes and a correct guess is returned at
 *          once; the roadmap's speculation cache.
 *   [SPS]  speculative-sampling project summary (sourcepulse.org 1842340),
 *          "How It Works": accept correct tokens, regenerate from the point of
 *          divergence; Google's and DeepMind's algorithms.
 *   [LKM]  the rule those algorithms share (Leviathan et al. 2023, Chen et
 *          al. 2023): accept x_i with probability min(1, p_i(x_i)/q_i(x_i));
 *          at the first rejection n draw from norm(max(0, p_n - q_n)); after
 *          k accepts draw the bonus token from p_k.
 *
 * Conventions shared by every call:
 *   - Tensor arguments are DEVICE pointers owned by the caller, unless a
 *     parameter says "host".  Nothing is allocated per call; scratch comes
 *     from a caller-supplied workspace (ssd_workspace_bytes) or from a
 *     speculation cache made once by ssd_spec_cache_create.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and the call returns after enqueueing.
 *   - Logits are row-major: row (b, i) of a [B, P, V] tensor starts at
 *     element b*bstride + i*V.  dtype is SSD_F32 or SSD_BF16; bf16 is widened
 *     to fp32 exactly before any arithmetic.
 *   - Every call returns an ssd_status; no call aborts or throws.  Argument
 *     errors are found on the host before anything is enqueued.  Errors in
 *     the DATA (invalid temperature, NaN logits, out-of-range tokens, a full
 *     cache) become per-row sentinels plus bits in a device error word, read
 *     by ssd_get_device_error.
 *   - Pointers need 4-byte alignment; logits, when the base pointer, V and
 *     bstride all give 16-byte aligned rows, are read with 16-byte vector
 *     loads, otherwise with scalar loads.
 *   - A workspace must be zero-filled once before its first use (cudaMemset
 *     or ssd_workspace_init); the calls keep it consistent afterwards.
 *   - Calls that share a workspace must not overlap on the GPU.
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ssd_stream_t; /* same type as cudaStream_t */

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,
    SSD_ERR_UNSUPPORTED_DTYPE = 2,
    SSD_ERR_CUDA = 3,
    SSD_ERR_CACHE_FULL = 4,
    SSD_ERR_TIMEOUT = 5,
    SSD_ERR_WORKSPACE = 6
} ssd_status;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* Bits of the device error word (ssd_get_device_error). */
#define SSD_DEVERR_BAD_TEMPERATURE 0x1 /* T < 0 or NaN: row sentinel -1   */
#define SSD_DEVERR_BAD_LOGITS 0x2      /* NaN (or +inf / all -inf at T>0) */
#define SSD_DEVERR_BAD_TOKEN 0x4       /* draft token outside [0, V): -2  */
#define SSD_DEVERR_CACHE_FULL 0x8      /* insert found no free slot       */
#define SSD_DEVERR_TIMEOUT 0x10        /* a bounded device wait ran out   */
#define SSD_DEVERR_FILTER_BAND 0x20    /* a filtered row's cut fell outside its collected
                                          bins; it was cut by bisection (results exact) */

/* Sentinels written to accept_len. */
#define SSD_ROW_INVALID (-1)
#define SSD_ROW_BAD_TOKEN (-2)

/* Limits checked on the host. */
#define SSD_MAX_K 31   /* draft length: one warp ballot holds k flags */
#define SSD_MAX_F 16   /* forked recovery fan-out                    */
#define SSD_MAX_M 64   /* masked tokens per (b, position)            */
#define SSD_MAX_TREE_NODES 64  /* nodes of one draft tree              */

SSD_API const char *ssd_status_string(ssd_status s);

/* Library version (major*10000 + minor*100 + patch). */
SSD_API int ssd_version(void);

/*
 * Streams, graphs, batch size.  Every call enqueues work on the caller's
 * stream and returns: no device allocation, no host synchronisation (except
 * the error-word reads, which say so).  The verify calls (all but
 * ssd_verify_noalloc) run the target-row and draft-row statistics on two
 * internal streams forked from and joined back to the caller's stream by
 * events (the draft-row stream at the device's greatest priority), and the
 * SSD round step inserts the forks into the cache on a third one, also at
 * the greatest priority, beside the draw; the streams and events are
 * created on the first such call on a device.  Calls can therefore be captured into a CUDA
 * graph (make one verify call on the device before capturing).  B may exceed
 * 65535: kernels launch in grids of 65535 batch rows.
 */

/*
 * Workspace bytes for ssd_verify / ssd_verify_fork / ssd_sample_residual /
 * ssd_forked_recovery on batch B, draft length k, vocabulary V and fan-out
 * f (0 if no forked recovery).  Returns 0 for invalid sizes.
 */
SSD_API size_t ssd_workspace_bytes(int B, int k, int V, int f);

/* Workspace bytes for ssd_softmax_temp on `rows` rows of V logits. */
SSD_API size_t ssd_softmax_workspace_bytes(int rows, int V);

/* Zero-fill `bytes` of workspace `ws` on `stream` (one cudaMemsetAsync). */
SSD_API ssd_status ssd_workspace_init(void *ws, size_t bytes, ssd_stream_t stream);

/*
 * Read (and, if clear != 0, reset) the device error word of a workspace or
 * of a speculation cache workspace.  Synchronises `stream`.  *out is a host
 * int32 receiving an OR of SSD_DEVERR_* bits.
 */
SSD_API ssd_status ssd_get_device_error(void *ws, ssd_stream_t stream, int32_t *out,
                                int clear);

/*
 * ssd_softmax_temp -- temperature softmax per row ([SUM] sampler: greedy at
 * temperature 0, stochastic otherwise).
 *   logits : [rows, V] (dtype)
 *   T      : [rows] fp32 temperatures.  T == 0 rows give the greedy
 *            distribution: a one-hot at the argmax (lowest index on ties),
 *            row_sum = 1.  T < 0 / NaN or an invalid row give m = S = NaN,
 *            argmax = -1, probs = NaN and set the error word.
 *   probs  : [rows, V] fp32 or NULL.  p_v = exp((z_v - m)/T) / S.
 *   row_max, row_sum : [rows] fp32, m = max z, S = sum exp((z - m)/T).
 *   row_argmax : [rows] int32.
 *   ws     : ssd_softmax_workspace_bytes(rows, V) bytes.
 */
SSD_API ssd_status ssd_softmax_temp(const void *logits, ssd_dtype dtype, int rows, int V,
                            const float *T, float *probs, float *row_max,
                            float *row_sum, int32_t *row_argmax, void *ws,
                            size_t ws_bytes, ssd_stream_t stream);

/*
 * ssd_verify -- acceptance, first-reject prefix and (optionally) the
 * recovery/bonus draw, in one call ([SSD] verify in one pass; [SPS] point of
 * divergence; [LKM] the rule).
 *   Z        : target logits [B, k+1, V], batch stride z_bstride elements.
 *   D        : draft logits [B, >=k, V], batch stride d_bstride; rows
 *              0..k-1 are read.
 *   x        : [B, k] int32 draft tokens.   T : [B] fp32 temperatures, used
 *              for target and draft rows alike; T == 0 is greedy.
 *   u_acc    : [B, k] fp32 uniforms in [0, 1).  Draft token i is accepted
 *              iff u_acc[b,i] < p_i(x_i) / q_i(x_i) (q == 0: iff p > 0);
 *              greedy rows accept iff x_i == argmax Z[b,i].
 *   accept_len : [B] int32 out: n in 0..k, or SSD_ROW_INVALID /
 *              SSD_ROW_BAD_TOKEN.
 *   p_at_x, q_at_x : [B, k] fp32 out or NULL: p_i(x_i), q_i(x_i) (greedy:
 *              1 if x_i is the argmax of that row, else 0).
 *   u_smp    : [B] fp32 uniforms, or NULL to skip the draw.
 *   out_tok  : [B, k+1] int32 out, required when u_smp is given: the n
 *              accepted tokens, then the drawn token, then -1.  The draw is
 *              the smallest j with C_j > u_smp * C_{V-1}, C the prefix sum of
 *              w = max(0, p_n - q_n) (n < k; if w is all zero, w = p_n) or of
 *              w = p_k (n == k); greedy rows take argmax Z[b,n].
 *   ws       : ssd_workspace_bytes(B, k, V, 0) bytes (or more).
 */
SSD_API ssd_status ssd_verify(const void *Z, int64_t z_bstride, const void *D,
                      int64_t d_bstride, ssd_dtype dtype, int B, int k, int V,
                      const int32_t *x, const float *T, const float *u_acc,
                      int32_t *accept_len, float *p_at_x, float *q_at_x,
                      const float *u_smp, int32_t *out_tok, void *ws,
                      size_t ws_bytes, ssd_stream_t stream);

/*
 * ssd_verify_noalloc -- ssd_verify for callers that cannot allocate device
 * memory (the pages have no counterpart; this is a deployment aid).  Some
 * callers cannot call cudaMalloc or an allocating library routine: code that
 * runs inside a framework that owns every allocation, or a process whose
 * device memory is fully pre-reserved.  This call takes no workspace: its
 * scratch is a file-scope device array of SSD_NOALLOC_SCRATCH_BYTES (8 MiB)
 * that every GPU which loads the library holds until exit.
 *   - Arguments and results are those of ssd_verify without ws/ws_bytes.
 *   - Sizes whose workspace (ssd_workspace_bytes(B, k, V, 0)) exceeds the
 *     array return SSD_ERR_WORKSPACE before anything is enqueued.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - Every call shares the one array, which keeps the last call's contents;
 *     each call writes every part it reads, so nothing needs clearing.  Calls
 *     that overlap on the GPU (other streams, other host threads) race.
 *   - The array's device error word is not exposed: data errors show as the
 *     accept_len sentinels.
 *   - u_smp may be NULL (out_tok then too): acceptance only.  T > 0 rows then
 *     get no recovery / bonus token (out_tok[b][n] = -1, if out_tok is
 *     given), and no later call can draw it, because ssd_sample_residual
 *     needs the statistics in a workspace this call does not expose.
 *   - Argument checks run before the array is touched: invalid sizes return
 *     SSD_ERR_INVALID_ARG, sizes beyond the array SSD_ERR_WORKSPACE, then
 *     null or misaligned pointers SSD_ERR_INVALID_ARG.
 */
#define SSD_NOALLOC_SCRATCH_BYTES (8u << 20)
SSD_API ssd_status ssd_verify_noalloc(const void *Z, int64_t z_bstride, const void *D,
                                      int64_t d_bstride, ssd_dtype dtype, int B, int k, int V,
                                      const int32_t *x, const float *T, const float *u_acc,
                                      int32_t *accept_len, float *p_at_x, float *q_at_x,
                                      const float *u_smp, int32_t *out_tok,
                                      ssd_stream_t stream);

/*
 * ssd_sample_residual -- the recovery/bonus draw alone, after an ssd_verify
 * call on the same workspace, inputs and sizes that was given u_smp = NULL.
 * accept_len may be that call's output or any values in 0..k (negative
 * entries are skipped).  Writes out_tok [B, k+1] as ssd_verify does.
 */
SSD_API ssd_status ssd_sample_residual(const void *Z, int64_t z_bstride, const void *D,
                               int64_t d_bstride, ssd_dtype dtype, int B, int k,
                               int V, const int32_t *x, const float *T,
                               const int32_t *accept_len, const float *u_smp,
                               int32_t *out_tok, void *ws, size_t ws_bytes,
                               ssd_stream_t stream);

/*
 * ssd_forked_recovery -- SSD's forked recovery tokens ([SUM]
 * get_forked_recovery_tokens_from_logits: top-k over logits with masking).
 *   L        : [B, P, V] logits, batch stride l_bstride.
 *   mask     : [B, P, M] int32 tokens to skip at each (b, j) (entries
 *              outside [0, V) skip nothing); may be NULL when M == 0.
 *   fork_tok : [B, P, f] int32 out, fork_logit : [B, P, f] fp32 out: the f
 *              largest unmasked logits of each row, logit descending then
 *              index ascending.  Missing candidates are (-1, -inf); a row
 *              holding a NaN gives (-1, NaN) and sets the error word.
 *   ws       : ssd_workspace_bytes(B, P-1, V, f) bytes (or more).
 */
SSD_API ssd_status ssd_forked_recovery(const void *L, int64_t l_bstride, ssd_dtype dtype,
                               int B, int P, int V, int f, const int32_t *mask,
                               int M, int32_t *fork_tok, float *fork_logit,
                               void *ws, size_t ws_bytes, ssd_stream_t stream);

/*
 * ssd_verify_fork -- ssd_verify and ssd_forked_recovery over the draft
 * buffer in one pass over the logits.  D must hold P = k+1 rows per batch
 * row (the SSD draft: rows 0..k-1 feed acceptance, rows 0..k the forked
 * recovery).  Arguments as in the two calls; ws: ssd_workspace_bytes(B, k,
 * V, f).
 */
SSD_API ssd_status ssd_verify_fork(const void *Z, int64_t z_bstride, const void *D,
                           int64_t d_bstride, ssd_dtype dtype, int B, int k,
                           int V, const int32_t *x, const float *T,
                           const float *u_acc, int32_t *accept_len,
                           float *p_at_x, float *q_at_x, const float *u_smp,
                           int32_t *out_tok, int f, const int32_t *mask, int M,
                           int32_t *fork_tok, float *fork_logit, void *ws,
                           size_t ws_bytes, ssd_stream_t stream);

/*
 * Variable fan-out ([SUM] get_forked_recovery_tokens_from_logits: selection
 * by fan-out strategy).  As ssd_forked_recovery / ssd_verify_fork with
 * F (<= SSD_MAX_F) in place of f, plus
 *   fanout   : [P] int32 device array, f_j tokens kept at position j
 *              (clamped to [0, F]).  fork_tok / fork_logit stay [B, P, F]:
 *              slots f_j .. F-1 of position j hold (-1, -inf), which the
 *              cache insert skips.  NULL keeps F everywhere.
 *   ws       : sized with f = F.
 */
SSD_API ssd_status ssd_forked_recovery_fanout(const void *L, int64_t l_bstride,
                                      ssd_dtype dtype, int B, int P, int V, int F,
                                      const int32_t *fanout, const int32_t *mask,
                                      int M, int32_t *fork_tok, float *fork_logit,
                                      void *ws, size_t ws_bytes, ssd_stream_t stream);
SSD_API ssd_status ssd_verify_fork_fanout(const void *Z, int64_t z_bstride,
                                  const void *D, int64_t d_bstride, ssd_dtype dtype,
                                  int B, int k, int V, const int32_t *x,
                                  const float *T, const float *u_acc,
                                  int32_t *accept_len, float *p_at_x, float *q_at_x,
                                  const float *u_smp, int32_t *out_tok, int F,
                                  const int32_t *fanout, const int32_t *mask, int M,
                                  int32_t *fork_tok, float *fork_logit, void *ws,
                                  size_t ws_bytes, ssd_stream_t stream);

/*
 * ssd_draft_sample -- the drafter's tokens, drawn on the GPU ([SUM] sampler:
 * greedy at temperature 0, stochastic otherwise; [SPS] the small model
 * proposes the draft), fused with the draft rows' statistics so that a later
 * ssd_verify_drafted reads only the target rows.
 *   D        : draft logits [B, >= row0+rows, V], batch stride d_bstride.
 *   k        : the verify call's draft length (sizes and places the
 *              statistics in ws); rows [row0, row0+rows) with
 *              row0 + rows <= k + 1 (row k: SSD's next-round token).
 *   T        : [B] fp32; the verify call must use the same temperatures.
 *   seed, offset : the draw of element v of row i of batch row b uses word
 *              v mod 4 of Philox4x32-10 (Salmon et al. 2011) at counter
 *              (v / 4, i, b, offset) under key (seed low, seed high 32 bits)
 *              and u = ((w >> 9) + 1/2) / 2^23.
 *   x_out    : x_out[b * x_bstride + (i - row0)] = the token: T > 0 the
 *              Gumbel-max draw argmax_v (z_v / T - ln(-ln u_v)) (an exact
 *              draw from softmax(z / T); ties to the lowest index); T == 0
 *              the argmax; -1 for T < 0 / NaN or an invalid row (device
 *              error word set).
 *   f, fork_tok, fork_logit : f >= 1 also writes [B, rows, f] forks: the f
 *              largest logits of each row other than its drafted token (SSD
 *              forked recovery with the drafter's token masked); f == 0
 *              writes none (pointers may be NULL).  f + 1 <= SSD_MAX_F.
 *   ws       : ssd_workspace_bytes(B, k, V, f > 0 ? f + 1 : 0) bytes; the
 *              same workspace goes to ssd_verify_drafted.
 */
SSD_API ssd_status ssd_draft_sample(const void *D, int64_t d_bstride, ssd_dtype dtype, int B,
                            int k, int V, int row0, int rows, const float *T,
                            uint64_t seed, uint32_t offset, int32_t *x_out,
                            int64_t x_bstride, int f, int32_t *fork_tok,
                            float *fork_logit, void *ws, size_t ws_bytes,
                            ssd_stream_t stream);

/*
 * ssd_verify_drafted -- ssd_verify whose draft rows 0..k-1 were already
 * summarised into ws by ssd_draft_sample calls (same B, k, V, T and ws):
 * the streaming pass reads only the k+1 target rows; D is still read at the
 * draft tokens and, for the recovery draw, at row n.  Arguments and results
 * as ssd_verify.
 */
SSD_API ssd_status ssd_verify_drafted(const void *Z, int64_t z_bstride, const void *D,
                              int64_t d_bstride, ssd_dtype dtype, int B, int k, int V,
                              const int32_t *x, const float *T, const float *u_acc,
                              int32_t *accept_len, float *p_at_x, float *q_at_x,
                              const float *u_smp, int32_t *out_tok, void *ws,
                              size_t ws_bytes, ssd_stream_t stream);

/*
 * ssd_verify_topk -- ssd_verify over top-k / top-p filtered distributions:
 * the target rows and the draft rows are filtered alike (order the tokens by
 * logit descending, index ascending; keep the first K; keep the shortest
 * prefix of those holding >= top_p[b] of their probability mass;
 * renormalise), and acceptance, the residual and the bonus draw use the
 * filtered p and q.  Greedy rows (T == 0) are unaffected.
 *   K        : K >= 1; K >= V keeps every token (top-p over the whole
 *              vocabulary).  min(K, V) <= 32: one pass over the 2k+1 rows
 *              keeps per-chunk top-K lists (no exponentials) and the rest
 *              works on at most K candidates per row.  Larger K: each row's
 *              kept set is found as a threshold on the token order (a row
 *              maximum pass, a histogram pass of x = (m - z) log2(e) / T in
 *              1/16 steps, a pass that sums the exact mass above the bins
 *              holding the cuts and collects those bins' tokens, an exact
 *              cut on them; see ssd_filter.cu), three reads of the rows in
 *              all.  A row whose cut bins hold more than 2048 tokens (e.g.
 *              thousands of equal logits) is cut by bisection on the token
 *              order, slower but exact.  V <= 2^21 on this path.
 *   top_p    : [B] fp32 device array, or NULL for 1 (no cut).  Values >= 1
 *              or NaN cut nothing.
 *   other arguments and results as ssd_verify (the draft tokens x must have
 *   been drawn from the filtered draft distribution for exactness).
 *   ws       : ssd_topk_workspace_bytes(B, k, V, K) bytes (0 for invalid
 *              sizes).
 * Mass sums and the top-p cut are exact to ~1e-12 relative (extended
 * precision exponentials, fixed-point sums), so a cut differs from an exact
 * computation only when the cumulative mass at the cut lies that close to
 * top_p times the kept tokens' mass.
 */
SSD_API size_t ssd_topk_workspace_bytes(int B, int k, int V, int K);
SSD_API ssd_status ssd_verify_topk(const void *Z, int64_t z_bstride, const void *D,
                           int64_t d_bstride, ssd_dtype dtype, int B, int k, int V,
                           const int32_t *x, const float *T, int K, const float *top_p,
                           const float *u_acc, int32_t *accept_len, float *p_at_x,
                           float *q_at_x, const float *u_smp, int32_t *out_tok, void *ws,
                           size_t ws_bytes, ssd_stream_t stream);

/*
 * ssd_verify_tree -- verification of a draft token tree per batch row (the
 * "tanishqkumar/ssd" summary's tree decoding), by the multi-step speculative
 * sampling of SpecInfer (Miao et al. 2024), which keeps the target's output
 * law when the children of a node were drawn independently from the
 * draft's q at that node:
 *   start at the root with r = p(root); try the children of the current
 *   node in increasing node index; child x is accepted when
 *   u_acc[b, child] < r(x) / q(x) (q(x) == 0: accepted iff r(x) > 0); an
 *   accepted child becomes the current node with r = its p; a rejection
 *   replaces r by norm(max(0, r - q)) (unchanged if that is all zero); when
 *   the children are exhausted the final token is drawn from r by inverse
 *   CDF with u_smp[b] (smallest v whose prefix sum exceeds u times the
 *   total).  T == 0 rows accept the first child whose token is the argmax
 *   (lowest index) of the current node's target row and end with that
 *   argmax.
 * One streaming pass over the N target rows and the inner nodes' draft rows
 * gives each row's maximum, argmax and sum; then a thread-block cluster per
 * batch row walks the tree, with one pass over the current node's two rows
 * per rejection (the next residual mass) and one for the final draw when it
 * is not already known.
 *   Z        : target logits at the nodes, row (b, j) at Z + b*z_bstride +
 *              j*V (the target's logits after node j's path; node 0 is the
 *              last committed position).  z_bstride >= N*V.
 *   D        : draft logits at the nodes, same layout (q of node j's
 *              children).  Only the rows of nodes that have children are
 *              read and checked: a leaf's q is never used.
 *   N        : nodes per tree, 1 <= N <= SSD_MAX_TREE_NODES.
 *   parent   : [B, N] int32 device: parent[b, 0] == -1, 0 <= parent[b, j] < j.
 *   tok      : [B, N] int32 device: node j's token (entry 0 unused).
 *   T        : [B] temperatures; u_acc: [B, N] uniforms in [0, 1), entry
 *              (b, j) tests node j (entry 0 unused); u_smp: [B].
 *   accept_len : [B] accepted nodes (path depth), or a sentinel: -1 for
 *              T < 0 or NaN or an invalid row (as ssd_verify), -2 for an
 *              invalid tree (parent or token out of range).
 *   out_tok  : [B, N]: the accepted tokens in path order, the final token,
 *              then -1 (all -1 on a sentinel).
 *   out_node : [B, N] or NULL: the accepted node ids, then -1.
 *   ws       : ssd_tree_workspace_bytes(B, N, V) bytes (its first word is
 *              the device error word, as for ssd_verify).  For V >= 32768
 *              it includes a cache of 16 (V + 32768) bytes per tree, where a
 *              node's first residual pass keeps each element's two
 *              exponentials for the later passes at that node.
 * Errors: SSD_ERR_INVALID_ARG for null required pointers, sizes out of
 * range, strides below N*V or misaligned pointers; SSD_ERR_WORKSPACE when
 * ws_bytes is too small; SSD_ERR_CUDA when a launch fails.
 */
SSD_API size_t ssd_tree_workspace_bytes(int B, int N, int V);
SSD_API ssd_status ssd_verify_tree(const void *Z, int64_t z_bstride, const void *D,
                           int64_t d_bstride, ssd_dtype dtype, int B, int N, int V,
                           const int32_t *parent, const int32_t *tok, const float *T,
                           const float *u_acc, const float *u_smp, int32_t *accept_len,
                           int32_t *out_tok, int32_t *out_node, void *ws, size_t ws_bytes,
                           ssd_stream_t stream);

/*
 * Speculation cache ([SSD] roadmap: the speculation cache; [SUM] cache
 * hits and misses).  An open-addressing table on the device mapping the key
 * (b, position, token) to `depth` draft tokens.  Keys compare exactly, so the
 * hash only decides slots, never results.  Inserts apply in input order (the
 * last duplicate wins, also across calls).  The call order is counted on the
 * device, so inserts into one cache must be ordered on one stream (or joined
 * by events); an insert captured in a CUDA graph keeps the rule on every
 * replay.  Probing is bounded by the capacity: an insert that finds no slot
 * is dropped and sets SSD_DEVERR_CACHE_FULL.  Limits: b < 2^24,
 * position < 256, token >= 0.
 */
typedef struct ssd_spec_cache ssd_spec_cache;

/* capacity: power of two >= 2; depth >= 1.  Allocates device memory once
 * (on the current device). */
SSD_API ssd_status ssd_spec_cache_create(int capacity, int depth, ssd_spec_cache **out);
SSD_API void ssd_spec_cache_destroy(ssd_spec_cache *cache);
SSD_API ssd_status ssd_spec_cache_clear(ssd_spec_cache *cache, ssd_stream_t stream);

/*
 * ssd_verify_fork_cache -- one SSD round step ([SSD] the drafter keeps
 * speculations for the likely verification outcomes; a correct guess is
 * returned at once): ssd_verify_fork, then (after clearing the cache when
 * clear != 0) the forks go into `cache` keyed (b, position, fork token) with
 * payload rows payload[((b*(k+1) + j)*f + r) * depth ..], and each row's
 * realised outcome (accept_len[b], out_tok[b, accept_len[b]]) is looked up:
 * hit[b] in {0, 1}, tok_out[b, 0..depth) (-1 on a miss).  With B >= 32 the
 * clear and the insert run on an internal stream while the recovery draw
 * runs.  Arguments otherwise as ssd_verify_fork (out_tok required); the
 * cache must live on the current device.
 */
SSD_API ssd_status ssd_verify_fork_cache(const void *Z, int64_t z_bstride, const void *D,
                                 int64_t d_bstride, ssd_dtype dtype, int B, int k, int V,
                                 const int32_t *x, const float *T, const float *u_acc,
                                 int32_t *accept_len, float *p_at_x, float *q_at_x,
                                 const float *u_smp, int32_t *out_tok, int f,
                                 const int32_t *mask, int M, int32_t *fork_tok,
                                 float *fork_logit, ssd_spec_cache *cache, int clear,
                                 const int32_t *payload, int32_t *hit, int32_t *tok_out,
                                 void *ws, size_t ws_bytes, ssd_stream_t stream);

/* n keys (b[i], pos[i], tok[i]) -> payload[i*depth .. +depth). */
SSD_API ssd_status ssd_spec_cache_insert(ssd_spec_cache *cache, const int32_t *b,
                                 const int32_t *pos, const int32_t *tok,
                                 const int32_t *payload, int n,
                                 ssd_stream_t stream);

/* hit[i] = 1 and tok_out[i*depth..] = payload on a hit; 0 and -1 on a miss
 * (keys with a negative token or out-of-range b/pos always miss). */
SSD_API ssd_status ssd_spec_cache_lookup(const ssd_spec_cache *cache, const int32_t *b,
                                 const int32_t *pos, const int32_t *tok, int n,
                                 int32_t *hit, int32_t *tok_out,
                                 ssd_stream_t stream);

/* Insert the forked recovery tokens directly: key (b, j, fork_tok[b,j,r])
 * -> payload[((b*P + j)*f + r)*depth ..] for every fork_tok >= 0. */
SSD_API ssd_status ssd_spec_cache_insert_forks(ssd_spec_cache *cache,
                                       const int32_t *fork_tok, int B, int P,
                                       int f, const int32_t *payload,
                                       ssd_stream_t stream);

/* Look up each row's realised outcome: key (b, n_b, out_tok[b, n_b]) with
 * n_b = accept_len[b] (rows with n_b < 0 miss).  hit [B], tok_out [B,depth]. */
SSD_API ssd_status ssd_spec_cache_lookup_outcome(const ssd_spec_cache *cache,
                                         const int32_t *accept_len,
                                         const int32_t *out_tok, int B, int k,
                                         int32_t *hit, int32_t *tok_out,
                                         ssd_stream_t stream);

/* Read (and optionally clear) the cache's device error word; syncs stream. */
SSD_API ssd_status ssd_spec_cache_get_error(ssd_spec_cache *cache, ssd_stream_t stream,
                                    int32_t *out, int clear);

SSD_API int ssd_spec_cache_capacity(const ssd_spec_cache *cache);
SSD_API int ssd_spec_cache_depth(const ssd_spec_cache *cache);

/*
 * Launch profiler (observability, not part of the method).  Between
 * ssd_profile_begin and ssd_profile_end every kernel the library launches
 * from this process is bracketed by a pair of CUDA events recorded on the
 * launch stream (at most max_launches launches; later ones go unrecorded but
 * are still counted).  ssd_profile_end waits for the recorded events and
 * fills out[0 .. *n_out) with one entry per kernel name: launches and total
 * device time.  Entries with launches == 0 are phases that span several
 * launches: "stats_pass" is the statistics pass of a batched verify, whose
 * target-row and draft-row kernels run concurrently on two internal streams,
 * from the fork to the join on the caller's stream; "stats_span" is the same
 * pass without the fork and join: from the earlier of its two launches'
 * begin events to the later of their end events.  Events are created at
 * begin and destroyed at end.
 */
typedef struct {
    char name[40];
    int launches;
    int timed;          /* launches with recorded events */
    double total_ms;    /* sum of event-measured durations of timed launches */
} ssd_profile_entry;

SSD_API ssd_status ssd_profile_begin(int max_launches);
SSD_API ssd_status ssd_profile_end(ssd_profile_entry *out, int cap, int *n_out);

/*
 * Vocabulary split override (tuning and tests; not part of the method).
 * Every logit row is split into chunks ("split-V") that CTAs stream and
 * whose partial statistics are merged in chunk order.  chunk_elems > 0 fixes
 * the chunk length (rounded up to a multiple of 8 and clamped to
 * [ceil(V / 256), 32 KB of logits]); chunks_per_cta > 0 fixes how many
 * consecutive chunks one statistics CTA streams (at most the chunk count).
 * 0 restores the built-in policy.  The setting is process-wide and read when
 * a call (or a workspace-size query) lays out its workspace, so query the
 * workspace size after setting it.  Integer results (accept lengths, tokens,
 * forks, cache lookups) do not depend on it; float outputs (p_at_x, q_at_x,
 * softmax sums) can differ in the last bits, because the chunk sums round
 * differently.  Returns SSD_ERR_INVALID_ARG for negative values.
 */
SSD_API ssd_status ssd_set_split(int chunk_elems, int chunks_per_cta);

/*
 * Small-batch schedule override (tuning and tests; not part of the method).
 * After the statistics pass, a verify call of at most max_b batch rows
 * (default 16) runs its finalisation, recovery / bonus draw and, in
 * ssd_verify_fork_cache, the cache insert and outcome lookup as one
 * cluster kernel: one thread-block cluster of up to 8 CTAs per batch row,
 * the row merges and the draw's pass over the vocabulary split over the
 * cluster, partial sums exchanged through distributed shared memory.
 * Larger batches launch the finalisation, draw and cache kernels
 * separately.  max_b = 0 disables the cluster kernel; negative restores the
 * default.  Process-wide, read at each call.  Accept lengths, p_at_x,
 * q_at_x and forks are the same bits on both schedules; a drawn token is
 * the same except where u falls within ~1e-12 relative of a boundary of the
 * inverse CDF (the two schedules round their fixed-point partial masses
 * over different ranges).  Returns SSD_OK.
 */
SSD_API ssd_status ssd_set_chain_batch(int max_b);

/*
 * Whole-call schedule override for the smallest batches (tuning and tests;
 * not part of the method).  A verify call of at most max_b batch rows
 * (default 4, at most 8) runs as one cooperative kernel: the statistics
 * pass, row merges and forks, acceptance, the draw's two exact passes over
 * rows n and the select, separated by grid-wide barriers among CTAs that
 * are all resident; in ssd_verify_fork_cache also the cache clear, insert
 * and outcome lookup.  max_b = 0 disables it, negative restores the default;
 * max_grid > 0 caps the CTAs of that kernel (0: as many as the GPU holds at
 * once).  If the launch is refused the call takes the launch-by-launch
 * schedule.  Every barrier wait is bounded: one that runs out sets
 * SSD_DEVERR_TIMEOUT and the kernel returns without finishing the call.
 * Accept lengths, p_at_x, q_at_x and forks are the same bits on every
 * schedule; a drawn token is the same except where u falls within ~1e-12
 * relative of a boundary of the inverse CDF.  Returns SSD_ERR_INVALID_ARG
 * for max_grid < 0, else SSD_OK.  Process-wide, read at each call.
 */
SSD_API ssd_status ssd_set_step_schedule(int max_b, int max_grid);

/*
 * Self-test hook for the library's extended-precision exponential (used by
 * the recovery draw): out[i] = 2^(x_hi[i] + x_lo[i]) in double, for
 * x_hi <= 0.  Device pointers, n >= 0.  Not part of the verify path.
 */
SSD_API ssd_status ssd_selftest_exp2(const float *x_hi, const float *x_lo, double *out,
                             int n, ssd_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SSD_GB300_H */
