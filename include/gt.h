/*
 * gt.h — C ABI of the GB300 (sm_103a) verify-and-graft step of tree speculative decoding.
 *
 * Sources, cited as page title + section:
 *   [Graft]     "浙江大学、阿里巴巴联手破解AI推理瓶颈" — write-up of the Graft paper.
 *               §二: calibrated prune at depths 0/1/5; the GPU-resident successor table
 *               ("adjacency matrix": row = token, its k most likely successors by rank);
 *               retrieval rooted at the current token and expanded by a stage-adaptive,
 *               asymmetric template into the freed slots (8/24/40 draft + 52/36/20
 *               retrieved of 60); flatten + tree position ids + mask + one parallel
 *               verify; online update of the row of every verified position.
 *               §四: batched serving keeps a fixed slot count per request and swaps
 *               low-confidence draft nodes for retrieved ones. §六: accepted and rejected
 *               positions both update the table.
 *   [TreeGraft] "TreeGraft 精读：多起草器共嫁接一棵草稿树，让投机解码跨越快与好的单选题".
 *               §一: accept the agreeing tokens, roll back at the first error.
 *               §三: cumulative path score s(v) = product of edge scores root..v; global
 *               prune to the verification budget Bver; tree-attention verification.
 *               §四 How: non-destructive graft, then one global prune to Bver = 63.
 *
 * Conventions shared by every entry point
 *   - Pointers named in the "device" list are caller-owned CUDA device pointers (or
 *     managed memory, except where an entry point says otherwise); the library never
 *     allocates, frees or keeps them. Host helpers at the end of the file take host
 *     pointers.
 *   - Trees are flattened in topological order: node 0 is the root (the current token),
 *     parent[0] = -1 and 0 <= parent[v] < v for v >= 1. Per-request arrays are
 *     row-major [B][stride]; entries at or beyond a request's node count are padding.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *     The return value reports what the host can see: bad arguments (GT_ERR_ARG), an
 *     unsupported shape (GT_ERR_SHAPE) or a failed launch (GT_ERR_CUDA). Problems only
 *     visible in device data (malformed tree, id out of range, non-monotone score, size
 *     stored on the device that exceeds a buffer) are written as the matching negative
 *     code into the device word *err with a compare-and-swap from 0, so the first error
 *     wins; the caller zeroes *err beforehand and reads it after its own synchronisation.
 *     err may be NULL (no device-side report). Requests with bad data get padded
 *     outputs (count 0 or -1 entries) and do not corrupt other requests.
 *   - Calls perform no host synchronisation and allocate nothing, so a sequence of them
 *     can be captured into a CUDA graph.
 */
#ifndef GT_H
#define GT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gt_stream_t;

typedef enum {
  GT_OK = 0,
  GT_ERR_ARG = -1,          /* null pointer, negative size, unsupported option          */
  GT_ERR_SHAPE = -2,        /* size outside what the kernels support                    */
  GT_ERR_CUDA = -3,         /* a CUDA launch or driver call failed                      */
  GT_ERR_TREE = -4,         /* device: not a rooted topological tree, id out of range   */
  GT_ERR_NONMONOTONE = -5,  /* device: a node's score exceeds its parent's, or is NaN   */
  GT_ERR_TIMEOUT = -6,      /* device: a bounded wait gave up                           */
  GT_ERR_RANGE = -7,        /* device: a stored count exceeds its buffer                */
  GT_ERR_IO = -8,           /* host: a file cannot be opened, read or written, or its    */
                            /* length differs from what its header states               */
  GT_ERR_CORRUPT = -9,      /* host: a file's magic, checksum or contents are invalid    */
  GT_ERR_VALUE = -10        /* device, checked builds only: a NaN where a number belongs */
} gt_status;

typedef enum { GT_F32 = 0, GT_BF16 = 1 } gt_dtype;

/* ---------------------------------------------------------------------------------------
 * a1. Prune to the verification budget.  [TreeGraft] §三, §四 How; [Graft] §二, §四.
 *
 * Keeps, per request b, the root and the best nodes by (score desc, index asc), at most
 * keep[b] nodes in total and, when thresh != NULL, only non-root nodes with
 * score >= thresh[b]. Kept nodes are renumbered in ascending old index and their parents
 * remapped, so the output is again a topological tree.
 *   device in : score  f32 [B][Nin]  cumulative path scores (root's value is ignored)
 *               parent i32 [B][Nin], tokens i32 [B][Nin]
 *               n_in   i32 [B] nodes per request (NULL: every request has Nin)
 *               keep   i32 [B] node budget incl. the root (>= 1)
 *               thresh f32 [B] confidence threshold (NULL: none)
 *   device out: out_parent, out_tokens i32 [B][Nout]; out_score f32 [B][Nout] (nullable);
 *               out_old_idx i32 [B][Nout] old index of each kept node (nullable);
 *               n_out i32 [B]. Entries >= n_out[b]: -1 (score 0).
 * Limits: 1 <= Nin <= 1024, Nout >= 1. Device errors: GT_ERR_TREE (bad parent),
 * GT_ERR_NONMONOTONE (score[v] > score[parent[v]] for a non-root parent, or NaN),
 * GT_ERR_RANGE (min(keep, n_in) > Nout, keep < 1, n_in outside [1, Nin]).
 * Output arrays must not alias the inputs.
 * ------------------------------------------------------------------------------------- */
int gt_prune_topB(const float *score, const int32_t *parent, const int32_t *tokens,
                  const int32_t *n_in, int B, int Nin, const int32_t *keep,
                  const float *thresh, int Nout, int32_t *out_parent, int32_t *out_tokens,
                  float *out_score, int32_t *out_old_idx, int32_t *n_out, int32_t *err,
                  gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * a2. Graft retrieved nodes into the freed slots.  [Graft] §二 (second gear), §四;
 *     Graft-TAIL: [Graft] §七 (the low-confidence tail of a block draft is replaced by
 *     retrieved candidates).
 *
 * In place on the kept trees. For request b with n = n_nodes[b] kept nodes, the
 * retrieved tree hangs from the anchor node a = anchor[b] (anchor NULL: a = 0, the root;
 * anchor[b] = -1: a = n - 1, the last kept node, i.e. the tail of a pruned chain). Template
 * nodes t = 0 .. R'-1, R' = min(R[b], Nmax - n, T), are tried in order: template parent
 * tpar[t] (-1 = the anchor, else an earlier template node) and successor rank
 * trank[t]; the node's token is table[token(parent)][trank[t]]. An empty entry (-1)
 * drops the node and all its template descendants. Survivors are appended at n, n+1, ...
 * in template order; slots from the new count to Nmax-1 are set to -1.
 *   device in/out: parent, tokens i32 [B][Nmax]; n_nodes i32 [B] (in: kept, out: total)
 *   device in    : tpar, trank i32 [T]; R i32 [B]; anchor i32 [B] (nullable);
 *                  table i32 [V][k] (entries in [-1, V))
 * Limits: 0 <= T <= 1024, k >= 1, V >= 1. Device errors: GT_ERR_TREE (template parent
 * not earlier, rank >= k, a token or table entry outside its range), GT_ERR_RANGE
 * (n_nodes outside [1, Nmax], or the anchor outside the kept tree: that request keeps its
 * tree and grafts nothing).
 * ------------------------------------------------------------------------------------- */
int gt_graft_expand(int32_t *parent, int32_t *tokens, int32_t *n_nodes, int B, int Nmax,
                    const int32_t *tpar, const int32_t *trank, int T, const int32_t *R,
                    const int32_t *anchor, const int32_t *table, int V, int k, int32_t *err,
                    gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * a3. Ancestor mask and tree position ids.  [Graft] §二 (third gear).
 *
 * depth[v] = number of edges from the root; pos[v] = prefix_len[b] + depth[v];
 * bit u of mask row v (word u/64, bit u%64) is set iff u is v or an ancestor of v.
 *   device in : parent i32 [B][N]; n_nodes i32 [B]; prefix_len i32 [B]
 *   device out: depth, pos i32 [B][N]; mask u64 [B][N][ceil(N/64)]
 *               Rows >= n_nodes[b]: depth = pos = -1, mask = 0.
 * Limits: 1 <= N <= 1024. Device errors: GT_ERR_TREE, GT_ERR_RANGE (n outside [1, N]).
 * ------------------------------------------------------------------------------------- */
int gt_tree_mask(const int32_t *parent, const int32_t *n_nodes, const int32_t *prefix_len,
                 int B, int N, int32_t *depth, int32_t *pos, uint64_t *mask, int32_t *err,
                 gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * a4. Tree-masked GQA attention of the tree's queries.  [Graft] §二 (third gear);
 *     [TreeGraft] §三 (tree-attention verification).
 *
 * O[b][i][h] = sum_j softmax_j(scale * Q[b][i][h] . K[b][h/g][j]) V[b][h/g][j], g = Hq/Hkv,
 * over keys j in [0, P) (the committed prefix, P = prefix_len[b]) and j = P + u for every
 * tree node u with bit u set in mask[b][i] (the tree's own K/V rows sit at P .. P+n-1).
 *   device in : Q  [B][N][Hq][d]   (dtype)
 *               K, V [B][Hkv][Lcap][d] (dtype) — the KV cache with the tree rows appended
 *               mask u64 [B][N][1] from gt_tree_mask; prefix_len, n_nodes i32 [B]
 *   device out: O [B][N][Hq][d] (dtype; fp32 accumulation, round to nearest even);
 *               rows i >= n_nodes[b] are zero.
 *   workspace : caller-owned device scratch of gt_tree_attn_workspace(...) bytes,
 *               256-byte aligned; contents need no initialisation and are clobbered.
 * dtype GT_BF16 runs on the tcgen05 tensor cores (bf16 operands, fp32 accumulators in
 * tensor memory, K/V tiles staged by TMA); GT_F32 runs on FP32 FMA units.
 * Q, K, V and O must be device memory of the current device (a cudaMalloc-family
 * allocation made there; the first and last byte of each are checked). Host, managed and
 * peer-device memory is refused with GT_ERR_ARG before anything is launched: the bf16
 * kernel streams K and V through cluster-multicast TMA loads, which this library issues
 * only over the memory of the GPU that runs them.
 * Limits: d = 128, 1 <= N <= 64, Hq % Hkv == 0, (Hq/Hkv)*N <= 512, Lcap >= 1, scale a
 * finite value > 0 (else GT_ERR_ARG); Q, K, V, O 16-byte aligned. Device errors:
 * GT_ERR_RANGE (prefix_len + n_nodes > Lcap, n_nodes outside [1, N], prefix_len < 0). Keys past a request's length are never read
 * into the result (cache rows there may hold anything, NaN included).
 * ------------------------------------------------------------------------------------- */
size_t gt_tree_attn_workspace(int B, int N, int Hq, int Hkv, int d, int Lcap);
int gt_tree_attn(const void *Q, const void *K, const void *V, const uint64_t *mask,
                 const int32_t *prefix_len, const int32_t *n_nodes, int B, int N, int Hq,
                 int Hkv, int d, int Lcap, int dtype, float scale, void *O,
                 void *workspace, size_t ws_bytes, int32_t *err, gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * a4 without caller scratch.  The pages have no counterpart: this is a convenience of
 * this library, not a step of the method.
 *
 * Same arguments, limits, results and device errors as gt_tree_attn, minus workspace and
 * ws_bytes. The scratch lives in one static device array of GT_ATTN_NOALLOC_SCRATCH_BYTES
 * (32 MiB) inside libgt, one copy per device, so the caller allocates nothing.
 * It is meant for callers that cannot hand over a workspace. One example is a C host
 * without a device allocator of its own. Another is a serving loop whose memory pool has
 * been given all of HBM, or that must not call cudaMalloc mid-step, because cudaMalloc
 * can synchronise the device.
 *   - Capacity: a shape whose gt_tree_attn_workspace(...) exceeds the array returns
 *     GT_ERR_SHAPE before anything is launched, with the sizes in gt_last_error(). With
 *     d = 128 the need is about 4*(SMs + B*Hkv)*ceil((Hq/Hkv)*N / 128)*128*128 bytes:
 *     e.g. B = 1, Hkv = 8, Hq/Hkv = 4, N = 60 needs about 21 MB and fits.
 *   - Memory held: every device that loads libgt's module holds the array until the
 *     process exits. Under lazy module loading (the CUDA default) that is every device on
 *     which any libgt kernel has run; under CUDA_MODULE_LOADING=EAGER it is every device
 *     with a context, whether or not this entry point is ever called.
 *   - Set-up: the first call in each context (with that device current) looks up the
 *     array's device address with cudaGetSymbolAddress, which may load the module, and
 *     caches it with the context's id; after cudaDeviceReset the next call looks it up
 *     again. Make that first call before any stream capture. A failed look-up returns
 *     GT_ERR_CUDA.
 *   - Sharing: every call on a device uses the same array. Nothing in it needs to start at
 *     zero; each call writes what it later reads. Calls ordered on one stream are
 *     safe. Calls that can overlap race on the array and give wrong results: concurrent
 *     streams, threads or processes sharing the context. Give such callers gt_tree_attn
 *     with a workspace each.
 * ------------------------------------------------------------------------------------- */
#define GT_ATTN_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int gt_tree_attn_noalloc(const void *Q, const void *K, const void *V, const uint64_t *mask,
                         const int32_t *prefix_len, const int32_t *n_nodes, int B, int N,
                         int Hq, int Hkv, int d, int Lcap, int dtype, float scale, void *O,
                         int32_t *err, gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * a5. Vocab-wide top-k per row (argmax = column 0).  [Graft] §二 (table rows hold the
 *     target's k most likely next tokens); [TreeGraft] §五 (greedy, temperature 0).
 *
 * Order: value descending, +0.0 equal to -0.0, NaN below -inf, ties to the lower index.
 *   device in : logits f32 [rows][V]
 *   device out: ids i32 [rows][k]; vals f32 [rows][k] (the logits' own bits)
 * Limits: 1 <= k <= 16, k <= V, rows >= 0.
 * ------------------------------------------------------------------------------------- */
int gt_vocab_topk(const float *logits, int rows, int V, int k, int32_t *ids, float *vals,
                  gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * a5 + a6. Greedy verification with commit indices.  [Graft] §二 (third gear);
 *     [TreeGraft] §一, §三.
 *
 * Runs gt_vocab_topk over all B*N rows, then per request: node v is accepted iff every
 * edge (p -> c) on its root path has tokens[c] == argmax[p]; v* = the deepest accepted
 * node (ties: smaller index); L = depth(v*). Outputs path = root .. v*, the committed
 * tokens (the path's draft tokens, then the bonus argmax[v*]) and the KV moves
 * kv_src[j] = P + path[j] -> kv_dst[j] = P + j.
 *   device in : logits f32 [B][N][V]; tokens, parent i32 [B][N]; n_nodes, prefix_len i32 [B]
 *   device out: topk_id i32 [B][N][k]; topk_val f32 [B][N][k]; acc_len i32 [B];
 *               path, kv_src, kv_dst i32 [B][N]; out_tok i32 [B][N+1]; entries past the
 *               accepted length are -1.
 * Limits: 1 <= N <= 1024, 1 <= k <= 16, k <= V. Device errors: GT_ERR_TREE, GT_ERR_RANGE.
 * ------------------------------------------------------------------------------------- */
int gt_verify_greedy(const float *logits, const int32_t *tokens, const int32_t *parent,
                     const int32_t *n_nodes, const int32_t *prefix_len, int B, int N, int V,
                     int k, int32_t *topk_id, float *topk_val, int32_t *acc_len,
                     int32_t *path, int32_t *out_tok, int32_t *kv_src, int32_t *kv_dst,
                     int32_t *err, gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * KV commit: compaction of the accepted path's cache rows.  [TreeGraft] §一 (keep the
 * agreeing prefix, drop the rest); [Graft] §二 third gear (the verified tokens join the
 * context).
 *
 * In place, for every request b and j = 0..acc_len[b]: row kv_dst[b][j] of every KV head
 * of K and V receives the row that was at kv_src[b][j] before the call (the outputs of
 * gt_verify_greedy / gt_verify_commit: src = prefix_len + path[j], dst = prefix_len + j).
 * Every source is read before any destination is written, so a destination may be the
 * source of another j. No other row changes.
 *   device in/out: K, V [B][Hkv][Lcap][d] (dtype), 16-byte aligned
 *   device in    : kv_src, kv_dst i32 [B][N]; acc_len i32 [B]
 * Limits: 1 <= N <= 64, d * element size a multiple of 16 bytes and at most 1024.
 * Device errors: GT_ERR_RANGE (acc_len outside [0, N), a row outside [0, Lcap)); such a
 * request's rows stay as they were.
 * ------------------------------------------------------------------------------------- */
int gt_kv_commit(void *K, void *V, const int32_t *kv_src, const int32_t *kv_dst,
                 const int32_t *acc_len, int B, int N, int Hkv, int d, int Lcap, int dtype,
                 int32_t *err, gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * a7. Online successor-table update.  [Graft] §二 (third gear), §六.
 *
 * For every verified node (b, v), v < n_nodes[b], accepted or not: row tokens[b][v] of
 * the table becomes topk_id[b][v][0..k). When several nodes share a token, the one with
 * the largest linear index b*N + v wins (the result of applying the writes in order).
 * Winners own distinct rows, so no atomics are used.
 *   device in/out: table i32 [V][k]
 *   device in    : tokens i32 [B][N]; topk_id i32 [B][N][k]; n_nodes i32 [B]
 * Limits: B*N <= 16384. Device errors: GT_ERR_TREE (token outside [0, V)),
 * GT_ERR_RANGE (n_nodes outside [0, N]).
 * ------------------------------------------------------------------------------------- */
int gt_succ_update(int32_t *table, int V, int k, const int32_t *tokens,
                   const int32_t *topk_id, const int32_t *n_nodes, int B, int N,
                   int32_t *err, gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Fused forms of the step (same results and device error codes as the calls they stand
 * for, fewer launches and global-memory round trips).
 *
 * gt_tree_build = gt_prune_topB (Nout = N) -> gt_graft_expand (Nmax = N) -> gt_tree_mask,
 *   one CTA per request holding the tree in shared memory. [TreeGraft] §三, §四 How;
 *   [Graft] §二, §四. Outputs: parent, tokens i32 [B][N] (final tree, -1 padded);
 *   out_score f32 / out_old_idx i32 [B][N] (kept nodes, nullable); n_nodes i32 [B] (final
 *   count); depth, pos i32 [B][N]; mask u64 [B][N][ceil(N/64)]. anchor i32 [B] (nullable)
 *   as in gt_graft_expand, counted in the pruned tree.
 *   Limits: 1 <= Nin, N <= 1024, 0 <= T <= 1024.
 * gt_verify_commit = gt_verify_greedy -> gt_succ_update on `table` i32 [V][k] (in place).
 *   [Graft] §二 (third gear), §六; [TreeGraft] §一, §三. Limits: N <= 1024, k <= 16,
 *   B*N <= 16384.
 * ------------------------------------------------------------------------------------- */
int gt_tree_build(const float *score, const int32_t *parent_in, const int32_t *tokens_in,
                  const int32_t *n_in, int B, int Nin, const int32_t *keep, const float *thresh,
                  const int32_t *tpar, const int32_t *trank, int T, const int32_t *R,
                  const int32_t *anchor, const int32_t *table, int V, int k,
                  const int32_t *prefix_len, int N,
                  int32_t *parent, int32_t *tokens, float *out_score, int32_t *out_old_idx,
                  int32_t *n_nodes, int32_t *depth, int32_t *pos, uint64_t *mask, int32_t *err,
                  gt_stream_t stream);
int gt_verify_commit(const float *logits, const int32_t *tokens, const int32_t *parent,
                     const int32_t *n_nodes, const int32_t *prefix_len, int B, int N, int V,
                     int k, int32_t *topk_id, float *topk_val, int32_t *acc_len, int32_t *path,
                     int32_t *out_tok, int32_t *kv_src, int32_t *kv_dst, int32_t *table,
                     int32_t *err, gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Verification at temperature T > 0.  [TreeGraft] §三 (the pruned tree goes to tree
 *     attention and rejection sampling), §七 (rejection sampling keeps the target's output
 *     distribution).
 *
 * The tree's proposals are point masses (drafters' top-m children, retrieved successors).
 * Rejection sampling of point masses has the distribution of one target draw y_u per node
 * followed by a walk into the first child (lowest index) whose token is y_u; the walk stops
 * at the first node with no such child and y_u there is the bonus token. These calls use
 * that form.
 *
 * gt_vocab_sample: sample[r] = argmax_j fl(fl(z[r][j] * fl(1/T)) + G(r, j)), ties to the
 *   lower index, NaN below -inf, +0.0 equal to -0.0 (a Gumbel-max draw from
 *   softmax(z[r] / T)). G(r, j) = -log(-log U) with U = ((x >> 9) + 0.5) * 2^-23 and
 *   x = (A << 24) | (B >> 8): A is byte j % 16 (little-endian) of the Philox-4x32-10 block
 *   (Salmon et al., SC 2011) at counter (j / 16, r, step mod 2^32, step / 2^32), B is word
 *   j % 4 of the block at counter (j / 4 + 2^31, r, step mod 2^32, step / 2^32), both with
 *   key (seed mod 2^32, seed / 2^32). log is the library's own float32
 *   routine: x = 2^e m, m in [sqrt(2)/2, sqrt(2)), s = (m-1)/(m+1), log m = (s + s) *
 *   (((( 1/9 z + 1/7) z + 1/5) z + 1/3) z + 1), z = s*s, log x = e * fl(ln 2) + log m, every
 *   float32 operation rounded to nearest once, so the draw is reproducible bit for bit.
 *   device in : logits f32 [rows][V]        device out: sample i32 [rows]
 *   Errors: GT_ERR_ARG for T not finite and > 0 or 1/T overflowing float32.
 * gt_verify_sample: gt_vocab_sample over the B*N rows (row b*N + v), then the sampled walk
 *   of each request. Outputs as gt_verify_greedy (acc_len, path, out_tok, kv_src, kv_dst).
 * gt_verify_sample_commit: gt_verify_sample plus gt_vocab_topk of the unscaled logits and
 *   the table update of gt_succ_update (the table keeps the target's k most likely tokens
 *   at every verified node, as at T = 0).
 *   device in : logits f32 [B][N][V]; tokens, parent i32 [B][N]; n_nodes, prefix_len i32 [B]
 *   device out: sample i32 [B][N]; topk_id i32 [B][N][k]; topk_val f32 [B][N][k]; the walk
 *               outputs as gt_verify_greedy; table i32 [V][k] in place.
 *   Limits: 1 <= N <= 1024, B*N <= 16384, 1 <= k <= 16, k <= V. Device errors: GT_ERR_TREE,
 *   GT_ERR_RANGE.
 * ------------------------------------------------------------------------------------- */
int gt_vocab_sample(const float *logits, int rows, int V, float temperature, uint64_t seed,
                    uint64_t step, int32_t *sample, gt_stream_t stream);
int gt_verify_sample(const float *logits, const int32_t *tokens, const int32_t *parent,
                     const int32_t *n_nodes, const int32_t *prefix_len, int B, int N, int V,
                     float temperature, uint64_t seed, uint64_t step, int32_t *sample,
                     int32_t *acc_len, int32_t *path, int32_t *out_tok, int32_t *kv_src,
                     int32_t *kv_dst, int32_t *err, gt_stream_t stream);
int gt_verify_sample_commit(const float *logits, const int32_t *tokens, const int32_t *parent,
                            const int32_t *n_nodes, const int32_t *prefix_len, int B, int N,
                            int V, int k, float temperature, uint64_t seed, uint64_t step,
                            int32_t *topk_id, float *topk_val, int32_t *sample, int32_t *acc_len,
                            int32_t *path, int32_t *out_tok, int32_t *kv_src, int32_t *kv_dst,
                            int32_t *table, int32_t *err, gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Drafting side of a tree step.  [TreeGraft] §一 (an n-gram small drafter and a neural mid
 *     drafter grow one shared tree), §三 (top-W frontier of a candidate pool by cumulative
 *     path score, top-m children per frontier node), §四 Where / How (pools; attach without
 *     overwriting), §七 item 6 (the n-gram drafter: the target's top-m cache of prefill and a
 *     context n-gram index).
 *
 * gt_frontier_select: frontier[b][0..n_frontier[b]) = the top-W pool nodes of request b by
 *   (score desc, index asc; NaN last, +0.0 equal to -0.0). Pool: nodes [pool_lo[b], n) (the
 *   small drafter's newest nodes) when pool_lo is given; else the nodes with
 *   visited[b][v] == 0 (the mid drafter), after which visited[b][v] = 1 for every v < n.
 *   Exactly one of pool_lo and visited is non-NULL.
 *   device in : score f32 [B][Nmax]; n_nodes i32 [B]; pool_lo i32 [B] | visited u8 [B][Nmax]
 *   device out: frontier i32 [B][W] (-1 padded); n_frontier i32 [B]
 *   Limits: Nmax <= 1024, 1 <= W <= 64. Device errors: GT_ERR_RANGE (n outside [1, Nmax]).
 * gt_ngram_draft: children of every frontier node from the n-gram drafter. The key of
 *   node f is the last q tokens of hist[b][0..hist_len[b]) followed by the tokens of the
 *   root-to-f path; the drafter finds the most recent position i with
 *   hist[i-q+1..i] = key, trying q = q_max first and backing off to 1, and returns row i of
 *   the top-m cache (the target's m most likely tokens for position i+1, with
 *   probabilities). No match: ids -1, probabilities 0.
 *   device in : hist i32 [B][Lh]; hist_len i32 [B]; cache_id i32 [B][Lh][m];
 *               cache_p f32 [B][Lh][m]; parent, tokens i32 [B][Nmax]; n_nodes i32 [B];
 *               frontier i32 [B][W]; n_frontier i32 [B]
 *   device out: child_id i32 [B][W][m]; child_p f32 [B][W][m]; match i32 [B][W][2]
 *               (matched position or -1, matched length q or 0; 8-byte aligned, also the
 *               call's scratch: the scan merges each key's best match into it)
 *   Limits: Nmax <= 1024, W <= 64, m <= 32, q_max <= 8. Device errors: GT_ERR_RANGE (n,
 *   hist_len, n_frontier or a frontier node out of range), GT_ERR_TREE (a parent not
 *   earlier than its child).
 * gt_tree_attach: non-destructive attach. The children with id >= 0 take the slots n, n+1,
 *   ... in (frontier order, child order) until Nmax; child score = fl(score(f) * p);
 *   existing nodes never change; slots past the new count are set to -1 / -1 / 0.
 *   n_nodes[b] becomes the new count and first_new[b] the old one (the next small step's
 *   pool).
 *   device in/out: parent, tokens i32 [B][Nmax]; score f32 [B][Nmax]; n_nodes i32 [B]
 *   device in    : frontier i32 [B][W]; n_frontier i32 [B]; child_id i32 [B][W][m];
 *                  child_p f32 [B][W][m]          device out: first_new i32 [B]
 *   Limits: Nmax <= 1024, W <= 64, m <= 32, W*m <= 1024. Device errors: GT_ERR_RANGE (n,
 *   n_frontier or a frontier node out of range), GT_ERR_TREE (a child id outside [-1, V));
 *   such a request keeps its tree.
 * ------------------------------------------------------------------------------------- */
int gt_frontier_select(const float *score, const int32_t *n_nodes, int B, int Nmax,
                       const int32_t *pool_lo, uint8_t *visited, int W, int32_t *frontier,
                       int32_t *n_frontier, int32_t *err, gt_stream_t stream);
int gt_ngram_draft(const int32_t *hist, const int32_t *hist_len, int B, int Lh,
                   const int32_t *cache_id, const float *cache_p, int m, const int32_t *parent,
                   const int32_t *tokens, const int32_t *n_nodes, int Nmax,
                   const int32_t *frontier, const int32_t *n_frontier, int W, int q_max,
                   int32_t *child_id, float *child_p, int32_t *match, int32_t *err,
                   gt_stream_t stream);
int gt_tree_attach(int32_t *parent, int32_t *tokens, float *score, int32_t *n_nodes, int B,
                   int Nmax, const int32_t *frontier, const int32_t *n_frontier, int W,
                   const int32_t *child_id, const float *child_p, int m, int V,
                   int32_t *first_new, int32_t *err, gt_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Successor-table files.  [Graft] §六 (the table warmed up in earlier runs is a prior that
 *     carries over to later ones: 0.37 MB after 5 warm-up rounds, 2.32 MB after 50).
 *
 * Host pointers, synchronous, no CUDA calls: copy a device table to the host before saving
 * and back after loading. File layout (little-endian): magic "GTSUCC" 0x00 0x01; uint32 V;
 * uint32 k; uint64 payload bytes (4 V k); uint32 CRC-32 of the payload; uint32 CRC-32 of
 * the 28 header bytes before it; then the table, int32 [V][k] row-major. CRC-32 is the
 * IEEE 802.3 checksum (reflected polynomial 0xEDB88320, initial value and final XOR
 * 0xFFFFFFFF).
 * gt_succ_save: writes table (host i32 [V][k], entries in [-1, V)) to path, through a
 *   temporary file "<path>.tmp" renamed over path, so path never names a partial file.
 *   Errors: GT_ERR_ARG (null, V or k < 1, an entry outside [-1, V)), GT_ERR_IO.
 * gt_succ_file_shape: V and k of the file at path (header checked, payload not read).
 *   Errors: GT_ERR_ARG, GT_ERR_IO (missing or shorter than a header), GT_ERR_CORRUPT.
 * gt_succ_load: reads the file into table (host i32 [V][k]). The table changes only when
 *   every check passes. Errors: GT_ERR_ARG, GT_ERR_IO (missing, shorter or longer than its
 *   header states), GT_ERR_SHAPE (the file's V or k differ from the arguments),
 *   GT_ERR_CORRUPT (magic, a checksum, or an entry outside [-1, V)).
 * ------------------------------------------------------------------------------------- */
int gt_succ_save(const char *path, const int32_t *table, int V, int k);
int gt_succ_file_shape(const char *path, int32_t *V, int32_t *k);
int gt_succ_load(const char *path, int32_t *table, int V, int k);

/* ---------------------------------------------------------------------------------------
 * Host helpers (host pointers, synchronous, no CUDA calls).
 *
 * gt_stage_budget: draft / retrieved split of `slots` for a prune at stage 0, 1 or 5
 *   ([Graft] §二: 8/52, 24/36, 40/20 of 60; the same proportions for other slot counts
 *   are not given by the pages, so slots must be 60). stage = -1: no prune, (slots, 0).
 * gt_default_template: the asymmetric retrieval template of T nodes, k ranks, depth <=
 *   max_depth (a reading of [Graft] §二: nodes chosen best-first by the integer weight
 *   prod(rank_i + 2), ties by depth then rank path; every prefix is ancestor-closed).
 * gt_status_string: a static description of a gt_status value.
 * ------------------------------------------------------------------------------------- */
int gt_stage_budget(int stage, int slots, int32_t *draft, int32_t *retrieved);
int gt_default_template(int T, int k, int max_depth, int32_t *tpar, int32_t *trank);
const char *gt_status_string(int status);

/* Host-side detail of the most recent GT_ERR_CUDA (or GT_ERR_ARG from a CUDA query) returned
 * on the calling thread: the failing CUDA call and its error string. Empty if none. The
 * pointer stays valid until the next libgt call on this thread. */
const char *gt_last_error(void);

/* Self-test of the bounded waits (no counterpart in the pages). One CTA waits on an
 * mbarrier that nothing arrives on, through the same bounded-wait helper the tcgen05 kernels
 * use, with a limit of limit_ns (1 ns .. 1 s); it sets GT_ERR_TIMEOUT in *err and, when
 * waited_ns (device, nullable) is given, stores the time it waited. The GPU context stays
 * usable afterwards. Host errors: GT_ERR_ARG (limit out of range, err NULL). */
int gt_selftest_wait_timeout(int64_t limit_ns, int32_t *err, int64_t *waited_ns,
                             gt_stream_t stream);

/* Records `event` (a cudaEvent_t) on `stream` as an externally visible node when the
 * stream is being captured into a CUDA graph (cudaEventRecordExternal), so a replayed
 * graph can time the work between two such records. Not part of the step. */
int gt_event_record_external(void *event, gt_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GT_H */
