/*
 * eagle.h -- C ABI of the EAGLE / EAGLE-2 tree-verify hot path on GB300
 * (sm_103a).  One verify step is:
 *
 *   eagle_draft_expand   (every level, then finalize) -> draft tree
 *                        (or eagle_draft_static: EAGLE-1's fixed template)
 *   eagle_tree_attn      tree-masked attention of every tree node
 *   eagle_lmhead_softmax LM-head logits, softmax statistics, argmax (and q)
 *   eagle_accept_greedy  | eagle_accept_stochastic(_logits) -> accepted tokens
 *
 * Sources, by page title and section:
 *   [S4000]   大模型推理效率突破：EAGLE推测解码算法在摩尔线程GPU的实践与优化
 *             (greedy-decoding and random-decoding paragraphs; "EAGLE的创新点"
 *             list item 2, tree attention)
 *   [EAGLE]   大模型推理效率无损提升3倍，滑铁卢大学、北京大学等机构发布EAGLE
 *             (speculative-sampling paragraph; workflow paragraph; "树状生成结构";
 *             "多轮投机采样")
 *   [EAGLE-2] EAGLE-2：動態草稿樹讓 LLM 推論加速 4 倍而不失精度
 *             (§2 "推測解碼的基礎原理"; §2 "EAGLE-2 的核心創新：動態草稿樹" items 1-3)
 *
 * Conventions shared by every entry point
 *   - Pointers named d_* are DEVICE pointers, owned by the caller, and must
 *     stay valid until the work queued on `stream` has finished.  The library
 *     allocates no memory and keeps no per-call state; scratch space is passed
 *     in by the caller (sizes from the *_bytes functions below).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream) and does no host synchronisation, so a whole step
 *     can be captured in a CUDA graph.
 *   - Host-checkable errors (NULL pointers, sizes out of range, unsupported
 *     shapes) are returned at once and nothing is queued.  Errors that only
 *     the device can see (malformed parent[] array, NaN/Inf or out-of-range
 *     probabilities, index out of range) are written to *d_status (device
 *     int, caller-zeroed; the first error code wins) and the outputs of that
 *     sequence are unspecified.  A failed kernel launch returns
 *     EAGLE_ERR_CUDA.
 *   - Trees: nodes of sequence b are tree_off[b] .. tree_off[b+1]-1 of every
 *     per-node array; parent[] holds LOCAL indices with parent[root] = -1 and
 *     0 <= parent[i] < i for i > 0 (the root is local node 0).
 *   - Row-major layouts everywhere; "[T,Hq,D]" means D is contiguous.
 */
#ifndef EAGLE_H_
#define EAGLE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define EAGLE_API __attribute__((visibility("default")))
#else
#define EAGLE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *eagle_stream_t; /* same handle as cudaStream_t */

typedef enum {
  EAGLE_OK = 0,
  EAGLE_ERR_INVALID_ARG = 1,  /* bad size, NULL pointer, index out of range  */
  EAGLE_ERR_INVALID_TREE = 2, /* parent[] is not a rooted, topological tree  */
  EAGLE_ERR_UNSUPPORTED = 3,  /* shape outside what the kernels implement    */
  EAGLE_ERR_NUMERIC = 4,      /* NaN/Inf or probability outside [0,1]        */
  EAGLE_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out          */
  EAGLE_ERR_CUDA = 6,         /* CUDA launch/runtime error                   */
  EAGLE_ERR_WORKSPACE = 7     /* workspace or pool smaller than required     */
} eagle_status;

typedef enum { EAGLE_F32 = 0, EAGLE_BF16 = 1 } eagle_dtype;
typedef enum {
  EAGLE_LMHEAD_GREEDY = 0,
  EAGLE_LMHEAD_PROB = 1,
  EAGLE_LMHEAD_LOGITS = 2
} eagle_lmhead_mode;
typedef enum { EAGLE_SAMPLE_REPLACE = 0, EAGLE_SAMPLE_NO_REPLACE = 1 } eagle_sample_mode;
typedef enum {
  EAGLE_EPI_STORE = 0,    /* y = A W^T, bf16                                  */
  EAGLE_EPI_ACCUM = 1,    /* accum += A W^T, fp32 (the residual stream)       */
  EAGLE_EPI_SWIGLU = 2,   /* y = silu(gate) * up, bf16                        */
  EAGLE_EPI_QKV_ROPE = 3  /* q, k rotated to their positions, v; bf16         */
} eagle_epilogue;

/* Limits of this implementation. */
#define EAGLE_MAX_TREE_NODES 256  /* nodes per sequence, root included       */
#define EAGLE_MAX_TOPK 32         /* EAGLE-2 top-k per expanded node          */
#define EAGLE_MAX_DEPTH 16        /* EAGLE-2 expansion levels                 */

/* Human-readable name of a status code (static string). */
EAGLE_API const char *eagle_status_string(int status);
/* Library version string (static). */
EAGLE_API const char *eagle_version(void);

/* ------------------------------------------------------------------------
 * eagle_tree_attn -- tree-masked attention of every draft-tree node.
 * [S4000] "EAGLE的创新点" item 2; [EAGLE] workflow paragraph: all root-to-leaf
 * paths are verified by ONE forward pass whose attention mask lets node i
 * see the cached context and exactly its own ancestors and itself.
 *
 *   out[t,h,:] = softmax_j( scale * q[t,h,:] . key_j ) value_j  over
 *   keys j = [k_cache rows of t's sequence | k_tree rows of t's root..t path],
 *   with kv head g = h / (Hq/Hkv) (grouped-query attention).
 *
 * dtype      EAGLE_BF16 (q, k_*, v_* bf16) or EAGLE_F32 (all fp32).
 * B          sequences (>= 1).            T  total tree nodes (= tree_off[B]).
 * Hq, Hkv    query / key-value heads; Hq % Hkv == 0.   D  head dim (64 or 128).
 * scale      softmax scale (usually 1/sqrt(D)).
 * max_nodes  upper bound on nodes of any one sequence (<= 256).
 * max_kv     upper bound on any sequence's cache length (>= 0).
 * kv_rows    rows held by d_k_cache / d_v_cache (= kv_off[B]); nothing past
 *            them is ever read.
 * d_q        [T,Hq,D];  d_k_tree, d_v_tree [T,Hkv,D] (K/V of the tree nodes).
 * d_k_cache, d_v_cache  packed caches [kv_off[B],Hkv,D].
 * d_kv_off   [B+1] int32, d_tree_off [B+1] int32, d_parent [T] int32 (local).
 * d_out      [T,Hq,D] fp32, written.
 * d_ws       scratch of eagle_tree_attn_workspace_bytes(...) bytes, 256-byte
 *            aligned (may be NULL if that size is 0); contents need no
 *            initialisation.
 * Device errors: INVALID_TREE (malformed parent[] or a sequence with more
 * than max_nodes nodes or a cache longer than max_kv).
 * Ordering: the first cache blocks are requested before the kernel waits
 * for the kernel queued just before it on `stream` (programmatic dependent
 * launch), so d_k_cache, d_v_cache and d_kv_off must not be written by that
 * immediately preceding kernel (any earlier one may write them).
 * ---------------------------------------------------------------------- */
EAGLE_API size_t eagle_tree_attn_workspace_bytes(int B, int T, int Hq, int Hkv, int D,
                                       int max_nodes, int max_kv);
EAGLE_API eagle_status eagle_tree_attn(eagle_dtype dtype, int B, int T, int Hq, int Hkv, int D,
                             float scale, int max_nodes, int max_kv, int kv_rows,
                             const void *d_q, const void *d_k_tree, const void *d_v_tree,
                             const void *d_k_cache, const void *d_v_cache,
                             const int32_t *d_kv_off, const int32_t *d_tree_off,
                             const int32_t *d_parent, float *d_out,
                             void *d_ws, size_t ws_bytes, int *d_status,
                             eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * eagle_tree_attn_paged -- eagle_tree_attn over a paged KV cache.
 * Same attention as eagle_tree_attn (same sources); only where the cached
 * keys live differs.  The cache is a pool of n_pages pages of page_size
 * positions, d_k_pages / d_v_pages [n_pages, page_size, Hkv, D]; sequence
 * b's cache position p is row p % page_size of page
 * d_block_table[b * max_pages + p / page_size], and its length is
 * d_kv_len[b] (<= max_kv <= max_pages * page_size).  Pages need not be
 * contiguous or in order, and a sequence grows by appending pages to its
 * table (the pages' fragmentation and batching problems named in [EAGLE-2]
 * §4, limitations).  bf16 with D = 128 runs on the tensor cores when
 * page_size is a multiple of 128; other page sizes and fp32 run the
 * CUDA-core kernel.  The cache is read only after the preceding kernel on
 * `stream` has finished, so a commit of accepted tokens may come right
 * before this call.  No scratch is needed.
 * Device errors: as eagle_tree_attn, plus INVALID_ARG for a table entry
 * outside [0, n_pages).
 * ---------------------------------------------------------------------- */
EAGLE_API eagle_status eagle_tree_attn_paged(eagle_dtype dtype, int B, int T, int Hq, int Hkv,
                                   int D, float scale, int max_nodes, int max_kv,
                                   int page_size, int n_pages, int max_pages, const void *d_q,
                                   const void *d_k_tree, const void *d_v_tree,
                                   const void *d_k_pages, const void *d_v_pages,
                                   const int32_t *d_block_table, const int32_t *d_kv_len,
                                   const int32_t *d_tree_off, const int32_t *d_parent,
                                   float *d_out, int *d_status, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * eagle_kv_commit_paged -- append a verify step's accepted tokens to a
 * paged KV cache.
 * [EAGLE] speculative-sampling paragraph: alpha accepted drafts give alpha+1
 * tokens; the tree's root (the last token of the previous step) and the
 * alpha accepted nodes join the context.  For every sequence b, path entry
 * i = 0 .. d_accept_len[b] (node d_accepted_nodes[b*(max_depth+1) + i], the
 * acceptance walk's output; entry 0 is the root) has its K and V rows of
 * d_k_tree / d_v_tree [T,Hkv,D] copied to cache position d_kv_len[b] + i of
 * the pages (layout as eagle_tree_attn_paged); then d_kv_len[b] grows by
 * d_accept_len[b] + 1.  The block table must already name pages for the
 * new length.  Rows are copied bit for bit (dtype gives the element size).
 * Device errors: INVALID_ARG (accept length outside [0, max_depth], a node
 * outside its tree, a position without a page); that sequence is left
 * unchanged.
 * ---------------------------------------------------------------------- */
EAGLE_API eagle_status eagle_kv_commit_paged(eagle_dtype dtype, int B, int Hkv, int D,
                                   int page_size, int n_pages, int max_pages, int max_depth,
                                   const int32_t *d_tree_off, const int32_t *d_accept_len,
                                   const int32_t *d_accepted_nodes, const void *d_k_tree,
                                   const void *d_v_tree, void *d_k_pages, void *d_v_pages,
                                   const int32_t *d_block_table, int32_t *d_kv_len,
                                   int *d_status, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * eagle_lmhead_softmax -- frozen LM head over every tree node.
 * [EAGLE] workflow paragraph: the frozen classification head gives each
 * node's next-token distribution, q = softmax(z / temperature), z = h W^T.
 *
 * dtype       EAGLE_BF16 (h, w bf16; fp32 accumulation) or EAGLE_F32.
 * T, H, V     rows (tree nodes), hidden size, vocabulary.
 * temperature > 0.
 * mode        EAGLE_LMHEAD_GREEDY: no [T,V] tensor is written.
 *             EAGLE_LMHEAD_PROB:   d_q [T,V] fp32 receives softmax(z/temp),
 *                                  each entry 2^fma(z, k2, -lse2) with
 *                                  k2 = rn(log2(e)/temp), lse2 =
 *                                  rn(row_lse * log2(e)) (rn: rounded to
 *                                  nearest), the power by the GPU's
 *                                  approximate base-2 exponential (relative
 *                                  error about 2^-22).
 *             EAGLE_LMHEAD_LOGITS: d_q [T,V] fp32 receives the logits z
 *                                  themselves; with d_row_lse they are what
 *                                  eagle_accept_stochastic_logits reads.
 * d_h         [T,H];  d_w [V,H] (vocabulary-major, as stored by LM heads).
 * d_argmax    [T] int32: argmax_v z[t,v], lowest index on ties.
 * d_row_max   [T] fp32: max_v z.         d_row_lse [T] fp32: log sum exp(z/temp).
 * d_top2_gap  [T] fp32: largest minus second-largest logit (0 on a tie).
 * d_q         [T,V] fp32 (16-byte aligned for the tensor-core path), or NULL
 *             in GREEDY mode.
 * d_ws        scratch of eagle_lmhead_workspace_bytes(T, V) bytes.
 * Device errors: NUMERIC (non-finite logit).
 * ---------------------------------------------------------------------- */
EAGLE_API size_t eagle_lmhead_workspace_bytes(int T, int V);
EAGLE_API eagle_status eagle_lmhead_softmax(eagle_dtype dtype, int T, int H, int V, float temperature,
                                  int mode, const void *d_h, const void *d_w,
                                  int32_t *d_argmax, float *d_row_max, float *d_row_lse,
                                  float *d_top2_gap, float *d_q, void *d_ws,
                                  size_t ws_bytes, int *d_status, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * eagle_lmhead_softmax_noalloc -- eagle_lmhead_softmax without a workspace
 * argument.  The paper has no counterpart to this entry point.
 *
 * Some callers cannot hand the library a scratch buffer: plain-C hosts
 * without an allocator of their own, or serving loops that run under a
 * framework's pooled allocator and may not allocate (or pay the device
 * synchronisation an allocation can cause) in the middle of a step.
 * This entry point keeps the LM head's per-row partial statistics in a
 * fixed array of the library's own device memory instead, and otherwise
 * takes the same arguments and produces the same results as
 * eagle_lmhead_softmax.  It calls no allocating routine.
 *
 *   - Limit: the call needs eagle_lmhead_workspace_bytes(T, V) bytes of
 *     scratch; above eagle_lmhead_noalloc_max_scratch_bytes() (16 MiB) it
 *     returns EAGLE_ERR_WORKSPACE and queues nothing.
 *   - Every GPU that loads the library holds the 16 MiB array until the
 *     process exits.
 *   - The first call on each device looks up the array's device address
 *     (with that device current) and keeps it for later calls.
 *   - All calls share the one array and it keeps the last call's contents.
 *     Calls whose work can overlap on a GPU (different streams without
 *     ordering between them) race on it and give undefined results; order
 *     them on one stream or with events.
 * ---------------------------------------------------------------------- */
EAGLE_API size_t eagle_lmhead_noalloc_max_scratch_bytes(void);
EAGLE_API eagle_status eagle_lmhead_softmax_noalloc(eagle_dtype dtype, int T, int H, int V,
                                          float temperature, int mode, const void *d_h,
                                          const void *d_w, int32_t *d_argmax,
                                          float *d_row_max, float *d_row_lse,
                                          float *d_top2_gap, float *d_q, int *d_status,
                                          eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * eagle_accept_greedy -- greedy tree walk.
 * [S4000] greedy-decoding paragraph: match the target's most probable token
 * from the first draft on and stop at the first mismatch; on a tree, move to
 * the child (lowest node index) whose token equals argmax[cur].
 * [EAGLE] speculative-sampling paragraph: alpha accepted -> alpha+1 tokens.
 *
 * d_tokens [T] int32 (token of every node; the root's is not compared),
 * d_argmax [T] int32 (target argmax after each node).
 * max_depth  output row width is max_depth+1; a walk deeper than max_depth
 *            is a device INVALID_ARG error.
 * Outputs (W = max_depth+1): d_accept_len [B] (alpha), d_accepted_nodes
 * [B,W] (local node ids: root, then accepted nodes; -1 padded), d_out_tokens
 * [B,W] (accepted tokens, then the bonus token; -1 padded).
 * ---------------------------------------------------------------------- */
EAGLE_API eagle_status eagle_accept_greedy(int B, int max_nodes, const int32_t *d_tree_off,
                                 const int32_t *d_parent, const int32_t *d_tokens,
                                 const int32_t *d_argmax, int max_depth,
                                 int32_t *d_accept_len, int32_t *d_accepted_nodes,
                                 int32_t *d_out_tokens, int *d_status,
                                 eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * eagle_accept_stochastic -- multi-round speculative sampling over the tree.
 * [S4000] random-decoding paragraph (accept with min(1, q/p), otherwise
 * resample from the corrected distribution); [EAGLE] "多轮投机采样" (applied
 * recursively over the tree with the recorded draft probabilities);
 * [EAGLE-2] §2 basic principle (output distribution equals the target's).
 *
 * At node cur: q_0 = q[cur], p_0 = p_rows[p_row_of_node[first child]]; for
 * each child c (ascending index, token t):
 *   accept iff (double)u_accept[c] * p_k[t] < (double)q_k[t];
 *   on reject:  W_j = trunc(max(0, q_k[j]-p_k[j]) * 2^40), Z = sum W (exact),
 *               q_{k+1}[j] = float(W_j) / float(Z), one IEEE fp32 division
 *               (kept as q_k if Z == 0);
 *               NO_REPLACE: P_j = trunc(p_k[j]*2^40), P_t = 0,
 *               p_{k+1}[j] = float(P_j) / float(sum P) (0 if the sum is 0);
 *               REPLACE: p_{k+1} = p_k.
 * When every child is rejected, or cur is a leaf, the bonus token is drawn
 * from q_final by inverse CDF over trunc(q*2^40): target =
 * (trunc(u_sample[cur]*2^24) * Z) >> 24, token = first j whose inclusive
 * prefix sum exceeds target.  All roundings are IEEE round-to-nearest, so
 * decisions and tokens are reproducible bit for bit on any IEEE machine.
 *
 * V          vocabulary; R rows in d_p_rows.
 * mode       EAGLE_SAMPLE_NO_REPLACE (siblings drawn without replacement, the
 *            EAGLE-2 case) or EAGLE_SAMPLE_REPLACE (siblings drawn i.i.d.).
 * d_q [T,V], d_p_rows [R,V] fp32 probabilities in [0,1];
 * d_p_row_of_node [T] int32 global row of the distribution node i was drafted
 * from; d_u_accept, d_u_sample [T] fp32 uniforms in [0,1).
 * Outputs as eagle_accept_greedy.
 * Device errors: NUMERIC (value outside [0,1] in a row the walk reads, or a
 * final distribution without mass), INVALID_ARG (token/row/uniform out of
 * range, walk deeper than max_depth), INVALID_TREE.
 * ---------------------------------------------------------------------- */
EAGLE_API eagle_status eagle_accept_stochastic(int B, int max_nodes, int V, int R, int mode,
                                     const int32_t *d_tree_off, const int32_t *d_parent,
                                     const int32_t *d_tokens, const float *d_q,
                                     const float *d_p_rows, const int32_t *d_p_row_of_node,
                                     const float *d_u_accept, const float *d_u_sample,
                                     int max_depth, int32_t *d_accept_len,
                                     int32_t *d_accepted_nodes, int32_t *d_out_tokens,
                                     int *d_status, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * eagle_accept_stochastic_logits -- eagle_accept_stochastic reading target
 * logits instead of probabilities.
 *
 * The walk reads q only for the nodes it visits (alpha + 1 of them per
 * sequence), so normalising every node's row beforehand is wasted work.
 * Here each visited row is normalised as it is loaded, with the same fp32
 * expression and the same instructions as eagle_lmhead_softmax's PROB mode
 * (see there), so given that call's d_row_lse the
 * probabilities, and with them every decision and token, are identical to
 * eagle_accept_stochastic fed with PROB mode's d_q.  Everything else is as
 * eagle_accept_stochastic.
 *
 * d_z [T,V] fp32 logits (EAGLE_LMHEAD_LOGITS output); d_row_lse [T] fp32;
 * temperature > 0, the value given to eagle_lmhead_softmax.
 * Device errors: as eagle_accept_stochastic (NUMERIC also for a non-finite
 * logit in a row the walk reads).
 * ---------------------------------------------------------------------- */
EAGLE_API eagle_status eagle_accept_stochastic_logits(
    int B, int max_nodes, int V, int R, int mode, const int32_t *d_tree_off,
    const int32_t *d_parent, const int32_t *d_tokens, const float *d_z, const float *d_row_lse,
    float temperature, const float *d_p_rows, const int32_t *d_p_row_of_node,
    const float *d_u_accept, const float *d_u_sample, int max_depth, int32_t *d_accept_len,
    int32_t *d_accepted_nodes, int32_t *d_out_tokens, int *d_status, eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * eagle_draft_expand -- EAGLE-2 dynamic draft tree: expand one level, or
 * finalize (rerank under the budget and emit the tree).
 * [EAGLE-2] §2 "EAGLE-2 的核心創新：動態草稿樹" items 1-3: per-node confidence,
 * adaptive expansion, greedy selection under a fixed draft-token budget.
 * A node's value is its cumulative draft log-prob.
 *
 * Expand (finalize == 0, level in [0, depth)): every frontier node takes the
 * top-k tokens of its draft row (log-prob descending, token ascending);
 * child score = fp32(parent score + logp); the next frontier is the top-k
 * children by (score desc, creation order).  Draft rows:
 *   d_draft_logp [B, R, V] fp32 with R = 1 + (depth-1)*k; level 0 reads row
 *   0 (the root's), level d >= 1 reads rows 1+(d-1)*k+f for frontier rank f.
 * Last level and finalize in one launch (finalize == 2, level == depth-1):
 * the CTA that completes a sequence's last level also finalizes it
 * (falls back to two launches when the pool is too large for that CTA's
 * shared memory); outputs as for finalize == 1.
 * Finalize (finalize == 1, after all `depth` levels): keep the top
 * d_budget[b] pool nodes by (score desc, creation order), number them by
 * (depth, score desc, creation order) after the root (node 0), and write
 *   d_tree_off [B+1], d_parent [T] (local), d_tokens [T] (root: d_root_token[b]),
 *   d_node_depth [T], d_score [T] (root 0), d_p_row_of_node [T] (global row
 *   b*R + local row; root -1),
 * where sequence b has min(budget[b], k + (depth-1)*k*k) + 1 nodes.
 *
 * d_pool: caller-owned scratch of eagle_draft_pool_bytes(B, k, depth, V)
 * bytes, reused by all levels of one tree build (level 0 resets it).
 * Arguments a role does not use may be NULL.  1 <= k <= min(32, V),
 * 1 <= depth <= 16.
 * Device errors: NUMERIC (non-finite log-prob), INVALID_ARG (negative budget).
 * ---------------------------------------------------------------------- */
EAGLE_API size_t eagle_draft_pool_bytes(int B, int k, int depth, int V);
EAGLE_API eagle_status eagle_draft_expand(int B, int V, int k, int depth, int level, int finalize,
                                const float *d_draft_logp, const int32_t *d_budget,
                                const int32_t *d_root_token, void *d_pool, size_t pool_bytes,
                                int32_t *d_tree_off, int32_t *d_parent, int32_t *d_tokens,
                                int32_t *d_node_depth, float *d_score,
                                int32_t *d_p_row_of_node, int *d_status,
                                eagle_stream_t stream);

/* eagle_draft_expand_all -- the whole EAGLE-2 tree build in one call: every
 * level (0 .. depth-1) and the finalize, with the same results as
 * eagle_draft_expand called for each level and then finalize (same
 * arguments, same outputs; budget, root_token and the tree outputs are
 * required).  Every level's draft rows must be ready before the previous
 * kernel on `stream` ends: one launch ranks the chunks of all levels at once,
 * then the levels are merged one launch each.  (Rows whose length is not a
 * multiple of 4 or that are not 16-byte aligned are built level by level.)
 * d_pool: eagle_draft_pool_bytes(B, k, depth, V) bytes, as above. */
EAGLE_API eagle_status eagle_draft_expand_all(int B, int V, int k, int depth,
                                    const float *d_draft_logp, const int32_t *d_budget,
                                    const int32_t *d_root_token, void *d_pool, size_t pool_bytes,
                                    int32_t *d_tree_off, int32_t *d_parent, int32_t *d_tokens,
                                    int32_t *d_node_depth, float *d_score,
                                    int32_t *d_p_row_of_node, int *d_status,
                                    eagle_stream_t stream);

/* eagle_draft_expand for draft rows written by the kernel queued just before
 * it on `stream` (the draft head of a draft -> verify loop): the same level
 * or finalize, with every row read only after that kernel has finished.
 * (eagle_draft_expand itself starts ranking a level's rows before the
 * previous kernel ends, which needs rows that were ready earlier.) */
EAGLE_API eagle_status eagle_draft_expand_dep(int B, int V, int k, int depth, int level,
                                    int finalize, const float *d_draft_logp,
                                    const int32_t *d_budget, const int32_t *d_root_token,
                                    void *d_pool, size_t pool_bytes, int32_t *d_tree_off,
                                    int32_t *d_parent, int32_t *d_tokens, int32_t *d_node_depth,
                                    float *d_score, int32_t *d_p_row_of_node, int *d_status,
                                    eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * The draft -> verify -> accept -> commit loop.
 * [EAGLE] workflow paragraph: the draft ("auto-regression") head reads the
 * target's feature and the embedding of the sampled token and predicts the
 * next feature; the frozen LM head gives the next-token distribution of
 * every draft node; the target verifies the whole tree in one pass; the
 * accepted tokens join the context.  A draft head is [f ; e] -> f' (one
 * matrix, eagle_gemm STORE) here, the LM head eagle_lmhead_softmax (LOGITS).
 * ---------------------------------------------------------------------- */

/* Input rows of the draft head for EAGLE-2 level `level` of a tree built by
 * eagle_draft_expand(_dep) in d_pool (same B, V, k, depth).  Level 0: row b
 * = [d_f_ctx[b] ; d_emb[d_root_token[b]]] (the root), d_node_cur[b] = -1.
 * Level d >= 1: the frontier the previous level left, by rank: row b*k + f =
 * [feature of the node's parent ; d_emb[node's token]], the parent's
 * feature taken from d_feat_prev [B*F_prev, H] bf16 (the previous call's
 * head output; F_prev = 1 at d = 1, else k) by matching the parent's pool
 * index in d_node_prev [B*F_prev]; d_node_cur [B*F] receives the rows' pool
 * indices.  d_a [B*F, 2H] bf16 (F = 1 at level 0, else k); d_emb [V, H]
 * bf16; d_f_ctx [B, H] bf16.  Device errors: INVALID_ARG. */
EAGLE_API eagle_status eagle_draft_head_input(int B, int V, int k, int depth, int level, int H,
                                    const void *d_pool, size_t pool_bytes,
                                    const int32_t *d_node_prev, int32_t *d_node_cur,
                                    const void *d_feat_prev, const void *d_f_ctx,
                                    const int32_t *d_root_token, const void *d_emb, void *d_a,
                                    int *d_status, eagle_stream_t stream);

/* Draft rows of one level from the LM head's logits of the level's B*F
 * draft nodes (d_z [B*F, V] fp32, d_lse [B*F]; F = 1 at level 0, else k):
 * row r = b*F + f becomes local row 0 (level 0) or 1 + (level-1)*k + f of
 * sequence b in d_logp [B, R, V] (R = 1 + (depth-1)*k) as z - lse (fp32),
 * and, if d_prob is given, in d_prob [B, R, V] as the probability with
 * eagle_lmhead_softmax's PROB-mode expression at temperature 1. */
EAGLE_API eagle_status eagle_draft_rows(int B, int V, int k, int depth, int level,
                                        const float *d_z, const float *d_lse, float *d_logp,
                                        float *d_prob, eagle_stream_t stream);

/* x [T, H] fp32 = d_emb[d_tokens[t]] (bf16 rows): the target's input rows
 * of the tree tokens.  Device errors: INVALID_ARG (token out of range). */
EAGLE_API eagle_status eagle_embed_rows(int T, int H, int V, const int32_t *d_tokens,
                                        const void *d_emb, float *d_x, int *d_status,
                                        eagle_stream_t stream);

/* After the acceptance walk: the next step's root token is the bonus token
 * d_out_tokens[b*(max_depth+1) + alpha], and its context feature
 * d_f_ctx [B, H] bf16 is the target's output (d_resid [T, H] fp32) at the
 * last accepted node.  Device errors: INVALID_ARG. */
EAGLE_API eagle_status eagle_loop_advance(int B, int H, int max_depth, const int32_t *d_tree_off,
                                          const int32_t *d_accept_len,
                                          const int32_t *d_accepted_nodes,
                                          const int32_t *d_out_tokens, const float *d_resid,
                                          void *d_f_ctx, int32_t *d_root_token, int *d_status,
                                          eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * eagle_draft_static -- EAGLE-1 static draft tree from a fixed template.
 * [EAGLE-2] §2 "EAGLE-2 的核心創新：動態草稿樹" (EAGLE-1's fixed top-k tree,
 * which the dynamic tree replaces); [S4000] "EAGLE的创新点" item 1 (the draft
 * keeps the top tokens at every step: K^m candidate paths for K per step
 * over m steps).
 *
 * The template (N nodes, root first, parents before children) is the same
 * for every sequence: node i >= 1 is the d_tmpl_rank[i]-th most probable
 * token (log-prob descending, token ascending) of the draft row that its
 * parent p = d_tmpl_parent[i] was expanded with, row d_tmpl_row[p] of the
 * sequence's rows.  Its score is fp32(score[p] + logp), as in
 * eagle_draft_expand.  Outputs use the template's numbering:
 *   d_tree_off [B+1] (= b*N), d_parent [B*N] (= the template), d_tokens
 *   (root: d_root_token[b]), d_node_depth, d_score (root 0),
 *   d_p_row_of_node (global row b*R + d_tmpl_row[p]; root -1).
 *
 * N          template nodes, 1 .. EAGLE_MAX_TREE_NODES.
 * R          draft rows per sequence: d_draft_logp is [B, R, V] fp32.
 * max_rank   every d_tmpl_rank[i] < max_rank <= min(EAGLE_MAX_TOPK, V).
 * d_tmpl_parent, d_tmpl_rank, d_tmpl_row [N] int32 (device); d_tmpl_row[i]
 *            is -1 (or anything) for a node without children.
 * Device errors: INVALID_TREE (template parents not topological),
 * INVALID_ARG (rank >= max_rank, an expanded node without a valid row),
 * NUMERIC (non-finite log-prob in a row that is read).
 * ---------------------------------------------------------------------- */
EAGLE_API eagle_status eagle_draft_static(int B, int V, int N, int R, int max_rank,
                                const int32_t *d_tmpl_parent, const int32_t *d_tmpl_rank,
                                const int32_t *d_tmpl_row, const float *d_draft_logp,
                                const int32_t *d_root_token, int32_t *d_tree_off,
                                int32_t *d_parent, int32_t *d_tokens, int32_t *d_node_depth,
                                float *d_score, int32_t *d_p_row_of_node, int *d_status,
                                eagle_stream_t stream);

/* ------------------------------------------------------------------------
 * The decoder layer around the tree attention.
 * [EAGLE] workflow paragraph; [S4000] "EAGLE的创新点" item 2: the verify pass
 * is one forward pass of the target model over every tree token.  The pages
 * name LLaMA-family targets without giving their layer, which is read here
 * as a pre-norm LLaMA layer:
 *     a  = rmsnorm(x) * g_attn                    eagle_rmsnorm
 *     q, k, v = a Wq^T, a Wk^T, a Wv^T, q and k rotated to each node's
 *               position (cache length + depth)  eagle_tree_rope_table +
 *                                                 eagle_gemm(QKV_ROPE)
 *     o  = tree attention                          eagle_tree_attn(_paged)
 *     h  = x + bf16(o) Wo^T                       eagle_cast_bf16 +
 *                                                 eagle_gemm(ACCUM)
 *     b  = rmsnorm(h) * g_mlp                     eagle_rmsnorm
 *     m  = silu(b Wg^T) * (b Wu^T)                eagle_gemm(SWIGLU)
 *     h += m Wd^T                                 eagle_gemm(ACCUM)
 * x, h are the fp32 residual stream [T, H]; every matrix-multiply operand and
 * q / k / v are bf16, accumulation fp32.
 * ---------------------------------------------------------------------- */

/* y [T,H] bf16 = x / sqrt(mean_j x[t,j]^2 + eps) * gain, x fp32 [T,H],
 * gain bf16 [H].  Device errors: NUMERIC (non-finite x). */
EAGLE_API eagle_status eagle_rmsnorm(int T, int H, float eps, const float *d_x,
                                     const void *d_gain, void *d_y, int *d_status,
                                     eagle_stream_t stream);

/* y[i] = bf16(x[i]) (round to nearest even), n elements. */
EAGLE_API eagle_status eagle_cast_bf16(size_t n, const float *d_x, void *d_y,
                                       eagle_stream_t stream);

/* Positions and rotations of the tree nodes.  Node i of sequence b sits at
 * position pos = L_b + depth(i) (where it would stand on its own
 * root-to-node path after the cache), L_b = kv_off[b+1] - kv_off[b] or
 * kv_len[b] (give exactly one of d_kv_off [B+1], d_kv_len [B]).  T =
 * tree_off[B] nodes.  Writes d_pos [T] and d_cos_sin [T, D/2, 2] fp32 =
 * (cos, sin) of pos * theta^(-2j/D): the angle formed and reduced modulo
 * 2 pi in fp64, sine and cosine in fp32 (within a few 1e-7).
 * Device errors: INVALID_TREE. */
EAGLE_API eagle_status eagle_tree_rope_table(int B, int T, int D, float theta,
                                             const int32_t *d_tree_off, const int32_t *d_parent,
                                             const int32_t *d_kv_off, const int32_t *d_kv_len,
                                             int32_t *d_pos, float *d_cos_sin, int *d_status,
                                             eagle_stream_t stream);

/* Tensor-core GEMM of the layer: Y = A W^T with A [T,K] bf16 (tree rows)
 * and W [N,K] bf16 (rows = output features, K contiguous), fp32
 * accumulation; N % 32 == 0, K % 8 == 0, pointers 16-byte aligned.  W is
 * streamed from memory once per 1024 rows of A.  The epilogue decides what
 * is written:
 *   EAGLE_EPI_STORE     d_y [T,N] bf16.
 *   EAGLE_EPI_ACCUM     d_accum [T,N] fp32 = R + Y with R = d_resid [T,N]
 *                       fp32 if given, else d_accum itself (in place).
 *   EAGLE_EPI_SWIGLU    W rows alternate 16 gate rows and the 16 matching
 *                       up rows; d_y [T,N/2] bf16 = silu(gate) * up.
 *   EAGLE_EPI_QKV_ROPE  N = (Hq + 2 Hkv) D; W = [Wq; Wk; Wv] with, inside
 *                       every q and k head, the rows of dimensions j and
 *                       j + D/2 adjacent (row 2j holds dimension j, row
 *                       2j+1 dimension j + D/2); q, k are rotated by
 *                       d_cos_sin (eagle_tree_rope_table) and written to
 *                       d_q [T,Hq,D], d_k [T,Hkv,D]; v to d_v [T,Hkv,D].
 * Arguments an epilogue does not use may be NULL / 0. */
EAGLE_API eagle_status eagle_gemm(int epilogue, int T, int N, int K, const void *d_a,
                                  const void *d_w, void *d_y, float *d_accum,
                                  const float *d_resid, void *d_q,
                                  void *d_k, void *d_v, const float *d_cos_sin, int Hq, int Hkv,
                                  int D, int *d_status, eagle_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* EAGLE_H_ */
