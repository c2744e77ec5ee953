/*
 * libjtree — one decode step of causal parallel tree drafting (JetSpec) on a
 * GB300 (sm_103a): per-depth top-W candidates, best-first tree expansion,
 * the tree-causal mask, tree attention for the verification pass, greedy
 * acceptance, the commit of the accepted path's K/V into the prefix cache,
 * and the draft LM head fused with the top-W selection.
 *
 * Sources (page title, site, section):
 *   [PL] "JetSpec: Breaking the Scaling Ceiling of Speculative Decoding with
 *        Parallel Tree Drafting", paperlayer.ai summary.
 *   [SM] the same paper, Korean review on startedourmission.github.io.
 *   [RB] the same paper, Chinese summary on paper.rainbus.top.
 *   [PP] "JetSpec++: Foresight Parallel Drafting with Self Refinements",
 *        paperlayer.ai summary.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every tensor pointer is a DEVICE pointer owned by the caller. The library
 *   never allocates, frees or synchronises (except jt_read_device_error).
 * - Every call is asynchronous on exec->stream and returns once the work is
 *   enqueued. A NULL exec means the legacy default stream, no device error
 *   word and no workspace.
 * - Arguments are validated on the host before anything is launched; a bad
 *   argument returns JT_ERR_INVALID_ARG or JT_ERR_UNSUPPORTED and launches
 *   nothing. A failed launch returns JT_ERR_CUDA.
 * - Values inside device buffers (parent ids, tokens, page ids, lengths) are
 *   checked on the device. A bad value ORs a JT_DEVERR_* flag into
 *   *exec->d_err (when non-NULL); the kernel then writes defined outputs
 *   (zeros, acc_len 0) and never traps. jt_read_device_error fetches and
 *   clears the word.
 * - Calls that need scratch memory take it from exec->workspace (device,
 *   caller-owned, 256-byte aligned, at least the size the matching
 *   jt_*_workspace_bytes query returns). Two calls in flight at the same
 *   time must not share a workspace.
 * - Tree node ids are 0..n-1 in creation order with parent[v] < v; parent -1
 *   means "child of the root". The root is the last prefix token, already in
 *   the KV cache; it is not a tree node.
 * - All pointers must be 16-byte aligned.
 * - The library keeps no global state except a per-process cache of the
 *   device's attributes, the wait budget of jt_set_wait_budget and the fixed
 *   array of jt_tree_accept_noalloc; it is safe to call from several host
 *   threads.
 */
#ifndef JTREE_H_
#define JTREE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define JT_API __attribute__((visibility("default")))
#else
#define JT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* jt_stream_t;

typedef enum {
  JT_OK = 0,
  JT_ERR_INVALID_ARG = 1,   /* null pointer, size out of range, misaligned pointer */
  JT_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement (e.g. head_dim 96) */
  JT_ERR_CUDA = 3,          /* a CUDA runtime call or launch failed */
  JT_ERR_DEVICE_DATA = 4,   /* jt_read_device_error found a device-side flag set */
  JT_ERR_TIMEOUT = 5,       /* a bounded device-side wait expired (flag JT_DEVERR_TIMEOUT) */
  JT_ERR_WORKSPACE = 6      /* exec->workspace missing or smaller than required */
} jt_status;

/* Bits of the device error word. */
#define JT_DEVERR_PARENT   0x01  /* parent[v] outside [-1, v) */
#define JT_DEVERR_TOKEN    0x02  /* a token id outside [0, vocab) */
#define JT_DEVERR_NNODES   0x04  /* n_nodes outside [0, B] */
#define JT_DEVERR_PAGE     0x08  /* a block-table page id outside the pool */
#define JT_DEVERR_PREFIX   0x10  /* prefix_len outside [0, max_prefix] */
#define JT_DEVERR_TIMEOUT  0x20  /* a bounded wait on an mbarrier ran out */
#define JT_DEVERR_PATH     0x40  /* acc_len outside [0, n_depth] or an accepted node outside [0, B) */

typedef struct {
  jt_stream_t stream;       /* stream every launch is enqueued on (NULL = default) */
  int32_t* d_err;           /* optional device int32 error word; NULL = no reporting */
  void* workspace;          /* optional caller-owned device scratch */
  size_t workspace_bytes;   /* its size */
} jt_exec;

JT_API const char* jt_status_str(jt_status s);

/* Synchronises exec->stream, copies *exec->d_err to *host_out and clears it.
 * Returns JT_OK when the word was zero, JT_ERR_TIMEOUT when the timeout flag
 * was set, JT_ERR_DEVICE_DATA for any other flag, JT_ERR_INVALID_ARG when
 * exec or exec->d_err is NULL. */
JT_API jt_status jt_read_device_error(const jt_exec* exec, int32_t* host_out);

/* Test hook, not part of the method (the pages have no counterpart).
 * Every wait of a kernel on an mbarrier (jt_tree_attn, jt_lmhead_topw) gives
 * up after a budget of SM clock cycles, about 2 s by default; the CTA then
 * sets JT_DEVERR_TIMEOUT in *exec->d_err, waits (again bounded, always with
 * the default budget) for the TMA loads and tensor-core operations it has
 * already issued, releases its tensor memory and finishes, leaving the
 * context usable. This call sets the budget given to kernels launched
 * afterwards by this process; cycles <= 0 restores the default. A budget of
 * a few cycles makes every such call report a timeout, which is how the
 * tests drive that path. Always returns JT_OK. */
JT_API jt_status jt_set_wait_budget(long long cycles);

/* ------------------------------------------------------------------------
 * jt_topw — top-W draft candidates per depth.
 * [PL] App. E "Drafting": the proposer extracts the top-k tokens and their
 * log-probabilities at each future position; [RB] "方法步骤详情": one draft
 * pass yields logits for every depth and the top W candidates per depth.
 *
 *   logits : fp32 [batch][n_depth][vocab], row-major, read only
 *   tok    : int32 [batch][n_depth][W]  token ids by logit, descending;
 *            equal logits rank the lower token id first
 *   logp   : fp32 [batch][n_depth][W]  log-softmax of those tokens over the
 *            full vocabulary, x - m - log(sum_j exp(x_j - m))
 * Limits: 1 <= W <= min(vocab, 32); vocab % 4 == 0; batch * n_depth >= 0.
 * NaN logits are undefined; -inf is allowed as long as a row has one finite
 * logit. Workspace: jt_topw_workspace_bytes (may be 0).
 * ------------------------------------------------------------------------ */
JT_API size_t jt_topw_workspace_bytes(int batch, int n_depth, int vocab, int W);
JT_API jt_status jt_topw(const float* logits, int batch, int n_depth, int vocab, int W,
                  int32_t* tok, float* logp, const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_topw_entropy — jt_topw plus the entropy of each depth's draft
 * distribution, from the same single pass over the logits.
 * [PL] App. C "Tree-Drafting Algorithm Ablation" and App. E "Drafting": the
 * proposer supports entropy-guided and hybrid scores built from the
 * per-depth (marginal) entropy; jt_tree_expand_scored consumes it.
 *
 *   entropy fp32 [batch][n_depth]: H = -sum_j p_j ln p_j (nats) with
 *           p = softmax(logits row); -inf logits contribute nothing; a row of
 *           all -inf reports 0.
 * Everything else (arguments, outputs, limits) as jt_topw. H is accumulated
 * in fp32 (online, rescaled with the running max): |error| <= 2e-4 nats for
 * rows of 151936 logits.
 * ------------------------------------------------------------------------ */
JT_API jt_status jt_topw_entropy(const float* logits, int batch, int n_depth, int vocab, int W,
                                 int32_t* tok, float* logp, float* entropy, const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_tree_expand — budget-B best-first tree construction.
 * [PL] App. B "Tree-Drafting Algorithm Details" (Algorithm 1) and §2 "Tree
 * Construction and Verification"; [RB] "方法步骤详情"; branch score =
 * cumulative draft log-probability, [SM] "How it works", s(π(v)) equation.
 *
 * Starting from the root (depth 0, score 0), repeatedly pop the expandable
 * node with the highest score (ties: lower node id; the root first) and
 * attach children r = 0..W-1 while fewer than B nodes exist. A child of a
 * depth-d node takes token tok[b][d][r] (depth d+1's rank-r candidate) and
 * score parent + logp[b][d][r] (one binary32 add). Children with depth < N
 * are pushed back; stop when B nodes exist or nothing is expandable.
 *
 *   tok, logp : [batch][n_depth][W] (the output of jt_topw)
 *   parent    : int32 [batch][B]  creation-order ids, -1 = child of root
 *   token     : int32 [batch][B]
 *   depth     : int32 [batch][B]  1..n_depth
 *   score     : fp32  [batch][B]  cumulative log-prob
 *   n_nodes   : int32 [batch]     nodes built (<= B); slots >= n_nodes hold
 *               parent -1, token -1, depth 0, score 0
 * Limits: 1 <= B <= 256, 1 <= n_depth <= 64, 1 <= W <= 32. No workspace.
 * ------------------------------------------------------------------------ */
JT_API jt_status jt_tree_expand(const int32_t* tok, const float* logp, int batch, int n_depth, int W,
                         int B, int32_t* parent, int32_t* token, int32_t* depth, float* score,
                         int32_t* n_nodes, const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_tree_expand_scored — jt_tree_expand with a choice of branch score.
 * [PL] App. C "Tree-Drafting Algorithm Ablation" and App. E "Drafting":
 * cumulative log-prob (the production default), entropy-guided and hybrid
 * scores, the hybrid weight alpha interpolating between the two (alpha -> 0
 * gives cumulative log-prob, alpha -> inf entropy-only). The pages give no
 * formula; this library reads it as the child's score increment
 *   JT_SCORE_LOGP    (0): logp[d][r]
 *   JT_SCORE_HYBRID  (1): logp[d][r] - alpha * H_d   (binary32 multiply, then subtract)
 *   JT_SCORE_ENTROPY (2): -H_d
 * for a child at depth d with candidate rank r, H_d from jt_topw_entropy,
 * so a hybrid score is cum_logp - alpha * sum of H over the path's depths.
 * Expansion, outputs, limits and device checks as jt_tree_expand (mode 0 is
 * exactly jt_tree_expand). entropy fp32 [batch][n_depth] may be NULL in mode 0;
 * alpha must be finite and >= 0 in mode 1.
 * ------------------------------------------------------------------------ */
typedef enum { JT_SCORE_LOGP = 0, JT_SCORE_HYBRID = 1, JT_SCORE_ENTROPY = 2 } jt_score_mode;
JT_API jt_status jt_tree_expand_scored(const int32_t* tok, const float* logp, const float* entropy,
                                       int batch, int n_depth, int W, int B, int mode, float alpha,
                                       int32_t* parent, int32_t* token, int32_t* depth,
                                       float* score, int32_t* n_nodes, const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_tree_mask — tree-causal attention mask as ancestor bitmasks.
 * [SM] "How it works", mask equation: M[v,u] = 0 iff u ∈ Anc(v) ∪ {v};
 * [PL] App. E "Verification": the mask is applied without a dense
 * per-request matrix.
 *
 *   parent  : int32 [batch][B], n_nodes : int32 [batch]
 *   mask    : uint32 [batch][B][(B+31)/32]; bit (u & 31) of word (u >> 5)
 *             of row v is set iff M[v,u] = 0. Rows v >= n_nodes are zero.
 * Device check: parent[v] outside [-1, v) sets JT_DEVERR_PARENT and zeroes
 * that sequence's rows. Limits: 1 <= B <= 256. No workspace.
 * ------------------------------------------------------------------------ */
JT_API jt_status jt_tree_mask(const int32_t* parent, const int32_t* n_nodes, int batch, int B,
                       uint32_t* mask, const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_tree_attn — tree-causal GQA attention for the verification pass.
 * [PL] §2 "Architecture" and App. E "Verification"; [SM] mask equation.
 *
 * For node v < n_nodes[b] and query head h (KV head h / (hq/hkv)):
 *   o = softmax(scale * q K^T + mask) V over the keys
 *       prefix[0 .. prefix_len[b])  ∪  { tree node u : mask[b][v] bit u }
 * fp32 softmax and accumulation, bf16 output. Rows v >= n_nodes[b] are zero.
 *
 *   q            bf16 [batch][B][hq][D]
 *   k_tree/v_tree bf16 [batch][B][hkv][D]   (the tree nodes' own K/V)
 *   contiguous prefix (block_table == NULL):
 *     k_cache/v_cache bf16 [batch][max_prefix][hkv][D]
 *   paged prefix (block_table != NULL):
 *     k_cache/v_cache bf16 [n_pages][page_size][hkv][D] pool,
 *     block_table int32 [batch][max_pages]; token j of sequence b lives in
 *     page block_table[b][j / page_size], slot j % page_size.
 *   prefix_len   int32 [batch], n_nodes int32 [batch]
 *   mask         uint32 [batch][B][(B+31)/32] (jt_tree_mask's output)
 *   out          bf16 [batch][B][hq][D]
 *   scale        > 0; 0 means 1/sqrt(D)
 * Limits: D in {64, 128}; hq % hkv == 0; hq/hkv in {1, 2, 4, 8, 16}; 1 <= B <= 256;
 * page_size == 16 when paged. Workspace: jt_tree_attn_workspace_bytes. Work
 * is cut into (sequence, KV head, 256-row block) units. When two CTAs per unit
 * fit on the SMs at once, each unit's key range is split over a cluster of up
 * to 8 CTAs whose fp32 partial outputs meet in this scratch (at most SM count
 * x (256 D + 1024) x 4 bytes; 0 when no split can apply). Otherwise the
 * units run longest first (an order of 8 bytes per unit in the scratch), and
 * while units are fewer than twice the SMs the long ones are cut into up to
 * ceil(2 SMs / units) chunks with one (256 D + 512) x 4-byte partial each.
 * Device checks: prefix_len beyond max_prefix (or max_pages*page_size), a page
 * id outside [0, n_pages) and n_nodes outside [0, B] set flags; the affected
 * sequence's output is zero.
 * ------------------------------------------------------------------------ */
typedef struct {
  int batch, B, hq, hkv, head_dim;
  float scale;
  const void* q;
  const void* k_tree;
  const void* v_tree;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;   /* NULL = contiguous prefix */
  int page_size, max_pages, n_pages;
  int max_prefix;               /* contiguous: cache length; paged: 0 or a bound on prefix_len */
  const int32_t* prefix_len;
  const int32_t* n_nodes;
  const uint32_t* mask;
  void* out;
} jt_attn_args;

JT_API size_t jt_tree_attn_workspace_bytes(const jt_attn_args* args);
JT_API jt_status jt_tree_attn(const jt_attn_args* args, const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_tree_accept — greedy (temperature 0) acceptance.
 * [PL] §2 "Tree Construction and Verification": accept the longest prefix
 * whose draft tokens meet the target's condition; [RB] "前置知识"; [PP] §3
 * "Preliminaries": commit the accepted prefix plus one bonus token.
 *
 *   target  fp32 [batch][B+1][vocab]: row 0 is the target's prediction at the
 *           root, row 1+v at node v. Argmax ties go to the lowest token id.
 *   Walk: a = argmax(row 0); while a child c of the current node has
 *   token[c] == a (the lowest id if several): accept c, a = argmax(row 1+c).
 *   acc_len    int32 [batch]            accepted draft tokens (0..n_depth)
 *   acc_tokens int32 [batch][n_depth]   their tokens, -1 beyond acc_len
 *   acc_nodes  int32 [batch][n_depth]   their node ids, -1 beyond acc_len
 *   bonus      int32 [batch]            the last argmax (committed too)
 * Committed tokens this step = acc_len + 1.
 * Limits: 1 <= B <= 256, 1 <= n_depth <= 64, vocab % 4 == 0.
 * Workspace: jt_tree_accept_workspace_bytes (0 when the tree is much wider
 * than a root path, (B+1) > 4(N+1): then only path rows are read, one
 * thread-block cluster per sequence). Device checks: bad parent, token
 * or n_nodes set a flag and give acc_len 0, bonus -1 for that sequence.
 * ------------------------------------------------------------------------ */
JT_API size_t jt_tree_accept_workspace_bytes(int batch, int B, int n_depth, int vocab);
JT_API jt_status jt_tree_accept(const float* target_logits, const int32_t* parent, const int32_t* token,
                         const int32_t* n_nodes, int batch, int B, int n_depth, int vocab,
                         int32_t* acc_len, int32_t* acc_tokens, int32_t* acc_nodes,
                         int32_t* bonus, const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_tree_accept_sampled — temperature-T (T > 0) acceptance.
 * [PP] App. F.3 "Lossless verification": every committed token is the
 * target's own draw at any temperature; a draft fixed before verification is
 * checked with point-mass proposals, each draft token accepted with the
 * target probability. [PP] App. F.1 gives the chain example: P(accept d1,
 * reject d2, draw b) = p(d1) p(b | d1) = 0.24.
 *
 * Walk (this library's reading for trees; for a chain it is the rule above):
 * at the current node draw y from softmax(target row / T); if a child has
 * token y, accept it and continue from it; otherwise y is the bonus token.
 * The draw is Gumbel-max, y = argmax_j (x_j * inv_T + G_j) (lowest j on
 * ties) with inv_T = 1.0f / temperature in binary32 and counter-based noise:
 *   k = ((b * (B+1) + r) << 32 | j) + 1   (r = 0: root row, 1+v: node v)
 *   h = output k of SplitMix64 seeded with `seed`
 *   U = ((h >> 41) + 0.5) * 2^-23,  G_j = -ln(-ln U)
 * with ln evaluated by the atanh series in binary32 (so results are exactly
 * reproducible from (seed, inputs)). The same seed on the same inputs gives
 * the same walk; a caller draws a fresh seed per round.
 * Arguments, outputs, limits, workspace (jt_tree_accept_workspace_bytes) and
 * device checks as jt_tree_accept; temperature must be finite and > 0 (use
 * jt_tree_accept for T = 0). A row whose logits are all -inf has no
 * distribution and gives an unspecified token.
 * ------------------------------------------------------------------------ */
JT_API jt_status jt_tree_accept_sampled(const float* target_logits, const int32_t* parent,
                                        const int32_t* token, const int32_t* n_nodes, int batch,
                                        int B, int n_depth, int vocab, float temperature,
                                        uint64_t seed, int32_t* acc_len, int32_t* acc_tokens,
                                        int32_t* acc_nodes, int32_t* bonus,
                                        const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_tree_accept_noalloc — jt_tree_accept for callers that cannot allocate.
 * The paper has no counterpart: this is a library convenience.
 *
 * Same arguments, results and device checks as jt_tree_accept, but the
 * scratch it needs (per-row argmaxes) comes from a fixed array inside the
 * library's device image instead of exec->workspace (which is ignored;
 * exec->stream and exec->d_err are used as by jt_tree_accept). It is meant
 * for callers that must not call cudaMalloc or any allocating routine — for
 * example runtimes whose device memory is entirely owned by another
 * allocator, plain C hosts with no device allocator at hand, or code that
 * cannot afford cudaMalloc's device synchronisation — so this call
 * allocates nothing.
 * Only chains and trees not much wider than a root path use the array:
 * when (B+1) > 4 (n_depth+1) the call walks the accepted path without any
 * scratch, and such calls neither touch nor race on the array.
 *
 * Limit: batch * (B + 1) <= 65536; larger requests return
 * JT_ERR_UNSUPPORTED without launching. The array (256 KiB) lives on every
 * GPU that loads the library until the process exits.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture that includes this entry point.
 * Every call on a device shares the one array and it keeps the last call's
 * contents; nothing in it needs to start at zero (each call writes every
 * entry it reads before reading it). Calls that overlap on the GPU (on
 * different streams, or from different host threads without ordering) race
 * on the array and give undefined results: serialise them.
 * ------------------------------------------------------------------------ */
JT_API jt_status jt_tree_accept_noalloc(const float* target_logits, const int32_t* parent,
                                        const int32_t* token, const int32_t* n_nodes, int batch,
                                        int B, int n_depth, int vocab, int32_t* acc_len,
                                        int32_t* acc_tokens, int32_t* acc_nodes, int32_t* bonus,
                                        const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_tree_commit_kv — append the accepted path's K/V to the prefix cache.
 * [PP] §3 "Preliminaries": a verification round commits the accepted prefix
 * plus one bonus token. The accepted draft nodes' K/V were produced by the
 * verification pass (rows of k_tree / v_tree), so committing them copies
 * those rows into the cache after the prefix, in path order. The bonus
 * token has no K/V yet (the next round produces it when it verifies that
 * token as its root) and is not written.
 *
 * For sequence b with L = prefix_len[b], a = acc_len[b] (from jt_tree_accept):
 *   cache position L + i  <-  tree row acc_nodes[b][i], i = 0 .. a-1, for
 *                              every KV head, K and V
 *   new_prefix_len[b] = L + a
 *
 *   k_tree, v_tree  bf16 [batch][B][hkv][D]        read only
 *   k_cache, v_cache: contiguous (block_table == NULL) bf16
 *                   [batch][max_prefix][hkv][D]; paged: pool
 *                   [n_pages][page_size][hkv][D] with block_table int32
 *                   [batch][max_pages] (token j of sequence b in page
 *                   block_table[b][j / page_size], slot j % page_size).
 *                   Only the committed slots are written.
 *   prefix_len      int32 [batch]
 *   acc_len         int32 [batch], acc_nodes int32 [batch][n_depth]
 *   new_prefix_len  int32 [batch]; may alias prefix_len (the call reads every
 *                   length before writing any)
 * Limits: 1 <= B <= 256, 1 <= n_depth <= 64, hkv >= 1, head_dim % 8 == 0,
 * hkv * head_dim <= 4096, page_size == 16 when paged. No workspace.
 * Device checks: a outside [0, n_depth] or an accepted node outside [0, B)
 * (JT_DEVERR_PATH), L < 0 or L + a beyond the cache (max_prefix, or
 * max_pages * page_size) (JT_DEVERR_PREFIX), a page id outside [0, n_pages)
 * among the slots to write (JT_DEVERR_PAGE): that sequence is left untouched
 * and new_prefix_len[b] = L.
 * ------------------------------------------------------------------------ */
typedef struct {
  int batch, B, n_depth, hkv, head_dim;
  const void* k_tree;
  const void* v_tree;
  void* k_cache;
  void* v_cache;
  const int32_t* block_table;   /* NULL = contiguous cache */
  int page_size, max_pages, n_pages;
  int max_prefix;               /* contiguous: positions per sequence */
  const int32_t* prefix_len;
  const int32_t* acc_len;
  const int32_t* acc_nodes;
  int32_t* new_prefix_len;
} jt_commit_args;

JT_API jt_status jt_tree_commit_kv(const jt_commit_args* args, const jt_exec* exec);

/* ------------------------------------------------------------------------
 * jt_lmhead_topw — draft logits through the LM head, reduced to top-W.
 * [PL] App. E "Training and evaluation details": the draft model reuses the
 * frozen target LM head, so depth d's draft logits are its hidden state times
 * the LM-head matrix; [PL] App. E "Drafting": the proposer keeps the top-k
 * tokens and log-probs per position. This call computes
 *   logits[r][v] = sum_k hidden[r][k] * w_lm[v][k]   (bf16 x bf16, fp32 sums)
 * and returns exactly what jt_topw (or jt_topw_entropy) returns for those
 * logits, without writing them to memory.
 *
 *   hidden   bf16 [rows][d]        (rows = batch * n_depth draft positions)
 *   w_lm     bf16 [vocab][d]       (the LM-head weight, row per token)
 *   tok      int32 [rows][W], logp fp32 [rows][W]   (as jt_topw)
 *   entropy  fp32 [rows] or NULL   (as jt_topw_entropy)
 * The logits are fp32 sums of exact bf16 products in the tensor cores'
 * order, so they differ from an exact dot product by rounding; top-W indices
 * agree with exact logits except between candidates closer than that.
 * Limits: d % 64 == 0, 1 <= W <= min(32, vocab). Workspace:
 * jt_lmhead_topw_workspace_bytes (one small partial per row and 512-token
 * slice of the vocabulary). No device-side data checks apply.
 * ------------------------------------------------------------------------ */
JT_API size_t jt_lmhead_topw_workspace_bytes(int rows, int d, int vocab, int W);
JT_API jt_status jt_lmhead_topw(const void* hidden, const void* w_lm, int rows, int d, int vocab,
                                int W, int32_t* tok, float* logp, float* entropy,
                                const jt_exec* exec);

#ifdef __cplusplus
}
#endif

#endif  /* JTREE_H_ */
