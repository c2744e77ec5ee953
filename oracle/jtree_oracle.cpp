// Oracle for one decode step of causal parallel tree drafting (JetSpec).
//
// TEST INFRASTRUCTURE ONLY. Nothing in the product path may link, import or
// call this file: only tests/, __graft_entry__.smoke() and bench.py's
// cpu_baseline / --impl reference legs use it. It shares no code, header,
// table or helper with the CUDA library; the two meet only at the seeded
// input bytes.
//
// Plain, slow, single-threaded C++17 written from the definitions on the
// pages (compiled with -O2 -ffp-contract=off, no fast-math):
//   orc_tree_mask    - the tree-causal mask M[v,u] (explicit ancestor walk)
//   orc_tree_attn    - attention with an explicit dense mask, fp64 softmax
//   orc_topw         - full stable sort of the vocabulary + fp64 log-softmax
//   orc_row_entropy  - fp64 Shannon entropy of softmax(row), in nats
//   orc_tree_expand  - best-first expansion on a std::priority_queue
//                      (orc_tree_expand_scored: hybrid / entropy-only scores)
//   orc_tree_accept  - sequential argmax + walk down the tree
//   orc_tree_commit_kv - append the accepted path's K/V rows to the prefix cache
//   orc_tree_accept_sampled - temperature-T acceptance, one target draw per node
//
// Sources (page title, site, section):
//   [PL]  "JetSpec: Breaking the Scaling Ceiling of Speculative Decoding with
//         Parallel Tree Drafting", paperlayer.ai summary.
//   [SM]  the same paper, Korean review on startedourmission.github.io.
//   [RB]  the same paper, Chinese summary on paper.rainbus.top.
//   [PP]  "JetSpec++: Foresight Parallel Drafting with Self Refinements",
//         paperlayer.ai summary.
//
// Every function returns 0 on success and a negative code on bad input
// (it never aborts), so tests can drive it with hand-made bad trees.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <numeric>
#include <queue>
#include <vector>

namespace {

constexpr int kBadArg = -1;
constexpr int kBadTree = -2;
constexpr int kBadToken = -3;

// SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
// generators", OOPSLA 2014): the state advances by the golden-ratio gamma and
// each output is the state passed through the 64-bit finaliser. Output k
// (k = 1, 2, ...) of the generator seeded with s is mix64(s + k * gamma), so
// any output can be computed directly from its index.
uint64_t splitmix64_output(uint64_t seed, uint64_t k) {
  uint64_t z = seed + k * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// Natural log of a positive normal binary32 from ln(m 2^e) = e ln2 +
// 2 atanh(f), f = (m-1)/(m+1), m in [sqrt(1/2), sqrt(2)), with the atanh
// series f + f^3/3 + ... + f^9/9 (|f| <= 0.172, truncation < 1e-8 relative).
// Every step is one binary32 operation (fused multiply-adds where written),
// so any implementation that takes the same steps gets the same bits.
float series_ln(float x) {
  uint32_t u;
  std::memcpy(&u, &x, sizeof u);
  int e = static_cast<int>(u >> 23) - 127;
  const uint32_t mb = (u & 0x7FFFFFu) | 0x3F800000u;
  float m;
  std::memcpy(&m, &mb, sizeof m);
  if (m > 1.41421356f) { m = m * 0.5f; e += 1; }
  const float f = (m - 1.0f) / (m + 1.0f);
  const float f2 = f * f;
  float p = std::fma(f2, 1.0f / 9.0f, 1.0f / 7.0f);
  p = std::fma(p, f2, 0.2f);
  p = std::fma(p, f2, 1.0f / 3.0f);
  p = std::fma(p, f2, 1.0f);
  const float lm = (2.0f * f) * p;
  return std::fma(static_cast<float>(e), 0.693147182f, lm);
}

// Gumbel(0,1) noise for draw index k of the stream `seed`: U from the top 23
// bits of the k-th SplitMix64 output, U = (bits + 1/2) 2^-23 in (0, 1), and
// G = -ln(-ln U) with series_ln.
float gumbel_noise(uint64_t seed, uint64_t k) {
  const uint64_t h = splitmix64_output(seed, k);
  const float u = (static_cast<float>(static_cast<uint32_t>(h >> 41)) + 0.5f) * 1.1920928955078125e-7f;
  return -series_ln(-series_ln(u));
}

double widen_bf16(uint16_t bits) {
  // A bf16 value is the top half of an IEEE binary32; widening is exact.
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

}  // namespace

extern "C" {

// ---------------------------------------------------------------------------
// Tree-causal mask. [SM] "How it works", mask equation:
//   M[v,u] = 0 if u in Anc(v) ∪ {v}, else -inf.
// [PL] §2 "Architecture": every node sees the prefix and its own ancestors,
// never descendants or unrelated siblings.
// Node ids are 0..n-1 in creation order; parent[v] = -1 means "child of the
// root" (the root is the last prefix token and is not a tree node).
// Output: for each node v a row of ceil(B/32) uint32 words, bit (u & 31) of
// word (u >> 5) set iff M[v,u] = 0. Rows v >= n are zero.
// Returns kBadTree if some parent[v] is outside [-1, v).
// ---------------------------------------------------------------------------
int orc_tree_mask(const int32_t* parent, const int32_t* n_nodes, int batch, int B,
                  uint32_t* mask) {
  if (batch < 0 || B < 0) return kBadArg;
  const int words = (B + 31) / 32;
  std::fill(mask, mask + static_cast<size_t>(batch) * B * words, 0u);
  for (int b = 0; b < batch; ++b) {
    const int n = n_nodes[b];
    if (n < 0 || n > B) return kBadTree;
    const int32_t* par = parent + static_cast<size_t>(b) * B;
    for (int v = 0; v < n; ++v)
      if (par[v] < -1 || par[v] >= v) return kBadTree;
    // Dense boolean matrix first, exactly as the definition reads.
    std::vector<char> visible(static_cast<size_t>(n) * n, 0);
    for (int v = 0; v < n; ++v) {
      visible[static_cast<size_t>(v) * n + v] = 1;  // u = v
      for (int u = par[v]; u != -1; u = par[u])      // u in Anc(v)
        visible[static_cast<size_t>(v) * n + u] = 1;
    }
    for (int v = 0; v < n; ++v)
      for (int u = 0; u < n; ++u)
        if (visible[static_cast<size_t>(v) * n + u])
          mask[(static_cast<size_t>(b) * B + v) * words + (u >> 5)] |= 1u << (u & 31);
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Tree-causal GQA attention for the verification pass.
// [PL] App. E "Verification": the target verifies every node in one forward
// pass using the tree attention mask; [PL] §2: each node attends to the
// prefix plus its ancestors and itself.
//
// For node v of sequence b and query head h (KV head h / (hq / hkv)):
//   keys  = prefix tokens 0..L_b-1  ∪  tree nodes u < n_b
//   s_j   = scale * <q, k_j>, plus the mask term (0 or -inf) for tree keys
//   out   = sum_j softmax(s)_j v_j
// Everything after widening the bf16 inputs is done in double.
//
// Layouts (element = bf16 bit pattern, uint16):
//   q, out rows : [batch][B][hq][D]   (out is double)
//   k/v_tree    : [batch][B][hkv][D]
//   contiguous prefix (block_table == NULL): [batch][max_prefix][hkv][D]
//   paged prefix: pool [pages][page_size][hkv][D], token j of sequence b in
//                 page block_table[b * max_pages + j / page_size], slot
//                 j % page_size.
// rows / n_rows: optional list of (b, v, h) triples to compute; out then has
// n_rows rows of D doubles. rows == NULL computes all batch*B*hq rows.
// Rows with v >= n_b are zero.
// ---------------------------------------------------------------------------
int orc_tree_attn(int batch, int B, int hq, int hkv, int D, double scale,
                  const uint16_t* q, const uint16_t* k_tree, const uint16_t* v_tree,
                  const uint16_t* k_cache, const uint16_t* v_cache,
                  const int32_t* block_table, int page_size, int max_pages,
                  int max_prefix, int n_pool_pages,
                  const int32_t* prefix_len, const int32_t* n_nodes,
                  const uint32_t* mask, const int32_t* rows, int n_rows, double* out) {
  if (batch < 0 || B < 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || D <= 0) return kBadArg;
  const int g = hq / hkv;
  const int words = (B + 31) / 32;
  if (scale == 0.0) scale = 1.0 / std::sqrt(static_cast<double>(D));
  const long total = rows ? n_rows : static_cast<long>(batch) * B * hq;

  std::vector<double> s, qv(D), acc(D);
  for (long r = 0; r < total; ++r) {
    int b, v, h;
    if (rows) {
      b = rows[3 * r]; v = rows[3 * r + 1]; h = rows[3 * r + 2];
      if (b < 0 || b >= batch || v < 0 || v >= B || h < 0 || h >= hq) return kBadArg;
    } else {
      b = static_cast<int>(r / (static_cast<long>(B) * hq));
      v = static_cast<int>((r / hq) % B);
      h = static_cast<int>(r % hq);
    }
    double* o = out + r * D;
    std::fill(o, o + D, 0.0);
    const int n = n_nodes[b];
    const int L = prefix_len[b];
    if (n < 0 || n > B) return kBadTree;
    if (v >= n) continue;  // unused budget slot: defined as zero
    if (L < 0 || (!block_table && L > max_prefix) ||
        (block_table && L > max_pages * page_size)) return kBadArg;
    const int kh = h / g;

    const uint16_t* qrow = q + ((static_cast<size_t>(b) * B + v) * hq + h) * D;
    for (int d = 0; d < D; ++d) qv[d] = widen_bf16(qrow[d]);

    auto prefix_row = [&](const uint16_t* base, int j) -> const uint16_t* {
      size_t tok;
      if (block_table) {
        const int page = block_table[static_cast<size_t>(b) * max_pages + j / page_size];
        if (page < 0 || page >= n_pool_pages) return nullptr;
        tok = static_cast<size_t>(page) * page_size + j % page_size;
      } else {
        tok = static_cast<size_t>(b) * max_prefix + j;
      }
      return base + (tok * hkv + kh) * D;
    };
    auto tree_row = [&](const uint16_t* base, int u) -> const uint16_t* {
      return base + ((static_cast<size_t>(b) * B + u) * hkv + kh) * D;
    };

    // Scores over all L + n keys; the dense mask term is explicit.
    const double neg_inf = -std::numeric_limits<double>::infinity();
    s.assign(static_cast<size_t>(L) + n, 0.0);
    for (int j = 0; j < L; ++j) {
      const uint16_t* kr = prefix_row(k_cache, j);
      if (!kr) return kBadArg;
      double dot = 0.0;
      for (int d = 0; d < D; ++d) dot += qv[d] * widen_bf16(kr[d]);
      s[j] = scale * dot;
    }
    const uint32_t* mrow = mask + (static_cast<size_t>(b) * B + v) * words;
    for (int u = 0; u < n; ++u) {
      const bool visible = (mrow[u >> 5] >> (u & 31)) & 1u;
      double dot = 0.0;
      const uint16_t* kr = tree_row(k_tree, u);
      for (int d = 0; d < D; ++d) dot += qv[d] * widen_bf16(kr[d]);
      s[L + u] = scale * dot + (visible ? 0.0 : neg_inf);
    }
    // Max-subtracted softmax; a row with no visible key stays zero.
    double m = neg_inf;
    for (double x : s) m = std::max(m, x);
    if (m == neg_inf) continue;
    double denom = 0.0;
    std::fill(acc.begin(), acc.end(), 0.0);
    for (size_t j = 0; j < s.size(); ++j) {
      if (s[j] == neg_inf) continue;
      const double p = std::exp(s[j] - m);
      denom += p;
      const uint16_t* vr = (static_cast<int>(j) < L) ? prefix_row(v_cache, static_cast<int>(j))
                                                       : tree_row(v_tree, static_cast<int>(j) - L);
      for (int d = 0; d < D; ++d) acc[d] += p * widen_bf16(vr[d]);
    }
    for (int d = 0; d < D; ++d) o[d] = acc[d] / denom;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Per-depth top-W candidates. [PL] App. E "Drafting": the proposer takes the
// top-k tokens and their log-probabilities at each future position;
// [RB] "方法步骤详情" (inference): one draft pass gives logits for every
// depth, and the top W candidates are extracted per depth.
//
// For each row (b, d) of V fp32 logits:
//   order  : full stable sort of token ids by logit, descending (ties keep
//            the lower id first), take the first W;
//   logp_i : x_i - m - log(sum_j exp(x_j - m)), m = max_j x_j, in double,
//            rounded once to float.
// ---------------------------------------------------------------------------
int orc_topw(const float* logits, int batch, int n_depth, int vocab, int W,
             int32_t* tok, float* logp) {
  if (batch < 0 || n_depth < 0 || vocab <= 0 || W <= 0 || W > vocab) return kBadArg;
  std::vector<int32_t> idx(vocab);
  for (long row = 0; row < static_cast<long>(batch) * n_depth; ++row) {
    const float* x = logits + row * static_cast<long>(vocab);
    double m = -std::numeric_limits<double>::infinity();
    for (int j = 0; j < vocab; ++j) m = std::max(m, static_cast<double>(x[j]));
    double Z = 0.0;
    for (int j = 0; j < vocab; ++j) Z += std::exp(static_cast<double>(x[j]) - m);
    const double logZ = std::log(Z);
    std::iota(idx.begin(), idx.end(), 0);
    std::stable_sort(idx.begin(), idx.end(), [x](int32_t a, int32_t c) { return x[a] > x[c]; });
    for (int r = 0; r < W; ++r) {
      tok[row * W + r] = idx[r];
      logp[row * W + r] = static_cast<float>(static_cast<double>(x[idx[r]]) - m - logZ);
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Per-depth entropy of the draft distribution. [PL] App. C "Tree-Drafting
// Algorithm Ablation" and App. E "Drafting": besides cumulative log-prob the
// proposer supports entropy-guided and hybrid scores built from the per-depth
// (marginal) entropy of the draft distribution.
//   H = -sum_j p_j ln p_j,  p = softmax(row)   (nats)
// computed in double as ln Z - sum_j (x_j - m) e^(x_j - m) / Z with m the row
// max and Z = sum_j e^(x_j - m); -inf logits contribute nothing (p ln p -> 0).
// A row of all -inf has no distribution; its entropy is reported as 0.
// ---------------------------------------------------------------------------
int orc_row_entropy(const float* rows, long n_rows, int vocab, float* entropy) {
  if (n_rows < 0 || vocab <= 0) return kBadArg;
  for (long r = 0; r < n_rows; ++r) {
    const float* x = rows + r * vocab;
    double m = -std::numeric_limits<double>::infinity();
    for (int j = 0; j < vocab; ++j) m = std::max(m, static_cast<double>(x[j]));
    if (m == -std::numeric_limits<double>::infinity()) { entropy[r] = 0.0f; continue; }
    double z = 0.0, s = 0.0;
    for (int j = 0; j < vocab; ++j) {
      if (x[j] == -std::numeric_limits<float>::infinity()) continue;
      const double d = static_cast<double>(x[j]) - m;
      const double e = std::exp(d);
      z += e;
      s += d * e;
    }
    entropy[r] = static_cast<float>(std::log(z) - s / z);
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Best-first tree expansion. [PL] App. B "Tree-Drafting Algorithm Details"
// (Algorithm 1) and [PL] §2 "Tree Construction and Verification"; [RB]
// "方法步骤详情": repeatedly pop the highest-scoring expandable node, attach
// up to W children, re-insert the children with updated scores, until the
// budget is full or no expandable node remains. Score = cumulative draft
// log-probability along the path, [SM] "How it works", s(π(v)) equation.
//
// Readings where the pages are silent:
//   * the budget B counts draft nodes, not the root;
//   * a child of a depth-d node takes its token and log-prob from depth
//     d+1's top-W list (rank order), shared by every depth-d node;
//   * children are attached in rank order while fewer than B nodes exist;
//     depth-N children are created but never pushed (not expandable);
//   * score(child) = score(parent) + increment in binary32 (the precision the
//     kernel ranks in), heap order = (score desc, node id asc), the root
//     (id -1, score 0) is popped first.
//
// Scores ([PL] App. C and App. E "Drafting"; the pages give the modes and
// the limits α -> 0 (cumulative log-prob) and α -> inf (entropy only), not
// the formula). The increment of a child at depth d with rank r is, in
// binary32 with H_d the entropy of depth d's draft distribution:
//   mode 0 (cumulative log-prob): logp[d][r]
//   mode 1 (hybrid):              logp[d][r] - (alpha * H_d)
//   mode 2 (entropy only):        -H_d
// so a hybrid score is cum_logp - alpha * sum_{d' <= d} H_d'.
// tok/logp: [batch][n_depth][W] as produced by orc_topw; entropy:
// [batch][n_depth] (unused in mode 0).
// Outputs per sequence: parent/token/depth/score [B] (slots >= n set to
// -1/-1/0/0), n_nodes.
// ---------------------------------------------------------------------------
int orc_tree_expand_scored(const int32_t* tok, const float* logp, const float* entropy,
                           int batch, int n_depth, int W, int B, int mode, float alpha,
                           int32_t* parent, int32_t* token, int32_t* depth, float* score,
                           int32_t* n_nodes) {
  if (batch < 0 || n_depth <= 0 || W <= 0 || B < 0) return kBadArg;
  if (mode < 0 || mode > 2 || (mode != 0 && !entropy)) return kBadArg;
  struct Entry { float score; int32_t id; int32_t depth; };
  struct Lower {  // "a ranks below c" for std::priority_queue (max-heap)
    bool operator()(const Entry& a, const Entry& c) const {
      if (a.score != c.score) return a.score < c.score;
      return a.id > c.id;
    }
  };
  for (int b = 0; b < batch; ++b) {
    int32_t* par = parent + static_cast<size_t>(b) * B;
    int32_t* tk = token + static_cast<size_t>(b) * B;
    int32_t* dp = depth + static_cast<size_t>(b) * B;
    float* sc = score + static_cast<size_t>(b) * B;
    for (int v = 0; v < B; ++v) { par[v] = -1; tk[v] = -1; dp[v] = 0; sc[v] = 0.0f; }
    const int32_t* tok_b = tok + static_cast<size_t>(b) * n_depth * W;
    const float* logp_b = logp + static_cast<size_t>(b) * n_depth * W;
    auto increment = [&](int d, int r) -> float {   // d = 1..N
      const float lp = logp_b[(d - 1) * W + r];
      if (mode == 0) return lp;
      const float h = entropy[static_cast<size_t>(b) * n_depth + d - 1];
      if (mode == 1) {
        const float t = alpha * h;   // one binary32 multiply
        return lp - t;               // one binary32 subtract
      }
      return -h;
    };

    std::priority_queue<Entry, std::vector<Entry>, Lower> heap;
    heap.push(Entry{0.0f, -1, 0});
    int count = 0;
    while (count < B && !heap.empty()) {
      const Entry u = heap.top();
      heap.pop();
      const int d = u.depth + 1;  // depth of the children, 1..N
      for (int r = 0; r < W && count < B; ++r) {
        const int v = count++;
        par[v] = u.id;
        tk[v] = tok_b[(d - 1) * W + r];
        dp[v] = d;
        sc[v] = u.score + increment(d, r);  // one binary32 add
        if (d < n_depth) heap.push(Entry{sc[v], v, d});
      }
    }
    n_nodes[b] = count;
  }
  return 0;
}

int orc_tree_expand(const int32_t* tok, const float* logp, int batch, int n_depth, int W, int B,
                    int32_t* parent, int32_t* token, int32_t* depth, float* score,
                    int32_t* n_nodes) {
  return orc_tree_expand_scored(tok, logp, nullptr, batch, n_depth, W, B, 0, 0.0f, parent, token,
                                depth, score, n_nodes);
}

// ---------------------------------------------------------------------------
// Greedy tree acceptance. [PL] §2 "Tree Construction and Verification":
// verification accepts the longest prefix whose draft tokens satisfy the
// target's acceptance condition; [RB] "前置知识": the target keeps the longest
// prefix consistent with its own predictions; [PP] §3 "Preliminaries": the
// accepted prefix is committed together with one bonus token.
// At temperature 0 the condition is "token == target argmax at the parent".
//
// target: [batch][B+1][V] fp32, row 0 = the root's prediction, row 1+v =
// node v's prediction. Argmax ties go to the lowest token id.
// Walk: a = argmax(row 0); while some child c of the current node has
// token[c] == a (the lowest such id if several): accept c, a = argmax(row
// 1+c). bonus = the last a. acc_tokens/acc_nodes: [batch][n_depth], unused
// entries -1. Returns kBadTree for a parent outside [-1, v).
// ---------------------------------------------------------------------------
int orc_tree_accept(const float* target, const int32_t* parent, const int32_t* token,
                    const int32_t* n_nodes, int batch, int B, int n_depth, int vocab,
                    int32_t* acc_len, int32_t* acc_tokens, int32_t* acc_nodes, int32_t* bonus) {
  if (batch < 0 || B < 0 || n_depth <= 0 || vocab <= 0) return kBadArg;
  auto argmax = [vocab](const float* row) {
    int best = 0;
    for (int j = 1; j < vocab; ++j)
      if (row[j] > row[best]) best = j;
    return best;
  };
  for (int b = 0; b < batch; ++b) {
    const int n = n_nodes[b];
    if (n < 0 || n > B) return kBadTree;
    const int32_t* par = parent + static_cast<size_t>(b) * B;
    const int32_t* tk = token + static_cast<size_t>(b) * B;
    for (int v = 0; v < n; ++v) {
      if (par[v] < -1 || par[v] >= v) return kBadTree;
      if (tk[v] < 0 || tk[v] >= vocab) return kBadToken;
    }
    const float* rows = target + static_cast<size_t>(b) * (B + 1) * vocab;
    int32_t* at = acc_tokens + static_cast<size_t>(b) * n_depth;
    int32_t* an = acc_nodes + static_cast<size_t>(b) * n_depth;
    for (int i = 0; i < n_depth; ++i) { at[i] = -1; an[i] = -1; }

    int cur = -1;
    int a = argmax(rows);
    int len = 0;
    while (true) {
      int next = -1;
      for (int c = 0; c < n; ++c)
        if (par[c] == cur && tk[c] == a) { next = c; break; }
      if (next < 0 || len >= n_depth) break;
      at[len] = a;
      an[len] = next;
      ++len;
      cur = next;
      a = argmax(rows + static_cast<size_t>(1 + next) * vocab);
    }
    acc_len[b] = len;
    bonus[b] = a;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Accepted-path K/V commit. [PP] §3 "Preliminaries": a verification round
// commits the accepted prefix plus one bonus token. The accepted draft nodes'
// K/V were produced by the verification pass (they are rows of the tree K/V),
// so committing them appends those rows to the sequence's prefix cache in path
// order. The bonus token has no K/V yet (the next round computes it when it
// verifies that token as its root), so it is not written.
//
// For sequence b with L = prefix_len[b] and a = acc_len[b]:
//   cache position L + i  <-  tree row acc_nodes[b][i], for i = 0 .. a-1
//                             (every KV head, K and V)
//   new_prefix_len[b] = L + a
// Layouts as in orc_tree_attn (elements are bf16 bit patterns). A sequence is
// left untouched, with new_prefix_len[b] = L, when a is outside [0, n_depth],
// an accepted node is outside [0, B), L is negative, L + a exceeds the cache
// (max_prefix, or max_pages * page_size when paged), or a page id it would
// write is outside [0, n_pool_pages); the call then returns kBadTree after
// processing every sequence. new_prefix_len may alias prefix_len.
// ---------------------------------------------------------------------------
int orc_tree_commit_kv(int batch, int B, int n_depth, int hkv, int D,
                       const uint16_t* k_tree, const uint16_t* v_tree,
                       uint16_t* k_cache, uint16_t* v_cache,
                       const int32_t* block_table, int page_size, int max_pages,
                       int n_pool_pages, int max_prefix,
                       const int32_t* prefix_len, const int32_t* acc_len,
                       const int32_t* acc_nodes, int32_t* new_prefix_len) {
  if (batch < 0 || B <= 0 || n_depth <= 0 || hkv <= 0 || D <= 0) return kBadArg;
  if (block_table && (page_size <= 0 || max_pages <= 0)) return kBadArg;
  const size_t row = static_cast<size_t>(hkv) * D;   // elements per token row
  const long capacity = block_table ? static_cast<long>(max_pages) * page_size : max_prefix;
  int rc = 0;
  for (int b = 0; b < batch; ++b) {
    const int L = prefix_len[b];
    const int a = acc_len[b];
    const int32_t* path = acc_nodes + static_cast<size_t>(b) * n_depth;
    bool ok = L >= 0 && a >= 0 && a <= n_depth && static_cast<long>(L) + a <= capacity;
    for (int i = 0; ok && i < a; ++i)
      if (path[i] < 0 || path[i] >= B) ok = false;
    // Where each committed token goes: its cache row index (element offset / row).
    std::vector<size_t> dst(ok ? a : 0);
    for (int i = 0; ok && i < a; ++i) {
      const long pos = static_cast<long>(L) + i;
      if (block_table) {
        const int page = block_table[static_cast<size_t>(b) * max_pages + pos / page_size];
        if (page < 0 || page >= n_pool_pages) { ok = false; break; }
        dst[i] = static_cast<size_t>(page) * page_size + pos % page_size;
      } else {
        dst[i] = static_cast<size_t>(b) * max_prefix + pos;
      }
    }
    if (!ok) {
      rc = kBadTree;
      new_prefix_len[b] = L;
      continue;
    }
    for (int i = 0; i < a; ++i) {
      const size_t src = (static_cast<size_t>(b) * B + path[i]) * row;
      for (size_t e = 0; e < row; ++e) {
        k_cache[dst[i] * row + e] = k_tree[src + e];
        v_cache[dst[i] * row + e] = v_tree[src + e];
      }
    }
    new_prefix_len[b] = L + a;
  }
  return rc;
}

// ---------------------------------------------------------------------------
// Temperature-T tree acceptance. [PP] App. F.3 "Lossless verification": every
// committed token is the target's own draw at any temperature; for a draft
// fixed before verification each draft token is checked with a point-mass
// proposal and accepted with the target probability. [PP] App. F.1: for a
// chain this gives P(accept d1, reject d2, draw b) = p(d1) (1 - p(d2|d1))
// p(b|d1) / (1 - p(d2|d1)) = p(d1) p(b|d1) (the 0.24 worked example).
//
// Reading for trees (the pages treat chains): at the current node draw one
// token y from softmax(target row / T); if a child carries y, accept it and
// continue from it, else y is the bonus token and the walk ends. For a chain
// this is exactly the point-mass rule above; for several children it is the
// same rule applied to the children in turn (each rejection removes that
// child's token from the residual), which again commits a draw of the target.
//
// The draw uses the Gumbel-max form: y = argmax_j (x_j / T + G_j), lowest j on
// ties, with G_j = gumbel_noise(seed, k) for draw index
//   k = ((b * (B+1) + r) << 32 | j) + 1      (r = 0 for the root row, 1+v
//                                            for node v's row)
// computed in binary32: t = x_j * (1/T) (one multiply by the binary32
// reciprocal inv_T the caller passes), key = t + G_j (one add).
// Everything else (layouts, validation, outputs) as orc_tree_accept.
// ---------------------------------------------------------------------------
int orc_tree_accept_sampled(const float* target, const int32_t* parent, const int32_t* token,
                            const int32_t* n_nodes, int batch, int B, int n_depth, int vocab,
                            float inv_T, uint64_t seed, int32_t* acc_len, int32_t* acc_tokens,
                            int32_t* acc_nodes, int32_t* bonus) {
  if (batch < 0 || B < 0 || n_depth <= 0 || vocab <= 0 || !(inv_T > 0.0f)) return kBadArg;
  auto draw = [&](int b, int r, const float* row) {
    const uint64_t base = (static_cast<uint64_t>(b) * (B + 1) + r) << 32;
    int best = -1;
    float bk = 0.0f;
    for (int j = 0; j < vocab; ++j) {
      if (row[j] == -std::numeric_limits<float>::infinity()) continue;
      const float t = row[j] * inv_T;
      const float key = t + gumbel_noise(seed, (base | static_cast<uint32_t>(j)) + 1);
      if (best < 0 || key > bk) { best = j; bk = key; }
    }
    return best;   // -1 only for a row of all -inf
  };
  for (int b = 0; b < batch; ++b) {
    const int n = n_nodes[b];
    if (n < 0 || n > B) return kBadTree;
    const int32_t* par = parent + static_cast<size_t>(b) * B;
    const int32_t* tk = token + static_cast<size_t>(b) * B;
    for (int v = 0; v < n; ++v) {
      if (par[v] < -1 || par[v] >= v) return kBadTree;
      if (tk[v] < 0 || tk[v] >= vocab) return kBadToken;
    }
    const float* rows = target + static_cast<size_t>(b) * (B + 1) * vocab;
    int32_t* at = acc_tokens + static_cast<size_t>(b) * n_depth;
    int32_t* an = acc_nodes + static_cast<size_t>(b) * n_depth;
    for (int i = 0; i < n_depth; ++i) { at[i] = -1; an[i] = -1; }
    int cur = -1, r = 0, len = 0;
    int a = draw(b, 0, rows);
    while (true) {
      int next = -1;
      for (int c = 0; c < n; ++c)
        if (par[c] == cur && tk[c] == a) { next = c; break; }
      if (next < 0 || len >= n_depth) break;
      at[len] = a;
      an[len] = next;
      ++len;
      cur = next;
      r = 1 + next;
      a = draw(b, r, rows + static_cast<size_t>(r) * vocab);
    }
    acc_len[b] = len;
    bonus[b] = a;
  }
  return 0;
}

// Test hooks for the pins: the log, the generator and the noise themselves.
void orc_series_ln(const float* x, long n, float* out) {
  for (long i = 0; i < n; ++i) out[i] = series_ln(x[i]);
}
void orc_splitmix64(uint64_t seed, const uint64_t* k, long n, uint64_t* out) {
  for (long i = 0; i < n; ++i) out[i] = splitmix64_output(seed, k[i]);
}
void orc_gumbel(uint64_t seed, const uint64_t* k, long n, float* out) {
  for (long i = 0; i < n; ++i) out[i] = gumbel_noise(seed, k[i]);
}

}  // extern "C"
