// jt_tree_expand: budget-B best-first tree construction.
//
// Algorithm (JetSpec summary on paperlayer.ai, App. B "Tree-Drafting
// Algorithm Details", Algorithm 1, and §2 "Tree Construction and
// Verification"; Chinese summary on paper.rainbus.top, "方法步骤详情"): pop the
// expandable node with the highest cumulative log-prob (JetSpec review on
// startedourmission.github.io, "How it works", s(π(v)) equation), attach up
// to W children, push them back, until B nodes exist or nothing is left.
//
// GPU design: one warp owns one sequence. Expansions of more than 16 pops
// go in rounds (tree_expand_rounds_kernel below: every node the heap would
// pop before any child created in the round pops at once); the one-pop-at-
// a-time form described here serves the others and width 1, where the tree
// is a chain. Each step of a pop is warp-parallel instead of a heap. The frontier (created, unpopped nodes with depth < N) lives in
// registers: node v occupies lane v & 31, slot v >> 5 (B <= 256 -> 8 slots).
// A pop is two warp reductions: __reduce_max_sync over an order-preserving
// uint32 key of the score, then __reduce_min_sync over the ids holding that
// key (ties -> lower id, as the heap order requires). The W children of a
// pop are created at once, each by the lane that will hold it; the popped
// node's score is recovered from its key and its depth comes by one shuffle
// from the lane that held it, so a pop touches no memory besides the
// candidate row of the next depth. Scores are binary32 sums (__fadd_rn), the
// same adds as the definition. The sequence's N x W candidates are staged in
// shared memory first, so no pop waits on a global load (the depth that
// selects the next candidate row is only known once the pop is done).
//
// Score modes (paperlayer.ai App. C "Tree-Drafting Algorithm Ablation" and
// App. E "Drafting": cumulative log-prob, entropy-guided and hybrid scores).
// A child at depth d with rank r adds, in binary32, logp[d][r] (mode 0),
// logp[d][r] - alpha * H_d (mode 1, one multiply and one subtract), or -H_d
// (mode 2). The increments are formed once while staging.
#include <climits>

#include "jt_internal.cuh"

namespace jt {
namespace {

constexpr int kWarpsPerBlock = 4;

// Inverse of order_key for the keys of real values (never 0 here).
__device__ __forceinline__ float key_score(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

template <int SLOTS>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
tree_expand_kernel(const int32_t* __restrict__ tok, const float* __restrict__ logp,
                   const float* __restrict__ entropy, int mode, float alpha, int batch,
                   int N, int W, int B, int32_t* __restrict__ parent_o,
                   int32_t* __restrict__ token_o, int32_t* __restrict__ depth_o,
                   float* __restrict__ score_o, int32_t* __restrict__ n_nodes_o) {
  extern __shared__ int32_t cand_s[];   // per warp: N*W tokens then N*W score increments
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + warp;
  if (b >= batch) return;  // whole warp leaves together
  constexpr unsigned kFull = 0xFFFFFFFFu;
  grid_dependency_sync();

  const int nw = N * W;
  int32_t* tk = cand_s + (size_t)warp * 2 * nw;
  float* lp = reinterpret_cast<float*>(tk + nw);
  for (int i = lane; i < nw; i += 32) {
    tk[i] = __ldg(tok + (size_t)b * nw + i);
    const float l = __ldg(logp + (size_t)b * nw + i);
    float inc = l;
    if (mode != 0) {
      const float h = __ldg(entropy + (size_t)b * N + i / W);
      inc = mode == 1 ? __fsub_rn(l, __fmul_rn(alpha, h)) : -h;
    }
    lp[i] = inc;
  }
  __syncwarp();
  int32_t* par = parent_o + (size_t)b * B;
  int32_t* tko = token_o + (size_t)b * B;
  int32_t* dpo = depth_o + (size_t)b * B;
  float* sco = score_o + (size_t)b * B;

  if (W == 1) {
    // Width 1: every pop finds exactly one frontier node, the last child, so
    // the expansion is the chain of min(B, N) nodes, node v = child of
    // v - 1 at depth v + 1 with the rank-0 candidate of that depth. Its
    // scores are the same binary32 sums, in the same order, from +0.
    const int n = min(B, N);
    for (int v = lane; v < B; v += 32) {
      const bool live = v < n;
      par[v] = live ? v - 1 : -1;
      tko[v] = live ? tk[v] : -1;
      dpo[v] = live ? v + 1 : 0;
      if (!live) sco[v] = 0.0f;
    }
    if (lane == 0) {
      float sc = 0.0f;
      for (int v = 0; v < n; ++v) {
        sc = __fadd_rn(sc, lp[v]);
        sco[v] = sc;
      }
      n_nodes_o[b] = n;
    }
    return;
  }

  // Frontier keys and depths of this lane's slots (node (slot << 5) | lane);
  // key 0 = empty. best_* cache the lane's own best (highest key, lowest
  // slot) and its depth.
  uint32_t fk[SLOTS];
  int fd[SLOTS];
#pragma unroll
  for (int k = 0; k < SLOTS; ++k) { fk[k] = 0u; fd[k] = 0; }
  uint32_t best_key = 0u;
  int best_slot = 0, best_depth = 0;

  int count = 0;
  int cur = -1;          // the node being expanded; the root first
  float cur_s = 0.0f;
  int cur_d = 0;
  while (true) {
    const int d = cur_d + 1;               // depth of the children
    const int nc = min(W, B - count);
    // Child r of this pop is node count + r, owned (and created) by lane
    // (count + r) & 31.
    const int r = (lane - count) & 31;
    if (r < nc) {
      const int v = count + r;
      const float csc = __fadd_rn(cur_s, lp[(d - 1) * W + r]);
      par[v] = cur;
      tko[v] = tk[(d - 1) * W + r];
      dpo[v] = d;
      sco[v] = csc;
      if (d < N) {
        const int slot = v >> 5;
        const uint32_t key = order_key(csc);
#pragma unroll
        for (int k = 0; k < SLOTS; ++k)
          if (k == slot) { fk[k] = key; fd[k] = d; }
        // A new node has a higher id than every node of its lane, so it
        // displaces the cached best only with a strictly higher key.
        if (key > best_key) { best_key = key; best_slot = slot; best_depth = d; }
      }
    }
    count += nc;
    if (count >= B) break;

    // Pop: best (key desc, id asc) over the frontier. The popped score is
    // the key's value (order_key is a bijection on the scores, which are
    // never -0: they start at +0 and a round-to-nearest sum is -0 only
    // when both terms are), and its depth comes from the owner lane.
    const uint32_t top = __reduce_max_sync(kFull, best_key);
    if (top == 0) break;  // nothing expandable
    const uint32_t id = __reduce_min_sync(
        kFull, best_key == top ? (uint32_t)((best_slot << 5) | lane) : 0xFFFFFFFFu);
    const int owner = (int)(id & 31u);
    cur_d = __shfl_sync(kFull, best_depth, owner);
    if (lane == owner) {
      // The owner drops the popped slot and rescans its remaining slots.
      const int ps = (int)(id >> 5);
#pragma unroll
      for (int k = 0; k < SLOTS; ++k)
        if (k == ps) fk[k] = 0u;
      best_key = 0u;
      best_slot = 0;
      best_depth = 0;
#pragma unroll
      for (int k = SLOTS - 1; k >= 0; --k)
        if (fk[k] >= best_key && fk[k] != 0u) { best_key = fk[k]; best_slot = k; best_depth = fd[k]; }
    }
    cur = (int)id;
    cur_s = key_score(top);
  }
  for (int v = count + lane; v < B; v += 32) {
    par[v] = -1;
    tko[v] = -1;
    dpo[v] = 0;
    sco[v] = 0.0f;
  }
  if (lane == 0) n_nodes_o[b] = count;
}

// ---------------------------------------------------------------------------
// Width >= 2: pops in rounds. One warp per sequence; node v is slot v >> 5
// of lane v & 31.
//
// A round looks at the whole frontier (created, unpopped nodes of depth
// < N). theta = the best score any child of a frontier node could get (its
// score plus the largest increment of the next depth, one binary32 add;
// children of depth N are never popped and bound nothing). Every frontier
// node scoring >= theta pops before any child created in this round: such
// a child scores at most theta, and on equal scores the older node (lower
// id) pops first. Those nodes are a prefix of the heap's key order (score
// desc, id asc), so the round pops all of them, in key order, up to the
// budget: pop rank q gives its children the ids count + q * W + r. If the
// prefix is empty (a score increment above 0), the round pops the frontier's
// best node alone, which is the heap's next pop whatever the increments.
// Drafts with a few dominant tokens per depth pop whole levels per round:
// two to four rounds per sequence instead of ceil(B / W) pops.
//
// The frontier lives in registers (the score's order key, 0 = not in the
// frontier; the depth; the order key of the best child score). A round is
// one warp reduction for theta, a ballot compaction of the prefix into
// shared memory, a pairwise rank of its elements (each lane ranks the
// elements it holds against the whole prefix), a rank table of the pops in
// shared memory, and the children created in parallel, each by the lane
// that will hold it.
// ---------------------------------------------------------------------------
// Shared memory of one warp, in 32-bit words: prefix keys (u64) first, so
// they stay 8-byte aligned; the total is even, so every warp's region is.
__host__ __device__ inline size_t rounds_words(int N, int W, int B) {
  const size_t w = (size_t)2 * B + B + 3 * (size_t)B + 2 * (size_t)N * W + N;
  return (w + 1) & ~(size_t)1;
}

template <int SLOTS>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
tree_expand_rounds_kernel(const int32_t* __restrict__ tok, const float* __restrict__ logp,
                          const float* __restrict__ entropy, int mode, float alpha, int batch,
                          int N, int W, int B, int32_t* __restrict__ parent_o,
                          int32_t* __restrict__ token_o, int32_t* __restrict__ depth_o,
                          float* __restrict__ score_o, int32_t* __restrict__ n_nodes_o) {
  extern __shared__ __align__(16) int32_t sm_rounds[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x >> 5) + warp;
  if (b >= batch) return;  // whole warp leaves together
  constexpr unsigned kFull = 0xFFFFFFFFu;
  grid_dependency_sync();

  const int nw = N * W;
  int32_t* base_s = sm_rounds + (size_t)warp * rounds_words(N, W, B);
  uint64_t* ak = reinterpret_cast<uint64_t*>(base_s);              // [B] prefix keys
  int32_t* ad = base_s + 2 * B;                                     // [B] prefix depths
  int32_t* pid = ad + B;                                            // [B] rank table: id,
  uint32_t* pkey = reinterpret_cast<uint32_t*>(pid + B);            //   score key,
  int32_t* pdep = reinterpret_cast<int32_t*>(pkey + B);             //   depth
  int32_t* tk = pdep + B;                                           // [N * W] tokens
  float* lp = reinterpret_cast<float*>(tk + nw);                    // [N * W] increments
  float* lpmax = lp + nw;                                           // [N] best increment

  for (int i = lane; i < nw; i += 32) {
    tk[i] = __ldg(tok + (size_t)b * nw + i);
    const float l = __ldg(logp + (size_t)b * nw + i);
    float inc = l;
    if (mode != 0) {
      const float h = __ldg(entropy + (size_t)b * N + i / W);
      inc = mode == 1 ? __fsub_rn(l, __fmul_rn(alpha, h)) : -h;
    }
    lp[i] = inc;
  }
  __syncwarp();
  for (int d = lane; d < N; d += 32) {
    float m = lp[d * W];
#pragma unroll 4
    for (int r = 1; r < W; ++r) m = fmaxf(m, lp[d * W + r]);
    lpmax[d] = m;
  }
  // x / W for 0 <= x <= 256 as one high multiply: the magic's excess over
  // 2^32 / W is below 1, so the error term x * excess / 2^32 < 2^-24 never
  // crosses the next multiple of 1 / W.
  const uint32_t w_magic = 0xFFFFFFFFu / (uint32_t)W + 1u;
  int32_t* par_g = parent_o + (size_t)b * B;
  int32_t* tok_g = token_o + (size_t)b * B;
  int32_t* dep_g = depth_o + (size_t)b * B;
  float* sco_g = score_o + (size_t)b * B;

  uint32_t fk[SLOTS], fb[SLOTS];
  int fd[SLOTS];
#pragma unroll
  for (int k = 0; k < SLOTS; ++k) { fk[k] = 0u; fb[k] = 0u; fd[k] = 0; }

  // The root's pop is rank 0 of the first round.
  if (lane == 0) { pid[0] = -1; pkey[0] = order_key(0.0f); pdep[0] = 0; }
  int count = 0, npop = 1;
  __syncwarp();
  while (true) {
    // Children of this round's pops: node u = count + q * W + r, held and
    // created by lane u & 31.
    const int stop = min(B, count + npop * W);
    for (int u = count + ((lane - count) & 31); u < stop; u += 32) {
      const int q = (int)__umulhi((uint32_t)(u - count), w_magic), r = u - count - q * W;
      const int pd = pdep[q];
      const float s = __fadd_rn(key_score(pkey[q]), lp[pd * W + r]);
      const int d = pd + 1;
      par_g[u] = pid[q];
      tok_g[u] = tk[pd * W + r];
      dep_g[u] = d;
      sco_g[u] = s;
      if (d < N) {
        const uint32_t key = order_key(s);
        const uint32_t bound = d + 1 < N ? order_key(__fadd_rn(s, lpmax[d])) : 0u;
        const int slot = u >> 5;
#pragma unroll
        for (int k = 0; k < SLOTS; ++k)
          if (k == slot) { fk[k] = key; fb[k] = bound; fd[k] = d; }
      }
    }
    count = stop;
    if (count >= B) break;

    uint32_t lb = 0u, lk = 0u;
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) { lb = max(lb, fb[k]); lk = max(lk, fk[k]); }
    const uint32_t theta = __reduce_max_sync(kFull, lb);
    uint32_t am = 0u;
#pragma unroll
    for (int k = 0; k < SLOTS; ++k)
      if (fk[k] != 0u && fk[k] >= theta) am |= 1u << k;
    int nA = __reduce_add_sync(kFull, (uint32_t)__popc(am));
    if (nA == 0) {
      const uint32_t top = __reduce_max_sync(kFull, lk);
      if (top == 0u) break;   // nothing expandable
      // The single best frontier node: key top, lowest id.
      int mine = 0x7FFFFFFF, mk = 0;
#pragma unroll
      for (int k = SLOTS - 1; k >= 0; --k)
        if (fk[k] == top) { mine = 32 * k + lane; mk = k; }
      const int id = (int)__reduce_min_sync(kFull, (uint32_t)mine);
      if (id == mine) am = 1u << mk;
      nA = 1;
    }
    // Compact the prefix (slot by slot, lane order) and drop it from the
    // frontier: if it is cut by the budget, this round is the last.
    int pos = 0;
#pragma unroll
    for (int k = 0; k < SLOTS; ++k) {
      const unsigned bal = __ballot_sync(kFull, (am >> k) & 1u);
      if ((am >> k) & 1u) {
        const int at = pos + __popc(bal & ((1u << lane) - 1u));
        ak[at] = ((uint64_t)(~fk[k]) << 32) | (uint32_t)(32 * k + lane);
        ad[at] = fd[k];
        fk[k] = 0u;
        fb[k] = 0u;
      }
      pos += __popc(bal);
    }
    __syncwarp();
    const int allowed = (B - count + W - 1) / W;
    npop = min(nA, allowed);
    // Rank of element j = number of prefix elements before it in key order.
    for (int j0 = 0; j0 < nA; j0 += 32) {
      const int j = j0 + lane;
      const uint64_t key = j < nA ? ak[j] : ~0ull;
      int rank = 0;
#pragma unroll 4
      for (int i = 0; i < nA; ++i) rank += ak[i] < key;
      if (j < nA && rank < npop) {
        pid[rank] = (int)(uint32_t)key;
        pkey[rank] = ~(uint32_t)(key >> 32);
        pdep[rank] = ad[j];
      }
    }
    __syncwarp();
  }
  for (int v = count + lane; v < B; v += 32) {
    par_g[v] = -1;
    tok_g[v] = -1;
    dep_g[v] = 0;
    sco_g[v] = 0.0f;
  }
  if (lane == 0) n_nodes_o[b] = count;
}

}  // namespace

cudaError_t launch_tree_expand(const Ctx& c, const int32_t* tok, const float* logp,
                               const float* entropy, int mode, float alpha, int batch,
                               int n_depth, int W, int B, int32_t* parent, int32_t* token,
                               int32_t* depth, float* score, int32_t* n_nodes) {
  if (batch == 0) return cudaSuccess;
  const int slots = (B + 31) / 32;
  // Rounds cost ~0.5 us each against ~0.15-0.25 us per pop: with at most 16
  // pops (tiny and mid-batch shapes: 2.2 vs 2.8 us, 3.9 vs 4.7 us) popping one
  // node at a time is faster; beyond that the rounds win (32 pops: 7.9 vs
  // 7.6 us, 64 pops: 16.9 vs 6.3 us).
  if (W >= 2 && (B + W - 1) / W > 16) {
    const size_t per_warp = rounds_words(n_depth, W, B) * sizeof(int32_t);   // <= 40 KiB
    const int warps = per_warp * kWarpsPerBlock <= 44 * 1024 ? kWarpsPerBlock : 1;
    const size_t smem = per_warp * warps;
    const dim3 grid((batch + warps - 1) / warps), block(warps * 32);
    auto kern = slots <= 1 ? tree_expand_rounds_kernel<1>
              : slots <= 2 ? tree_expand_rounds_kernel<2>
              : slots <= 4 ? tree_expand_rounds_kernel<4>
                           : tree_expand_rounds_kernel<8>;
    return launch_kernel(kern, grid, block, smem, c.stream, 1, tok, logp, entropy, mode, alpha,
                         batch, n_depth, W, B, parent, token, depth, score, n_nodes);
  }
  // Candidates staged per warp: 8 bytes each, at most 64 x 32 (16 KiB).
  const int warps = (size_t)n_depth * W * 8 * kWarpsPerBlock <= 44 * 1024 ? kWarpsPerBlock : 1;
  const size_t smem = (size_t)warps * n_depth * W * 8;
  const dim3 grid((batch + warps - 1) / warps), block(warps * 32);
  auto kern = slots <= 1 ? tree_expand_kernel<1>
            : slots <= 2 ? tree_expand_kernel<2>
            : slots <= 4 ? tree_expand_kernel<4>
                         : tree_expand_kernel<8>;
  return launch_kernel(kern, grid, block, smem, c.stream, 1, tok, logp, entropy, mode, alpha,
                       batch, n_depth, W, B, parent, token, depth, score, n_nodes);
}

}  // namespace jt
