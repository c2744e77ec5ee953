// jt_tree_expand: budget-B best-first tree construction.
//
// Algorithm (JetSpec summary on paperlayer.ai, App. B "Tree-Drafting
// Algorithm Details", Algorithm 1, and §2 "Tree Construction and
// Verification"; Chinese summary on paper.rainbus.top, "方法步骤详情"): pop the
// expandable node with the highest cumulative log-prob (JetSpec review on
// startedourmission.github.io, "How it works", s(π(v)) equation), attach up
// to W children, push them back, until B nodes exist or nothing is left.
//
// GPU design: the expansion is inherently serial, so one warp owns one
// sequence and makes every step of a pop warp-parallel instead of using a
// heap. The frontier (created, unpopped nodes with depth < N) lives in
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

}  // namespace

cudaError_t launch_tree_expand(const Ctx& c, const int32_t* tok, const float* logp,
                               const float* entropy, int mode, float alpha, int batch,
                               int n_depth, int W, int B, int32_t* parent, int32_t* token,
                               int32_t* depth, float* score, int32_t* n_nodes) {
  if (batch == 0) return cudaSuccess;
  const int slots = (B + 31) / 32;
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
