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
// pop are created by W lanes at once; each is handed to its owner lane by a
// shuffle. Scores are binary32 sums (__fadd_rn), the same adds as the
// definition. The sequence's N x W candidates are staged in shared memory
// first, so no pop waits on a global load (the depth that selects the next
// candidate row is only known once the pop is done).
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

template <int SLOTS>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
tree_expand_kernel(const int32_t* __restrict__ tok, const float* __restrict__ logp,
                   const float* __restrict__ entropy, int mode, float alpha, int batch,
                   int N, int W, int B, int32_t* __restrict__ parent_o,
                   int32_t* __restrict__ token_o, int32_t* __restrict__ depth_o,
                   float* __restrict__ score_o, int32_t* __restrict__ n_nodes_o) {
  __shared__ float score_s[kWarpsPerBlock][kMaxB];
  __shared__ uint8_t depth_s[kWarpsPerBlock][kMaxB];
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
  float* scs = score_s[warp];
  uint8_t* dep = depth_s[warp];

  // Frontier keys of this lane's slots (node (slot << 5) | lane); 0 = empty.
  // best_key / best_slot cache the lane's own best (highest key, lowest slot).
  uint32_t fk[SLOTS];
#pragma unroll
  for (int k = 0; k < SLOTS; ++k) fk[k] = 0u;
  uint32_t best_key = 0u;
  int best_slot = 0;

  int count = 0;
  int cur = -1;          // the node being expanded; the root first
  float cur_s = 0.0f;
  int cur_d = 0;
  while (true) {
    const int d = cur_d + 1;               // depth of the children
    const int nc = min(W, B - count);
    float csc = 0.0f;
    if (lane < nc) {                       // lane r creates child r
      const int v = count + lane;
      const int t = tk[(d - 1) * W + lane];
      csc = __fadd_rn(cur_s, lp[(d - 1) * W + lane]);
      par[v] = cur;
      tko[v] = t;
      dpo[v] = d;
      sco[v] = csc;
      scs[v] = csc;
      dep[v] = (uint8_t)d;
    }
    // Owner lane of child v = count + r is lane v & 31, i.e. r = (lane - count) & 31.
    const int r = (lane - count) & 31;
    const float sv = __shfl_sync(kFull, csc, r);
    if (d < N && r < nc) {
      const int slot = (count + r) >> 5;
      const uint32_t key = order_key(sv);
#pragma unroll
      for (int k = 0; k < SLOTS; ++k)
        if (k == slot) fk[k] = key;
      // A new node has a higher id than every node of its lane, so it
      // displaces the cached best only with a strictly higher key.
      if (key > best_key) { best_key = key; best_slot = slot; }
    }
    count += nc;
    __syncwarp();
    if (count >= B) break;

    // Pop: best (key desc, id asc) over the frontier.
    const uint32_t top = __reduce_max_sync(kFull, best_key);
    if (top == 0) break;  // nothing expandable
    const uint32_t id = __reduce_min_sync(
        kFull, best_key == top ? (uint32_t)((best_slot << 5) | lane) : 0xFFFFFFFFu);
    if ((int)(id & 31u) == lane) {
      // The owner drops the popped slot and rescans its remaining slots.
      const int ps = (int)(id >> 5);
#pragma unroll
      for (int k = 0; k < SLOTS; ++k)
        if (k == ps) fk[k] = 0u;
      best_key = 0u;
      best_slot = 0;
#pragma unroll
      for (int k = SLOTS - 1; k >= 0; --k)
        if (fk[k] >= best_key && fk[k] != 0u) { best_key = fk[k]; best_slot = k; }
    }
    cur = (int)id;
    cur_s = scs[cur];
    cur_d = dep[cur];
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
