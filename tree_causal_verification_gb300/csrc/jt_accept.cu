// jt_tree_accept: greedy (temperature 0) tree acceptance.
//
// Accept the longest root path whose every token equals the target's argmax
// at its parent, then commit one bonus token (JetSpec summary on
// paperlayer.ai, §2 "Tree Construction and Verification"; Chinese summary on
// paper.rainbus.top, "前置知识"; JetSpec++ summary on paperlayer.ai, §3
// "Preliminaries"). Argmax ties go to the lowest token id.
//
// Two launches:
//  1. argmax of every live target row (row 0 and rows 1+v, v < n_nodes), one
//     HBM pass with the same clustered row scan as jt_topw (K = 1, no
//     log-sum-exp); the per-row argmax goes to the workspace;
//  2. the walk: one warp per sequence, each step a warp-wide search for the
//     child whose token matches (__reduce_min_sync picks the lowest id).
#include "jt_rowscan.cuh"

namespace jt {
namespace {

__global__ void __launch_bounds__(kScanThreads)
accept_argmax_kernel(const float* __restrict__ target, const int32_t* __restrict__ n_nodes,
                     int B, int V, int S, int32_t* __restrict__ am) {
  __shared__ ScanPartial<1> warp_parts[kScanWarps];
  __shared__ ScanPartial<1> part;
  const int row = blockIdx.x / S;
  const int seg = blockIdx.x % S;
  const int b = row / (B + 1), j = row % (B + 1);
  const int n = n_nodes[b];
  // Uniform over the cluster (same row): dead rows skip the scan entirely.
  if (n < 0 || n > B || j > n) return;
  const int v4 = V >> 2;
  const int per = (v4 + S - 1) / S;
  const int lo = min(v4, seg * per), hi = min(v4, lo + per);
  TopK<1> top;
  top.init();
  Lse lse;
  lse.init();
  scan_segment<1, false>(target + (size_t)row * V, lo, hi, top, lse);
  block_reduce<1, false>(top, lse, &part, warp_parts);
  if (cluster_reduce<1, false>(&part, S, top, lse)) am[row] = top.i[0];
}

constexpr int kWalkWarps = 4;

__global__ void __launch_bounds__(kWalkWarps * 32)
accept_walk_kernel(const int32_t* __restrict__ am, const int32_t* __restrict__ parent,
                   const int32_t* __restrict__ token, const int32_t* __restrict__ n_nodes,
                   int batch, int B, int N, int V, int32_t* __restrict__ acc_len,
                   int32_t* __restrict__ acc_tokens, int32_t* __restrict__ acc_nodes,
                   int32_t* __restrict__ bonus, int32_t* d_err) {
  __shared__ int32_t par_s[kWalkWarps][kMaxB];
  __shared__ int32_t tok_s[kWalkWarps][kMaxB];
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWalkWarps + warp;
  if (b >= batch) return;
  const int n = n_nodes[b];
  int32_t* at = acc_tokens + (size_t)b * N;
  int32_t* an = acc_nodes + (size_t)b * N;
  bool bad = (n < 0 || n > B);
  int flag = bad ? JT_DEVERR_NNODES : 0;
  if (!bad) {
    for (int v = lane; v < n; v += 32) {
      const int p = parent[(size_t)b * B + v];
      const int t = token[(size_t)b * B + v];
      if (p < -1 || p >= v) flag |= JT_DEVERR_PARENT;
      if (t < 0 || t >= V) flag |= JT_DEVERR_TOKEN;
      par_s[warp][v] = p;
      tok_s[warp][v] = t;
    }
    flag = __reduce_or_sync(kFull, flag);
    bad = flag != 0;
  }
  __syncwarp();
  int len = 0, a = -1;
  if (!bad) {
    const int32_t* am_b = am + (size_t)b * (B + 1);
    a = am_b[0];
    int cur = -1;
    while (len < N) {
      uint32_t cand = 0xFFFFFFFFu;
      for (int v = lane; v < n; v += 32)
        if (par_s[warp][v] == cur && tok_s[warp][v] == a) cand = min(cand, (uint32_t)v);
      const uint32_t c = __reduce_min_sync(kFull, cand);
      if (c == 0xFFFFFFFFu) break;
      if (lane == 0) { at[len] = a; an[len] = (int)c; }
      ++len;
      cur = (int)c;
      a = am_b[1 + cur];
    }
  } else if (lane == 0) {
    raise_flag(d_err, flag);
  }
  for (int i = len + lane; i < N; i += 32) { at[i] = -1; an[i] = -1; }
  if (lane == 0) {
    acc_len[b] = len;
    bonus[b] = a;
  }
}

}  // namespace

size_t accept_workspace_bytes(int batch, int B, int vocab) {
  (void)vocab;
  return align_up((size_t)batch * (B + 1) * sizeof(int32_t), 256);
}

cudaError_t launch_tree_accept(const Ctx& c, const float* target, const int32_t* parent,
                               const int32_t* token, const int32_t* n_nodes, int batch, int B,
                               int n_depth, int vocab, int32_t* acc_len, int32_t* acc_tokens,
                               int32_t* acc_nodes, int32_t* bonus) {
  if (batch == 0) return cudaSuccess;
  int32_t* am = static_cast<int32_t*>(c.workspace);
  const long rows = (long)batch * (B + 1);
  const int S = pick_row_split(rows, vocab / 4, c.num_sms, 16);
  cudaError_t e = launch_clustered(accept_argmax_kernel, (int)(rows * S), S, c.stream, target,
                                   n_nodes, B, vocab, S, am);
  if (e != cudaSuccess) return e;
  accept_walk_kernel<<<(batch + kWalkWarps - 1) / kWalkWarps, kWalkWarps * 32, 0, c.stream>>>(
      am, parent, token, n_nodes, batch, B, n_depth, vocab, acc_len, acc_tokens, acc_nodes, bonus,
      c.d_err);
  return cudaGetLastError();
}

}  // namespace jt
