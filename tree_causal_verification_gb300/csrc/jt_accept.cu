// jt_tree_accept: greedy (temperature 0) tree acceptance.
//
// Accept the longest root path whose every token equals the target's argmax
// at its parent, then commit one bonus token (JetSpec summary on
// paperlayer.ai, §2 "Tree Construction and Verification"; Chinese summary on
// paper.rainbus.top, "前置知识"; JetSpec++ summary on paperlayer.ai, §3
// "Preliminaries"). Argmax ties go to the lowest token id.
//
// Two strategies, chosen per call from the shape:
//  * path walk (trees much larger than one root path, (B+1) > 4(N+1)): one
//    thread-block cluster per sequence walks down the tree. At each level
//    every CTA scans its segment of the current node's target row, the CTAs
//    exchange (max, index) partials through distributed shared memory, and
//    each CTA finds the matching child itself. Only the rows on the accepted
//    path (at most N+1 per sequence) are read. When the batch is small, the
//    rows of the current node's children are prefetched into L2 while the
//    current row is scanned, hiding the next level's DRAM latency.
//  * all rows (chains and small trees, where nearly every row may be on the
//    path): (1) argmax of every live target row with the row scan of jt_topw
//    (K = 1, no log-sum-exp) into the workspace, clustered, or for few long
//    rows as 32 segment partials per row that the walk reduces when it
//    reaches the row, then (2) one warp per sequence walks, each step a
//    warp-wide search for the matching child (__reduce_min_sync picks the
//    lowest id).
#include "jt_rowscan.cuh"
#include "jt_sample.cuh"

namespace jt {
namespace {

// A segment's best (value, lowest index); i == INT_MAX: no element.
struct ArgPart {
  float v;
  int i;
};

// Few long rows: kFlatParts CTAs per live row, no cluster; each writes its
// segment's argmax to the scratch and the walk reduces a row's partials when
// it reaches that row.
template <bool SAMPLED, bool RES>
__global__ void __launch_bounds__(kScanThreads)
accept_argmax_flat_kernel(const float* __restrict__ target, const int32_t* __restrict__ n_nodes,
                          int B, int V, float inv_t, uint64_t seed, ArgPart* __restrict__ parts) {
  __shared__ ScanPartial<1> warp_parts[kScanWarps];
  __shared__ ScanPartial<1> part;
  const int row = blockIdx.x / kFlatParts;
  const int seg = blockIdx.x % kFlatParts;
  const int b = row / (B + 1), j = row % (B + 1);
  grid_dependency_sync();
  const int n = n_nodes[b];
  if (n < 0 || n > B || j > n) return;   // a row the walk never reads
  const int v4 = V >> 2;
  const int per = (v4 + kFlatParts - 1) / kFlatParts;
  const int lo = min(v4, seg * per), hi = min(v4, lo + per);
  if (SAMPLED)
    scan_to_partial<1, false, false, RES, GumbelKeys, true>(target + (size_t)row * V, lo, hi, &part,
                                                       warp_parts,
                                                       GumbelKeys{seed, (uint64_t)row << 32, inv_t});
  else
    scan_to_partial<1, false, false, RES, IdentityXf, true>(target + (size_t)row * V, lo, hi, &part,
                                                       warp_parts);
  if (threadIdx.x == 0) parts[blockIdx.x] = ArgPart{part.v[0], part.i[0]};
}

template <bool SAMPLED, bool RES>
__global__ void __launch_bounds__(kScanThreads)
accept_argmax_kernel(const float* __restrict__ target, const int32_t* __restrict__ n_nodes,
                     int B, int V, int S, float inv_t, uint64_t seed, int32_t* __restrict__ am) {
  __shared__ ScanPartial<1> warp_parts[kScanWarps];
  __shared__ ScanPartial<1> part;
  const int row = blockIdx.x / S;
  const int seg = blockIdx.x % S;
  const int b = row / (B + 1), j = row % (B + 1);
  grid_dependency_sync();
  const int n = n_nodes[b];
  // Uniform over the cluster (same row): dead rows skip the scan entirely.
  if (n < 0 || n > B || j > n) return;
  const int v4 = V >> 2;
  const int per = (v4 + S - 1) / S;
  const int lo = min(v4, seg * per), hi = min(v4, lo + per);
  if (SAMPLED)
    scan_to_partial<1, false, false, RES, GumbelKeys>(target + (size_t)row * V, lo, hi, &part,
                                                 warp_parts,
                                                 GumbelKeys{seed, (uint64_t)row << 32, inv_t});
  else
    scan_to_partial<1, false, false, RES, IdentityXf, true>(target + (size_t)row * V, lo, hi, &part,
                                                       warp_parts);
  TopK<1> top;
  Lse lse;
  if (cluster_reduce<1, false>(&part, S, top, lse)) am[row] = top.i[0];
}

constexpr int kWalkWarps = 4;

// Argmax of row `row` from the scratch: one index per row (nparts == 1) or
// the warp-wide best of the row's kFlatParts segment partials (value desc,
// index asc, as everywhere else).
__device__ __forceinline__ int row_argmax(const void* am, int nparts, size_t row, int lane) {
  constexpr unsigned kFull = 0xFFFFFFFFu;
  if (nparts == 1) return static_cast<const int32_t*>(am)[row];
  ArgPart q{-INFINITY, INT_MAX};
  if (lane < nparts) q = static_cast<const ArgPart*>(am)[row * nparts + lane];
  const uint32_t key = q.i == INT_MAX ? 0u : order_key(q.v);
  const uint32_t top = __reduce_max_sync(kFull, key);
  return (int)__reduce_min_sync(kFull, (key == top && q.i != INT_MAX) ? (uint32_t)q.i : 0xFFFFFFFFu);
}

__global__ void __launch_bounds__(kWalkWarps * 32)
accept_walk_kernel(const void* __restrict__ am, int nparts, const int32_t* __restrict__ parent,
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
  grid_dependency_sync();
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
    const size_t row0 = (size_t)b * (B + 1);
    a = row_argmax(am, nparts, row0, lane);
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
      a = row_argmax(am, nparts, row0 + 1 + cur, lane);
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

constexpr int kPathThreads = 256;
constexpr int kPathUnroll = 8;   // float4 loads in flight per thread (4: MoE-shaped 31.3 us, 8: 27.8, 16: 30.9)

__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <bool SAMPLED>
__global__ void __launch_bounds__(kPathThreads)
accept_path_kernel(const float* __restrict__ target, const int32_t* __restrict__ parent,
                   const int32_t* __restrict__ token, const int32_t* __restrict__ n_nodes, int B,
                   int N, int V, int S, int prefetch, float inv_t, uint64_t seed,
                   int32_t* __restrict__ acc_len,
                   int32_t* __restrict__ acc_tokens, int32_t* __restrict__ acc_nodes,
                   int32_t* __restrict__ bonus, int32_t* d_err) {
  __shared__ int32_t par_s[kMaxB], tok_s[kMaxB];
  __shared__ ArgPart part[2];                     // this CTA's partial, by level parity
  __shared__ ArgPart warp_best[kPathThreads / 32];
  __shared__ int a_s, child_s;
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x / S, rank = blockIdx.x % S;
  grid_dependency_sync();
  const int n = n_nodes[b];

  // Validate and stage the tree (every CTA of the cluster reaches the same verdict).
  int flag = (n < 0 || n > B) ? JT_DEVERR_NNODES : 0;
  if (!flag) {
    for (int v = tid; v < n; v += kPathThreads) {
      const int pv = parent[(size_t)b * B + v], t = token[(size_t)b * B + v];
      if (pv < -1 || pv >= v) flag |= JT_DEVERR_PARENT;
      if (t < 0 || t >= V) flag |= JT_DEVERR_TOKEN;
      par_s[v] = pv;
      tok_s[v] = t;
    }
  }
  const int bad = __syncthreads_or(flag);
  int32_t* at = acc_tokens + (size_t)b * N;
  int32_t* an = acc_nodes + (size_t)b * N;
  if (bad) {  // uniform over the cluster: nobody touches DSMEM
    if (rank == 0) {
      if (flag) raise_flag(d_err, flag);
      for (int i = tid; i < N; i += kPathThreads) { at[i] = -1; an[i] = -1; }
      if (tid == 0) { acc_len[b] = 0; bonus[b] = -1; }
    }
    return;
  }

  cg::cluster_group cluster = cg::this_cluster();
  const int v4 = V >> 2;
  const int per = (v4 + S - 1) / S;
  const int lo = min(v4, rank * per), hi = min(v4, lo + per);
  const float* rows = target + (size_t)b * (B + 1) * V;
  int cur = -1, row = 0, len = 0, a = -1;
  for (int level = 0;; ++level) {
    // Prefetch this CTA's segment of every child row (one of them is next).
    if (prefetch && tid < n && par_s[tid] == cur && hi > lo)
      prefetch_l2_bulk(rows + (size_t)(1 + tid) * V + 4 * lo, (uint32_t)(hi - lo) * 16u);
    // Scan this CTA's segment of the current row: max, lowest index on ties.
    const float4* r4 = reinterpret_cast<const float4*>(rows + (size_t)row * V);
    const GumbelKeys gk{seed, ((uint64_t)b * (B + 1) + row) << 32, inv_t};
    float bv = -INFINITY;
    int bi = INT_MAX;
    for (int j0 = lo + tid; j0 < hi; j0 += kPathUnroll * kPathThreads) {
      float4 x[kPathUnroll];
#pragma unroll
      for (int u = 0; u < kPathUnroll; ++u) {
        const int j = j0 + u * kPathThreads;
        x[u] = j < hi ? ld_stream(r4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
      if (SAMPLED) {
#pragma unroll
        for (int u = 0; u < kPathUnroll; ++u)
          if (j0 + u * kPathThreads < hi) x[u] = gk(x[u], j0 + u * kPathThreads);
      }
#pragma unroll
      for (int u = 0; u < kPathUnroll; ++u) {
        const int j = j0 + u * kPathThreads;
        if (j < hi) {
          if (x[u].x > bv || bi == INT_MAX) { bv = x[u].x; bi = 4 * j; }
          if (x[u].y > bv) { bv = x[u].y; bi = 4 * j + 1; }
          if (x[u].z > bv) { bv = x[u].z; bi = 4 * j + 2; }
          if (x[u].w > bv) { bv = x[u].w; bi = 4 * j + 3; }
        }
      }
    }
    {
      const uint32_t key = bi == INT_MAX ? 0u : order_key(bv);
      const uint32_t top = __reduce_max_sync(kFull, key);
      const uint32_t idx = __reduce_min_sync(kFull, (key == top && bi != INT_MAX) ? (uint32_t)bi : 0xFFFFFFFFu);
      const float wvv = __shfl_sync(kFull, bv, __ffs(__ballot_sync(kFull, key == top && (uint32_t)bi == idx && bi != INT_MAX)) - 1);
      if (lane == 0) warp_best[warp] = ArgPart{top == 0 ? -INFINITY : wvv, top == 0 ? INT_MAX : (int)idx};
    }
    __syncthreads();
    if (warp == 0) {
      const ArgPart wp = lane < kPathThreads / 32 ? warp_best[lane] : ArgPart{-INFINITY, INT_MAX};
      const uint32_t key = wp.i == INT_MAX ? 0u : order_key(wp.v);
      const uint32_t top = __reduce_max_sync(kFull, key);
      const uint32_t idx = __reduce_min_sync(kFull, (key == top && wp.i != INT_MAX) ? (uint32_t)wp.i : 0xFFFFFFFFu);
      const float wvv = __shfl_sync(kFull, wp.v, __ffs(__ballot_sync(kFull, key == top && (uint32_t)wp.i == idx && wp.i != INT_MAX)) - 1);
      if (lane == 0) part[level & 1] = ArgPart{top == 0 ? -INFINITY : wvv, top == 0 ? INT_MAX : (int)idx};
    }
    cluster.sync();  // every CTA's partial for this level is visible
    if (warp == 0) {
      ArgPart rp = {-INFINITY, INT_MAX};
      if (lane < S) rp = cluster.map_shared_rank(part, lane)[level & 1];
      const uint32_t key = rp.i == INT_MAX ? 0u : order_key(rp.v);
      const uint32_t top = __reduce_max_sync(kFull, key);
      const uint32_t idx = __reduce_min_sync(kFull, (key == top && rp.i != INT_MAX) ? (uint32_t)rp.i : 0xFFFFFFFFu);
      if (lane == 0) { a_s = (int)idx; child_s = INT_MAX; }
    }
    __syncthreads();
    a = a_s;
    if (tid < n && par_s[tid] == cur && tok_s[tid] == a) atomicMin(&child_s, tid);
    __syncthreads();
    const int c = child_s;
    if (c == INT_MAX || len >= N) break;   // uniform over the cluster
    if (rank == 0 && tid == 0) { at[len] = a; an[len] = c; }
    ++len;
    cur = c;
    row = 1 + c;
    __syncthreads();   // child_s / a_s are rewritten next level
  }
  if (rank == 0) {
    for (int i = len + tid; i < N; i += kPathThreads) { at[i] = -1; an[i] = -1; }
    if (tid == 0) { acc_len[b] = len; bonus[b] = a; }
  }
  cluster.sync();  // keep this CTA's partials alive until every rank has read them
}

bool use_path_walk(int B, int n_depth) { return (B + 1) > 4 * (n_depth + 1); }

}  // namespace

size_t accept_workspace_bytes(int batch, int B, int n_depth, int vocab, int num_sms) {
  if (use_path_walk(B, n_depth)) return 0;
  const long rows = (long)batch * (B + 1);
  if (use_flat_rows(rows, vocab, num_sms))
    return align_up((size_t)rows * kFlatParts * sizeof(ArgPart), 256);
  return align_up((size_t)rows * sizeof(int32_t), 256);
}

cudaError_t launch_tree_accept(const Ctx& c, const float* target, const int32_t* parent,
                               const int32_t* token, const int32_t* n_nodes, int batch, int B,
                               int n_depth, int vocab, int32_t* acc_len, int32_t* acc_tokens,
                               int32_t* acc_nodes, int32_t* bonus, bool sampled, float inv_t,
                               uint64_t seed) {
  if (batch == 0) return cudaSuccess;
  if (use_path_walk(B, n_depth)) {
    // Cluster size: enough CTAs for ~4 per SM, at most 16 per sequence.
    int S = 1;
    while (S < 16 && (long)batch * S * 2 <= 4L * c.num_sms && (vocab / 4) / (2 * S) >= 1024) S *= 2;
    const int prefetch = (long)batch * B <= 64L * 64 ? 1 : 0;
    auto kern = sampled ? accept_path_kernel<true> : accept_path_kernel<false>;
    return launch_kernel(kern, dim3(batch * S), dim3(kPathThreads), 0, c.stream, S, target, parent,
                         token, n_nodes, B, n_depth, vocab, S, prefetch, inv_t, seed, acc_len,
                         acc_tokens, acc_nodes, bonus, c.d_err);
  }
  const long rows = (long)batch * (B + 1);
  cudaError_t e;
  int nparts = 1;
  if (use_flat_rows(rows, vocab, c.num_sms)) {
    nparts = kFlatParts;
    const bool res = use_resident(1, (vocab / 4 + kFlatParts - 1) / kFlatParts);
    auto kern = sampled ? (res ? accept_argmax_flat_kernel<true, true>
                               : accept_argmax_flat_kernel<true, false>)
                        : (res ? accept_argmax_flat_kernel<false, true>
                               : accept_argmax_flat_kernel<false, false>);
    e = launch_kernel(kern, dim3((unsigned)(rows * kFlatParts)), dim3(kScanThreads), 0, c.stream,
                      1, target, n_nodes, B, vocab, inv_t, seed,
                      static_cast<ArgPart*>(c.workspace));
  } else {
    const int S = pick_row_split(rows, vocab / 4, c.num_sms, 16);
    const bool res = use_resident(1, (vocab / 4 + S - 1) / S);
    auto kern = sampled ? (res ? accept_argmax_kernel<true, true> : accept_argmax_kernel<true, false>)
                        : (res ? accept_argmax_kernel<false, true> : accept_argmax_kernel<false, false>);
    e = launch_clustered(kern, (int)(rows * S), S, c.stream, target, n_nodes, B, vocab, S, inv_t,
                         seed, static_cast<int32_t*>(c.workspace));
  }
  if (e != cudaSuccess) return e;
  return launch_kernel(accept_walk_kernel, dim3((batch + kWalkWarps - 1) / kWalkWarps),
                       dim3(kWalkWarps * 32), 0, c.stream, 1, (const void*)c.workspace, nparts,
                       parent, token, n_nodes, batch, B, n_depth, vocab, acc_len, acc_tokens,
                       acc_nodes, bonus, c.d_err);
}

}  // namespace jt
