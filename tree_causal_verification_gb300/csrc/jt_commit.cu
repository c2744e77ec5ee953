// jt_tree_commit_kv: append the accepted path's K/V rows to the prefix cache.
//
// "JetSpec++: Foresight Parallel Drafting with Self Refinements" (paperlayer.ai
// summary), §3 "Preliminaries": a verification round commits the accepted
// prefix plus one bonus token. The accepted draft nodes' K/V rows, produced by
// the verification pass, become cache positions L .. L+a-1 in path order; the
// bonus token's K/V does not exist yet and is not written.
//
// GPU design: a gather/scatter of at most n_depth token rows (hkv * D bf16 per
// tensor) per sequence, bound by HBM (2 * a * hkv * D * 2 bytes read and the
// same written per sequence). One CTA per sequence validates the whole path
// and every destination slot first, so a rejected sequence is left untouched,
// then all threads copy 16-byte chunks with kUnroll chunks of K and of V in
// flight each. Thread 0 writes the new length after the CTA barrier that
// follows every thread's read of the old one, so the two may alias.
#include "jt_internal.cuh"

namespace jt {
namespace {

constexpr int kCommitThreads = 256;
constexpr int kUnroll = 4;

__global__ void __launch_bounds__(kCommitThreads)
tree_commit_kernel(const uint4* __restrict__ k_tree, const uint4* __restrict__ v_tree,
                   uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                   const int32_t* __restrict__ block_table, int B, int n_depth, int chunks,
                   int page_size, int max_pages, int n_pages, long capacity, int max_prefix,
                   const int32_t* prefix_len, const int32_t* __restrict__ acc_len,
                   const int32_t* __restrict__ acc_nodes, int32_t* new_prefix_len,
                   int32_t* d_err) {
  __shared__ long long dst_s[kMaxDepth];   // destination token row of committed token i
  __shared__ int src_s[kMaxDepth];         // its tree node
  const int b = blockIdx.x, tid = threadIdx.x;
  grid_dependency_sync();
  const int L = prefix_len[b];
  const int a = acc_len[b];
  int flag = 0;
  if (a < 0 || a > n_depth) flag = JT_DEVERR_PATH;
  else if (L < 0 || (long)L + a > capacity) flag = JT_DEVERR_PREFIX;
  if (flag == 0 && tid < a) {               // n_depth <= kMaxDepth <= kCommitThreads
    const int v = acc_nodes[(size_t)b * n_depth + tid];
    if (v < 0 || v >= B) flag |= JT_DEVERR_PATH;
    const long pos = (long)L + tid;
    long long row = (long long)b * max_prefix + pos;
    if (block_table) {
      const int page = block_table[(size_t)b * max_pages + pos / page_size];
      if (page < 0 || page >= n_pages) flag |= JT_DEVERR_PAGE;
      row = (long long)page * page_size + pos % page_size;
    }
    dst_s[tid] = row;
    src_s[tid] = v;
  }
  if (__syncthreads_or(flag)) {
    if (flag) raise_flag(d_err, flag);
    if (tid == 0) new_prefix_len[b] = L;
    return;
  }
  const int total = a * chunks;
  for (int i0 = tid; i0 < total; i0 += kCommitThreads * kUnroll) {
    uint4 kx[kUnroll], vx[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kCommitThreads;
      if (i < total) {
        const int t = i / chunks, c = i % chunks;
        const size_t src = ((size_t)b * B + src_s[t]) * chunks + c;
        kx[u] = k_tree[src];
        vx[u] = v_tree[src];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = i0 + u * kCommitThreads;
      if (i < total) {
        const int t = i / chunks, c = i % chunks;
        const size_t dst = (size_t)dst_s[t] * chunks + c;
        k_cache[dst] = kx[u];
        v_cache[dst] = vx[u];
      }
    }
  }
  if (tid == 0) new_prefix_len[b] = L + a;
}

}  // namespace

cudaError_t launch_tree_commit(const Ctx& c, const jt_commit_args& a) {
  if (a.batch == 0) return cudaSuccess;
  const int chunks = a.hkv * a.head_dim / 8;
  const bool paged = a.block_table != nullptr;
  const long capacity = paged ? (long)a.max_pages * a.page_size : (long)a.max_prefix;
  return launch_kernel(tree_commit_kernel, dim3(a.batch), dim3(kCommitThreads), 0, c.stream, 1,
                       static_cast<const uint4*>(a.k_tree), static_cast<const uint4*>(a.v_tree),
                       static_cast<uint4*>(a.k_cache), static_cast<uint4*>(a.v_cache),
                       a.block_table, a.B, a.n_depth, chunks, paged ? a.page_size : 1,
                       a.max_pages, a.n_pages, capacity, a.max_prefix, a.prefix_len, a.acc_len,
                       a.acc_nodes, a.new_prefix_len, c.d_err);
}

}  // namespace jt
