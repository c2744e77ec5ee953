// jt_tree_mask: ancestor bitmasks for the tree-causal attention mask.
//
// Definition: M[v,u] = 0 iff u ∈ Anc(v) ∪ {v} (JetSpec review on
// startedourmission.github.io, "How it works", mask equation). The mask is
// kept as one bit per (v, u), never as a dense matrix (JetSpec summary on
// paperlayer.ai, App. E "Verification").
//
// One CTA per sequence, one thread per node. Thread v follows its parent
// chain (length = depth(v) <= B) through a shared-memory copy of the parent
// array, setting one bit per visited node in registers, then stores its
// ceil(B/32)-word row. parent[v] < v is checked first for every node of the
// sequence, so every walk strictly decreases and ends.
#include "jt_internal.cuh"

namespace jt {
namespace {

template <int WORDS>
__global__ void __launch_bounds__(256) tree_mask_kernel(const int32_t* __restrict__ parent,
                                                        const int32_t* __restrict__ n_nodes,
                                                        int B, uint32_t* __restrict__ mask,
                                                        int32_t* d_err) {
  __shared__ int32_t par_s[kMaxB];
  const int b = blockIdx.x;
  const int v = threadIdx.x;
  grid_dependency_sync();
  const int n = n_nodes[b];
  const bool n_ok = (n >= 0 && n <= B);
  int p = -1;
  bool bad = !n_ok;
  if (v < B) {
    p = parent[(size_t)b * B + v];
    if (n_ok && v < n && (p < -1 || p >= v)) bad = true;
    par_s[v] = p;
  }
  bad = __syncthreads_or(bad);
  if (v >= B) return;
  if (bad && threadIdx.x == 0) raise_flag(d_err, n_ok ? JT_DEVERR_PARENT : JT_DEVERR_NNODES);

  uint32_t w[WORDS];
#pragma unroll
  for (int i = 0; i < WORDS; ++i) w[i] = 0u;
  if (!bad && v < n) {
    for (int u = v; u != -1; u = par_s[u]) {
      const int wi = u >> 5;
      const uint32_t bit = 1u << (u & 31);
#pragma unroll
      for (int i = 0; i < WORDS; ++i)
        if (i == wi) w[i] |= bit;
    }
  }
  const int words = (B + 31) >> 5;
  uint32_t* row = mask + ((size_t)b * B + v) * words;
#pragma unroll
  for (int i = 0; i < WORDS; ++i)
    if (i < words) row[i] = w[i];
}

}  // namespace

cudaError_t launch_tree_mask(const Ctx& c, const int32_t* parent, const int32_t* n_nodes,
                             int batch, int B, uint32_t* mask) {
  if (batch == 0) return cudaSuccess;
  const int words = (B + 31) / 32;
  const dim3 grid(batch), block(B < 32 ? 32 : B);
  auto kern = words <= 1 ? tree_mask_kernel<1>
            : words <= 2 ? tree_mask_kernel<2>
            : words <= 4 ? tree_mask_kernel<4>
                         : tree_mask_kernel<8>;
  return launch_kernel(kern, grid, block, 0, c.stream, 1, parent, n_nodes, B, mask, c.d_err);
}

}  // namespace jt
