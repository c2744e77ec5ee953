// jt_tree_attn: tree-causal GQA attention for the verification pass.
//
// Node v of sequence b, query head h (KV head h / g) attends to the prefix
// KV and to the tree nodes u with M[v,u] = 0, i.e. its ancestors and itself
// (JetSpec summary on paperlayer.ai, §2 "Architecture" and App. E
// "Verification"; JetSpec review on startedourmission.github.io, "How it
// works", mask equation). The mask is read as ancestor bitmasks.
//
// This translation unit holds the first, CUDA-core version: one CTA per
// (sequence, KV head, 16 query rows), key tiles of 32 staged through shared
// memory, online softmax in fp32.
#include "jt_internal.cuh"

namespace jt {
namespace {

constexpr int kRows = 16;
constexpr int kKeys = 32;
constexpr int kThreads = 128;

__device__ __forceinline__ float bf2f(__nv_bfloat16 x) { return __bfloat162float(x); }

template <int D>
__global__ void __launch_bounds__(kThreads)
attn_simple_kernel(jt_attn_args a, int32_t* d_err) {
  constexpr int DL = D / 32;  // output dims per lane
  __shared__ float q_s[kRows][D];
  __shared__ float k_s[kKeys][D + 1];
  __shared__ float v_s[kKeys][D];
  const int b = blockIdx.z, kh = blockIdx.y;
  const int g = a.hq / a.hkv;
  const int row0 = blockIdx.x * kRows;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = a.n_nodes[b];
  const int L = a.prefix_len[b];
  const bool paged = a.block_table != nullptr;
  const int words = (a.B + 31) >> 5;

  // Validate this sequence (every CTA of the sequence reaches the same verdict).
  int flag = 0;
  if (n < 0 || n > a.B) flag |= JT_DEVERR_NNODES;
  const int Lmax = paged ? a.max_pages * kPageSize : a.max_prefix;
  if (L < 0 || L > Lmax) flag |= JT_DEVERR_PREFIX;
  if (paged && !(flag & JT_DEVERR_PREFIX)) {
    const int np = (L + kPageSize - 1) / kPageSize;
    for (int p = threadIdx.x; p < np; p += kThreads) {
      const int pg = a.block_table[(size_t)b * a.max_pages + p];
      if (pg < 0 || pg >= a.n_pages) flag |= JT_DEVERR_PAGE;
    }
  }
  flag = __syncthreads_or(flag) ? (flag | 0x40000000) : flag;
  const bool bad = (flag & 0x40000000) != 0;
  if (bad && (flag & ~0x40000000)) raise_flag(d_err, flag & ~0x40000000);

  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);
  const __nv_bfloat16* kc = static_cast<const __nv_bfloat16*>(a.k_cache);
  const __nv_bfloat16* vc = static_cast<const __nv_bfloat16*>(a.v_cache);
  const __nv_bfloat16* kt = static_cast<const __nv_bfloat16*>(a.k_tree);
  const __nv_bfloat16* vt = static_cast<const __nv_bfloat16*>(a.v_tree);
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out);
  const float scale = a.scale != 0.0f ? a.scale : rsqrtf((float)D);

  // Query rows: row r = v * g + j (node-major), head h = kh * g + j.
  for (int i = threadIdx.x; i < kRows * D; i += kThreads) {
    const int r = i / D, d = i % D;
    const int row = row0 + r;
    const int v = row / g, j = row % g;
    float x = 0.0f;
    if (!bad && v < n) x = bf2f(q[(((size_t)b * a.B + v) * a.hq + kh * g + j) * D + d]);
    q_s[r][d] = x;
  }

  float m[4], l[4], o[4][DL];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.0f;
#pragma unroll
    for (int dd = 0; dd < DL; ++dd) o[r][dd] = 0.0f;
  }
  uint32_t mrow[4][kMaxWords];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = row0 + warp * 4 + r;
    const int v = row / g;
#pragma unroll
    for (int w = 0; w < kMaxWords; ++w)
      mrow[r][w] = (!bad && v < n && w < words) ? a.mask[((size_t)b * a.B + v) * words + w] : 0u;
  }

  const int n_pre_tiles = bad ? 0 : (L + kKeys - 1) / kKeys;
  const int n_tree_tiles = bad ? 0 : (n + kKeys - 1) / kKeys;
  for (int t = 0; t < n_pre_tiles + n_tree_tiles; ++t) {
    const bool tree = t >= n_pre_tiles;
    const int k0 = tree ? (t - n_pre_tiles) * kKeys : t * kKeys;
    const int kend = tree ? n : L;
    __syncthreads();
    for (int i = threadIdx.x; i < kKeys * D; i += kThreads) {
      const int kk = i / D, d = i % D;
      const int key = k0 + kk;
      float xk = 0.0f, xv = 0.0f;
      if (key < kend) {
        size_t off;
        if (tree) {
          off = (((size_t)b * a.B + key) * a.hkv + kh) * D + d;
          xk = bf2f(kt[off]);
          xv = bf2f(vt[off]);
        } else {
          size_t tokpos;
          if (paged) {
            const int pg = a.block_table[(size_t)b * a.max_pages + key / kPageSize];
            tokpos = (size_t)pg * kPageSize + key % kPageSize;
          } else {
            tokpos = (size_t)b * a.max_prefix + key;
          }
          off = (tokpos * a.hkv + kh) * D + d;
          xk = bf2f(kc[off]);
          xv = bf2f(vc[off]);
        }
      }
      k_s[kk][d] = xk;
      v_s[kk][d] = xv;
    }
    __syncthreads();
    const int key = k0 + lane;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int lr = warp * 4 + r;
      float s = 0.0f;
#pragma unroll 8
      for (int d = 0; d < D; ++d) s += q_s[lr][d] * k_s[lane][d];
      s *= scale;
      bool vis = key < kend;
      if (tree && vis) vis = (mrow[r][key >> 5] >> (key & 31)) & 1u;
      if (!vis) s = -INFINITY;
      float tmax = s;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xFFFFFFFFu, tmax, off));
      const float mn = fmaxf(m[r], tmax);
      if (mn == -INFINITY) continue;  // nothing visible yet for this row
      const float corr = (m[r] == -INFINITY) ? 0.0f : __expf(m[r] - mn);
      const float p = (s == -INFINITY) ? 0.0f : __expf(s - mn);
      float psum = p;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xFFFFFFFFu, psum, off);
      l[r] = l[r] * corr + psum;
      m[r] = mn;
#pragma unroll
      for (int dd = 0; dd < DL; ++dd) o[r][dd] *= corr;
      for (int kk = 0; kk < kKeys; ++kk) {
        const float pk = __shfl_sync(0xFFFFFFFFu, p, kk);
#pragma unroll
        for (int dd = 0; dd < DL; ++dd) o[r][dd] += pk * v_s[kk][lane + 32 * dd];
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = row0 + warp * 4 + r;
    const int v = row / g, j = row % g;
    if (v >= a.B) continue;
    const float inv = (v < n && l[r] > 0.0f) ? 1.0f / l[r] : 0.0f;  // unused slots: zero
#pragma unroll
    for (int dd = 0; dd < DL; ++dd)
      out[(((size_t)b * a.B + v) * a.hq + kh * g + j) * D + lane + 32 * dd] =
          __float2bfloat16_rn(o[r][dd] * inv);
  }
}

}  // namespace

size_t attn_workspace_bytes(const jt_attn_args& a, int num_sms) {
  (void)a;
  (void)num_sms;
  return 0;
}

cudaError_t launch_tree_attn(const Ctx& c, const jt_attn_args& a) {
  if (a.batch == 0) return cudaSuccess;
  const int g = a.hq / a.hkv;
  dim3 grid((a.B * g + kRows - 1) / kRows, a.hkv, a.batch), block(kThreads);
  if (a.head_dim == 64)
    attn_simple_kernel<64><<<grid, block, 0, c.stream>>>(a, c.d_err);
  else
    attn_simple_kernel<128><<<grid, block, 0, c.stream>>>(a, c.d_err);
  return cudaGetLastError();
}

}  // namespace jt
