// Internal declarations shared by libjtree's translation units.
// Not part of the public ABI (that is include/jtree.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/jtree.h"

namespace jt {

constexpr int kMaxB = 256;        // tree budget limit (8 mask words per row)
constexpr int kMaxWords = kMaxB / 32;
constexpr int kMaxDepth = 64;
constexpr int kMaxW = 32;
constexpr int kPageSize = 16;
constexpr int kNumSMs = 152;      // GB300; the launchers query the real count

// Cycle budget of the bounded device-side waits on mbarriers (about 2 s at
// 2 GHz). jt_set_wait_budget may shorten it for kernels launched afterwards;
// the waits that drain a CTA's own copies and MMAs after it gave up always
// use this default.
constexpr long long kDefaultWaitBudget = 4000000000LL;
long long wait_budget();   // the budget kernels launched now are given

// ---------------------------------------------------------------------------
// Device error word.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_flag(int32_t* d_err, int32_t bit) {
  if (d_err) atomicOr(d_err, bit);
}

// Float -> uint32 key whose unsigned order is the float order, with -0 == +0
// (the caller folds -0 to +0 first). NaN is outside the contract.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// (value, index) ranking used by every top-W / argmax in the library:
// a ranks before b iff a.v > b.v, or a.v == b.v and a.i < b.i.
__device__ __forceinline__ bool ranks_before(float av, int ai, float bv, int bi) {
  return av > bv || (av == bv && ai < bi);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. Every kernel of the library is launched with
// programmatic stream serialization, so it may be scheduled while the grid
// before it in the stream is still draining. Each kernel therefore calls
// wait_prior_grids() before its first global-memory access (read or write),
// which blocks until that grid has completed and its writes are visible;
// only data-independent set-up (shared-memory barriers, TMEM allocation)
// comes before it. Right after the wait the kernel lets its own dependent
// grid be scheduled. On a launch without the attribute both are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void wait_prior_grids() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void release_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_sync() {
  wait_prior_grids();
  release_dependents();
}

// ---------------------------------------------------------------------------
// Launch plumbing shared by jt_api.cu and the kernel files.
// ---------------------------------------------------------------------------
struct Ctx {
  cudaStream_t stream;
  int32_t* d_err;
  void* workspace;
  size_t workspace_bytes;
  int num_sms;
  int device;
};

// Device attributes are cached per device (the only process-wide state).
int device_sm_count(int device);

// Launchers (defined next to their kernels). They assume validated args and
// return the cudaError_t of the launch.
cudaError_t launch_tree_mask(const Ctx&, const int32_t* parent, const int32_t* n_nodes, int batch,
                             int B, uint32_t* mask);
cudaError_t launch_tree_expand(const Ctx&, const int32_t* tok, const float* logp,
                               const float* entropy, int mode, float alpha, int batch,
                               int n_depth, int W, int B, int32_t* parent, int32_t* token,
                               int32_t* depth, float* score, int32_t* n_nodes);
cudaError_t launch_topw(const Ctx&, const float* logits, int rows, int vocab, int W, int32_t* tok,
                        float* logp, float* entropy);
size_t accept_workspace_bytes(int batch, int B, int n_depth, int vocab, int num_sms);
cudaError_t launch_tree_accept(const Ctx&, const float* target, const int32_t* parent,
                               const int32_t* token, const int32_t* n_nodes, int batch, int B,
                               int n_depth, int vocab, int32_t* acc_len, int32_t* acc_tokens,
                               int32_t* acc_nodes, int32_t* bonus, bool sampled = false,
                               float inv_t = 1.0f, uint64_t seed = 0);
cudaError_t launch_tree_commit(const Ctx&, const jt_commit_args& a);
size_t lmhead_workspace_bytes(int rows, int vocab, int W);
cudaError_t launch_lmhead_topw(const Ctx&, const void* hidden, const void* w_lm, int rows, int d,
                               int vocab, int W, int32_t* tok, float* logp, float* entropy);
size_t attn_workspace_bytes(const jt_attn_args& a, int num_sms);
cudaError_t launch_tree_attn(const Ctx&, const jt_attn_args& a);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launches `kernel` on `stream` with programmatic stream serialization and,
// when cluster > 1, 1-D clusters of `cluster` CTAs (sizes above 8 opt in to
// non-portable clusters).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cluster;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (cluster > 8) {
      cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace jt
