// Full-vocabulary row scans: top-K (value desc, index asc) and the
// log-sum-exp of a row of fp32 logits, streamed once from HBM.
//
// Layout of the work: a row of V floats is cut into S segments (S = the
// cluster size, 1..16). The S CTAs of a thread-block cluster each stream one
// segment with 128-bit non-allocating loads, UNROLL float4s per thread in
// flight, keeping per thread a sorted top-K list in registers and an online
// (max, sum exp) pair. Lists are merged warp-wide with xor shuffles (a
// bitonic half-cleaner keeps the better half of two sorted lists, then
// log2 K compare-exchange stages re-sort it), then across warps through
// shared memory, then across the cluster: after a cluster barrier, CTA rank
// 0 reads the other CTAs' partials straight out of their shared memory
// (distributed shared memory) and finishes the row. No global scratch, no
// atomics, no second launch.
#pragma once

#include <cooperative_groups.h>

#include "jt_internal.cuh"

namespace jt {

namespace cg = cooperative_groups;

constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kScanUnroll = 8;

template <int K>
struct TopK {
  float v[K];
  int i[K];

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int k = 0; k < K; ++k) { v[k] = -INFINITY; i[k] = INT_MAX; }
  }

  __device__ __forceinline__ void push(float x, int idx) {
    if (!ranks_before(x, idx, v[K - 1], i[K - 1])) return;
    v[K - 1] = x;
    i[K - 1] = idx;
#pragma unroll
    for (int k = K - 1; k > 0; --k) {
      if (ranks_before(v[k], i[k], v[k - 1], i[k - 1])) {
        const float tv = v[k]; v[k] = v[k - 1]; v[k - 1] = tv;
        const int ti = i[k]; i[k] = i[k - 1]; i[k - 1] = ti;
      }
    }
  }

  // Keep the best K of (this ∪ other); both sorted, result sorted.
  __device__ __forceinline__ void merge(const float (&ov)[K], const int (&oi)[K]) {
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (ranks_before(ov[K - 1 - k], oi[K - 1 - k], v[k], i[k])) {
        v[k] = ov[K - 1 - k];
        i[k] = oi[K - 1 - k];
      }
    }
    // v is now bitonic; sort descending with half-cleaners.
#pragma unroll
    for (int j = K / 2; j > 0; j >>= 1) {
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const int p = k ^ j;
        if (p > k && ranks_before(v[p], i[p], v[k], i[k])) {
          const float tv = v[k]; v[k] = v[p]; v[p] = tv;
          const int ti = i[k]; i[k] = i[p]; i[p] = ti;
        }
      }
    }
  }

  __device__ __forceinline__ void warp_merge(unsigned mask = 0xFFFFFFFFu) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float ov[K];
      int oi[K];
#pragma unroll
      for (int k = 0; k < K; ++k) {
        ov[k] = __shfl_xor_sync(mask, v[k], off);
        oi[k] = __shfl_xor_sync(mask, i[k], off);
      }
      merge(ov, oi);
    }
  }
};

// Online log-sum-exp: the row's running max m and s = sum exp(x - m).
struct Lse {
  float m, s;
  __device__ __forceinline__ void init() { m = -INFINITY; s = 0.0f; }
  __device__ __forceinline__ void combine(float m2, float s2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; s = s2; return; }
    if (m2 > m) { s = s * __expf(m - m2) + s2; m = m2; }
    else { s = s + s2 * __expf(m2 - m); }
  }
  __device__ __forceinline__ void warp_reduce() {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
      const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, off);
      combine(m2, s2);
    }
  }
};

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

// Per-CTA partial result kept in shared memory for the cluster merge.
template <int K>
struct ScanPartial {
  float v[K];
  int i[K];
  float m, s;
};

// Streams floats [lo4*4, hi4*4) of `row` into per-thread state.
template <int K, bool LSE>
__device__ __forceinline__ void scan_segment(const float* __restrict__ row, int lo4, int hi4,
                                             TopK<K>& top, Lse& lse) {
  const float4* r4 = reinterpret_cast<const float4*>(row);
  for (int base = lo4 + (int)threadIdx.x; base < hi4; base += kScanThreads * kScanUnroll) {
    float4 x[kScanUnroll];
#pragma unroll
    for (int u = 0; u < kScanUnroll; ++u) {
      const int j = base + u * kScanThreads;
      x[u] = (j < hi4) ? ld_stream(r4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    if (LSE) {
      float bm = -INFINITY;
#pragma unroll
      for (int u = 0; u < kScanUnroll; ++u)
        bm = fmaxf(bm, fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w)));
      if (bm > lse.m) {
        lse.s = (lse.m == -INFINITY) ? 0.0f : lse.s * __expf(lse.m - bm);
        lse.m = bm;
      }
      if (lse.m != -INFINITY) {
        float acc = 0.0f;
#pragma unroll
        for (int u = 0; u < kScanUnroll; ++u)
          acc += __expf(x[u].x - lse.m) + __expf(x[u].y - lse.m) + __expf(x[u].z - lse.m) +
                 __expf(x[u].w - lse.m);
        lse.s += acc;
      }
    }
#pragma unroll
    for (int u = 0; u < kScanUnroll; ++u) {
      const int j = base + u * kScanThreads;
      if (j < hi4) {
        top.push(x[u].x, 4 * j);
        top.push(x[u].y, 4 * j + 1);
        top.push(x[u].z, 4 * j + 2);
        top.push(x[u].w, 4 * j + 3);
      }
    }
  }
}

// Reduces the CTA's per-thread state into `out` (valid in thread 0's view of
// shared memory after the trailing __syncthreads).
template <int K, bool LSE>
__device__ __forceinline__ void block_reduce(TopK<K>& top, Lse& lse, ScanPartial<K>* out,
                                             ScanPartial<K>* warp_parts) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  top.warp_merge();
  if (LSE) lse.warp_reduce();
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) { warp_parts[warp].v[k] = top.v[k]; warp_parts[warp].i[k] = top.i[k]; }
    warp_parts[warp].m = lse.m;
    warp_parts[warp].s = lse.s;
  }
  __syncthreads();
  if (warp == 0) {
    TopK<K> t;
    Lse l;
    if (lane < kScanWarps) {
#pragma unroll
      for (int k = 0; k < K; ++k) { t.v[k] = warp_parts[lane].v[k]; t.i[k] = warp_parts[lane].i[k]; }
      l.m = warp_parts[lane].m;
      l.s = warp_parts[lane].s;
    } else {
      t.init();
      l.init();
    }
    t.warp_merge();
    if (LSE) l.warp_reduce();
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < K; ++k) { out->v[k] = t.v[k]; out->i[k] = t.i[k]; }
      out->m = l.m;
      out->s = l.s;
    }
  }
  __syncthreads();
}

// Merge the cluster's partials in CTA rank 0 (warp 0). Returns true in the
// thread that holds the final result (lane 0 of warp 0 of rank 0).
template <int K, bool LSE>
__device__ __forceinline__ bool cluster_reduce(ScanPartial<K>* mine, int S, TopK<K>& top,
                                               Lse& lse) {
  if (S == 1) {
    if (threadIdx.x != 0) return false;
#pragma unroll
    for (int k = 0; k < K; ++k) { top.v[k] = mine->v[k]; top.i[k] = mine->i[k]; }
    lse.m = mine->m;
    lse.s = mine->s;
    return true;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();  // every CTA's partial is in its shared memory
  bool holder = false;
  if (cluster.block_rank() == 0 && threadIdx.x < 32) {
    const int lane = threadIdx.x;
    if (lane < S) {
      const ScanPartial<K>* p = cluster.map_shared_rank(mine, lane);
#pragma unroll
      for (int k = 0; k < K; ++k) { top.v[k] = p->v[k]; top.i[k] = p->i[k]; }
      lse.m = p->m;
      lse.s = p->s;
    } else {
      top.init();
      lse.init();
    }
    top.warp_merge();
    if (LSE) lse.warp_reduce();
    holder = (lane == 0);
  }
  cluster.sync();  // keep every CTA's shared memory alive until rank 0 has read it
  return holder;
}

// Picks the cluster size (segments per row) for `rows` rows of `v4` float4s:
// enough CTAs to cover the SMs a few times, segments of >= 2048 float4s.
inline int pick_row_split(long rows, int v4, int num_sms, int max_split) {
  int s = 1;
  while (s < max_split && rows * s < 2L * num_sms && (v4 / (2 * s)) >= 2048) s *= 2;
  return s;
}

template <typename Kernel, typename... Args>
cudaError_t launch_clustered(Kernel kernel, int grid, int cluster, cudaStream_t stream,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kScanThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 8) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace jt
