// Full-vocabulary row scans: top-K (value desc, index asc) and the
// log-sum-exp of a row of fp32 logits, streamed once from HBM.
//
// Work layout: a row of V floats is cut into S segments (S = the cluster
// size, 1..16); each CTA of a thread-block cluster streams one segment with
// 128-bit non-allocating loads, two batches of float4s per thread in flight.
// Per thread: a sorted top-K list in registers, guarded by a one-compare
// rejection test of each float4's maximum against the current K-th value,
// and an online log-sum-exp in the log2 domain (optionally with the sum that
// gives the distribution's entropy).
//
// Selection (warp, then block, then cluster) runs K rounds of a warp-wide
// argmax: every lane offers its best remaining candidate; __reduce_max_sync
// over an order-preserving uint32 key of the value picks the winning value,
// __reduce_min_sync over the indices holding it breaks ties towards the
// lower token id, and the winning lane advances to its next candidate.
// The cluster's CTAs hand their partials to CTA rank 0 through distributed
// shared memory. No global scratch, no atomics, no second launch.
#pragma once

#include <cooperative_groups.h>

#include "jt_internal.cuh"

namespace jt {

namespace cg = cooperative_groups;

constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kScanBatch = 4;     // float4s per thread per batch (two batches in flight)
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int K>
struct TopK {
  float v[K];
  int i[K];
  int n;      // real elements inserted so far (the first K always enter)
  float thr;  // v[K-1] once K elements are in, NaN before (every test passes)
  // Warp-wide pruning bound: the K-th best value of the warp so far (over
  // the union of the lanes' lists). An element strictly below it ranks after
  // K elements the warp already holds, so it cannot be in the warp's top K.
  float wthr;

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int k = 0; k < K; ++k) { v[k] = -INFINITY; i[k] = INT_MAX; }
    n = 0;
    thr = __int_as_float(0x7fffffff);
    wthr = -INFINITY;
  }

  // Elements must arrive in increasing index order within a thread, so a
  // later element that ties the K-th value never displaces it.
  __device__ __forceinline__ void push(float x, int idx) {
    if (x <= thr) return;   // false for the NaN sentinel: the first K always enter
    ++n;
    v[K - 1] = x;
    i[K - 1] = idx;
#pragma unroll
    for (int k = K - 1; k > 0; --k) {
      if (ranks_before(v[k], i[k], v[k - 1], i[k - 1])) {
        const float tv = v[k]; v[k] = v[k - 1]; v[k - 1] = tv;
        const int ti = i[k]; i[k] = i[k - 1]; i[k - 1] = ti;
      }
    }
    if (n >= K) thr = v[K - 1];
  }
};

// Online log-sum-exp in log2 units: with u = x*log2e, the row's running max
// m of u, s = sum 2^(u - m) and (entropy scans only) t = sum (u - m) 2^(u - m).
// Then ln Z = m ln2 + ln s and the entropy of softmax(x) is ln s - ln2 * t/s
// nats. When m grows by -d (d = m_old - m_new < 0), s' = s 2^d and
// t' = (t + d s) 2^d.
struct Lse {
  float m, s, t;
  __device__ __forceinline__ void init() { m = -INFINITY; s = 0.0f; t = 0.0f; }
  __device__ __forceinline__ void combine(float m2, float s2, float t2) {
    if (m2 == -INFINITY) return;
    if (m == -INFINITY) { m = m2; s = s2; t = t2; return; }
    if (m2 > m) {
      const float d = m - m2, f = fast_ex2(d);
      t = fmaf(fmaf(d, s, t), f, t2);
      s = fmaf(s, f, s2);
      m = m2;
    } else {
      const float d = m2 - m, f = fast_ex2(d);
      t = fmaf(fmaf(d, s2, t2), f, t);
      s = fmaf(s2, f, s);
    }
  }
  __device__ __forceinline__ void warp_reduce() {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
      const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, off);
      const float t2 = __shfl_xor_sync(0xFFFFFFFFu, t, off);
      combine(m2, s2, t2);
    }
  }
  // Raises the running max to bm (> m), rescaling s (and t when ENT).
  template <bool ENT>
  __device__ __forceinline__ void raise(float bm) {
    if (m == -INFINITY) {
      s = 0.0f;
      t = 0.0f;
    } else {
      const float d = m - bm, f = fast_ex2(d);
      if (ENT) t = fmaf(d, s, t) * f;
      s *= f;
    }
    m = bm;
  }
  // Adds one element with u - m = a (a <= 0; -inf for a -inf logit).
  template <bool ENT>
  __device__ __forceinline__ float term(float a, float& tacc) const {
    const float e = fast_ex2(a);
    // a = -inf (or below the flush range) gives e = 0: the clamp keeps 0 * a finite.
    if (ENT) tacc = fmaf(fmaxf(a, -126.0f), e, tacc);
    return e;
  }
};

// Element transform applied to each float4 as it is loaded (float4 index j4):
// the identity for plain scans.
struct IdentityXf {
  __device__ __forceinline__ float4 operator()(float4 x, int) const { return x; }
};

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
               : "l"(p));
  return r;
}

// A candidate list handed between selection levels.
template <int K>
struct ScanPartial {
  float v[K];
  int i[K];
  float m, s, t;
};

// K rounds of warp-wide argmax. Lane l offers the sorted list (cv, ci) of
// length `len`; on return every lane holds the warp's best K in out_v/out_i.
template <int K, int L>
__device__ __forceinline__ void warp_select(const float (&cv)[L], const int (&ci)[L], int len,
                                            float (&out_v)[K], int (&out_i)[K]) {
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31;
  int head = 0;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    float hv = -INFINITY;
    int hi = INT_MAX;
#pragma unroll
    for (int q = 0; q < L; ++q)
      if (q == head && q < len) { hv = cv[q]; hi = ci[q]; }
    const bool live = head < len;
    // key 0 = nothing left in this lane; every real value maps above 0.
    const uint32_t key = live ? order_key(hv) : 0u;
    const uint32_t top = __reduce_max_sync(kFull, key);
    const uint32_t idx = __reduce_min_sync(kFull, (live && key == top) ? (uint32_t)hi : 0xFFFFFFFFu);
    // The winner: the lane whose head has that key and index.
    const bool win = live && key == top && (uint32_t)hi == idx;
    const float wv = __shfl_sync(kFull, hv, __ffs(__ballot_sync(kFull, win)) - 1);
    out_v[k] = top == 0 ? -INFINITY : wv;
    out_i[k] = top == 0 ? INT_MAX : (int)idx;
    if (win) ++head;
    (void)lane;
  }
}

// Inverse of order_key for keys of real values (key 0 = none -> -inf).
__device__ __forceinline__ float key_value(uint32_t key) {
  if (key == 0u) return -INFINITY;
  const uint32_t u = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
  return __uint_as_float(u);
}

// One batch of kScanBatch float4s (element index 4*j of float4 j = j0 + u*T).
// refresh: every lane of the warp processes a batch in this call and the
// warp-wide pruning bound is recomputed afterwards (K rounds of warp argmax,
// so it is done only while the bound is still tightening quickly).
template <int K, bool LSE, bool ENT>
__device__ __forceinline__ void scan_batch(const float4 (&x)[kScanBatch], int j0, TopK<K>& top,
                                           Lse& lse, bool refresh) {
  float mx[kScanBatch];
#pragma unroll
  for (int u = 0; u < kScanBatch; ++u)
    mx[u] = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
  if (LSE) {
    const float bm2 = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * kLog2e;
    if (bm2 > lse.m) lse.raise<ENT>(bm2);
    if (lse.m != -INFINITY) {
      const float nm = -lse.m;
      float a0 = 0.0f, a1 = 0.0f, t0 = 0.0f, t1 = 0.0f;
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) {
        a0 += lse.term<ENT>(fmaf(x[u].x, kLog2e, nm), t0) +
              lse.term<ENT>(fmaf(x[u].y, kLog2e, nm), t1);
        a1 += lse.term<ENT>(fmaf(x[u].z, kLog2e, nm), t0) +
              lse.term<ENT>(fmaf(x[u].w, kLog2e, nm), t1);
      }
      lse.s += a0 + a1;
      if (ENT) lse.t += t0 + t1;
    }
  }
#pragma unroll
  for (int u = 0; u < kScanBatch; ++u) {
    // Some element of this float4 may enter: above the lane's own K-th value
    // and not below the warp's bound.
    if (mx[u] >= top.wthr && !(mx[u] <= top.thr)) {
      const int e = 4 * (j0 + u * kScanThreads);
      top.push(x[u].x, e);
      top.push(x[u].y, e + 1);
      top.push(x[u].z, e + 2);
      top.push(x[u].w, e + 3);
    }
  }
  if (refresh) {
    float wv[K];
    int wi[K];
    warp_select<K, K>(top.v, top.i, min(top.n, K), wv, wi);
    top.wthr = wv[K - 1];   // -inf while the warp holds fewer than K elements
  }
}

// Streams float4s [lo4, hi4) of `row` into per-thread state: full batches
// without bounds checks, ping-ponging two register buffers so that one batch
// is in flight while the other is processed, then a checked tail.
// EARLY_TAIL: a segment of at most two full batches issues its tail's loads
// together with them (one round trip to memory instead of two); measured to
// pay off for the plain argmax only, the log-sum-exp and keyed scans lose.
template <int K, bool LSE, bool ENT = false, class Xf = IdentityXf, bool EARLY_TAIL = false>
__device__ __forceinline__ void scan_segment(const float* __restrict__ row, int lo4, int hi4,
                                             TopK<K>& top, Lse& lse, const Xf& xf = Xf()) {
  const float4* r4 = reinterpret_cast<const float4*>(row);
  constexpr int STEP = kScanThreads * kScanBatch;
  const int tid = (int)threadIdx.x;
  const int full_end = lo4 + ((hi4 - lo4) / STEP) * STEP;
  float4 a[kScanBatch], b[kScanBatch];
  int base = lo4;
  // Full batches are uniform over the CTA; the warp bound is refreshed after
  // batches 1, 2, 4, 8, ... (a stale bound is still a valid, looser bound).
  int nbatch = 0;
  auto refresh = [&]() { ++nbatch; return (nbatch & (nbatch - 1)) == 0; };
  if (base < full_end) {
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) a[u] = ld_stream(r4 + base + tid + u * kScanThreads);
  }
  const bool early_tail = EARLY_TAIL && full_end - lo4 <= 2 * STEP && full_end < hi4;
  float4 tl[kScanBatch];
  if (early_tail) {
    if (base + STEP < full_end) {
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) b[u] = ld_stream(r4 + base + STEP + tid + u * kScanThreads);
    }
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) {
      const int j = full_end + tid + u * kScanThreads;
      tl[u] = j < hi4 ? ld_stream(r4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
  }
  while (base < full_end) {
    const bool nb = base + STEP < full_end;
    if (nb && !(early_tail && base == lo4)) {   // the early tail loaded batch 1 already
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) b[u] = ld_stream(r4 + base + STEP + tid + u * kScanThreads);
    }
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) a[u] = xf(a[u], base + tid + u * kScanThreads);
    scan_batch<K, LSE, ENT>(a, base + tid, top, lse, refresh());
    base += STEP;
    if (!nb) break;
    const bool na = base + STEP < full_end;
    if (na) {
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) a[u] = ld_stream(r4 + base + STEP + tid + u * kScanThreads);
    }
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) b[u] = xf(b[u], base + tid + u * kScanThreads);
    scan_batch<K, LSE, ENT>(b, base + tid, top, lse, refresh());
    base += STEP;
    if (!na) break;
  }
  // Tail: fewer than STEP float4s, padded with -inf (which never enters the
  // top-K ahead of a real element and adds 0 to the sum).
  if (full_end < hi4) {
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) {
      const int j = full_end + tid + u * kScanThreads;
      a[u] = j < hi4 ? xf(early_tail ? tl[u] : ld_stream(r4 + j), j) : ninf;
    }
    if (full_end + tid < hi4) {
      // Lanes whose whole batch is padding skip it (their padding would
      // otherwise occupy top-K slots as if they were real -inf elements).
      float4 x[kScanBatch];
      int cnt = 0;
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) {
        const int j = full_end + tid + u * kScanThreads;
        x[u] = a[u];
        cnt += j < hi4;
      }
      if (cnt == kScanBatch) {
        scan_batch<K, LSE, ENT>(x, full_end + tid, top, lse, false);
      } else {
        // Partial batch: element-wise, in index order.
        if (LSE) {
          float bm = -INFINITY;
#pragma unroll
          for (int u = 0; u < kScanBatch; ++u)
            if (u < cnt) bm = fmaxf(bm, fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w)));
          const float bm2 = bm * kLog2e;
          if (bm2 > lse.m) lse.raise<ENT>(bm2);
          if (lse.m != -INFINITY) {
            const float nm = -lse.m;
            float acc = 0.0f, tacc = 0.0f;
#pragma unroll
            for (int u = 0; u < kScanBatch; ++u)
              if (u < cnt)
                acc += lse.term<ENT>(fmaf(x[u].x, kLog2e, nm), tacc) +
                       lse.term<ENT>(fmaf(x[u].y, kLog2e, nm), tacc) +
                       lse.term<ENT>(fmaf(x[u].z, kLog2e, nm), tacc) +
                       lse.term<ENT>(fmaf(x[u].w, kLog2e, nm), tacc);
            lse.s += acc;
            if (ENT) lse.t += tacc;
          }
        }
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) {
          if (u < cnt) {
            const int e = 4 * (full_end + tid + u * kScanThreads);
            top.push(x[u].x, e);
            top.push(x[u].y, e + 1);
            top.push(x[u].z, e + 2);
            top.push(x[u].w, e + 3);
          }
        }
      }
    }
  }
}

// Short segments: at most kResident float4s per thread, every load issued
// at once (one round trip to memory) and the elements kept in registers.
// The log-sum-exp runs over them as in scan_batch; the warp's top K is then
// taken by K rounds of warp argmax over each lane's best remaining element,
// the round's winner blanking that element (NaN, which is outside the input
// contract and which fmaxf ignores) and rescanning its per-float4 maxima.
// No per-element insertion (whose lane divergence dominated short scans).
constexpr int kResident = 12;

template <int K, bool LSE, bool ENT, class Xf>
__device__ __forceinline__ void scan_resident(const float* __restrict__ row, int lo4, int hi4,
                                              float (&wv)[K], int (&wi)[K], Lse& lse,
                                              const Xf& xf) {
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const float4* r4 = reinterpret_cast<const float4*>(row);
  const int tid = (int)threadIdx.x;
  const float nan = __int_as_float(0x7fffffff);
  float4 x[kResident];
#pragma unroll
  for (int u = 0; u < kResident; ++u) {
    const int j = lo4 + tid + u * kScanThreads;
    x[u] = j < hi4 ? ld_stream(r4 + j) : make_float4(nan, nan, nan, nan);
  }
#pragma unroll
  for (int u = 0; u < kResident; ++u) {
    const int j = lo4 + tid + u * kScanThreads;
    if (j < hi4) x[u] = xf(x[u], j);
  }
  float sm[kResident];   // slot maxima; NaN for padding (and, later, emptied slots)
#pragma unroll
  for (int u = 0; u < kResident; ++u) sm[u] = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
  if (LSE) {
    float bm = -INFINITY;
#pragma unroll
    for (int u = 0; u < kResident; ++u) bm = fmaxf(bm, sm[u]);
    const float bm2 = bm * kLog2e;
    if (bm2 > lse.m) lse.raise<ENT>(bm2);
    if (lse.m != -INFINITY) {
      const float nm = -lse.m;
      float a0 = 0.0f, a1 = 0.0f, t0 = 0.0f, t1 = 0.0f;
#pragma unroll
      for (int u = 0; u < kResident; ++u) {
        if (lo4 + tid + u * kScanThreads < hi4) {
          a0 += lse.term<ENT>(fmaf(x[u].x, kLog2e, nm), t0) +
                lse.term<ENT>(fmaf(x[u].y, kLog2e, nm), t1);
          a1 += lse.term<ENT>(fmaf(x[u].z, kLog2e, nm), t0) +
                lse.term<ENT>(fmaf(x[u].w, kLog2e, nm), t1);
        }
      }
      lse.s += a0 + a1;
      if (ENT) lse.t += t0 + t1;
    }
  }
  // The lane's best remaining element: the first slot with the highest
  // maximum (slots rise with the element index), then its first element
  // equal to that maximum. bu < 0: nothing left.
  int bu = -1;
  float bmx = 0.0f;
  auto find_best = [&]() {
    bu = -1;
#pragma unroll
    for (int u = 0; u < kResident; ++u)
      if (sm[u] == sm[u] && (bu < 0 || sm[u] > bmx)) { bmx = sm[u]; bu = u; }
  };
  find_best();
#pragma unroll
  for (int k = 0; k < K; ++k) {
    int idx = INT_MAX, c = 0;
    if (bu >= 0) {
      float4 q = x[0];
#pragma unroll
      for (int u = 1; u < kResident; ++u)
        if (u == bu) q = x[u];
      c = q.x == bmx ? 0 : q.y == bmx ? 1 : q.z == bmx ? 2 : 3;
      idx = 4 * (lo4 + tid + bu * kScanThreads) + c;
    }
    const uint32_t key = bu >= 0 ? order_key(bmx) : 0u;
    const uint32_t top = __reduce_max_sync(kFull, key);
    const uint32_t win = __reduce_min_sync(kFull, (bu >= 0 && key == top) ? (uint32_t)idx : 0xFFFFFFFFu);
    wv[k] = top == 0 ? -INFINITY : key_value(top);
    wi[k] = top == 0 ? INT_MAX : (int)win;
    if (k + 1 < K && bu >= 0 && (uint32_t)idx == win) {
#pragma unroll
      for (int u = 0; u < kResident; ++u) {
        if (u == bu) {
          if (c == 0) x[u].x = nan;
          else if (c == 1) x[u].y = nan;
          else if (c == 2) x[u].z = nan;
          else x[u].w = nan;
          sm[u] = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
        }
      }
      find_best();
    }
  }
}

// Reduces the warps' sorted top-K lists (identical in every lane of a warp)
// and the threads' log-sum-exp states into `out` (valid after the trailing
// __syncthreads).
template <int K, bool LSE>
__device__ __forceinline__ void block_reduce_lists(const float (&wv)[K], const int (&wi)[K],
                                                   Lse& lse, ScanPartial<K>* out,
                                                   ScanPartial<K>* warp_parts) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (LSE) lse.warp_reduce();
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < K; ++k) { warp_parts[warp].v[k] = wv[k]; warp_parts[warp].i[k] = wi[k]; }
    warp_parts[warp].m = lse.m;
    warp_parts[warp].s = lse.s;
    warp_parts[warp].t = lse.t;
  }
  __syncthreads();
  if (warp == 0) {
    // kScanWarps lists of K: lane l takes list l (the lists are sorted).
    float cv[K];
    int ci[K];
    Lse l;
    int len = 0;
    if (lane < kScanWarps) {
#pragma unroll
      for (int k = 0; k < K; ++k) { cv[k] = warp_parts[lane].v[k]; ci[k] = warp_parts[lane].i[k]; }
      len = K;
      l.m = warp_parts[lane].m;
      l.s = warp_parts[lane].s;
      l.t = warp_parts[lane].t;
    } else {
#pragma unroll
      for (int k = 0; k < K; ++k) { cv[k] = -INFINITY; ci[k] = INT_MAX; }
      l.init();
    }
    // Short lists (fewer than K real elements) end in sentinels: count the rest.
    len = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) len += (ci[k] != INT_MAX);
    float bv[K];
    int bi[K];
    warp_select<K, K>(cv, ci, len, bv, bi);
    if (LSE) l.warp_reduce();
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < K; ++k) { out->v[k] = bv[k]; out->i[k] = bi[k]; }
      out->m = l.m;
      out->s = l.s;
      out->t = l.t;
    }
  }
  __syncthreads();
}

// Reduces the CTA's per-thread state into `out` (valid after the trailing
// __syncthreads).
template <int K, bool LSE>
__device__ __forceinline__ void block_reduce(TopK<K>& top, Lse& lse, ScanPartial<K>* out,
                                             ScanPartial<K>* warp_parts) {
  float wv[K];
  int wi[K];
  warp_select<K, K>(top.v, top.i, min(top.n, K), wv, wi);
  block_reduce_lists<K, LSE>(wv, wi, lse, out, warp_parts);
}

// Whether segments of seg4 float4s take the register-resident scan (a
// separate kernel instance, so that the streaming one keeps its registers).
inline bool use_resident(int K, int seg4) { return K <= 8 && seg4 <= kResident * kScanThreads; }

// A CTA's scan of [lo4, hi4) of a row into `part`: the register-resident
// scan (RES, segments of at most kResident float4s per thread) or the
// streaming scan.
template <int K, bool LSE, bool ENT, bool RES, class Xf = IdentityXf, bool EARLY_TAIL = false>
__device__ __forceinline__ void scan_to_partial(const float* __restrict__ row, int lo4, int hi4,
                                                ScanPartial<K>* part, ScanPartial<K>* warp_parts,
                                                const Xf& xf = Xf()) {
  Lse lse;
  lse.init();
  if (RES) {
    float wv[K];
    int wi[K];
    scan_resident<K, LSE, ENT>(row, lo4, hi4, wv, wi, lse, xf);
    block_reduce_lists<K, LSE>(wv, wi, lse, part, warp_parts);
  } else {
    TopK<K> top;
    top.init();
    scan_segment<K, LSE, ENT, Xf, EARLY_TAIL>(row, lo4, hi4, top, lse, xf);
    block_reduce<K, LSE>(top, lse, part, warp_parts);
  }
}

// Merges the cluster's partials in CTA rank 0 (warp 0). Returns true in the
// thread that holds the final result (lane 0 of warp 0 of rank 0), with the
// list in top.v/top.i and the log-sum-exp state in lse.
template <int K, bool LSE>
__device__ __forceinline__ bool cluster_reduce(ScanPartial<K>* mine, int S, TopK<K>& top,
                                               Lse& lse) {
  if (S == 1) {
    if (threadIdx.x != 0) return false;
#pragma unroll
    for (int k = 0; k < K; ++k) { top.v[k] = mine->v[k]; top.i[k] = mine->i[k]; }
    lse.m = mine->m;
    lse.s = mine->s;
    lse.t = mine->t;
    return true;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();  // every CTA's partial is in its shared memory
  bool holder = false;
  if (cluster.block_rank() == 0 && threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float cv[K];
    int ci[K];
    int len = 0;
    if (lane < S) {
      const ScanPartial<K>* p = cluster.map_shared_rank(mine, lane);
#pragma unroll
      for (int k = 0; k < K; ++k) { cv[k] = p->v[k]; ci[k] = p->i[k]; }
      len = K;
      lse.m = p->m;
      lse.s = p->s;
      lse.t = p->t;
    } else {
#pragma unroll
      for (int k = 0; k < K; ++k) { cv[k] = -INFINITY; ci[k] = INT_MAX; }
      lse.init();
    }
    len = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) len += (ci[k] != INT_MAX);
    warp_select<K, K>(cv, ci, len, top.v, top.i);
    if (LSE) lse.warp_reduce();
    holder = (lane == 0);
  }
  // Keep every CTA's shared memory alive until rank 0 has read it. Rank 0
  // has consumed every value it loaded before it arrives, so the barrier
  // needs no memory ordering: a relaxed arrive skips the release fence.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  return holder;
}

// Few long rows (fewer than two waves of 16-CTA clusters, rows of at least
// 64K elements) are cut into kFlatParts segments with no cluster: each CTA's
// segment is then at most one full batch plus a tail, all loaded in one
// round trip, and its partial goes to global scratch for a later merge.
constexpr int kFlatParts = 32;

inline bool use_flat_rows(long rows, int V, int num_sms) {
  return rows * 16 < 2L * num_sms && V / 4 >= 16 * 1024;
}

// Picks the cluster size (segments per row) for `rows` rows of `v4` float4s:
// enough CTAs to cover the SMs twice, segments of >= 2048 float4s.
inline int pick_row_split(long rows, int v4, int num_sms, int max_split) {
  int s = 1;
  while (s < max_split && rows * s < 2L * num_sms && (v4 / (2 * s)) >= 2048) s *= 2;
  return s;
}

template <typename Kernel, typename... Args>
cudaError_t launch_clustered(Kernel kernel, int grid, int cluster, cudaStream_t stream,
                             Args... args) {
  return launch_kernel(kernel, dim3(grid), dim3(kScanThreads), 0, stream, cluster, args...);
}

}  // namespace jt
