// Full-vocabulary row scans: top-K (value desc, index asc) and the
// log-sum-exp of a row of fp32 logits, streamed once from HBM.
//
// Work layout: a row of V floats is cut into S segments (S = the cluster
// size, 1..16); each CTA of a thread-block cluster streams one segment with
// 128-bit non-allocating loads: short segments all at once into registers,
// long ones two batches of float4s per thread in flight (in registers, or
// more through a per-thread shared-memory ring filled by cp.async).
// Long segments keep one sorted top-K list per warp (entry k in lane k): a
// batch costs one vote unless some float4's maximum can beat the list's K-th
// entry, and an insertion is a warp-uniform ballot and one-lane shift.
// Every thread keeps an online log-sum-exp in the log2 domain (optionally
// with the sum that gives the distribution's entropy).
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

  __device__ __forceinline__ void init() {
#pragma unroll
    for (int k = 0; k < K; ++k) { v[k] = -INFINITY; i[k] = INT_MAX; }
    n = 0;
    thr = __int_as_float(0x7fffffff);
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

// The warp's best K elements so far for the streaming scans, one list per
// warp: entry k (k-th by rank) in lane k, lanes >= K unused; (tv, ti) is
// entry K-1 in every lane, the sentinel (-inf, INT_MAX) until K elements
// have entered. A float4 is offered to the list only when it can hold an
// element ranking before entry K-1, so after the first batches almost every
// batch costs one vote; an insertion is warp-uniform (a ballot and a shift
// by one lane), never a divergent per-lane sort.
template <int K>
struct WarpTopK {
  static_assert(K >= 1 && K <= 32, "one entry per lane");
  float v, tv;
  int i, ti;

  __device__ __forceinline__ void init() {
    v = -INFINITY; i = INT_MAX;
    tv = -INFINITY; ti = INT_MAX;
  }

  // Inserts (x, e); every lane passes the same pair.
  __device__ __forceinline__ void insert(float x, int e) {
    constexpr unsigned kFull = 0xFFFFFFFFu;
    const int lane = threadIdx.x & 31;
    // The entries are sorted, so the ones (x, e) ranks before are a suffix.
    const uint32_t bm = __ballot_sync(kFull, lane < K && ranks_before(x, e, v, i));
    if (bm == 0) return;
    const int pos = __ffs(bm) - 1;
    const float pv = __shfl_up_sync(kFull, v, 1);
    const int pi = __shfl_up_sync(kFull, i, 1);
    if (lane == pos) {
      v = x; i = e;
    } else if (lane > pos && lane < K) {
      v = pv; i = pi;
    }
    tv = __shfl_sync(kFull, v, K - 1);
    ti = __shfl_sync(kFull, i, K - 1);
  }

  // The K-th largest of the warp's valid float4 maxima (-inf if there are
  // fewer than K): K float4s each hold an element at least that large, so
  // no element below it can end in the warp's top K.
  __device__ __forceinline__ static float kth_max(const float (&mx)[kScanBatch], uint32_t valid) {
    constexpr unsigned kFull = 0xFFFFFFFFu;
    static_assert(kScanBatch == 4, "sorting network for four values");
    float s0 = (valid & 1u) ? mx[0] : -INFINITY, s1 = (valid & 2u) ? mx[1] : -INFINITY;
    float s2 = (valid & 4u) ? mx[2] : -INFINITY, s3 = (valid & 8u) ? mx[3] : -INFINITY;
    float t;
    t = fmaxf(s0, s1); s1 = fminf(s0, s1); s0 = t;
    t = fmaxf(s2, s3); s3 = fminf(s2, s3); s2 = t;
    t = fmaxf(s0, s2); s2 = fminf(s0, s2); s0 = t;
    t = fmaxf(s1, s3); s3 = fminf(s1, s3); s1 = t;
    t = fmaxf(s1, s2); s2 = fminf(s1, s2); s1 = t;
    const int n = __popc(valid);
    int h = 0;
    uint32_t top = 0;
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const float hv = h == 0 ? s0 : h == 1 ? s1 : h == 2 ? s2 : s3;
      const uint32_t key = h < n ? order_key(hv) : 0u;
      top = __reduce_max_sync(kFull, key);
      if (top == 0u) return -INFINITY;
      const uint32_t win = __ballot_sync(kFull, key == top);
      if ((threadIdx.x & 31) == __ffs(win) - 1) ++h;
    }
    return key_value(top);
  }

  // Offers the valid float4s of one batch (float4 u of this lane has index
  // j0 + u*T, its maximum mx[u]).
  __device__ __forceinline__ void offer(const float4 (&x)[kScanBatch], const float (&mx)[kScanBatch],
                                        uint32_t valid, int j0) {
    constexpr unsigned kFull = 0xFFFFFFFFu;
    const int lane = threadIdx.x & 31;
    const float bound = ti == INT_MAX ? kth_max(mx, valid) : tv;
    float bm = -INFINITY;
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u)
      if ((valid >> u) & 1u) bm = fmaxf(bm, mx[u]);
    // One vote per batch while no lane's batch maximum reaches the bound.
    if (!__any_sync(kFull, (valid != 0u) && bm >= bound)) return;
    // Float4s that can hold an element ranking before entry K-1: a larger
    // maximum, or an equal one whose first index is lower.
    uint32_t m = 0;
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u)
      m |= (uint32_t)(((valid >> u) & 1u) && mx[u] >= bound &&
                      (mx[u] > tv || 4 * (j0 + u * kScanThreads) < ti)) << u;
    for (;;) {
      const uint32_t lanes = __ballot_sync(kFull, m != 0);
      if (lanes == 0) break;
      const int src = __ffs(lanes) - 1;
      const int u = __shfl_sync(kFull, __ffs(m) - 1, src);
      float4 q = x[0];
#pragma unroll
      for (int w = 1; w < kScanBatch; ++w)
        if (w == u) q = x[w];
      const float qv[4] = {__shfl_sync(kFull, q.x, src), __shfl_sync(kFull, q.y, src),
                           __shfl_sync(kFull, q.z, src), __shfl_sync(kFull, q.w, src)};
      const int e = 4 * (__shfl_sync(kFull, j0, src) + u * kScanThreads);
#pragma unroll
      for (int c = 0; c < 4; ++c)   // warp-uniform test: most elements of the float4 fail it
        if (qv[c] > tv || (qv[c] == tv && e + c < ti)) insert(qv[c], e + c);
      if (lane == src) m &= m - 1;
    }
  }
};

// Adds the valid float4s of a batch (bits of `valid`; all of them when
// valid == 0xF) to the thread's log-sum-exp.
template <bool ENT>
__device__ __forceinline__ void lse_batch(const float4 (&x)[kScanBatch], const float (&mx)[kScanBatch],
                                          uint32_t valid, Lse& lse) {
  float bm = -INFINITY;
#pragma unroll
  for (int u = 0; u < kScanBatch; ++u)
    if ((valid >> u) & 1u) bm = fmaxf(bm, mx[u]);
  const float bm2 = bm * kLog2e;
  if (bm2 > lse.m) lse.raise<ENT>(bm2);
  if (lse.m != -INFINITY) {
    const float nm = -lse.m;
    float a0 = 0.0f, a1 = 0.0f, t0 = 0.0f, t1 = 0.0f;
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) {
      if ((valid >> u) & 1u) {
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

// One full batch of kScanBatch float4s (float4 j0 + u*T for u < kScanBatch);
// warp-collective.
template <int K, bool LSE, bool ENT>
__device__ __forceinline__ void scan_batch(const float4 (&x)[kScanBatch], int j0, WarpTopK<K>& top,
                                           Lse& lse) {
  float mx[kScanBatch];
#pragma unroll
  for (int u = 0; u < kScanBatch; ++u)
    mx[u] = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
  if (LSE) lse_batch<ENT>(x, mx, 0xFu, lse);
  top.offer(x, mx, 0xFu, j0);
}

// The last, partial batch of a segment: float4s full_end + tid + u*T below
// hi4 hold data, the rest is padding that neither enters the list nor the
// sums. Warp-collective: every lane calls it, lanes with padding only too.
template <int K, bool LSE, bool ENT>
__device__ __forceinline__ void scan_tail(const float4 (&x)[kScanBatch], int full_end, int hi4,
                                          WarpTopK<K>& top, Lse& lse) {
  const int tid = (int)threadIdx.x;
  uint32_t valid = 0;
  float mx[kScanBatch];
#pragma unroll
  for (int u = 0; u < kScanBatch; ++u) {
    const bool ok = full_end + tid + u * kScanThreads < hi4;
    valid |= (uint32_t)ok << u;
    mx[u] = ok ? fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w)) : -INFINITY;
  }
  if (LSE) lse_batch<ENT>(x, mx, valid, lse);
  top.offer(x, mx, valid, full_end + tid);
}

// Streams float4s [lo4, hi4) of `row` into the warp lists and the threads'
// sums: full batches without bounds checks, ping-ponging two register
// buffers so that one batch is in flight while the other is processed, then
// a checked tail. Every lane of a warp runs the same batches (the warp-wide
// list needs the whole warp).
// EARLY_TAIL: a segment of at most two full batches issues its tail's loads
// together with them (one round trip to memory instead of two); measured to
// pay off for the plain argmax only, the log-sum-exp and keyed scans lose.
template <int K, bool LSE, bool ENT = false, class Xf = IdentityXf, bool EARLY_TAIL = false>
__device__ __forceinline__ void scan_segment(const float* __restrict__ row, int lo4, int hi4,
                                             WarpTopK<K>& top, Lse& lse, const Xf& xf = Xf()) {
  const float4* r4 = reinterpret_cast<const float4*>(row);
  constexpr int STEP = kScanThreads * kScanBatch;
  const int tid = (int)threadIdx.x;
  const int full_end = lo4 + ((hi4 - lo4) / STEP) * STEP;
  float4 a[kScanBatch], b[kScanBatch];
  int base = lo4;
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
    scan_batch<K, LSE, ENT>(a, base + tid, top, lse);
    base += STEP;
    if (!nb) break;
    const bool na = base + STEP < full_end;
    if (na) {
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) a[u] = ld_stream(r4 + base + STEP + tid + u * kScanThreads);
    }
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) b[u] = xf(b[u], base + tid + u * kScanThreads);
    scan_batch<K, LSE, ENT>(b, base + tid, top, lse);
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
    scan_tail<K, LSE, ENT>(a, full_end, hi4, top, lse);
  }
}

// 16-byte asynchronous copy global -> shared that bypasses L1 (cp.async.cg);
// its completion is tracked per thread by commit groups.
__device__ __forceinline__ void cp_async16(float4* dst, const float4* src) {
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's commit groups are still pending.
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Dynamic shared memory of the ring scan: NST stages of one batch.
template <int NST>
constexpr size_t ring_smem_bytes() {
  return (size_t)NST * kScanBatch * kScanThreads * sizeof(float4);
}

// scan_segment with the batches staged in shared memory instead of
// registers: every thread copies its own float4s of batch c into stage
// c mod NST with cp.async and reads them back once the copy has landed, so
// NST batches (NST x 16 KB per CTA) are in flight without holding registers.
// No thread reads another's data, so the only synchronisation is the
// thread's own cp.async.wait_group. The tail (the last, partial batch) goes
// through the ring as well. `ring` holds NST * kScanBatch * kScanThreads
// float4s.
template <int K, bool LSE, bool ENT, int NST>
__device__ __forceinline__ void scan_segment_ring(const float* __restrict__ row, int lo4, int hi4,
                                                  WarpTopK<K>& top, Lse& lse, float4* ring) {
  static_assert(NST >= 2, "the ring needs two stages at least");
  const float4* r4 = reinterpret_cast<const float4*>(row);
  constexpr int STEP = kScanThreads * kScanBatch;
  const int tid = (int)threadIdx.x;
  const int nfull = (hi4 - lo4) / STEP;
  const int full_end = lo4 + nfull * STEP;
  const int nb = nfull + (full_end < hi4 ? 1 : 0);
  float4* mine = ring + tid;
  // Batch c -> stage c mod NST; the thread's float4 u of a stage sits at
  // (stage * kScanBatch + u) * kScanThreads (consecutive threads, consecutive
  // 16-byte words: no bank conflicts).
  auto issue = [&](int c, int stage) {
    if (c < nb) {
      const int j0 = lo4 + c * STEP + tid;
#pragma unroll
      for (int u = 0; u < kScanBatch; ++u) {
        const int j = j0 + u * kScanThreads;
        if (c < nfull || j < hi4) cp_async16(mine + (stage * kScanBatch + u) * kScanThreads, r4 + j);
      }
    }
    cp_async_commit();   // an empty group past the end keeps the count uniform
  };
#pragma unroll
  for (int c = 0; c < NST - 1; ++c) issue(c, c);
  int stage = 0, fill = NST - 1;
  for (int c = 0; c < nfull; ++c) {
    // Stage `fill` held batch c - 1, which this thread has consumed.
    issue(c + NST - 1, fill);
    fill = fill + 1 == NST ? 0 : fill + 1;
    cp_async_wait<NST - 1>();   // batch c has landed
    float4 x[kScanBatch];
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) x[u] = mine[(stage * kScanBatch + u) * kScanThreads];
    stage = stage + 1 == NST ? 0 : stage + 1;
    scan_batch<K, LSE, ENT>(x, lo4 + c * STEP + tid, top, lse);
  }
  cp_async_wait<0>();
  if (full_end < hi4) {
    float4 x[kScanBatch];
#pragma unroll
    for (int u = 0; u < kScanBatch; ++u) {
      const int j = full_end + tid + u * kScanThreads;
      x[u] = j < hi4 ? mine[(stage * kScanBatch + u) * kScanThreads]
                     : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    }
    scan_tail<K, LSE, ENT>(x, full_end, hi4, top, lse);
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

// Reduces the warps' lists and the threads' sums into `out` (valid after
// the trailing __syncthreads).
template <int K, bool LSE>
__device__ __forceinline__ void block_reduce(const WarpTopK<K>& top, Lse& lse,
                                             ScanPartial<K>* out, ScanPartial<K>* warp_parts) {
  float wv[K];
  int wi[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    wv[k] = __shfl_sync(0xFFFFFFFFu, top.v, k);
    wi[k] = __shfl_sync(0xFFFFFFFFu, top.i, k);
  }
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
    WarpTopK<K> top;
    top.init();
    scan_segment<K, LSE, ENT, Xf, EARLY_TAIL>(row, lo4, hi4, top, lse, xf);
    block_reduce<K, LSE>(top, lse, part, warp_parts);
  }
}

// The streaming scan of [lo4, hi4) through a shared-memory ring (NST
// stages at `ring`) into `part`.
template <int K, bool LSE, bool ENT, int NST>
__device__ __forceinline__ void scan_to_partial_ring(const float* __restrict__ row, int lo4,
                                                     int hi4, ScanPartial<K>* part,
                                                     ScanPartial<K>* warp_parts, float4* ring) {
  Lse lse;
  lse.init();
  WarpTopK<K> top;
  top.init();
  scan_segment_ring<K, LSE, ENT, NST>(row, lo4, hi4, top, lse, ring);
  block_reduce<K, LSE>(top, lse, part, warp_parts);
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
