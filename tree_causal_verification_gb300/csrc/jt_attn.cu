// jt_tree_attn: tree-causal GQA attention for the verification pass.
//
// Node v of sequence b, query head h (KV head h / g) attends to the prefix
// KV and to the tree nodes u with M[v,u] = 0, i.e. its ancestors and itself
// (JetSpec summary on paperlayer.ai, §2 "Architecture" and App. E
// "Verification"; JetSpec review on startedourmission.github.io, "How it
// works", mask equation). The mask arrives as ancestor bitmasks and is
// applied in registers; no dense mask exists anywhere.
//
// Kernel design (sm_100 family, tcgen05 + TMA)
// --------------------------------------------
// Rows are node-major, row = v*g + j: 128/g consecutive tree nodes times the
// g query heads sharing KV head kh make one 128-row M tile, so every K/V
// tile streamed from HBM serves all of them (GQA folded into MMA M).
// Work unit = (sequence b, KV head kh, pair of M tiles A and B = 256 rows).
// The unit's keys are the prefix tiles (128 keys; paged through 16-token
// pages or contiguous) then the tree tiles holding its nodes' ancestors.
//
// One CTA per unit (or per slice of its key tiles when units are too few to
// fill the GPU: split-KV over a cluster of S = 2..8 CTAs, whose fp32
// partials meet in an L2-resident workspace across one cluster barrier). 384 threads = 3 warpgroups; setmaxnreg moves registers
// from the third (producer / MMA, 104 each) to the two softmax warpgroups
// (200 each) for the main loop; 384 x 168 = 256 x 200 + 128 x 104:
//   warps 0-3  softmax of tile A, warps 4-7 softmax of tile B: thread r of a
//              warpgroup owns TMEM lane r (= query row). It loads the row's
//              128 scores of S from TMEM once, applies the prefix bound /
//              ancestor bits / scale in registers, takes the row max, forms
//              P = 2^(s - m) and writes it back over S in TMEM as packed bf16.
//              O is rescaled in TMEM only when a row max grows by more than
//              2^8 (lazy rescaling; the final 1/l uses the same stale max);
//   warp 8     TMA producer of Q_A, Q_B (once) and of K tiles into a 2-slot ring;
//   warp 10    TMA producer of V tiles into a second 2-slot ring. A K slot is
//              released as soon as both tiles' S MMAs have read it, a V slot
//              after both P V MMAs, so K tile j+2 streams in while tile j+1
//              is still being processed;
//   warp 11    idle (completes the third warpgroup);
//   warp 9     TMEM owner and MMA issuer, per K/V tile j:
//              PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), where
//              S_X = Q_X K^T (M=128, N=128, K=D, operands in shared memory)
//              O_X += P_X V  (M=128, N=D, K=128 keys; P from TMEM, V from
//                             shared memory, MN-major)
//              so one tile's softmax overlaps the other tile's MMAs. Tensor
//              ops retire in issue order, so the commit after S_X(j+1) also
//              certifies that PV_X(j) has finished with P_X / O_X. The whole
//              warp runs the loop and elect.sync inside each MMA / commit
//              picks the issuing lane: issued from a lane-0 branch instead,
//              the MMAs fell behind the tensor pipe once the softmax warps
//              shared the warp's scheduler;
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,256+D),
// O_B [256+D', ...) with D' = 128 for D = 128 (384..511).
// Key-split instance (KSPLIT, chosen when the budget fits one M tile): tile
// B has no live node, so warpgroup G (0 or 1) takes the key tiles G, G+2, ...
// of tile A's rows into the S_G / O_G columns, the MMA order per key tile t
// being PV_G(t), S_G(t+2); the two (m, l, O) states merge in the epilogue.
// In the softmax the exponent argument and the row sum run two columns per
// packed fp32x2 instruction and the row max uses the three-input max: the
// softmax warps are bound by instruction issue, not by the exponential unit.
// Every mbarrier wait is bounded; on expiry the CTA raises JT_DEVERR_TIMEOUT,
// waits (bounded again) for the TMA loads it issued and for its outstanding
// MMAs, frees TMEM and finishes.
#include <cooperative_groups.h>
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "jt_internal.cuh"
#include "jt_sm100.cuh"
#include "jt_tmamap.h"

namespace jt {
namespace {

namespace cg = cooperative_groups;
using namespace sm100;

constexpr int kThreads = 384;
constexpr uint32_t kRegsSoftmax = 200, kRegsOther = 104, kRegsLaunch = 168;
static_assert(256 * kRegsSoftmax + 128 * kRegsOther == 384 * kRegsLaunch,
              "the setmaxnreg split must use exactly the launch allocation");
constexpr int kWarpTMA = 8, kWarpMMA = 9, kWarpTMAV = 10;
constexpr int kTile = 128;                 // query rows per M tile = keys per K/V tile
constexpr int kStages = 2;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr int kPrefetchPages = 3;          // block-table entries per thread loaded with the sequence sizes

struct AttnParams {
  int batch, B, hq, hkv, g, npt, n_mpairs, S;
  // Balanced schedule (kernel template flag BAL): block i runs work item
  // perm[i] = unit * S + chunk (items sorted by length, longest first, -1
  // past the last); a unit of t tiles is cut into min(S, ceil(t /
  // chunk_tiles)) chunks (nparts[unit], written by its chunk 0) whose
  // partials attn_merge_kernel combines after the grid. Otherwise unit =
  // blockIdx / S and the S CTAs of a cluster split its key tiles.
  int units, chunk_tiles;
  int32_t* perm;
  int32_t* nparts;
  int paged, max_pages, n_pages, Lbound, words;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* n_nodes;
  const uint32_t* mask;
  __nv_bfloat16* out;
  float* part;        // split-KV partials, kPartFloats per CTA (S > 1 only)
  float scale_log2;
  long long wait_budget;   // cycles per bounded wait (kDefaultWaitBudget unless a test shortens it)
  int32_t* d_err;
};

// Split-KV partial of one CTA in the workspace: O as [D/4][256] float4s,
// then m[256] and l[256]. Rows are stored rank-contiguous: row R of the unit
// at slot (R % S) * (256 / S) + R / S, so that the rows rank k finishes
// (k, k + S, k + 2S, ...) are one contiguous run in every rank's partial.
template <int D>
__host__ __device__ constexpr int part_floats() { return 2 * kTile * D + 4 * kTile; }

struct Bars {
  uint64_t q_full, k_full[kStages], k_empty[kStages], v_full[kStages], v_empty[kStages];
  uint64_t s_full[2], p_full[2], pv_done[2], drain;
  uint32_t tmem_base;
  int abort;
  int unit, rank, split;   // this CTA's work, reloaded by the epilogue
};

// The epilogue reloads the CTA's coordinates from shared memory instead of
// keeping them live in registers through the main loop.
__device__ __forceinline__ int ld_shared_volatile(const int* p) {
  return *reinterpret_cast<const volatile int*>(p);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 two = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&two);
}

// Split-KV merge of one unit by rank `rank` of its SS CTAs: rows
// rank, rank + SS, rank + 2 SS, ... of the unit's 256 (live rows come first
// in a unit, so the round-robin share spreads them evenly). Row R's result
// is sum_s e^(m_s - M) O_s / sum_s e^(m_s - M) l_s over the SS partials,
// M = max_s m_s (m in the log2 domain). Every partial load bypasses L1 and U
// items are kept in flight per thread; rows of unused slots are zeros.
template <int D, int SS, int U>
__device__ __forceinline__ void merge_split(const AttnParams& p, const float* part0, float* fac,
                                            int rank, int n_live, int v0, int b, int kh, int tid) {
  constexpr int RR = 2 * kTile / SS;
  constexpr int PF4 = part_floats<D>() / 4;
  const int g = p.g;
  const int nl = n_live > rank ? (n_live - rank + SS - 1) / SS : 0;   // live rows of this rank
  if (tid < nl) {
    const float* ml = part0 + 2 * kTile * D + rank * RR + tid;
    float ms[SS], ls[SS];
#pragma unroll
    for (int s2 = 0; s2 < SS; ++s2) {
      ms[s2] = __ldcg(ml + (size_t)s2 * part_floats<D>());
      ls[s2] = __ldcg(ml + (size_t)s2 * part_floats<D>() + 2 * kTile);
    }
    float M = -INFINITY;
#pragma unroll
    for (int s2 = 0; s2 < SS; ++s2) M = fmaxf(M, ms[s2]);
    float lsum = 0.0f, f[SS];
#pragma unroll
    for (int s2 = 0; s2 < SS; ++s2) {
      f[s2] = (ms[s2] == -INFINITY) ? 0.0f : ex2(ms[s2] - M);
      lsum += f[s2] * ls[s2];
    }
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
#pragma unroll
    for (int s2 = 0; s2 < SS; ++s2) fac[tid * SS + s2] = f[s2] * inv;
  }
  __syncthreads();
  // Live rows: item i = (row rl = i % nl, float4 column c4 = i / nl); a warp
  // reads runs of nl consecutive slots of each partial.
  const float4* src0 = reinterpret_cast<const float4*>(part0) + rank * RR;
  const int items = nl * (D / 4);
  for (int i0 = tid; i0 < items; i0 += U * kThreads) {
    float4 x[U][SS];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kThreads;
      if (i < items) {
        const float4* src = src0 + (i / nl) * (2 * kTile) + i % nl;
#pragma unroll
        for (int s2 = 0; s2 < SS; ++s2) x[u][s2] = __ldcg(src + (size_t)s2 * PF4);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kThreads;
      if (i < items) {
        const int rl = i % nl, c4 = i / nl;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int s2 = 0; s2 < SS; ++s2) {
          const float f = fac[rl * SS + s2];
          acc.x += f * x[u][s2].x; acc.y += f * x[u][s2].y;
          acc.z += f * x[u][s2].z; acc.w += f * x[u][s2].w;
        }
        const int row = rank + SS * rl;
        const int vv = v0 + row / g, jh = row % g;
        reinterpret_cast<uint2*>(p.out + (((size_t)b * p.B + vv) * p.hq + kh * g + jh) * D)[c4] =
            make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
      }
    }
  }
  // Rows of unused budget slots of this rank (node < B): zeros.
  for (int i = tid; i < (RR - nl) * (D / 8); i += kThreads) {
    const int row = rank + SS * (nl + i / (D / 8));
    const int vv = v0 + row / g, jh = row % g;
    if (vv < p.B)
      reinterpret_cast<uint4*>(p.out + (((size_t)b * p.B + vv) * p.hq + kh * g + jh) * D)[i % (D / 8)] =
          make_uint4(0, 0, 0, 0);
  }
}

// Balanced schedule, after the attention grid: combine the k = nparts[unit]
// (<= 8) chunk partials of every split unit with the same formula as
// merge_split; kMergeSlices CTAs per unit, each a slice of its 256 rows, so
// the merges of all units run side by side across the SMs. Partials are
// row-ordered (slot = row) and read past L1; every thread keeps UN items x
// KMAX loads in flight. Units with k < 2 wrote their output directly.
constexpr int kMergeThreads = 256;
constexpr int kMergeSlices = 4;
constexpr int kMergeRows = 2 * kTile / kMergeSlices;

template <int D, int UN, int KMAX>
__device__ __forceinline__ void merge_rows(const AttnParams& p, const float* part0, int k,
                                           int r0, int r1, int v0, int b, int kh,
                                           const float* fac, uint2* tile) {
  constexpr int PF4 = part_floats<D>() / 4;
  const int g = p.g, rows = r1 - r0, items = rows * (D / 4);
  const float4* src0 = reinterpret_cast<const float4*>(part0);
  for (int i0 = threadIdx.x; i0 < items; i0 += UN * kMergeThreads) {
    float4 x[UN][KMAX];
#pragma unroll
    for (int u = 0; u < UN; ++u) {
      const int i = i0 + u * kMergeThreads;
      if (i < items) {
        const int r = r0 + i % rows, c4 = i / rows;
#pragma unroll
        for (int s2 = 0; s2 < KMAX; ++s2)
          if (s2 < k) x[u][s2] = __ldcg(src0 + (size_t)s2 * PF4 + c4 * (2 * kTile) + r);
      }
    }
#pragma unroll
    for (int u = 0; u < UN; ++u) {
      const int i = i0 + u * kMergeThreads;
      if (i < items) {
        const int r = r0 + i % rows, c4 = i / rows;
        float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int s2 = 0; s2 < KMAX; ++s2) {
          if (s2 < k) {
            const float f = fac[(r - r0) * 8 + s2];
            acc.x += f * x[u][s2].x; acc.y += f * x[u][s2].y;
            acc.z += f * x[u][s2].z; acc.w += f * x[u][s2].w;
          }
        }
        tile[(r - r0) * (D / 4) + c4] = make_uint2(pack_bf16(acc.x, acc.y), pack_bf16(acc.z, acc.w));
      }
    }
  }
  // The partials are read row-contiguous; the output rows are written whole
  // (16-byte stores, consecutive threads along a row) from the staged tile.
  __syncthreads();
  for (int i = threadIdx.x; i < rows * (D / 8); i += kMergeThreads) {
    const int rr = i / (D / 8), q = i % (D / 8), r = r0 + rr;
    const int vv = v0 + r / g, jh = r % g;
    reinterpret_cast<uint4*>(p.out + (((size_t)b * p.B + vv) * p.hq + kh * g + jh) * D)[q] =
        reinterpret_cast<const uint4*>(tile + rr * (D / 4))[q];
  }
}

template <int D>
__global__ void __launch_bounds__(kMergeThreads) attn_merge_kernel(const AttnParams p) {
  __shared__ float fac[kMergeRows * 8];
  __shared__ uint2 tile[kMergeRows * (D / 4)];   // the slice's output rows, bf16
  constexpr int PF = part_floats<D>();
  grid_dependency_sync();
  const int unit = blockIdx.x / kMergeSlices, slice = blockIdx.x % kMergeSlices;
  const int k = p.nparts[unit];
  if (k < 2) return;   // no partials: the unit's output is already written
  const int mp = unit % p.n_mpairs, bk = unit / p.n_mpairs;
  const int kh = bk % p.hkv, b = bk / p.hkv;
  const int g = p.g, v0 = mp * 2 * p.npt;
  const int n = p.n_nodes[b];   // valid: a unit with partials passed the checks
  const int n_live = min(2 * kTile, (n - v0) * g);
  const int r0 = slice * kMergeRows, r1 = min(n_live, r0 + kMergeRows);
  const float* part0 = p.part + (size_t)unit * p.S * PF;
  for (int r = r0 + threadIdx.x; r < r1; r += kMergeThreads) {
    float ms[8], ls[8];
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2) {
      ms[s2] = s2 < k ? __ldcg(part0 + (size_t)s2 * PF + 2 * kTile * D + r) : -INFINITY;
      ls[s2] = s2 < k ? __ldcg(part0 + (size_t)s2 * PF + 2 * kTile * D + 2 * kTile + r) : 0.0f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2) M = fmaxf(M, ms[s2]);
    float lsum = 0.0f, f[8];
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2) {
      f[s2] = (ms[s2] == -INFINITY) ? 0.0f : ex2(ms[s2] - M);
      lsum += f[s2] * ls[s2];
    }
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
#pragma unroll
    for (int s2 = 0; s2 < 8; ++s2) fac[(r - r0) * 8 + s2] = f[s2] * inv;
  }
  __syncthreads();
  if (r1 > r0) {
    if (k <= 2) merge_rows<D, 4, 2>(p, part0, k, r0, r1, v0, b, kh, fac, tile);
    else if (k <= 4) merge_rows<D, 2, 4>(p, part0, k, r0, r1, v0, b, kh, fac, tile);
    else merge_rows<D, 1, 8>(p, part0, k, r0, r1, v0, b, kh, fac, tile);
  }
  // This slice's rows of unused budget slots (node < B): zeros.
  const int z0 = max(r0, n_live), z1 = r0 + kMergeRows;
  for (int i = threadIdx.x; i < max(0, z1 - z0) * (D / 8); i += kMergeThreads) {
    const int r = z0 + i / (D / 8);
    const int vv = v0 + r / g, jh = r % g;
    if (vv < p.B)
      reinterpret_cast<uint4*>(p.out + (((size_t)b * p.B + vv) * p.hq + kh * g + jh) * D)[i % (D / 8)] =
          make_uint4(0, 0, 0, 0);
  }
}

// Balanced schedule, before the attention grid: list the work items (unit,
// chunk) of every unit, chunk count min(S, ceil(t / chunk_tiles)) for a unit
// of t key tiles, ordered by chunk length, longest first, into
// perm[0 .. units*S), -1 past the last item; and zero the per-unit partial
// counts (a unit whose chunk 0 never runs is then left alone by the merge).
// The order is a counting sort on the length (one shared-memory atomic per
// item for its place within its length, a block-wide scan of the counts, a
// scatter): items of equal length may come in any order, which changes only
// the schedule, never a result. Beyond kPlanMaxSort slots the items stay
// unsorted. The counts only order the work: the attention kernel recomputes
// and validates everything itself (it can only find fewer chunks, never
// more, so every chunk it runs has an item).
constexpr int kPlanThreads = 1024;
constexpr int kPlanMaxSort = 8192;
constexpr int kPlanBuckets = 2 * kPlanThreads;   // lengths >= kPlanBuckets - 1 share the first

__global__ void __launch_bounds__(kPlanThreads) attn_plan_kernel(const AttnParams p) {
  extern __shared__ int plan_s[];   // [kPlanBuckets] counts, then [slots] (bucket << 16 | place)
  __shared__ int warp_tot[kPlanThreads / 32];
  grid_dependency_sync();
  const int units = p.units, S = p.S, slots = units * S, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  if (slots > kPlanMaxSort) {
    for (int i = tid; i < slots; i += kPlanThreads) p.perm[i] = i;
  } else {
    int* cnt = plan_s;
    int* rec = plan_s + kPlanBuckets;
    for (int i = tid; i < kPlanBuckets; i += kPlanThreads) cnt[i] = 0;
    __syncthreads();
    for (int i = tid; i < slots; i += kPlanThreads) {
      int r = -1;
      const int u = i / S, c = i % S;
      const int mp = u % p.n_mpairs, b = (u / p.n_mpairs) / p.hkv;
      const int n = p.n_nodes[b], L = p.prefix_len[b];
      int t = 0;
      if (n >= 0 && n <= p.B && L >= 0 && L <= p.Lbound) {
        const int v0 = mp * 2 * p.npt;
        if (v0 < n) t = (L + kTile - 1) / kTile + (min(v0 + 2 * p.npt, n) - 1 + kTile) / kTile;
      }
      const int k = min(S, max(1, (t + p.chunk_tiles - 1) / p.chunk_tiles));
      if (c < k) {
        const int len = (t + k - 1) / k;
        const int d = kPlanBuckets - 1 - min(len, kPlanBuckets - 1);   // longest first
        r = (d << 16) | atomicAdd(&cnt[d], 1);
      }
      rec[i] = r;
    }
    __syncthreads();
    // Exclusive scan of the counts: buckets 2 tid and 2 tid + 1 per thread.
    const int c0 = cnt[2 * tid], c1 = cnt[2 * tid + 1];
    int x = c0 + c1;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_tot[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
        if (lane >= o) w += y;
      }
      warp_tot[lane] = w;   // inclusive over warps
    }
    __syncthreads();
    const int excl = x - (c0 + c1) + (warp > 0 ? warp_tot[warp - 1] : 0);
    const int items = warp_tot[kPlanThreads / 32 - 1];
    __syncthreads();   // every count read before the offsets overwrite them
    cnt[2 * tid] = excl;
    cnt[2 * tid + 1] = excl + c0;
    __syncthreads();
    for (int i = tid; i < slots; i += kPlanThreads) {
      const int r = rec[i];
      if (r >= 0) p.perm[cnt[r >> 16] + (r & 0xFFFF)] = i;
    }
    for (int i = items + tid; i < slots; i += kPlanThreads) p.perm[i] = -1;
  }
  if (p.nparts)
    for (int i = tid; i < units; i += kPlanThreads) p.nparts[i] = 0;
}

template <int D, bool BAL, bool KSPLIT>
__global__ void __launch_bounds__(kThreads, 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mkc,
                    const __grid_constant__ CUtensorMap mvc, const __grid_constant__ CUtensorMap mkt,
                    const __grid_constant__ CUtensorMap mvt, const AttnParams p) {
  constexpr int CH = D / 64;               // 64-element (128-byte) chunks of the head dim
  constexpr int QB = kTile * D * 2;        // bytes of one Q, K or V tile
  constexpr int CHB = kTile * 128;         // bytes of one 64-column chunk of a tile
  constexpr int KS = 4 * CH;               // K=16 steps of Q K^T
  constexpr int OSTRIDE = D == 128 ? 128 : 64;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(sm + 2 * QB + kStages * 2 * QB);
  auto sQ = [&](int X) { return sm + X * QB; };
  auto sK = [&](int st) { return sm + 2 * QB + st * 2 * QB; };
  auto sV = [&](int st) { return sm + 3 * QB + st * 2 * QB; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.S;
  const int g = p.g, npt = p.npt;
  // Cluster schedule: unit and rank come from the block index (recomputed
  // wherever needed); balanced schedule (BAL): from the plan, after the wait.
  int rank = (int)(blockIdx.x % (unsigned)S);
  int unit = (int)(blockIdx.x / (unsigned)S);

  // ---- set-up (independent of the sequence's data, so it overlaps the
  // drain of the previous grid and the latency of the loads below):
  // barriers, TMEM ----
  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->k_full[i], 1);
      mbar_init(&bars->k_empty[i], 1);
      mbar_init(&bars->v_full[i], 1);
      mbar_init(&bars->v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->p_full[i], 4);
      mbar_init(&bars->pv_done[i], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (lane == 0 && warp == kWarpTMA) {   // the maps live in parameter space
    tma_prefetch_desc(&mq);
    tma_prefetch_desc(&mkc);
    tma_prefetch_desc(&mkt);
  } else if (lane == 0 && warp == kWarpTMAV) {
    tma_prefetch_desc(&mvc);
    tma_prefetch_desc(&mvt);
  }

  grid_dependency_sync();

  bool no_item = false;   // balanced schedule: a grid slot past the last item
  if (BAL) {
    const int item = p.perm[blockIdx.x];
    no_item = item < 0 || item >= p.units * S;
    unit = no_item ? 0 : item / S;
    rank = no_item ? 0 : item % S;
    if (tid == 0) {
      bars->unit = unit;
      bars->rank = rank;
    }
  }
  const int mp = unit % p.n_mpairs;
  const int bk = unit / p.n_mpairs;
  const int kh = bk % p.hkv, b = bk / p.hkv;
  const int v0 = mp * 2 * npt;

  // ---- validate the sequence (same verdict in every CTA of the sequence) ----
  // The first kPrefetchPages * kThreads block-table entries of the sequence
  // are loaded together with its node count and prefix length (they lie in
  // the sequence's row of the table whatever the length), so that the page
  // check costs no extra round trip; longer tables read the rest after.
  int pre[kPrefetchPages];
#pragma unroll
  for (int q = 0; q < kPrefetchPages; ++q) {
    const int i = tid + q * kThreads;
    pre[q] = (p.paged && !no_item && i < p.max_pages) ? p.block_table[(size_t)b * p.max_pages + i] : 0;
  }
  const int n_raw = p.n_nodes[b];
  const int L = p.prefix_len[b];
  int flag = 0;
  if (n_raw < 0 || n_raw > p.B) flag |= JT_DEVERR_NNODES;
  if (L < 0 || L > p.Lbound) flag |= JT_DEVERR_PREFIX;
  if (p.paged && !no_item && !(flag & JT_DEVERR_PREFIX)) {
    const int np = (L + kPageSize - 1) / kPageSize;
#pragma unroll
    for (int q = 0; q < kPrefetchPages; ++q)
      if (tid + q * kThreads < np && (pre[q] < 0 || pre[q] >= p.n_pages)) flag |= JT_DEVERR_PAGE;
    for (int i = tid + kPrefetchPages * kThreads; i < np; i += kThreads) {
      const int pg = p.block_table[(size_t)b * p.max_pages + i];
      if (pg < 0 || pg >= p.n_pages) flag |= JT_DEVERR_PAGE;
    }
  }
  tc_fence_before();
  const int bad = __syncthreads_or(flag);   // also publishes the barriers and the TMEM base
  tc_fence_after();
  if (BAL && no_item) {
    if (warp == kWarpMMA) tmem_dealloc(bars->tmem_base, kTmemCols);
    return;
  }
  if (flag && rank == 0) raise_flag(p.d_err, flag);
  const int n = bad ? 0 : n_raw;

  const bool has_rows = v0 < n;
  const bool twoB = v0 + npt < n;          // tile B holds at least one live node
  const int p_tiles = has_rows ? (L + kTile - 1) / kTile : 0;
  const int v_last = min(v0 + 2 * npt, n) - 1;
  const int t_tree = has_rows ? (v_last + kTile) / kTile : 0;
  const int t_tot = p_tiles + t_tree;
  // CTAs sharing this unit's key tiles: the cluster, or this unit's chunks.
  const int split = BAL ? min(S, max(1, (t_tot + p.chunk_tiles - 1) / p.chunk_tiles)) : S;
  if (BAL && tid == 0) {
    bars->split = split;
    if (rank == 0 && p.nparts) p.nparts[unit] = split;   // read by attn_merge_kernel
  }
  if (BAL && rank >= split) {   // a chunk slot this unit does not need
    if (warp == kWarpMMA) tmem_dealloc(bars->tmem_base, kTmemCols);
    return;
  }
  const int t_begin = (int)((long)rank * t_tot / split);
  const int t_end = (int)((long)(rank + 1) * t_tot / split);
  const int T = t_end - t_begin;

  if (!has_rows) {
    // Every row of this unit is an unused budget slot: zeros. The unit's
    // CTAs split the rows; in a cluster they still join its barrier.
    if (warp == kWarpMMA) tmem_dealloc(bars->tmem_base, kTmemCols);
    const int R = 2 * kTile / split;
    for (int i = tid; i < R * (D / 8); i += kThreads) {
      const int r = rank * R + i / (D / 8), u = i % (D / 8);
      const int v = v0 + r / g, j = r % g;
      if (v < p.B)
        reinterpret_cast<uint4*>(p.out + (((size_t)b * p.B + v) * p.hq + kh * g + j) * D)[u] =
            make_uint4(0, 0, 0, 0);
    }
    if (!BAL && S > 1) cg::this_cluster().sync();
    return;
  }

  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  auto fail = [&]() {
    if (atomicExch(&bars->abort, 1) == 0) raise_flag(p.d_err, JT_DEVERR_TIMEOUT);
  };
  // Every lane of the calling warp polls; the verdict is made warp-uniform so
  // that warp-collective tcgen05 / vote instructions never see divergence.
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort, p.wait_budget)) != 0;
  };
  // Valid keys of tile t (prefix tiles first, then tree tiles).
  auto tile_valid = [&](int t) {
    return t < p_tiles ? min(kTile, L - t * kTile) : min(kTile, n - (t - p_tiles) * kTile);
  };

  // Key split: when tile B holds no live node, both softmax warpgroups serve
  // tile A's rows, warpgroup G taking the key tiles jt = G, G + 2, ... into
  // its own S/P and O columns (S_G = Q_A K^T), so that the S MMA and the
  // softmax of one key tile overlap those of the next; their two (m, l, O)
  // states are merged in the epilogue.
  const bool ks = KSPLIT && !twoB && T >= 2;
  // Softmax state, read by the common epilogue.
  float m_run = -INFINITY, l_run = 0.0f;
  const int G = warp >> 2;                  // TMEM column group (S/P and O)
  const int X = ks ? 0 : G;                 // M tile of this thread's row
  const int r = tid & 127;
  const int R = X * kTile + r;              // row within the unit's 256
  const int v = v0 + R / g;
  const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t s_col = tmem + lane_base + G * 128;
  const uint32_t o_col = tmem + lane_base + 256 + G * OSTRIDE;
  const bool tile_live = X == 0 || twoB;
  const int j_first = ks ? G : 0, j_step = ks ? 2 : 1;
  const int T_own = ks ? (T - G + 1) / 2 : T;   // key tiles this warpgroup processes
  bool sm_ok = true;
  int issued = 0;   // producers: K (warp 8) or V (warp 10) tiles whose loads were issued

  if (warp >= 8) {
  // Third warpgroup: producer, MMA issuer, two idle warps. Lean registers.
  regs_dec<kRegsOther>();
  if (warp == kWarpTMA || warp == kWarpTMAV) {
    // =================== TMA producers (warp 8: Q and K, warp 10: V) ===================
    const bool is_v = warp == kWarpTMAV;
    if (lane == 0 && T > 0) {
      if (!is_v) {
        mbar_arrive_expect_tx(&bars->q_full, (twoB ? 2 : 1) * QB);
        for (int X2 = 0; X2 < (twoB ? 2 : 1); ++X2)
#pragma unroll
          for (int ch = 0; ch < CH; ++ch)
            tma_load_4d(sQ(X2) + ch * CHB, &mq, &bars->q_full, ch * 64, kh * g, v0 + X2 * npt, b);
      }
      const CUtensorMap* mc = is_v ? &mvc : &mkc;
      const CUtensorMap* mtr = is_v ? &mvt : &mkt;
      uint64_t* full = is_v ? bars->v_full : bars->k_full;
      uint64_t* empty = is_v ? bars->v_empty : bars->k_empty;
      const int np = (L + kPageSize - 1) / kPageSize;
      // Page ids of a paged prefix tile: all eight loaded together, one tile
      // ahead (right after the current tile's copies have taken theirs), so
      // that they are in flight while the producer waits for the next ring
      // slot (one at a time, each load sat between TMA issues).
      constexpr int kPagesPerTile = kTile / kPageSize;
      int pg_cur[kPagesPerTile];
      auto load_pages = [&](int t, int (&ids)[kPagesPerTile]) {
        if (p.paged && t < p_tiles) {
#pragma unroll
          for (int q = 0; q < kPagesPerTile; ++q) {
            const int pi = t * kPagesPerTile + q;
            ids[q] = pi < np ? p.block_table[(size_t)b * p.max_pages + pi] : 0;
          }
        }
      };
      load_pages(t_begin, pg_cur);
      for (int jt = 0; jt < T; ++jt) {
        const int t = t_begin + jt, st = jt % kStages;
        if (jt >= kStages &&
            !mbar_wait(&empty[st], ((jt / kStages) + 1) & 1, abort, p.wait_budget)) {
          fail();
          break;
        }
        mbar_arrive_expect_tx(&full[st], QB);
        issued = jt + 1;
        uint8_t* dst = is_v ? sV(st) : sK(st);
        if (t < p_tiles) {
          const int key0 = t * kTile;
          if (p.paged) {
#pragma unroll
            for (int pg = 0; pg < kPagesPerTile; ++pg) {
#pragma unroll
              for (int ch = 0; ch < CH; ++ch)
                tma_load_4d(dst + ch * CHB + pg * (kPageSize * 128), mc, &full[st], ch * 64, kh, 0,
                            pg_cur[pg]);
            }
          } else {
#pragma unroll
            for (int ch = 0; ch < CH; ++ch)
              tma_load_4d(dst + ch * CHB, mc, &full[st], ch * 64, kh, key0, b);
          }
        } else {
          const int u0 = (t - p_tiles) * kTile;
#pragma unroll
          for (int ch = 0; ch < CH; ++ch)
            tma_load_4d(dst + ch * CHB, mtr, &full[st], ch * 64, kh, u0, b);
        }
        if (jt + 1 < T) load_pages(t + 1, pg_cur);
      }
    }
  } else if (warp == kWarpMMA) {
    // =================== MMA issuer ===================
    constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t id_o = idesc_bf16(128, D, 0, 1);   // N = D: one MMA per K step
    // Descriptor bases (start address in the low 14 bits); each K step adds
    // a constant byte offset >> 4, so no descriptor is rebuilt in the loop.
    const uint64_t qd[2] = {sdesc_sw128(smem_u32(sQ(0)), 16, 1024), sdesc_sw128(smem_u32(sQ(1)), 16, 1024)};
    const uint64_t kd[2] = {sdesc_sw128(smem_u32(sK(0)), 16, 1024), sdesc_sw128(smem_u32(sK(1)), 16, 1024)};
    const uint64_t vd[2] = {sdesc_sw128(smem_u32(sV(0)), CHB, 1024), sdesc_sw128(smem_u32(sV(1)), CHB, 1024)};
    // S of column group Gd from Q tile Xq and K slot st.
    auto issue_s = [&](int Xq, int st, int Gd) {
      const uint64_t q = qd[Xq], k = kd[st];
      const uint32_t d = tmem + Gd * 128;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * CHB + (kk & 3) * 32) >> 4);
        mma_bf16_ss_warp(d, q + off, k + off, id_s, kk > 0);
      }
      mma_commit_warp(&bars->s_full[Gd]);
    };
    // O_Gd (+)= P_Gd V, V from the slot of key tile jt; `first` starts O.
    // Only a group's last P V is committed to pv_done (one phase per
    // launch): the epilogue is its one reader.
    auto issue_pv = [&](int Gd, int jt, bool first, bool last) {
      const uint64_t v = vd[jt % kStages];
      const uint32_t d = tmem + 256 + Gd * OSTRIDE, a = tmem + Gd * 128;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_bf16_ts_warp(d, a + kk * 8, v + (uint64_t)(kk * (2048 >> 4)), id_o, !first || kk > 0);
      if (last) mma_commit_warp(&bars->pv_done[Gd]);
    };
    // Rows of V past a tile's valid keys that the TMA read from memory may
    // hold anything (NaN included); P is 0 there but 0 * NaN is NaN, so they
    // are zeroed before P V reads them. Rows outside the tensor arrive as
    // zeros already (contiguous cache past max_prefix, tree rows past B).
    auto zero_v_tail = [&](int jt) {
      const int t = t_begin + jt;
      const int valid = tile_valid(t);
      const int loaded = t < p_tiles ? (p.paged ? kTile : min(kTile, p.Lbound - t * kTile))
                                     : min(kTile, p.B - (t - p_tiles) * kTile);
      if (valid < loaded) {
        uint8_t* vt = sV(jt % kStages);
        for (int i = lane; i < (loaded - valid) * CH * 8; i += 32) {
          const int r = valid + i / (CH * 8), rem = i % (CH * 8);
          *reinterpret_cast<uint4*>(vt + (rem / 8) * CHB + r * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
    };
    bool ok = T > 0 && warp_wait(&bars->q_full, 0) && warp_wait(&bars->k_full[0], 0);
    if (T > 0 && !ok) fail();
    if (ok && ks) {
      // Key split, per key tile t (column group t & 1, local index t >> 1):
      // S(0), S(1), then PV(t), S(t + 2) for t = 0, 1, 2, ...
      tc_fence_after();
      issue_s(0, 0, 0);
      mma_commit_warp(&bars->k_empty[0]);
      if (!warp_wait(&bars->k_full[1], 0)) { fail(); ok = false; }
      if (ok) {
        tc_fence_after();
        issue_s(0, 1, 1);
        mma_commit_warp(&bars->k_empty[1]);
      }
      for (int t = 0; ok && t < T; ++t) {
        const int Gt = t & 1, st = t % kStages;
        if (!warp_wait(&bars->p_full[Gt], (t >> 1) & 1)) { fail(); ok = false; break; }
        if (!warp_wait(&bars->v_full[st], (t / kStages) & 1)) { fail(); ok = false; break; }
        zero_v_tail(t);
        tc_fence_after();
        issue_pv(Gt, t, t < 2, t + 2 >= T);
        mma_commit_warp(&bars->v_empty[st]);
        if (t + 2 < T) {
          if (!warp_wait(&bars->k_full[st], ((t + 2) / kStages) & 1)) { fail(); ok = false; break; }
          tc_fence_after();
          issue_s(0, st, Gt);
          mma_commit_warp(&bars->k_empty[st]);
        }
      }
    } else if (ok) {
      // Tile pair, per key tile jt: PV_A(jt), S_A(jt+1), PV_B(jt), S_B(jt+1).
      tc_fence_after();
      issue_s(0, 0, 0);
      if (twoB) issue_s(1, 0, 1);
      mma_commit_warp(&bars->k_empty[0]);   // K tile 0 is no longer needed
    }
    for (int jt = 0; ok && !ks && jt < T; ++jt) {
      const int st = jt % kStages;
      const bool more = jt + 1 < T;
      const int st1 = (jt + 1) % kStages;
      // The loads run well ahead of the MMAs: observe V(jt) and K(jt+1)
      // first, so that only the MMAs follow the wait for P_A (the tile's
      // softmax -> P V -> S -> softmax chain sets the pace).
      // One combined test (both normally landed long ago); the bounded
      // waits only when it fails.
      const bool kv = mbar_test_wait(&bars->v_full[st], (jt / kStages) & 1) &
                      (!more || mbar_test_wait(&bars->k_full[st1], ((jt + 1) / kStages) & 1));
      if (!__all_sync(0xFFFFFFFFu, kv)) {
        if (!warp_wait(&bars->v_full[st], (jt / kStages) & 1)) { fail(); ok = false; break; }
        if (more && !warp_wait(&bars->k_full[st1], ((jt + 1) / kStages) & 1)) {
          fail(); ok = false; break;
        }
      }
      zero_v_tail(jt);
      if (!warp_wait(&bars->p_full[0], jt & 1)) { fail(); ok = false; break; }
      tc_fence_after();
      issue_pv(0, jt, jt == 0, !more);
      if (more) {
        issue_s(0, st1, 0);
        if (!twoB) mma_commit_warp(&bars->k_empty[st1]);
      }
      if (twoB) {
        if (!warp_wait(&bars->p_full[1], jt & 1)) { fail(); ok = false; break; }
        tc_fence_after();
        issue_pv(1, jt, jt == 0, !more);
      }
      mma_commit_warp(&bars->v_empty[st]);
      if (twoB && more) {
        issue_s(1, st1, 1);
        mma_commit_warp(&bars->k_empty[st1]);
      }
    }
  }
  } else {
  // =================== softmax (warps 0-7, tile X = warp / 4) ===================
  regs_inc<kRegsSoftmax>();
  if (tile_live) {
    const bool row_valid = v < n;
    // This row's ancestor words, read for the tree tiles only (one or two
    // per CTA), before the wait for S so that the load overlaps it.
    const uint32_t* mrow = p.mask + ((size_t)b * p.B + (row_valid ? v : 0)) * p.words;
    const float sl2 = p.scale_log2;
    for (int jt = j_first, it = 0; jt < T; jt += j_step, ++it) {
      const int t = t_begin + jt;
      // Which keys of this tile the row sees: c < lim, and for tree tiles the
      // ancestor bit of key u0 + c.
      const bool tree = t >= p_tiles;
      const int lim = tree ? n - (t - p_tiles) * kTile : L - t * kTile;
      const int wb = tree && ((t - p_tiles) * kTile) >= 128 ? 4 : 0;
      uint32_t ws0 = 0xFFFFFFFFu, ws1 = 0xFFFFFFFFu, ws2 = 0xFFFFFFFFu, ws3 = 0xFFFFFFFFu;
      if (tree) {
        ws0 = row_valid && wb + 0 < p.words ? __ldg(mrow + wb + 0) : 0u;
        ws1 = row_valid && wb + 1 < p.words ? __ldg(mrow + wb + 1) : 0u;
        ws2 = row_valid && wb + 2 < p.words ? __ldg(mrow + wb + 2) : 0u;
        ws3 = row_valid && wb + 3 < p.words ? __ldg(mrow + wb + 3) : 0u;
      }
      if (!warp_wait(&bars->s_full[G], it & 1)) { fail(); sm_ok = false; break; }
      tc_fence_after();
      auto word_of = [&](int c) {   // ancestor bits of keys 32c..32c+31 of this tile
        const uint32_t w01 = (c & 1) ? ws1 : ws0, w23 = (c & 1) ? ws3 : ws2;
        return (c & 2) ? w23 : w01;
      };
      // All 128 scores of the row at once (one wait), then the row max of the
      // visible raw scores (scaling by sl2 > 0 commutes with the max; it is
      // folded into the exponent below). A prefix tile whose 128 keys are all
      // visible needs no per-key test; otherwise one word per 32 keys holds
      // the visibility bits (ancestor bits and c < lim).
      const bool full = !tree && lim >= kTile;
      float x[kTile];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float tmp[32];
        tmem_ld32(s_col + c * 32, tmp);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = tmp[i];
      }
      tmem_wait_ld();
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (!full) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int rem = lim - c * 32;
          const uint32_t lim_bits = rem >= 32 ? 0xFFFFFFFFu : rem <= 0 ? 0u : (1u << rem) - 1u;
          const uint32_t vw = word_of(c) & lim_bits;
#pragma unroll
          for (int i = 0; i < 32; ++i) x[c * 32 + i] = ((vw >> i) & 1u) ? x[c * 32 + i] : -INFINITY;
        }
      }
#pragma unroll
      for (int i = 0; i < kTile; i += 2) m4[(i >> 1) & 3] = fmax3(m4[(i >> 1) & 3], x[i], x[i + 1]);
      const float tmax = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * sl2;
      const float mnew = fmaxf(m_run, tmax);
      const bool need = mnew > m_run + kRescaleLog2;
      float corr = 1.0f;
      if (need) {
        corr = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mnew);
        l_run *= corr;
        m_run = mnew;
      }
      if (it >= 1 && __any_sync(0xFFFFFFFFu, need)) {
        // This group's previous P V is complete: the commit behind s_full covers it.
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(o_col + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= corr;
          tmem_st32(o_col + c * 32, o);
        }
      }
      // P = 2^(s sl2 - m) as bf16 pairs over the S columns (all already read);
      // the exponent argument and the row sum go two columns per packed
      // fp32x2 instruction.
      const float muse = (m_run == -INFINITY) ? 0.0f : m_run;
      const uint64_t sl2x2 = f32x2(sl2, sl2), negm2 = f32x2(-muse, -muse);
      uint64_t ls2[2] = {f32x2(0.0f, 0.0f), f32x2(0.0f, 0.0f)};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float y0, y1;
          f32x2_split(ffma2(f32x2(x[c * 32 + 2 * i], x[c * 32 + 2 * i + 1]), sl2x2, negm2), y0, y1);
          const float p0 = ex2(y0), p1 = ex2(y1);
          ls2[i & 1] = fadd2(ls2[i & 1], f32x2(p0, p1));
          pk[i] = pack_bf16(p0, p1);
        }
        tmem_st16(s_col + c * 16, pk);
      }
      float l0, l1, l2, l3;
      f32x2_split(ls2[0], l0, l1);
      f32x2_split(ls2[1], l2, l3);
      const float lsum = (l0 + l1) + (l2 + l3);
      tmem_wait_st();
      l_run += lsum;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[G]);
    }
    if (sm_ok && T_own > 0) {
      if (warp_wait(&bars->pv_done[G], 0)) tc_fence_after();
      else { fail(); sm_ok = false; }
    }
  }
  regs_dec<kRegsLaunch>();
  }
  // Only once both softmax warpgroups have handed their extra registers back
  // may the third warpgroup take its share again: setmaxnreg.inc waits
  // without bound, so an earlier request (e.g. from the idle warps) could
  // take registers a softmax warpgroup still needs to grow, and deadlock.
  __syncthreads();
  if (warp >= 8) regs_inc<kRegsLaunch>();
  // A CTA that gave up (every failing wait precedes the barrier above) may
  // still have TMA loads landing in its shared memory. Before that memory is
  // reused below or released at exit, each producer waits for its last load
  // into each ring slot (a slot's earlier loads were consumed, or it would
  // not have been refilled) and for Q, with the default budget.
  if (*abort && lane == 0 && (warp == kWarpTMA || warp == kWarpTMAV) && T > 0) {
    uint64_t* full = warp == kWarpTMAV ? bars->v_full : bars->k_full;
    bool drained = warp == kWarpTMAV || mbar_wait_drain(&bars->q_full, 0, kDefaultWaitBudget);
    for (int st = 0; st < kStages; ++st) {
      if (issued > st) {
        const int last = st + kStages * ((issued - 1 - st) / kStages);
        drained &= mbar_wait_drain(&full[st], (last / kStages) & 1, kDefaultWaitBudget);
      }
    }
    (void)drained;   // a load that never lands has already been reported as a timeout
  }
  const bool have_o = warp < 8 && tile_live && sm_ok && T_own > 0;
  if (!have_o) { m_run = -INFINITY; l_run = 0.0f; }
  // Every live tile has seen its last P V complete, so the tensor pipe and
  // the K/V ring are idle from here on: the merge buffer may overlay them.
  __syncthreads();

  // Key split: the two warpgroups swap (m, l) through the unused Q_B tile and
  // each merges one half of the head dimension of the same rows:
  // O = f_0 O_0 + f_1 O_1, l = f_0 l_0 + f_1 l_1, f_G = 2^(m_G - M), M = max_G m_G.
  // Each group has waited only for its own last P V: the tcgen05 fences
  // around the barrier order the other group's MMAs before the TMEM loads.
  float f0 = 1.0f, f1 = 0.0f;
  if (ks) {
    float2* ml = reinterpret_cast<float2*>(sQ(1));
    if (warp < 8) ml[G * kTile + r] = make_float2(m_run, l_run);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp < 8) {
      const float2 a0 = ml[r], a1 = ml[kTile + r];
      const float M = fmaxf(a0.x, a1.x);
      f0 = a0.x == -INFINITY ? 0.0f : ex2(a0.x - M);
      f1 = a1.x == -INFINITY ? 0.0f : ex2(a1.x - M);
      l_run = f0 * a0.y + f1 * a1.y;
      m_run = M;
    }
  }
  // Columns 32c .. 32c + 31 of this row's O (zeros without one); in a key
  // split both groups' O, merged 16 columns at a time.
  const uint32_t o0_col = tmem + lane_base + 256;
  auto load_o = [&](int c, float (&o)[32]) {
    if (ks) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float a[16], bb[16];
        tmem_ld16(o0_col + c * 32 + h * 16, a);
        tmem_ld16(o0_col + OSTRIDE + c * 32 + h * 16, bb);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o[h * 16 + i] = (f0 != 0.0f ? a[i] * f0 : 0.0f) + (f1 != 0.0f ? bb[i] * f1 : 0.0f);
      }
    } else if (have_o) {
      tmem_ld32(o_col + c * 32, o);
      tmem_wait_ld();
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = 0.0f;
    }
  };
  // 32-column chunks of O this thread writes (a key split halves them).
  const int c_lo = ks ? G * (D / 64) : 0, c_hi = ks ? c_lo + D / 64 : D / 32;

  // ---- output (S == 1) or publish partials (S > 1); both read O from TMEM ----
  const int unit_e = BAL ? ld_shared_volatile(&bars->unit) : unit;
  const int rank_e = BAL ? ld_shared_volatile(&bars->rank) : rank;
  const int split_e = BAL ? ld_shared_volatile(&bars->split) : split;
  const int bk_e = unit_e / p.n_mpairs;
  const int kh_e = bk_e % p.hkv, b_e = bk_e / p.hkv;
  const int v0_e = (unit_e % p.n_mpairs) * 2 * npt;
  const int n_live = min(2 * kTile, (n - v0_e) * g);   // rows of live nodes come first
  if (warp < 8) {
    const int j = R % g;
    const bool write_row = v < p.B;
    const float inv = (v < n && l_run > 0.0f) ? 1.0f / l_run : 0.0f;
    if (split_e > 1) {
      // Only rows that some rank will merge are written; coalesced per column
      // (a warp's 32 rows land in 32 / S runs of whole 32-byte sectors). The
      // TMEM load is warp-collective, so the whole warp takes it whenever any
      // of its rows is live, and only the stores are per row. The balanced
      // schedule's single merging CTA reads rows in order (slot = R).
      if ((R & ~31) < n_live) {
        const bool live = R < n_live;
        const size_t pidx = BAL ? (size_t)unit_e * S + rank_e : (size_t)blockIdx.x;
        float* part = p.part + pidx * part_floats<D>();
        const int sig = BAL ? 1 : S;
        const int slot = (R % sig) * (2 * kTile / sig) + R / sig;
        float4* po = reinterpret_cast<float4*>(part);
#pragma unroll 1
        for (int c = c_lo; c < c_hi; ++c) {
          float o[32];
          load_o(c, o);
          if (live) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              __stcg(po + (c * 8 + i / 4) * (2 * kTile) + slot,
                     make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]));
          }
        }
        if (live && (!ks || G == 0)) {
          __stcg(part + 2 * kTile * D + slot, m_run);
          __stcg(part + 2 * kTile * D + 2 * kTile + slot, l_run);
        }
      }
    } else {
      uint4* dst = reinterpret_cast<uint4*>(p.out + (((size_t)b_e * p.B + v) * p.hq + kh_e * g + j) * D);
#pragma unroll
      for (int c = c_lo; c < c_hi; ++c) {
        float o[32];
        load_o(c, o);
        if (write_row) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[c * 4 + q] = make_uint4(pack_bf16(o[8 * q] * inv, o[8 * q + 1] * inv),
                                        pack_bf16(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                                        pack_bf16(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                                        pack_bf16(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
        }
      }
    }
  }

  // Key split with direct output: tile B's rows hold no live node; the
  // third warpgroup writes the zeros of those inside the budget (the split-KV
  // merges zero every unused row themselves).
  if (ks && split_e == 1 && warp >= 8) {
    const int Rb = kTile + (tid - 256);
    const int vb = v0_e + Rb / g;
    if (vb < p.B) {
      uint4* dst = reinterpret_cast<uint4*>(p.out + (((size_t)b_e * p.B + vb) * p.hq + kh_e * g + Rb % g) * D);
#pragma unroll
      for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
    }
  }

  // ---- release TMEM (after draining outstanding MMAs on the abort path) ----
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMMA) {
    tc_fence_after();
    if (*abort) {
      // The elected lane issued every MMA, so it also commits the drain.
      mma_commit_warp(&bars->drain);
      const long long t0 = clock64();
      while (!mbar_try_wait(&bars->drain, 0) && clock64() - t0 < kDefaultWaitBudget) {
      }
    }
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (split_e == 1) return;

  if (BAL) return;   // attn_merge_kernel combines the chunks after the grid

  // ---- split-KV merge through L2 (the cluster barrier, reached by every CTA
  // of the split, orders the partial writes above before the reads) ----
  cg::this_cluster().sync();
  float* fac = reinterpret_cast<float*>(sm);   // over the dead Q tile
  const float* part0 = p.part + (size_t)(blockIdx.x - rank_e) * part_floats<D>();
  switch (S) {
    case 2: merge_split<D, 2, 4>(p, part0, fac, rank_e, n_live, v0_e, b_e, kh_e, tid); break;
    case 4: merge_split<D, 4, 2>(p, part0, fac, rank_e, n_live, v0_e, b_e, kh_e, tid); break;
    default: merge_split<D, 8, 1>(p, part0, fac, rank_e, n_live, v0_e, b_e, kh_e, tid); break;
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps, split choice, launch.
// ---------------------------------------------------------------------------
AttnParams make_params(const jt_attn_args& a) {
  AttnParams p = {};
  p.batch = a.batch;
  p.B = a.B;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.g = a.hq / a.hkv;
  p.npt = kTile / p.g;
  p.n_mpairs = ((a.B + p.npt - 1) / p.npt + 1) / 2;
  p.paged = a.block_table != nullptr;
  p.max_pages = a.max_pages;
  p.n_pages = a.n_pages;
  p.Lbound = p.paged ? a.max_pages * kPageSize : a.max_prefix;
  if (p.paged && a.max_prefix > 0 && a.max_prefix < p.Lbound) p.Lbound = a.max_prefix;
  p.words = (a.B + 31) / 32;
  p.block_table = a.block_table;
  p.prefix_len = a.prefix_len;
  p.n_nodes = a.n_nodes;
  p.mask = a.mask;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  const float scale = a.scale != 0.0f ? a.scale : 1.0f / sqrtf((float)a.head_dim);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.wait_budget = wait_budget();
  return p;
}

// Largest split (power of two, at most 8) before residency is checked: the
// grid stays within the SMs and no rank is left without a key tile.
int split_limit(const jt_attn_args& a, const AttnParams& p, int num_sms) {
  const int units = a.batch * a.hkv * p.n_mpairs;
  const int tiles_max = (p.Lbound + kTile - 1) / kTile + (a.B + kTile - 1) / kTile;
  int s = 1;
  while (s < 8 && (long)units * (2 * s) <= num_sms && 2 * s <= tiles_max) s *= 2;
  return s;
}

// Schedule choice, a function of the shapes only (so that the workspace
// query and the launch agree). Few units (two or more CTAs per unit fit in
// one wave): cluster split. Otherwise the balanced schedule, with up to
// ceil(2 SMs / units) chunks per unit (1 when the units alone cover the SMs
// twice) and chunks of ceil(tiles_max / S) tiles.
struct Schedule {
  int balanced, S, chunk_tiles, units;
};

Schedule pick_schedule(const jt_attn_args& a, const AttnParams& p, int num_sms) {
  Schedule sc{0, 1, 0, a.batch * a.hkv * p.n_mpairs};
  if ((long)sc.units * 2 <= num_sms) return sc;   // cluster split (S chosen at launch)
  const int tiles_max = (p.Lbound + kTile - 1) / kTile + (a.B + kTile - 1) / kTile;
  sc.balanced = 1;
  sc.S = (int)std::min<long>(8, std::max<long>(1, (2L * num_sms + sc.units - 1) / sc.units));
  sc.S = std::min(sc.S, std::max(1, tiles_max));
  sc.chunk_tiles = std::max(1, (tiles_max + sc.S - 1) / sc.S);
  return sc;
}

size_t balanced_meta_bytes(int units, int S) {
  return align_up((size_t)units * (S + 1) * sizeof(int32_t), 256);   // items, then part counts
}

template <int D>
size_t smem_bytes() { return (2 + 2 * kStages) * (size_t)kTile * D * 2 + 256 + 1024; }

// Registers per thread a kernel launches with (queried once per kernel).
cudaError_t kernel_regs(const void* kern, int* regs) {
  static std::mutex mu;
  static const void* keys[16] = {};
  static int vals[16] = {};
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < 16 && keys[i]; ++i)
    if (keys[i] == kern) { *regs = vals[i]; return cudaSuccess; }
  cudaFuncAttributes fa = {};
  const cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  *regs = fa.numRegs;
  for (int i = 0; i < 16; ++i)
    if (!keys[i]) { keys[i] = kern; vals[i] = fa.numRegs; break; }
  return cudaSuccess;
}

template <int D>
cudaError_t launch_d(const Ctx& c, const jt_attn_args& a, AttnParams& p) {
  const size_t smem = smem_bytes<D>();
  const int units = a.batch * a.hkv * p.n_mpairs;
  const Schedule sc = pick_schedule(a, p, c.num_sms);
  // Residency queries use the plain variant (both variants have the same
  // shared memory and threads).
  auto kern = sc.balanced ? tree_attn_tc_kernel<D, true, false> : tree_attn_tc_kernel<D, false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;

  if (sc.balanced) {
    const size_t meta = balanced_meta_bytes(units, sc.S);
    const size_t need = meta + (sc.S > 1 ? align_up((size_t)units * sc.S * part_floats<D>() *
                                                        sizeof(float), 256) : 0);
    if (!c.workspace || c.workspace_bytes < need) return cudaErrorInvalidValue;
    p.units = units;
    p.S = sc.S;
    p.chunk_tiles = sc.chunk_tiles;
    p.perm = static_cast<int32_t*>(c.workspace);
    p.nparts = sc.S > 1 ? p.perm + (size_t)units * sc.S : nullptr;
    p.part = sc.S > 1 ? reinterpret_cast<float*>(static_cast<char*>(c.workspace) + meta) : nullptr;
    const size_t plan_smem =
        units * sc.S <= kPlanMaxSort ? (size_t)(kPlanBuckets + units * sc.S) * sizeof(int) : 0;
    if (plan_smem > 48 * 1024) {
      e = cudaFuncSetAttribute(attn_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)plan_smem);
      if (e != cudaSuccess) return e;
    }
    e = launch_kernel(attn_plan_kernel, dim3(1), dim3(kPlanThreads), plan_smem, c.stream, 1, p);
    if (e != cudaSuccess) return e;
  }
  // Cluster split: only when the workspace holds the partials.
  const bool have_part = !sc.balanced && p.part != nullptr &&
                         c.workspace_bytes >= (size_t)c.num_sms * part_floats<D>() * sizeof(float);
  const int limit = have_part ? split_limit(a, p, c.num_sms) : 1;
  // Largest split whose clusters are all resident at once (one wave).
  int S = sc.balanced ? sc.S : 1;
  cudaLaunchConfig_t occ = {};
  cudaLaunchAttribute occ_attr[1];
  occ.blockDim = dim3(kThreads);
  occ.dynamicSmemBytes = smem;
  occ.stream = c.stream;
  occ_attr[0].id = cudaLaunchAttributeClusterDimension;
  occ_attr[0].val.clusterDim.y = 1;
  occ_attr[0].val.clusterDim.z = 1;
  occ.attrs = occ_attr;
  occ.numAttrs = 1;
  for (int cand = 2; !sc.balanced && cand <= limit; cand *= 2) {
    occ_attr[0].val.clusterDim.x = cand;
    occ.gridDim = dim3(units * cand);
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &occ) != cudaSuccess) {
      cudaGetLastError();
      break;
    }
    if (nclusters < units) break;
    S = cand;
  }
  p.S = S;
  // Key split variant: no unit can have a live tile B (the budget fits one M
  // tile, B <= 128 / g) and some CTA gets two key tiles or more.
  const int tiles_max = (p.Lbound + kTile - 1) / kTile + (a.B + kTile - 1) / kTile;
  const int cta_tiles = sc.balanced ? sc.chunk_tiles : (tiles_max + S - 1) / S;
  if (a.B <= p.npt && cta_tiles >= 2) {
    kern = sc.balanced ? tree_attn_tc_kernel<D, true, true> : tree_attn_tc_kernel<D, false, true>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }

  // setmaxnreg.inc waits without bound for the registers it asks for, and
  // the split draws on the block's launch allocation: a build whose kernel
  // got fewer than kRegsLaunch registers per thread would never finish.
  // Refuse it instead.
  int regs = 0;
  e = kernel_regs(reinterpret_cast<const void*>(kern), &regs);
  if (e != cudaSuccess) return e;
  if (regs * kThreads < 256 * (int)kRegsSoftmax + 128 * (int)kRegsOther)
    return cudaErrorInvalidConfiguration;

  CUtensorMap mq, mkc, mvc, mkt, mvt;
  const uint64_t D64 = D;
  if (!make_map(&mq, a.q, {D64, (uint64_t)a.hq, (uint64_t)a.B, (uint64_t)a.batch},
                {64, (uint32_t)p.g, (uint32_t)p.npt, 1}))
    return cudaErrorInvalidValue;
  if (a.block_table) {
    if (!make_map(&mkc, a.k_cache, {D64, (uint64_t)a.hkv, (uint64_t)kPageSize, (uint64_t)a.n_pages},
                  {64, 1, (uint32_t)kPageSize, 1}) ||
        !make_map(&mvc, a.v_cache, {D64, (uint64_t)a.hkv, (uint64_t)kPageSize, (uint64_t)a.n_pages},
                  {64, 1, (uint32_t)kPageSize, 1}))
      return cudaErrorInvalidValue;
  } else {
    if (!make_map(&mkc, a.k_cache, {D64, (uint64_t)a.hkv, (uint64_t)a.max_prefix, (uint64_t)a.batch},
                  {64, 1, (uint32_t)kTile, 1}) ||
        !make_map(&mvc, a.v_cache, {D64, (uint64_t)a.hkv, (uint64_t)a.max_prefix, (uint64_t)a.batch},
                  {64, 1, (uint32_t)kTile, 1}))
      return cudaErrorInvalidValue;
  }
  if (!make_map(&mkt, a.k_tree, {D64, (uint64_t)a.hkv, (uint64_t)a.B, (uint64_t)a.batch},
                {64, 1, (uint32_t)kTile, 1}) ||
      !make_map(&mvt, a.v_tree, {D64, (uint64_t)a.hkv, (uint64_t)a.B, (uint64_t)a.batch},
                {64, 1, (uint32_t)kTile, 1}))
    return cudaErrorInvalidValue;
  e = launch_kernel(kern, dim3(units * S), dim3(kThreads), smem, c.stream,
                    sc.balanced ? 1 : S, mq, mkc, mvc, mkt, mvt, p);
  if (e != cudaSuccess || !sc.balanced || sc.S < 2) return e;
  return launch_kernel(attn_merge_kernel<D>, dim3(units * kMergeSlices), dim3(kMergeThreads), 0,
                       c.stream, 1, p);
}

}  // namespace

size_t attn_workspace_bytes(const jt_attn_args& a, int num_sms) {
  if (a.batch == 0) return 0;
  AttnParams p = make_params(a);
  const size_t per = (a.head_dim == 64 ? part_floats<64>() : part_floats<128>()) * sizeof(float);
  const Schedule sc = pick_schedule(a, p, num_sms);
  if (sc.balanced) {
    // item order and per-unit part counts, then one partial per chunk slot
    return balanced_meta_bytes(sc.units, sc.S) +
           (sc.S > 1 ? align_up((size_t)sc.units * sc.S * per, 256) : 0);
  }
  // A cluster split never exceeds the SMs (one CTA per SM, one wave), so
  // num_sms partials always suffice; none are needed when no split fits.
  if (split_limit(a, p, num_sms) < 2) return 0;
  return align_up((size_t)num_sms * per, 256);
}

cudaError_t launch_tree_attn(const Ctx& c, const jt_attn_args& a) {
  if (a.batch == 0) return cudaSuccess;
  AttnParams p = make_params(a);
  p.part = static_cast<float*>(c.workspace);
  p.d_err = c.d_err;
  return a.head_dim == 64 ? launch_d<64>(c, a, p) : launch_d<128>(c, a, p);
}

}  // namespace jt
