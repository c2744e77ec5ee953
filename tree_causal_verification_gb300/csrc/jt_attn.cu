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
// Work unit = (sequence b, KV head kh, M-tile of 128 query rows). Rows are
// node-major, row = v*g + j, so one unit's 128 rows are 128/g consecutive
// tree nodes times all g query heads that share KV head kh: every K/V tile
// streamed from HBM is used by all of them (GQA folded into the MMA M
// dimension). The unit's keys are the prefix tiles (128 keys each, paged
// through 16-token pages or contiguous) followed by the tree tiles (only
// those holding ancestors of the tile's nodes).
//
// One CTA per unit (or per slice of its key tiles when the unit count is too
// small to fill the GPU: split-KV across a thread-block cluster, merged in
// distributed shared memory). 192 threads:
//   warps 0-3  softmax: thread r owns query row r = TMEM lane r. Reads S from
//              TMEM, applies prefix bound / ancestor bits and the scale,
//              online softmax in the log2 domain with lazy O rescaling (only
//              when the row max grows by more than 8, i.e. 2^8), writes P as
//              bf16 into a 128B-swizzled shared tile;
//   warp 4     TMA producer: Q once, then K and V tiles into a 2-stage ring;
//   warp 5     TMEM owner and MMA issuer (one thread):
//              S[j&1] = Q K_j^T   (M=128, N=128, K=D; S double-buffered)
//              O     += P_j V_j   (M=128, N=64 per half of D, K=128 keys)
// TMEM: S0 cols [0,128), S1 [128,256), O [256, 256+D) (512 allocated).
// Every mbarrier wait is bounded; on expiry the CTA raises JT_DEVERR_TIMEOUT,
// drains its outstanding MMAs, frees TMEM and finishes.
#include <cooperative_groups.h>
#include <cuda.h>

#include <mutex>

#include "jt_internal.cuh"
#include "jt_sm100.cuh"

namespace jt {
namespace {

namespace cg = cooperative_groups;
using namespace sm100;

constexpr int kThreads = 192;
constexpr int kTile = 128;                 // query rows per unit = keys per tile
constexpr uint32_t kTmemCols = 512;
constexpr long long kWaitBudget = 4000000000LL;   // ~2 s at 2 GHz
constexpr float kRescaleLog2 = 8.0f;

struct AttnParams {
  int batch, B, hq, hkv, g, npt, n_mtiles, S;
  int paged, max_pages, n_pages, Lbound, words;
  const int32_t* block_table;
  const int32_t* prefix_len;
  const int32_t* n_nodes;
  const uint32_t* mask;
  __nv_bfloat16* out;
  float scale_log2;
  int32_t* d_err;
};

struct Bars {
  uint64_t q_full, kv_full[2], kv_empty[2], s_full[2], s_free[2], p_full, pv_done, drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__device__ __forceinline__ void store_row(const AttnParams& p, int b, int kh, int v, int j,
                                          const float* o, float inv) {
  uint4* dst = reinterpret_cast<uint4*>(p.out + (((size_t)b * p.B + v) * p.hq + kh * p.g + j) * D);
#pragma unroll
  for (int u = 0; u < D / 8; ++u) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 two = __floats2bfloat162_rn(o[8 * u + 2 * e] * inv, o[8 * u + 2 * e + 1] * inv);
      w[e] = *reinterpret_cast<uint32_t*>(&two);
    }
    dst[u] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
tree_attn_tc_kernel(const __grid_constant__ CUtensorMap mq, const __grid_constant__ CUtensorMap mkc,
                    const __grid_constant__ CUtensorMap mvc, const __grid_constant__ CUtensorMap mkt,
                    const __grid_constant__ CUtensorMap mvt, const AttnParams p) {
  constexpr int CH = D / 64;               // 64-element (128-byte) chunks of the head dim
  constexpr int QB = kTile * D * 2;        // bytes of one Q, K or V tile
  constexpr int PB = kTile * kTile * 2;    // bytes of the P tile
  constexpr uint32_t kTxKV = 2 * QB;
  constexpr int KS = 4 * CH;               // K=16 steps of Q K^T

  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm;
  uint8_t* sP = sm + 5 * QB;
  Bars* bars = reinterpret_cast<Bars*>(sm + 5 * QB + PB);
  auto sK = [&](int st) { return sm + QB + st * 2 * QB; };
  auto sV = [&](int st) { return sm + 2 * QB + st * 2 * QB; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.S;
  const int rank = (int)(blockIdx.x % (unsigned)S);
  const int unit = (int)(blockIdx.x / (unsigned)S);
  const int mt = unit % p.n_mtiles;
  const int bk = unit / p.n_mtiles;
  const int kh = bk % p.hkv, b = bk / p.hkv;
  const int g = p.g, npt = p.npt;
  const int v0 = mt * npt;

  // ---- validate the sequence (same verdict in every CTA of the sequence) ----
  const int n_raw = p.n_nodes[b];
  const int L = p.prefix_len[b];
  int flag = 0;
  if (n_raw < 0 || n_raw > p.B) flag |= JT_DEVERR_NNODES;
  if (L < 0 || L > p.Lbound) flag |= JT_DEVERR_PREFIX;
  if (p.paged && !(flag & JT_DEVERR_PREFIX)) {
    const int np = (L + kPageSize - 1) / kPageSize;
    for (int i = tid; i < np; i += kThreads) {
      const int pg = p.block_table[(size_t)b * p.max_pages + i];
      if (pg < 0 || pg >= p.n_pages) flag |= JT_DEVERR_PAGE;
    }
  }
  const int bad = __syncthreads_or(flag);
  if (flag && rank == 0) raise_flag(p.d_err, flag);
  const int n = bad ? 0 : n_raw;

  const bool has_rows = v0 < n;
  const int p_tiles = has_rows ? (L + kTile - 1) / kTile : 0;
  const int v_last = min(v0 + npt, n) - 1;
  const int t_tree = has_rows ? (v_last + kTile) / kTile : 0;
  const int t_tot = p_tiles + t_tree;
  const int t_begin = (int)((long)rank * t_tot / S);
  const int t_end = (int)((long)(rank + 1) * t_tot / S);
  const int T = t_end - t_begin;

  if (!has_rows) {
    // Every row of this unit belongs to an unused budget slot: zeros. The
    // cluster's CTAs split the rows; no CTA of the cluster touches DSMEM.
    const int R = kTile / S;
    for (int i = tid; i < R * (D / 8); i += kThreads) {
      const int r = rank * R + i / (D / 8), u = i % (D / 8);
      const int v = v0 + r / g, j = r % g;
      if (v < p.B)
        reinterpret_cast<uint4*>(p.out + (((size_t)b * p.B + v) * p.hq + kh * g + j) * D)[u] =
            make_uint4(0, 0, 0, 0);
    }
    return;
  }

  // ---- set-up: barriers, TMEM ----
  if (tid == 0) {
    mbar_init(&bars->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 4);
    }
    mbar_init(&bars->p_full, 4);
    mbar_init(&bars->pv_done, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  auto fail = [&]() {
    if (atomicExch(&bars->abort, 1) == 0) raise_flag(p.d_err, JT_DEVERR_TIMEOUT);
  };
  // Every lane of the calling warp polls; the verdict is made warp-uniform so
  // that warp-collective tcgen05 / vote instructions never see divergence.
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort, kWaitBudget)) != 0;
  };

  // Valid keys of tile t (prefix tiles first, then tree tiles).
  auto tile_valid = [&](int t) {
    return t < p_tiles ? min(kTile, L - t * kTile) : min(kTile, n - (t - p_tiles) * kTile);
  };

  float o_acc[D];
  float m_run = -INFINITY, l_run = 0.0f;

  if (warp == 4) {
    // =================== TMA producer ===================
    if (lane == 0 && T > 0) {
      tma_prefetch_desc(&mq);
      tma_prefetch_desc(&mkc);
      tma_prefetch_desc(&mvc);
      tma_prefetch_desc(&mkt);
      tma_prefetch_desc(&mvt);
      mbar_arrive_expect_tx(&bars->q_full, QB);
#pragma unroll
      for (int ch = 0; ch < CH; ++ch)
        tma_load_4d(sQ + ch * (kTile * 128), &mq, &bars->q_full, ch * 64, kh * g, v0, b);
      const int np = (L + kPageSize - 1) / kPageSize;
      for (int jt = 0; jt < T; ++jt) {
        const int t = t_begin + jt, st = jt & 1;
        if (jt >= 2 && !mbar_wait(&bars->kv_empty[st], ((jt >> 1) + 1) & 1, abort, kWaitBudget)) {
          fail();
          break;
        }
        mbar_arrive_expect_tx(&bars->kv_full[st], kTxKV);
        uint8_t* dk = sK(st);
        uint8_t* dv = sV(st);
        if (t < p_tiles) {
          const int key0 = t * kTile;
          if (p.paged) {
#pragma unroll 1
            for (int pg = 0; pg < kTile / kPageSize; ++pg) {
              const int pi = key0 / kPageSize + pg;
              const int page = pi < np ? p.block_table[(size_t)b * p.max_pages + pi] : 0;
#pragma unroll
              for (int ch = 0; ch < CH; ++ch) {
                tma_load_4d(dk + ch * (kTile * 128) + pg * (kPageSize * 128), &mkc,
                            &bars->kv_full[st], ch * 64, kh, 0, page);
                tma_load_4d(dv + ch * (kTile * 128) + pg * (kPageSize * 128), &mvc,
                            &bars->kv_full[st], ch * 64, kh, 0, page);
              }
            }
          } else {
#pragma unroll
            for (int ch = 0; ch < CH; ++ch) {
              tma_load_4d(dk + ch * (kTile * 128), &mkc, &bars->kv_full[st], ch * 64, kh, key0, b);
              tma_load_4d(dv + ch * (kTile * 128), &mvc, &bars->kv_full[st], ch * 64, kh, key0, b);
            }
          }
        } else {
          const int u0 = (t - p_tiles) * kTile;
#pragma unroll
          for (int ch = 0; ch < CH; ++ch) {
            tma_load_4d(dk + ch * (kTile * 128), &mkt, &bars->kv_full[st], ch * 64, kh, u0, b);
            tma_load_4d(dv + ch * (kTile * 128), &mvt, &bars->kv_full[st], ch * 64, kh, u0, b);
          }
        }
      }
    }
  } else if (warp == 5) {
    // =================== MMA issuer ===================
    constexpr uint32_t id_s = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t id_o = idesc_bf16(128, 64, 0, 1);
    const uint32_t q_addr = smem_u32(sQ), p_addr = smem_u32(sP);
    auto issue_pv = [&](int jt) {
      const uint32_t v_addr = smem_u32(sV(jt & 1));
#pragma unroll
      for (int h = 0; h < CH; ++h)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t aoff = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
          const uint32_t boff = h * (kTile * 128) + kk * 2048;
          mma_bf16_ss(tmem + 256 + 64 * h, sdesc_sw128(p_addr + aoff, 16, 1024),
                      sdesc_sw128(v_addr + boff, kTile * 128, 1024), id_o, jt > 0 || kk > 0);
        }
      mma_commit(&bars->kv_empty[jt & 1]);
      mma_commit(&bars->pv_done);
    };
    bool ok = T > 0 && warp_wait(&bars->q_full, 0);
    if (T > 0 && !ok) fail();
    for (int jt = 0; ok && jt < T; ++jt) {
      const int st = jt & 1;
      if (!warp_wait(&bars->kv_full[st], (jt >> 1) & 1)) { fail(); ok = false; break; }
      // Rows of V past the tile's valid keys may hold anything (NaN included);
      // P is 0 there, but 0 * NaN is NaN, so zero them before P V reads them.
      const int valid = tile_valid(t_begin + jt);
      if (valid < kTile) {
        uint8_t* vt = sV(st);
        for (int i = lane; i < (kTile - valid) * CH * 8; i += 32) {
          const int r = valid + i / (CH * 8), rem = i % (CH * 8);
          const int ch = rem / 8, u = rem % 8;
          *reinterpret_cast<uint4*>(vt + ch * (kTile * 128) + r * 128 + u * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (jt >= 2 && !warp_wait(&bars->s_free[st], ((jt >> 1) + 1) & 1)) {
        fail(); ok = false; break;
      }
      tc_fence_after();
      if (lane == 0) {
        const uint32_t k_addr = smem_u32(sK(st));
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const uint32_t off = (kk >> 2) * (kTile * 128) + (kk & 3) * 32;
          mma_bf16_ss(tmem + st * 128, sdesc_sw128(q_addr + off, 16, 1024),
                      sdesc_sw128(k_addr + off, 16, 1024), id_s, kk > 0);
        }
        mma_commit(&bars->s_full[st]);
      }
      __syncwarp();
      if (jt >= 1) {
        if (!warp_wait(&bars->p_full, (jt - 1) & 1)) { fail(); ok = false; break; }
        tc_fence_after();
        if (lane == 0) issue_pv(jt - 1);
        __syncwarp();
      }
    }
    if (ok) {
      if (warp_wait(&bars->p_full, (T - 1) & 1)) {
        tc_fence_after();
        if (lane == 0) issue_pv(T - 1);
        __syncwarp();
      } else {
        fail();
      }
    }
  } else {
    // =================== softmax (warps 0-3) ===================
    const int r = tid;
    const int v = v0 + r / g;
    const bool row_valid = v < n;
    uint32_t mrow[kMaxWords];
#pragma unroll
    for (int w = 0; w < kMaxWords; ++w)
      mrow[w] = (row_valid && w < p.words) ? p.mask[((size_t)b * p.B + v) * p.words + w] : 0u;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    uint8_t* prow = sP + r * 128;
    const int rsw = r & 7;
    bool ok = true;
    for (int jt = 0; jt < T; ++jt) {
      const int t = t_begin + jt, sb = jt & 1;
      if (!warp_wait(&bars->s_full[sb], (jt >> 1) & 1)) { fail(); ok = false; break; }
      tc_fence_after();
      float x[kTile];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float tmp[32];
        tmem_ld32(tmem + lane_base + sb * 128 + c * 32, tmp);
#pragma unroll
        for (int i = 0; i < 32; ++i) x[c * 32 + i] = tmp[i];
      }
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->s_free[sb]);
      // Mask and scale into the log2 domain.
      float tmax = -INFINITY;
      if (t < p_tiles) {
        const int kv = L - t * kTile;
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          x[c] = (c < kv) ? x[c] * sl2 : -INFINITY;
          tmax = fmaxf(tmax, x[c]);
        }
      } else {
        const int u0 = (t - p_tiles) * kTile;
        const int wb = u0 >> 5;
        uint32_t wsel[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) wsel[i] = (wb == 0) ? mrow[i] : mrow[4 + i];
        const int ncap = n - u0;
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          const bool vis = ((wsel[c >> 5] >> (c & 31)) & 1u) && c < ncap;
          x[c] = vis ? x[c] * sl2 : -INFINITY;
          tmax = fmaxf(tmax, x[c]);
        }
      }
      const float mnew = fmaxf(m_run, tmax);
      if (jt >= 1) {
        if (!warp_wait(&bars->pv_done, (jt - 1) & 1)) { fail(); ok = false; break; }
        tc_fence_after();
      }
      const bool need = mnew > m_run + kRescaleLog2;
      float corr = 1.0f;
      if (need) {
        corr = (m_run == -INFINITY) ? 0.0f : ex2(m_run - mnew);
        l_run *= corr;
        m_run = mnew;
      }
      if (jt >= 1 && __any_sync(0xFFFFFFFFu, need)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float tmp[32];
          tmem_ld32(tmem + lane_base + 256 + c * 32, tmp);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) tmp[i] *= corr;
          tmem_st32(tmem + lane_base + 256 + c * 32, tmp);
        }
        tmem_wait_st();
      }
      const float muse = (m_run == -INFINITY) ? 0.0f : m_run;
      float lsum = 0.0f;
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = ch * 64 + u * 8 + 2 * e;
            const float p0 = ex2(x[c] - muse), p1 = ex2(x[c + 1] - muse);
            lsum += p0 + p1;
            __nv_bfloat162 two = __floats2bfloat162_rn(p0, p1);
            w[e] = *reinterpret_cast<uint32_t*>(&two);
          }
          *reinterpret_cast<uint4*>(prow + ch * (kTile * 128) + ((u ^ rsw) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      l_run += lsum;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full);
    }
    // Final accumulator.
    if (ok && T > 0 && warp_wait(&bars->pv_done, (T - 1) & 1)) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float tmp[32];
        tmem_ld32(tmem + lane_base + 256 + c * 32, tmp);
#pragma unroll
        for (int i = 0; i < 32; ++i) o_acc[c * 32 + i] = tmp[i];
      }
      tmem_wait_ld();
    } else {
      if (ok && T > 0) fail();
#pragma unroll
      for (int i = 0; i < D; ++i) o_acc[i] = 0.0f;
      if (T == 0) { m_run = -INFINITY; l_run = 0.0f; }
    }
  }

  // ---- release TMEM (after draining outstanding MMAs on the abort path) ----
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    if (*abort && lane == 0) {
      mma_commit(&bars->drain);
      mbar_try_wait(&bars->drain, 0);
      const long long t0 = clock64();
      while (!mbar_try_wait(&bars->drain, 0) && clock64() - t0 < kWaitBudget) {
      }
    }
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
  }

  // ---- output ----
  if (S == 1) {
    if (tid < kTile) {
      const int r = tid, v = v0 + r / g, jh = r % g;
      if (v < p.B) store_row<D>(p, b, kh, v, jh, o_acc, (v < n && l_run > 0.0f) ? 1.0f / l_run : 0.0f);
    }
    return;
  }
  // Split-KV: publish (O, m, l) of every row in shared memory, then rank k
  // merges rows [k*R, (k+1)*R) across the cluster through DSMEM.
  float* o_s = reinterpret_cast<float*>(sm + QB);          // [128][D], over the K/V ring
  float* m_s = o_s + kTile * D;
  float* l_s = m_s + kTile;
  float* fac = l_s + kTile;                                 // [R][S] = 128 floats
  if (tid < kTile) {
#pragma unroll
    for (int i = 0; i < D; i += 4)
      *reinterpret_cast<float4*>(o_s + tid * D + i) =
          make_float4(o_acc[i], o_acc[i + 1], o_acc[i + 2], o_acc[i + 3]);
    m_s[tid] = m_run;
    l_s[tid] = l_run;
  }
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  const int R = kTile / S;
  if (tid < R) {
    const int row = rank * R + tid;
    float M = -INFINITY;
    for (int s = 0; s < S; ++s) M = fmaxf(M, cluster.map_shared_rank(m_s, s)[row]);
    float lsum = 0.0f;
    for (int s = 0; s < S; ++s) {
      const float ms = cluster.map_shared_rank(m_s, s)[row];
      const float f = (ms == -INFINITY) ? 0.0f : ex2(ms - M);
      fac[tid * S + s] = f;
      lsum += f * cluster.map_shared_rank(l_s, s)[row];
    }
    const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
    for (int s = 0; s < S; ++s) fac[tid * S + s] *= inv;
  }
  __syncthreads();
  for (int i = tid; i < R * (D / 8); i += kThreads) {
    const int rl = i / (D / 8), u = i % (D / 8);
    const int row = rank * R + rl;
    const int v = v0 + row / g, jh = row % g;
    if (v >= p.B) continue;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    if (v < n) {
      for (int s = 0; s < S; ++s) {
        const float f = fac[rl * S + s];
        const float4* src = reinterpret_cast<const float4*>(cluster.map_shared_rank(o_s, s) + row * D + u * 8);
        const float4 a = src[0], c4 = src[1];
        acc[0] += f * a.x; acc[1] += f * a.y; acc[2] += f * a.z; acc[3] += f * a.w;
        acc[4] += f * c4.x; acc[5] += f * c4.y; acc[6] += f * c4.z; acc[7] += f * c4.w;
      }
    }
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      __nv_bfloat162 two = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
      w[e] = *reinterpret_cast<uint32_t*>(&two);
    }
    reinterpret_cast<uint4*>(p.out + (((size_t)b * p.B + v) * p.hq + kh * g + jh) * D)[u] =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
  cluster.sync();  // keep this CTA's shared memory alive until every rank has read it
}

// ---------------------------------------------------------------------------
// Host side: tensor maps, split choice, launch.
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 4-D bf16 map, dims innermost first, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, const uint64_t (&dims)[4],
              const uint32_t (&box)[4]) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t gd[4], gs[3];
  cuuint32_t bx[4], es[4] = {1, 1, 1, 1};
  for (int i = 0; i < 4; ++i) { gd[i] = dims[i] ? dims[i] : 1; bx[i] = box[i]; }
  gs[0] = gd[0] * 2;
  gs[1] = gs[0] * gd[1];
  gs[2] = gs[1] * gd[2];
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gd, gs, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
size_t smem_bytes() { return 5 * (size_t)kTile * D * 2 + (size_t)kTile * kTile * 2 + 256 + 1024; }

template <int D>
cudaError_t launch_d(const Ctx& c, const jt_attn_args& a, AttnParams& p) {
  const size_t smem = smem_bytes<D>();
  auto kern = tree_attn_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;

  const int units = a.batch * a.hkv * p.n_mtiles;
  const int tiles_max = (p.Lbound + kTile - 1) / kTile + (a.B + kTile - 1) / kTile;
  int S = 1;
  while (S < 16 && units * S * 2 <= c.num_sms && S * 2 <= tiles_max) S *= 2;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  while (S > 1) {  // largest split the hardware can co-schedule as a cluster
    attr[0].val.clusterDim.x = S;
    cfg.gridDim = dim3(units * S);
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, kern, &cfg) == cudaSuccess && nclusters > 0)
      break;
    cudaGetLastError();
    S >>= 1;
  }
  p.S = S;
  attr[0].val.clusterDim.x = S;
  cfg.gridDim = dim3(units * S);

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
  return cudaLaunchKernelEx(&cfg, kern, mq, mkc, mvc, mkt, mvt, p);
}

}  // namespace

size_t attn_workspace_bytes(const jt_attn_args& a, int num_sms) {
  (void)a;
  (void)num_sms;
  return 0;
}

cudaError_t launch_tree_attn(const Ctx& c, const jt_attn_args& a) {
  if (a.batch == 0) return cudaSuccess;
  AttnParams p = {};
  p.batch = a.batch;
  p.B = a.B;
  p.hq = a.hq;
  p.hkv = a.hkv;
  p.g = a.hq / a.hkv;
  p.npt = kTile / p.g;
  p.n_mtiles = (a.B + p.npt - 1) / p.npt;
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
  p.d_err = c.d_err;
  return a.head_dim == 64 ? launch_d<64>(c, a, p) : launch_d<128>(c, a, p);
}

}  // namespace jt
