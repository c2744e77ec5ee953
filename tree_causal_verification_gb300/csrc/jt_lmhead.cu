// jt_lmhead_topw: draft logits through the LM head, reduced to the top-W
// tokens, their log-probs and (optionally) the entropy of every row, without
// writing the logits.
//
// JetSpec summary on paperlayer.ai, App. E "Training and evaluation details":
// the draft model reuses the frozen target LM head, so a depth's draft logits
// are its hidden state times the LM-head matrix; App. E "Drafting": the
// proposer keeps the top-k tokens and log-probs at every future position.
//
// GPU design (sm_100 family): logits = hidden [R][d] x w_lm [V][d]^T with
// bf16 operands and fp32 accumulation in TMEM. One block computes a 128-row x
// 512-vocab tile (two M128 x N256 accumulators, all 512 TMEM columns),
// streaming d in 64-wide chunks through a 2-stage TMA ring (A 16 KB + B 2 x
// 32 KB per stage, 128-byte swizzle, K-major); one thread issues the MMAs.
// Epilogue threads own one row each (TMEM lane = row) and reduce the tile's
// 512 logits to a sorted top-K list and the online log-sum-exp (and entropy
// sum) of jt_rowscan.cuh, written as one small partial per (row, vocabulary
// slice). A second kernel merges each row's partials over all slices (one
// warp per row). Blocks that share a vocabulary slice are adjacent in the
// grid (row tiles fastest), so a slice's weights come from HBM once and from
// L2 for the other row tiles.
#include "jt_rowscan.cuh"
#include "jt_sm100.cuh"
#include "jt_tmamap.h"

namespace jt {
namespace {

using namespace sm100;

constexpr int kLmThreads = 192;            // warps 0-3 epilogue, 4 TMA producer, 5 MMA issuer
constexpr int kLmRows = 128;               // rows per block (MMA M)
constexpr int kLmN = 256;                  // vocabulary per accumulator (MMA N)
constexpr int kLmVocab = 2 * kLmN;         // vocabulary per block
constexpr int kLmK = 64;                   // d per stage: one 128-byte swizzle row
constexpr int kLmStages = 2;
constexpr int kLmABytes = kLmRows * kLmK * 2;
constexpr int kLmBBytes = kLmN * kLmK * 2;
constexpr int kLmStageBytes = kLmABytes + 2 * kLmBBytes;
constexpr uint32_t kLmTmemCols = 512;
constexpr int kMergeWarps = 8;

struct LmBars {
  uint64_t full[kLmStages], empty[kLmStages], done;
  uint32_t tmem_base;
  int abort;
};

size_t lm_smem_bytes() { return (size_t)kLmStages * kLmStageBytes + sizeof(LmBars) + 1024; }

template <int K, bool ENT>
__global__ void __launch_bounds__(kLmThreads, 1)
lmhead_tile_kernel(const __grid_constant__ CUtensorMap ma, const __grid_constant__ CUtensorMap mb,
                   int R, int d, int V, int m_tiles, int n_slices, long long budget,
                   ScanPartial<K>* __restrict__ part, int32_t* d_err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  LmBars* bars = reinterpret_cast<LmBars*>(sm + kLmStages * kLmStageBytes);
  auto sA = [&](int st) { return sm + st * kLmStageBytes; };
  auto sB = [&](int st, int n) { return sm + st * kLmStageBytes + kLmABytes + n * kLmBBytes; };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = (int)(blockIdx.x / (unsigned)m_tiles), mt = (int)(blockIdx.x % (unsigned)m_tiles);
  const int r0 = mt * kLmRows, v0 = slice * kLmVocab, nk = d / kLmK;

  if (tid == 0) {
    for (int i = 0; i < kLmStages; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    mbar_init(&bars->done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, kLmTmemCols);
    tmem_relinquish();
  }
  grid_dependency_sync();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  auto fail = [&]() {
    if (atomicExch(&bars->abort, 1) == 0) raise_flag(d_err, JT_DEVERR_TIMEOUT);
  };

  int issued = 0;   // producer: stages of A/B loads issued
  if (warp == 4) {
    // ---- TMA producer ----
    if (lane == 0) {
      tma_prefetch_desc(&ma);
      tma_prefetch_desc(&mb);
      for (int c = 0; c < nk; ++c) {
        const int st = c % kLmStages;
        if (c >= kLmStages &&
            !mbar_wait(&bars->empty[st], ((c / kLmStages) + 1) & 1, abort, budget)) {
          fail();
          break;
        }
        mbar_arrive_expect_tx(&bars->full[st], kLmStageBytes);
        issued = c + 1;
        tma_load_4d(sA(st), &ma, &bars->full[st], c * kLmK, r0, 0, 0);
        tma_load_4d(sB(st, 0), &mb, &bars->full[st], c * kLmK, v0, 0, 0);
        tma_load_4d(sB(st, 1), &mb, &bars->full[st], c * kLmK, v0 + kLmN, 0, 0);
      }
    }
  } else if (warp == 5) {
    // ---- MMA issuer: D_n += A B_n^T, n = 0, 1 (K-major operands, K = 16 per MMA) ----
    // The whole warp runs the loop; elect.sync inside each MMA / commit picks
    // the issuing lane (the same one every time), so no divergent branch
    // surrounds the issue.
    constexpr uint32_t idesc = idesc_bf16(kLmRows, kLmN, 0, 0);
    for (int c = 0; c < nk; ++c) {
      const int st = c % kLmStages;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(&bars->full[st], (c / kLmStages) & 1, abort, budget))) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const uint64_t a = sdesc_sw128(smem_u32(sA(st)), 16, 1024);
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        const uint64_t bdesc = sdesc_sw128(smem_u32(sB(st, n)), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kLmK / 16; ++kk)   // +32 bytes along K = +2 in the descriptor
          mma_bf16_ss_warp(tmem + n * kLmN, a + 2 * kk, bdesc + 2 * kk, idesc, c > 0 || kk > 0);
      }
      mma_commit_warp(&bars->empty[st]);
    }
    mma_commit_warp(&bars->done);   // also after a failure: completes once issued MMAs retire
    __syncwarp();
  } else {
    // ---- epilogue: thread tid owns row r0 + tid (TMEM lane tid) ----
    TopK<K> top;
    top.init();
    Lse lse;
    lse.init();
    // After a failure elsewhere in the CTA the accumulators are incomplete:
    // the partial then holds no candidates (defined, and flagged).
    const bool done = __all_sync(0xFFFFFFFFu, mbar_wait(&bars->done, 0, abort, budget)) != 0;
    if (!done) fail();
    const bool ok = __all_sync(0xFFFFFFFFu, done && !*abort) != 0;
    tc_fence_after();
    const int row = r0 + tid;
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    if (ok) {
#pragma unroll 1
      for (int c = 0; c < kLmVocab / 32; ++c) {
        float x[32];
        tmem_ld32(tmem + lane_base + c * 32, x);
        tmem_wait_ld();
        const int vb = v0 + c * 32;
        float mx = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          if (vb + i >= V) x[i] = -INFINITY;   // vocabulary past V (zero-filled weights)
          mx = fmaxf(mx, x[i]);
        }
        if (row < R && mx != -INFINITY) {
          const float bm2 = mx * kLog2e;
          if (bm2 > lse.m) lse.raise<ENT>(bm2);
          const float nm = -lse.m;
          float a0 = 0.0f, tacc = 0.0f;
#pragma unroll
          for (int i = 0; i < 32; ++i) a0 += lse.term<ENT>(fmaf(x[i], kLog2e, nm), tacc);
          lse.s += a0;
          if (ENT) lse.t += tacc;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (vb + i < V) top.push(x[i], vb + i);
        }
      }
    }
    if (row < R) {
      ScanPartial<K> q;
#pragma unroll
      for (int k = 0; k < K; ++k) {
        const bool real = k < top.n;
        q.v[k] = real ? top.v[k] : -INFINITY;
        q.i[k] = real ? top.i[k] : INT_MAX;
      }
      q.m = lse.m;
      q.s = lse.s;
      q.t = lse.t;
      part[(size_t)row * n_slices + slice] = q;
    }
  }

  tc_fence_before();
  __syncthreads();
  // After a failed wait (all of them precede the barrier above) TMA loads
  // may still be landing in shared memory: the producer waits for the last
  // load of each stage (earlier ones were consumed) before the CTA exits.
  if (*abort && warp == 4 && lane == 0) {
    for (int st = 0; st < kLmStages; ++st) {
      if (issued > st) {
        const int last = st + kLmStages * ((issued - 1 - st) / kLmStages);
        mbar_wait_drain(&bars->full[st], (last / kLmStages) & 1, kDefaultWaitBudget);
      }
    }
  }
  if (warp == 5) {
    tc_fence_after();
    if (*abort && lane == 0)   // retire every issued MMA before TMEM is released
      mbar_wait_drain(&bars->done, 0, kDefaultWaitBudget);
    __syncwarp();
    tmem_dealloc(tmem, kLmTmemCols);
  }
}

// One warp per row: lane l merges the partials of slices l, l+32, ... (their
// vocabulary ranges increase, as TopK requires), then K rounds of warp argmax.
template <int K, bool ENT>
__global__ void __launch_bounds__(kMergeWarps * 32)
lmhead_merge_kernel(const ScanPartial<K>* __restrict__ part, int R, int n_slices, int W,
                    int32_t* __restrict__ tok, float* __restrict__ logp,
                    float* __restrict__ entropy) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kMergeWarps + warp;
  if (row >= R) return;
  grid_dependency_sync();
  TopK<K> top;
  top.init();
  Lse lse;
  lse.init();
  for (int sl = lane; sl < n_slices; sl += 32) {
    const ScanPartial<K>& q = part[(size_t)row * n_slices + sl];
#pragma unroll
    for (int k = 0; k < K; ++k)
      if (q.i[k] != INT_MAX) top.push(q.v[k], q.i[k]);
    lse.combine(q.m, q.s, q.t);
  }
  float wv[K];
  int wi[K];
  warp_select<K, K>(top.v, top.i, min(top.n, K), wv, wi);
  lse.warp_reduce();
  if (lane == 0) {
    const float ln_s = logf(lse.s);
    const float lnZ = fmaf(lse.m, 0.6931471805599453f, ln_s);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (k < W) {
        tok[(size_t)row * W + k] = wi[k];
        logp[(size_t)row * W + k] = wv[k] - lnZ;
      }
    }
    if (ENT) entropy[row] = lse.s > 0.0f ? fmaf(-0.6931471805599453f, lse.t / lse.s, ln_s) : 0.0f;
  }
}

int pow2_k(int W) {
  int k = 1;
  while (k < W) k <<= 1;
  return k;
}

template <int K, bool ENT>
cudaError_t launch_k(const Ctx& c, const void* hidden, const void* w_lm, int R, int d, int V,
                     int W, int32_t* tok, float* logp, float* entropy) {
  const int m_tiles = (R + kLmRows - 1) / kLmRows;
  const int n_slices = (V + kLmVocab - 1) / kLmVocab;
  CUtensorMap ma, mb;
  if (!make_map(&ma, hidden, {(uint64_t)d, (uint64_t)R, 1, 1}, {kLmK, kLmRows, 1, 1}) ||
      !make_map(&mb, w_lm, {(uint64_t)d, (uint64_t)V, 1, 1}, {kLmK, kLmN, 1, 1}))
    return cudaErrorInvalidValue;
  auto part = static_cast<ScanPartial<K>*>(c.workspace);
  auto tile = lmhead_tile_kernel<K, ENT>;
  cudaError_t e = cudaFuncSetAttribute(tile, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)lm_smem_bytes());
  if (e != cudaSuccess) return e;
  e = launch_kernel(tile, dim3(m_tiles * n_slices), dim3(kLmThreads), lm_smem_bytes(), c.stream, 1,
                    ma, mb, R, d, V, m_tiles, n_slices, wait_budget(), part, c.d_err);
  if (e != cudaSuccess) return e;
  return launch_kernel(lmhead_merge_kernel<K, ENT>, dim3((R + kMergeWarps - 1) / kMergeWarps),
                       dim3(kMergeWarps * 32), 0, c.stream, 1, (const ScanPartial<K>*)part, R,
                       n_slices, W, tok, logp, entropy);
}

template <int K>
cudaError_t launch_e(const Ctx& c, const void* hidden, const void* w_lm, int R, int d, int V,
                     int W, int32_t* tok, float* logp, float* entropy) {
  return entropy ? launch_k<K, true>(c, hidden, w_lm, R, d, V, W, tok, logp, entropy)
                 : launch_k<K, false>(c, hidden, w_lm, R, d, V, W, tok, logp, entropy);
}

}  // namespace

size_t lmhead_workspace_bytes(int R, int V, int W) {
  const size_t slices = (size_t)((V + kLmVocab - 1) / kLmVocab);
  const int K = pow2_k(W);
  const size_t per = 2 * sizeof(float) * K + 3 * sizeof(float);   // sizeof(ScanPartial<K>)
  return align_up((size_t)R * slices * per, 256);
}

cudaError_t launch_lmhead_topw(const Ctx& c, const void* hidden, const void* w_lm, int R, int d,
                               int V, int W, int32_t* tok, float* logp, float* entropy) {
  if (R == 0) return cudaSuccess;
  switch (pow2_k(W)) {
    case 1: return launch_e<1>(c, hidden, w_lm, R, d, V, W, tok, logp, entropy);
    case 2: return launch_e<2>(c, hidden, w_lm, R, d, V, W, tok, logp, entropy);
    case 4: return launch_e<4>(c, hidden, w_lm, R, d, V, W, tok, logp, entropy);
    case 8: return launch_e<8>(c, hidden, w_lm, R, d, V, W, tok, logp, entropy);
    case 16: return launch_e<16>(c, hidden, w_lm, R, d, V, W, tok, logp, entropy);
    default: return launch_e<32>(c, hidden, w_lm, R, d, V, W, tok, logp, entropy);
  }
}

}  // namespace jt
