// jt_topw: top-W draft candidates and their log-probabilities per depth.
//
// The proposer takes the top-k tokens and their log-probabilities at every
// future position (JetSpec summary on paperlayer.ai, App. E "Drafting"; the
// Chinese summary on paper.rainbus.top, "方法步骤详情": top-W candidates per
// depth from one draft pass). logp = x - m - log(sum_j exp(x_j - m)) over
// the full vocabulary; ranking (x desc, token id asc).
//
// The row is read exactly once: the top-W selection and the log-sum-exp run
// in the same pass (jt_rowscan.cuh), and so does the entropy of the depth's
// draft distribution when it is asked for (entropy-guided and hybrid tree
// scores, paperlayer.ai App. C "Tree-Drafting Algorithm Ablation" and App. E
// "Drafting"): H = ln s - ln2 * t / s from the same online sums. Rows are split over a thread-block
// cluster when there are too few rows to fill the GPU (batch 1: 16 rows of
// 151936 logits -> 16-CTA clusters), and the cluster merges its partials in
// distributed shared memory.
#include <atomic>

#include "jt_rowscan.cuh"

namespace jt {
namespace {

// NST > 0: the streaming scan stages its batches in an NST-stage shared-
// memory ring (dynamic shared memory) instead of registers.
template <int K, bool ENT, bool RES, int NST>
__global__ void __launch_bounds__(kScanThreads)
topw_kernel(const float* __restrict__ logits, int V, int W, int S, int32_t* __restrict__ tok,
            float* __restrict__ logp, float* __restrict__ entropy) {
  __shared__ ScanPartial<K> warp_parts[kScanWarps];
  __shared__ ScanPartial<K> part;
  extern __shared__ __align__(16) float4 ring[];
  const int row = blockIdx.x / S;
  const int seg = blockIdx.x % S;
  const int v4 = V >> 2;
  const int per = (v4 + S - 1) / S;
  const int lo = min(v4, seg * per), hi = min(v4, lo + per);
  grid_dependency_sync();
  if constexpr (NST > 0)
    scan_to_partial_ring<K, true, ENT, NST>(logits + (size_t)row * V, lo, hi, &part, warp_parts,
                                            ring);
  else
    scan_to_partial<K, true, ENT, RES>(logits + (size_t)row * V, lo, hi, &part, warp_parts);
  TopK<K> top;
  Lse lse;
  if (cluster_reduce<K, true>(&part, S, top, lse)) {
    // lse.m is the max of x*log2(e) and lse.s = sum 2^(x*log2(e) - m), so
    // ln Z = m * ln 2 + ln s.
    const float ln_s = logf(lse.s);
    const float lnZ = fmaf(lse.m, 0.6931471805599453f, ln_s);
#pragma unroll
    for (int k = 0; k < K; ++k) {
      if (k < W) {
        tok[(size_t)row * W + k] = top.i[k];
        logp[(size_t)row * W + k] = top.v[k] - lnZ;
      }
    }
    if (ENT)
      entropy[row] = lse.s > 0.0f ? fmaf(-0.6931471805599453f, lse.t / lse.s, ln_s) : 0.0f;
  }
}

// The shared-memory ring: kRingStages batches of 16 KB per CTA, two CTAs per
// SM. It is used for streaming scans whose rows fill at most two CTAs per SM
// (one wave of few, long segments), where the two register batches of the
// plain streaming scan keep too few bytes in flight per CTA; such rows are
// then cut into as many segments as keep that bound.
constexpr int kRingStages = 6;
constexpr int kRingCtasPerSm = 2;

template <int K, bool ENT>
cudaError_t launch_ring(const Ctx& c, const float* logits, int rows, int V, int W, int S,
                        int32_t* tok, float* logp, float* entropy) {
  auto kern = topw_kernel<K, ENT, false, kRingStages>;
  constexpr size_t smem = ring_smem_bytes<kRingStages>();
  // Devices 0..63 the shared-memory limit was raised on (others raise it on
  // every launch).
  static std::atomic<uint64_t> opted{0};
  const uint64_t bit = (c.device >= 0 && c.device < 64) ? 1ull << c.device : 0ull;
  if (!bit || !(opted.load(std::memory_order_relaxed) & bit)) {
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    opted.fetch_or(bit, std::memory_order_relaxed);
  }
  return launch_kernel(kern, dim3(rows * S), dim3(kScanThreads), smem, c.stream, S, logits, V, W,
                       S, tok, logp, entropy);
}

template <int K>
cudaError_t launch_k(const Ctx& c, const float* logits, int rows, int V, int W, int32_t* tok,
                     float* logp, float* entropy) {
  const int v4 = V / 4;
  const long ring_ctas = (long)kRingCtasPerSm * c.num_sms;
  if (K <= 16 && rows <= ring_ctas) {   // (K = 32 takes too many registers for two CTAs per SM)
    const int S = pick_row_split(rows, v4, c.num_sms, 16);
    int Sr = 1;
    while (2 * Sr <= S && (long)rows * 2 * Sr <= ring_ctas) Sr *= 2;
    if (!use_resident(K, (v4 + Sr - 1) / Sr))
      return entropy ? launch_ring<K, true>(c, logits, rows, V, W, Sr, tok, logp, entropy)
                     : launch_ring<K, false>(c, logits, rows, V, W, Sr, tok, logp, entropy);
  }
  const int S = pick_row_split(rows, v4, c.num_sms, 16);
  const bool res = use_resident(K, (v4 + S - 1) / S);
  auto kern = entropy ? (res ? topw_kernel<K, true, true, 0> : topw_kernel<K, true, false, 0>)
                      : (res ? topw_kernel<K, false, true, 0> : topw_kernel<K, false, false, 0>);
  return launch_clustered(kern, rows * S, S, c.stream, logits, V, W, S, tok, logp, entropy);
}

}  // namespace

cudaError_t launch_topw(const Ctx& c, const float* logits, int rows, int V, int W, int32_t* tok,
                        float* logp, float* entropy) {
  if (rows == 0) return cudaSuccess;
  if (W <= 1) return launch_k<1>(c, logits, rows, V, W, tok, logp, entropy);
  if (W <= 2) return launch_k<2>(c, logits, rows, V, W, tok, logp, entropy);
  if (W <= 4) return launch_k<4>(c, logits, rows, V, W, tok, logp, entropy);
  if (W <= 8) return launch_k<8>(c, logits, rows, V, W, tok, logp, entropy);
  if (W <= 16) return launch_k<16>(c, logits, rows, V, W, tok, logp, entropy);
  return launch_k<32>(c, logits, rows, V, W, tok, logp, entropy);
}

}  // namespace jt
