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
#include "jt_rowscan.cuh"

namespace jt {
namespace {

template <int K, bool ENT, bool RES>
__global__ void __launch_bounds__(kScanThreads)
topw_kernel(const float* __restrict__ logits, int V, int W, int S, int32_t* __restrict__ tok,
            float* __restrict__ logp, float* __restrict__ entropy) {
  __shared__ ScanPartial<K> warp_parts[kScanWarps];
  __shared__ ScanPartial<K> part;
  const int row = blockIdx.x / S;
  const int seg = blockIdx.x % S;
  const int v4 = V >> 2;
  const int per = (v4 + S - 1) / S;
  const int lo = min(v4, seg * per), hi = min(v4, lo + per);
  grid_dependency_sync();
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

template <int K>
cudaError_t launch_k(const Ctx& c, const float* logits, int rows, int V, int W, int32_t* tok,
                     float* logp, float* entropy) {
  const int S = pick_row_split(rows, V / 4, c.num_sms, 16);
  const bool res = use_resident(K, (V / 4 + S - 1) / S);
  auto kern = entropy ? (res ? topw_kernel<K, true, true> : topw_kernel<K, true, false>)
                      : (res ? topw_kernel<K, false, true> : topw_kernel<K, false, false>);
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
