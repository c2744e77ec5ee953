// libjtree C ABI: host-side argument validation and dispatch to the kernels.
// Declarations and the contract of every call: include/jtree.h.
#include <atomic>
#include <mutex>

#include "jt_internal.cuh"

namespace jt {

namespace {
std::atomic<long long> g_wait_budget{kDefaultWaitBudget};
}  // namespace

long long wait_budget() { return g_wait_budget.load(std::memory_order_relaxed); }

int device_sm_count(int device) {
  static std::mutex mu;
  static int cached[64] = {0};
  if (device < 0 || device >= 64) return kNumSMs;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || n <= 0)
      n = kNumSMs;
    cached[device] = n;
  }
  return cached[device];
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

jt_status make_ctx(const jt_exec* exec, Ctx* c) {
  c->stream = exec ? reinterpret_cast<cudaStream_t>(exec->stream) : nullptr;
  c->d_err = exec ? exec->d_err : nullptr;
  c->workspace = exec ? exec->workspace : nullptr;
  c->workspace_bytes = exec ? exec->workspace_bytes : 0;
  if (c->d_err && (reinterpret_cast<uintptr_t>(c->d_err) & 3u)) return JT_ERR_INVALID_ARG;
  if (cudaGetDevice(&c->device) != cudaSuccess) return JT_ERR_CUDA;
  c->num_sms = device_sm_count(c->device);
  return JT_OK;
}

jt_status need_workspace(const Ctx& c, size_t bytes) {
  if (bytes == 0) return JT_OK;
  if (!c.workspace || c.workspace_bytes < bytes) return JT_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(c.workspace) & 255u) return JT_ERR_INVALID_ARG;
  return JT_OK;
}

jt_status from_cuda(cudaError_t e) { return e == cudaSuccess ? JT_OK : JT_ERR_CUDA; }

}  // namespace
}  // namespace jt

using namespace jt;

extern "C" {

const char* jt_status_str(jt_status s) {
  switch (s) {
    case JT_OK: return "JT_OK";
    case JT_ERR_INVALID_ARG: return "JT_ERR_INVALID_ARG: bad argument (null, size or alignment)";
    case JT_ERR_UNSUPPORTED: return "JT_ERR_UNSUPPORTED: request outside what the library implements";
    case JT_ERR_CUDA: return "JT_ERR_CUDA: a CUDA call or kernel launch failed";
    case JT_ERR_DEVICE_DATA: return "JT_ERR_DEVICE_DATA: a device-side data check failed";
    case JT_ERR_TIMEOUT: return "JT_ERR_TIMEOUT: a bounded device-side wait expired";
    case JT_ERR_WORKSPACE: return "JT_ERR_WORKSPACE: workspace missing or too small";
  }
  return "unknown jt_status";
}

jt_status jt_read_device_error(const jt_exec* exec, int32_t* host_out) {
  if (!exec || !exec->d_err || !host_out) return JT_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(exec->stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, exec->d_err, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return JT_ERR_CUDA;
  if (cudaMemsetAsync(exec->d_err, 0, sizeof v, s) != cudaSuccess) return JT_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return JT_ERR_CUDA;
  *host_out = v;
  if (v == 0) return JT_OK;
  return (v & JT_DEVERR_TIMEOUT) ? JT_ERR_TIMEOUT : JT_ERR_DEVICE_DATA;
}

jt_status jt_set_wait_budget(long long cycles) {
  g_wait_budget.store(cycles > 0 ? cycles : kDefaultWaitBudget, std::memory_order_relaxed);
  return JT_OK;
}

size_t jt_topw_workspace_bytes(int batch, int n_depth, int vocab, int W) {
  (void)batch; (void)n_depth; (void)vocab; (void)W;
  return 0;
}

namespace {

jt_status topw_impl(const float* logits, int batch, int n_depth, int vocab, int W, int32_t* tok,
                    float* logp, float* entropy, const jt_exec* exec) {
  if (batch < 0 || n_depth < 0 || vocab <= 0 || W < 1 || W > kMaxW || W > vocab)
    return JT_ERR_INVALID_ARG;
  if (vocab % 4 != 0) return JT_ERR_UNSUPPORTED;
  const long rows = (long)batch * n_depth;
  if (rows * 16 > 0x7FFFFFFFL) return JT_ERR_UNSUPPORTED;
  if (rows > 0 && (!logits || !tok || !logp)) return JT_ERR_INVALID_ARG;
  if (!aligned16(logits) || !aligned16(tok) || !aligned16(logp) || !aligned16(entropy))
    return JT_ERR_INVALID_ARG;
  Ctx c;
  jt_status st = make_ctx(exec, &c);
  if (st != JT_OK) return st;
  return from_cuda(launch_topw(c, logits, (int)rows, vocab, W, tok, logp, entropy));
}

jt_status expand_impl(const int32_t* tok, const float* logp, const float* entropy, int batch,
                      int n_depth, int W, int B, int mode, float alpha, int32_t* parent,
                      int32_t* token, int32_t* depth, float* score, int32_t* n_nodes,
                      const jt_exec* exec) {
  if (batch < 0 || n_depth < 1 || n_depth > kMaxDepth || W < 1 || W > kMaxW || B < 1 || B > kMaxB)
    return JT_ERR_INVALID_ARG;
  if (mode < JT_SCORE_LOGP || mode > JT_SCORE_ENTROPY) return JT_ERR_INVALID_ARG;
  if (mode == JT_SCORE_HYBRID && !(alpha >= 0.0f && alpha <= 3.0e38f)) return JT_ERR_INVALID_ARG;
  if (batch > 0 && (!tok || !logp || !parent || !token || !depth || !score || !n_nodes ||
                    (mode != JT_SCORE_LOGP && !entropy)))
    return JT_ERR_INVALID_ARG;
  const void* ptrs[] = {tok, logp, entropy, parent, token, depth, score, n_nodes};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JT_ERR_INVALID_ARG;
  Ctx c;
  jt_status st = make_ctx(exec, &c);
  if (st != JT_OK) return st;
  return from_cuda(launch_tree_expand(c, tok, logp, mode == JT_SCORE_LOGP ? nullptr : entropy,
                                      mode, alpha, batch, n_depth, W, B, parent, token, depth,
                                      score, n_nodes));
}

}  // namespace

jt_status jt_topw(const float* logits, int batch, int n_depth, int vocab, int W, int32_t* tok,
                  float* logp, const jt_exec* exec) {
  return topw_impl(logits, batch, n_depth, vocab, W, tok, logp, nullptr, exec);
}

jt_status jt_topw_entropy(const float* logits, int batch, int n_depth, int vocab, int W,
                          int32_t* tok, float* logp, float* entropy, const jt_exec* exec) {
  if ((long)batch * n_depth > 0 && !entropy) return JT_ERR_INVALID_ARG;
  return topw_impl(logits, batch, n_depth, vocab, W, tok, logp, entropy, exec);
}

jt_status jt_tree_expand(const int32_t* tok, const float* logp, int batch, int n_depth, int W,
                         int B, int32_t* parent, int32_t* token, int32_t* depth, float* score,
                         int32_t* n_nodes, const jt_exec* exec) {
  return expand_impl(tok, logp, nullptr, batch, n_depth, W, B, JT_SCORE_LOGP, 0.0f, parent, token,
                     depth, score, n_nodes, exec);
}

jt_status jt_tree_expand_scored(const int32_t* tok, const float* logp, const float* entropy,
                                int batch, int n_depth, int W, int B, int mode, float alpha,
                                int32_t* parent, int32_t* token, int32_t* depth, float* score,
                                int32_t* n_nodes, const jt_exec* exec) {
  return expand_impl(tok, logp, entropy, batch, n_depth, W, B, mode, alpha, parent, token, depth,
                     score, n_nodes, exec);
}

jt_status jt_tree_mask(const int32_t* parent, const int32_t* n_nodes, int batch, int B,
                       uint32_t* mask, const jt_exec* exec) {
  if (batch < 0 || B < 1 || B > kMaxB) return JT_ERR_INVALID_ARG;
  if (batch > 0 && (!parent || !n_nodes || !mask)) return JT_ERR_INVALID_ARG;
  if (!aligned16(parent) || !aligned16(n_nodes) || !aligned16(mask)) return JT_ERR_INVALID_ARG;
  Ctx c;
  jt_status st = make_ctx(exec, &c);
  if (st != JT_OK) return st;
  return from_cuda(launch_tree_mask(c, parent, n_nodes, batch, B, mask));
}

static jt_status check_attn(const jt_attn_args* a) {
  if (!a) return JT_ERR_INVALID_ARG;
  if (a->batch < 0 || a->B < 1 || a->B > kMaxB || a->hq < 1 || a->hkv < 1 || a->hq % a->hkv)
    return JT_ERR_INVALID_ARG;
  if (a->head_dim != 64 && a->head_dim != 128) return JT_ERR_UNSUPPORTED;
  if (!(a->scale >= 0.0f)) return JT_ERR_INVALID_ARG;  // negative or NaN
  if (a->hq / a->hkv > 16 || 128 % (a->hq / a->hkv) != 0) return JT_ERR_UNSUPPORTED;
  if (a->batch == 0) return JT_OK;
  if (!a->q || !a->k_tree || !a->v_tree || !a->k_cache || !a->v_cache || !a->prefix_len ||
      !a->n_nodes || !a->mask || !a->out)
    return JT_ERR_INVALID_ARG;
  const void* ptrs[] = {a->q, a->k_tree, a->v_tree, a->k_cache, a->v_cache, a->prefix_len,
                        a->n_nodes, a->mask, a->out, a->block_table};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JT_ERR_INVALID_ARG;
  if (a->block_table) {
    if (a->page_size != kPageSize) return JT_ERR_UNSUPPORTED;
    if (a->max_pages < 1 || a->n_pages < 1) return JT_ERR_INVALID_ARG;
  } else if (a->max_prefix < 0) {
    return JT_ERR_INVALID_ARG;
  }
  return JT_OK;
}

size_t jt_tree_attn_workspace_bytes(const jt_attn_args* args) {
  if (check_attn(args) != JT_OK) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  return attn_workspace_bytes(*args, device_sm_count(dev));
}

jt_status jt_tree_attn(const jt_attn_args* args, const jt_exec* exec) {
  jt_status st = check_attn(args);
  if (st != JT_OK) return st;
  Ctx c;
  st = make_ctx(exec, &c);
  if (st != JT_OK) return st;
  st = need_workspace(c, attn_workspace_bytes(*args, c.num_sms));
  if (st != JT_OK) return st;
  return from_cuda(launch_tree_attn(c, *args));
}

jt_status jt_tree_commit_kv(const jt_commit_args* a, const jt_exec* exec) {
  if (!a) return JT_ERR_INVALID_ARG;
  if (a->batch < 0 || a->B < 1 || a->B > kMaxB || a->n_depth < 1 || a->n_depth > kMaxDepth ||
      a->hkv < 1 || a->head_dim < 1 || (long)a->hkv * a->head_dim > 4096)
    return JT_ERR_INVALID_ARG;
  if (a->head_dim % 8 != 0) return JT_ERR_UNSUPPORTED;
  const void* ptrs[] = {a->k_tree, a->v_tree, a->k_cache, a->v_cache, a->prefix_len,
                        a->acc_len, a->acc_nodes, a->new_prefix_len};
  for (const void* p : ptrs)
    if (!p || !aligned16(p)) return JT_ERR_INVALID_ARG;
  if (a->block_table) {
    if (!aligned16(a->block_table)) return JT_ERR_INVALID_ARG;
    if (a->page_size != kPageSize) return JT_ERR_UNSUPPORTED;
    if (a->max_pages < 1 || a->n_pages < 1) return JT_ERR_INVALID_ARG;
  } else if (a->max_prefix < 0) {
    return JT_ERR_INVALID_ARG;
  }
  Ctx c;
  jt_status st = make_ctx(exec, &c);
  if (st != JT_OK) return st;
  return from_cuda(launch_tree_commit(c, *a));
}

size_t jt_lmhead_topw_workspace_bytes(int rows, int d, int vocab, int W) {
  if (rows < 0 || d < 64 || vocab < 1 || W < 1 || W > kMaxW || W > vocab) return 0;
  return lmhead_workspace_bytes(rows, vocab, W);
}

jt_status jt_lmhead_topw(const void* hidden, const void* w_lm, int rows, int d, int vocab, int W,
                         int32_t* tok, float* logp, float* entropy, const jt_exec* exec) {
  if (rows < 0 || d < 64 || vocab < 1 || W < 1 || W > kMaxW || W > vocab)
    return JT_ERR_INVALID_ARG;
  if (d % 64 != 0) return JT_ERR_UNSUPPORTED;
  if ((long)rows * ((vocab + 511) / 512) > 0x7FFFFFFFL / 64) return JT_ERR_UNSUPPORTED;
  if (rows > 0 && (!hidden || !w_lm || !tok || !logp)) return JT_ERR_INVALID_ARG;
  const void* ptrs[] = {hidden, w_lm, tok, logp, entropy};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JT_ERR_INVALID_ARG;
  Ctx c;
  jt_status st = make_ctx(exec, &c);
  if (st != JT_OK) return st;
  st = need_workspace(c, lmhead_workspace_bytes(rows, vocab, W));
  if (st != JT_OK) return st;
  return from_cuda(launch_lmhead_topw(c, hidden, w_lm, rows, d, vocab, W, tok, logp, entropy));
}

size_t jt_tree_accept_workspace_bytes(int batch, int B, int n_depth, int vocab) {
  if (batch < 0 || B < 1 || B > kMaxB || n_depth < 1 || n_depth > kMaxDepth || vocab < 1) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  return accept_workspace_bytes(batch, B, n_depth, vocab, device_sm_count(dev));
}

namespace {

jt_status accept_impl(const float* target_logits, const int32_t* parent, const int32_t* token,
                      const int32_t* n_nodes, int batch, int B, int n_depth, int vocab,
                      int32_t* acc_len, int32_t* acc_tokens, int32_t* acc_nodes, int32_t* bonus,
                      bool sampled, float inv_t, uint64_t seed, const jt_exec* exec) {
  if (batch < 0 || B < 1 || B > kMaxB || n_depth < 1 || n_depth > kMaxDepth || vocab < 1)
    return JT_ERR_INVALID_ARG;
  if (vocab % 4 != 0) return JT_ERR_UNSUPPORTED;
  if ((long)batch * (B + 1) * 16 > 0x7FFFFFFFL) return JT_ERR_UNSUPPORTED;
  if (batch > 0 && (!target_logits || !parent || !token || !n_nodes || !acc_len || !acc_tokens ||
                    !acc_nodes || !bonus))
    return JT_ERR_INVALID_ARG;
  const void* ptrs[] = {target_logits, parent, token, n_nodes, acc_len, acc_tokens, acc_nodes, bonus};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JT_ERR_INVALID_ARG;
  Ctx c;
  jt_status st = make_ctx(exec, &c);
  if (st != JT_OK) return st;
  st = need_workspace(c, accept_workspace_bytes(batch, B, n_depth, vocab, c.num_sms));
  if (st != JT_OK) return st;
  return from_cuda(launch_tree_accept(c, target_logits, parent, token, n_nodes, batch, B, n_depth,
                                      vocab, acc_len, acc_tokens, acc_nodes, bonus, sampled,
                                      inv_t, seed));
}

}  // namespace

jt_status jt_tree_accept(const float* target_logits, const int32_t* parent, const int32_t* token,
                         const int32_t* n_nodes, int batch, int B, int n_depth, int vocab,
                         int32_t* acc_len, int32_t* acc_tokens, int32_t* acc_nodes,
                         int32_t* bonus, const jt_exec* exec) {
  return accept_impl(target_logits, parent, token, n_nodes, batch, B, n_depth, vocab, acc_len,
                     acc_tokens, acc_nodes, bonus, false, 1.0f, 0, exec);
}

jt_status jt_tree_accept_sampled(const float* target_logits, const int32_t* parent,
                                 const int32_t* token, const int32_t* n_nodes, int batch, int B,
                                 int n_depth, int vocab, float temperature, uint64_t seed,
                                 int32_t* acc_len, int32_t* acc_tokens, int32_t* acc_nodes,
                                 int32_t* bonus, const jt_exec* exec) {
  if (!(temperature > 0.0f) || !(temperature <= 3.0e38f)) return JT_ERR_INVALID_ARG;
  const float inv_t = 1.0f / temperature;   // binary32 reciprocal, the multiplier of every key
  if (!(inv_t <= 3.0e38f)) return JT_ERR_INVALID_ARG;
  return accept_impl(target_logits, parent, token, n_nodes, batch, B, n_depth, vocab, acc_len,
                     acc_tokens, acc_nodes, bonus, true, inv_t, seed, exec);
}

}  // extern "C"
