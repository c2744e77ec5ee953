// jt_tree_accept_noalloc: greedy acceptance without a caller workspace.
//
// jt_tree_accept needs batch * (B + 1) int32 of scratch (the argmax of every
// live target row, for chains and trees not much wider than a root path) and
// takes it from exec->workspace. Some callers have no way to provide that:
// code that must not call cudaMalloc (it synchronises the device), hosts
// whose device memory is fully planned by an allocator they do not control,
// or plain C embedders with no allocator at all. This entry point serves
// them: the scratch is a fixed array in the library's own device memory
// image, so the call allocates nothing.
//
// The array is a file-scope __device__ symbol. In host code its name is only
// a host-side stand-in, so the device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) and passed to the
// kernels. Every GPU that loads the library holds the array until the
// process exits.
#include <mutex>

#include "jt_internal.cuh"

namespace jt {
namespace {

// batch * (B + 1) must not exceed this (256 KiB of int32 scratch).
constexpr int kNoAllocMaxRows = 65536;
static __device__ __align__(256) int32_t g_accept_scratch[kNoAllocMaxRows];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_accept_scratch on the current device (looked up once).
jt_status scratch_on_current_device(int* device, void** out) {
  if (cudaGetDevice(device) != cudaSuccess) return JT_ERR_CUDA;
  if (*device < 0 || *device >= kMaxDevices) return JT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[*device]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_accept_scratch);
    if (e != cudaSuccess || p == nullptr) {
      // Clear the (non-sticky) error so that the caller's next, unrelated
      // CUDA error check does not report it.
      cudaGetLastError();
      return JT_ERR_CUDA;
    }
    g_scratch_ptr[*device] = p;
  }
  *out = g_scratch_ptr[*device];
  return JT_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace jt

using namespace jt;

extern "C" jt_status jt_tree_accept_noalloc(const float* target_logits, const int32_t* parent,
                                            const int32_t* token, const int32_t* n_nodes,
                                            int batch, int B, int n_depth, int vocab,
                                            int32_t* acc_len, int32_t* acc_tokens,
                                            int32_t* acc_nodes, int32_t* bonus,
                                            const jt_exec* exec) {
  if (batch < 0 || B < 1 || B > kMaxB || n_depth < 1 || n_depth > kMaxDepth || vocab < 1)
    return JT_ERR_INVALID_ARG;
  if (vocab % 4 != 0) return JT_ERR_UNSUPPORTED;
  if ((long)batch * (B + 1) > kNoAllocMaxRows) return JT_ERR_UNSUPPORTED;  // beyond the array
  if (batch > 0 && (!target_logits || !parent || !token || !n_nodes || !acc_len || !acc_tokens ||
                    !acc_nodes || !bonus))
    return JT_ERR_INVALID_ARG;
  const void* ptrs[] = {target_logits, parent, token, n_nodes, acc_len, acc_tokens, acc_nodes, bonus};
  for (const void* p : ptrs)
    if (!aligned16(p)) return JT_ERR_INVALID_ARG;
  Ctx c;
  c.stream = exec ? reinterpret_cast<cudaStream_t>(exec->stream) : nullptr;
  c.d_err = exec ? exec->d_err : nullptr;
  if (c.d_err && (reinterpret_cast<uintptr_t>(c.d_err) & 3u)) return JT_ERR_INVALID_ARG;
  void* scratch = nullptr;
  const jt_status st = scratch_on_current_device(&c.device, &scratch);
  if (st != JT_OK) return st;
  c.workspace = scratch;
  c.workspace_bytes = sizeof(int32_t) * (size_t)kNoAllocMaxRows;
  c.num_sms = device_sm_count(c.device);
  // Whatever layout the call picks (one index per row, or per-segment
  // partials for a few long rows) must fit the array.
  if (accept_workspace_bytes(batch, B, n_depth, vocab, c.num_sms) > c.workspace_bytes)
    return JT_ERR_UNSUPPORTED;
  if (batch == 0) return JT_OK;
  return launch_tree_accept(c, target_logits, parent, token, n_nodes, batch, B, n_depth, vocab,
                            acc_len, acc_tokens, acc_nodes, bonus) == cudaSuccess
             ? JT_OK
             : JT_ERR_CUDA;
}
