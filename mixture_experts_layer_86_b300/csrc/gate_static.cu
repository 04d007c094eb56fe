// moe_gate_topk_static: moe_gate_topk for callers that cannot allocate
// device memory.
//
// Some callers only ever hold the input and output buffers of a call and a
// stream -- for example a plugin inside another inference engine whose
// enqueue hook hands over tensors and nothing else, or a service that bans
// device allocation once it has started serving.  They have no way to
// provide the scratch workspace moe_gate_topk asks for.  This entry point
// gives them the same gate and routing with the scratch taken from a fixed
// array compiled into the library instead.
//
// The array is a file-scope device variable, so every GPU that loads the
// library reserves it until the process exits.  In host code its name is
// only a stand-in for the device object, never a usable pointer: the device
// address is looked up with cudaGetSymbolAddress, once per device, with
// that device current, and handed to the kernels as the workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "moe_b300.h"

// 16 MiB of routing / logits scratch shared by every call on a device.
static constexpr size_t kGateStaticScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_gate_static_scratch[kGateStaticScratchBytes];

namespace {

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device; looked up on
// the first call made on each device and cached.
moe_status static_scratch_address(void **out) {
  static void *addr[kMaxDevices] = {nullptr};
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_gate_static_scratch);
    if (e != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
  return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_gate_topk_static(const moe_config *cfg, const void *x,
                                           const void *w_gate, const float *logit_bias,
                                           float *logits, float *probs, int32_t *topk_idx,
                                           float *topk_w, int32_t *slot, int32_t *routed_cnt,
                                           int32_t *kept_cnt, int32_t *expert_offsets,
                                           int32_t *row_src, float *l_aux, moe_stream_t stream) {
  size_t need = 0;
  moe_status st = moe_workspace_size(cfg, 0, &need);
  if (st != MOE_OK) return st;
  if (need > kGateStaticScratchBytes) return MOE_ERR_WORKSPACE;  // config too large
  void *scratch = nullptr;
  st = static_scratch_address(&scratch);
  if (st != MOE_OK) return st;
  // Every scratch word the routing kernels read is written earlier in the
  // same call, so the previous call's contents need no clearing.
  return moe_gate_topk(cfg, x, w_gate, logit_bias, logits, probs, topk_idx, topk_w, slot,
                       routed_cnt, kept_cnt, expert_offsets, row_src, l_aux, scratch,
                       kGateStaticScratchBytes, stream);
}
