// ditango_attn_step_static_workspace: the attention step with its scratch memory taken from a
// fixed array inside this library instead of a caller-supplied workspace.
//
// Some callers of this library cannot call cudaMalloc at all: plugins whose host framework
// forbids device allocation inside their execute call, processes whose memory pool has
// already claimed the GPU's free memory, and latency-critical loops that cannot afford
// cudaMalloc's implicit device synchronisation. They still own their inputs, outputs and state
// cache; only the step's scratch (the rotated q and k written by the RoPE prologue) has nowhere
// to live. This entry point gives that scratch a home in a file-scope device array.
//
// The array costs kStaticWorkspaceBytes of device memory on every GPU where the library's
// device code is loaded, held until the process exits.
#include <cstdint>
#include <mutex>

#include "ditango_internal.h"
#include "plan_internal.h"

namespace {

// 64 MiB: rotated q and k for up to 2^24 bf16 (2^23 fp32) elements each (B * N * H * d).
constexpr size_t kStaticWorkspaceBytes = size_t{64} << 20;

static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
void* g_static_ptr[kMaxDevices] = {};
std::mutex g_static_mutex;

// Device address of g_static_workspace on the current device. In host code the array's name
// only stands for the symbol, so its address is looked up once per device, with that device
// current, and cached.
int static_workspace_ptr(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DITANGO_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
    if (e != cudaSuccess || p == nullptr) return DITANGO_ERR_CUDA;
    g_static_ptr[dev] = p;
  }
  *out = g_static_ptr[dev];
  return DITANGO_OK;
}

}  // namespace

extern "C" int ditango_attn_step_static_workspace(
    ditango_plan_t plan, const ditango_tensor* q, const ditango_tensor* k, const ditango_tensor* v,
    const ditango_rope* rope, const uint8_t* reuse_mask, const ditango_state_cache* cache,
    const ditango_tensor* out, const ditango_tensor* out_lse, float softmax_scale, void* stream) {
  if (plan == nullptr || q == nullptr) return DITANGO_ERR_INVALID_ARG;
  // the shape checks ditango_attn_step makes before it looks at the workspace, so that a bad
  // shape is reported as SHAPE here too rather than sizing the scratch from it
  if (q->ndim != 4) return DITANGO_ERR_SHAPE;
  for (int a = 0; a < 4; ++a)
    if (q->shape[a] < 1) return DITANGO_ERR_SHAPE;
  if (q->shape[1] != plan->N) return DITANGO_ERR_SHAPE;
  if (static_cast<double>(q->shape[0]) * static_cast<double>(q->shape[1]) *
          static_cast<double>(q->shape[2]) > 2147483648.0)
    return DITANGO_ERR_SHAPE;
  const size_t need = ditango_attn_step_workspace_size(plan, q->shape[0], q->shape[2],
                                                       static_cast<int32_t>(q->shape[3]), q->dtype,
                                                       rope != nullptr ? 1 : 0);
  if (need > kStaticWorkspaceBytes) return DITANGO_ERR_WORKSPACE;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  if (need > 0) {
    const int st = static_workspace_ptr(&ws);
    if (st != DITANGO_OK) return st;
    ws_bytes = kStaticWorkspaceBytes;
  }
  return ditango_attn_step(plan, q, k, v, rope, reuse_mask, cache, out, out_lse, softmax_scale, ws,
                           ws_bytes, stream);
}
