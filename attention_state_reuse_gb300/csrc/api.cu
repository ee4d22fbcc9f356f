// C ABI entry points: argument validation, TMA descriptor set-up and kernel launches.
//
// One attention-layer step (DiTango, gist.science/paper/2607.15650, Methodology 1-2):
//   1. validate the reuse mask against the plan's cache bookkeeping (host);
//   2. optional 3D RoPE: k (and q for fp32) into the caller's workspace (rope.cu); for bf16
//      the pair kernel rotates each Q tile in shared memory after loading it (pair_tc.cu);
//   3. fresh states for the computed pairs only, written into the state cache (pair_tc.cu for
//      bf16, pair_f32.cu for fp32), over a schedule that lists computed pairs only;
//   4. merge of every query row's states (merge.cu): its computed states with its reused
//      ones, or with one group state per row composed from them (rebuilt when stale);
//   5. record the computed pairs as valid at this step.
// Every device buffer belongs to the caller; nothing here allocates device memory.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "ditango_internal.h"
#include "plan_internal.h"

namespace ditango {
namespace {

// Set by kernels when a bounded barrier wait gives up; read and cleared by
// ditango_device_status.
__device__ int g_device_error;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  int* err_ptr = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mutex;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DITANGO_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DITANGO_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return DITANGO_ERR_CUDA;
    d.err_ptr = static_cast<int*>(p);
    d.ready = true;
  }
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        fn == nullptr)
      return DITANGO_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = &d;
  return DITANGO_OK;
}

size_t elem_size(int32_t dtype) { return dtype == DITANGO_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks a [B, N, H, d] tensor with d contiguous.
int check_bnhd(const ditango_tensor* t, int64_t B, int64_t N, int64_t H, int64_t d, int32_t dtype) {
  if (t == nullptr || t->ptr == nullptr) return DITANGO_ERR_INVALID_ARG;
  if (t->ndim != 4) return DITANGO_ERR_SHAPE;
  if (t->shape[0] != B || t->shape[1] != N || t->shape[2] != H || t->shape[3] != d)
    return DITANGO_ERR_SHAPE;
  if (t->dtype != dtype) return DITANGO_ERR_DTYPE;
  if (t->stride[3] != 1) return DITANGO_ERR_SHAPE;
  const int64_t vec = 16 / static_cast<int64_t>(elem_size(dtype));
  if (!aligned16(t->ptr)) return DITANGO_ERR_ALIGN;
  for (int a = 0; a < 3; ++a)
    if (t->stride[a] <= 0 || t->stride[a] % vec != 0) return DITANGO_ERR_ALIGN;
  return DITANGO_OK;
}

// Every stride of the first `n` dims at least 1 (no aliasing of distinct elements through a
// zero stride, no negative offsets).
bool positive_strides(const ditango_tensor* t, int n) {
  for (int a = 0; a < n; ++a)
    if (t->stride[a] < 1) return false;
  return true;
}

bool contiguous(const ditango_tensor* t) {
  int64_t s = 1;
  for (int a = t->ndim - 1; a >= 0; --a) {
    if (t->shape[a] != 1 && t->stride[a] != s) return false;
    s *= t->shape[a];
  }
  return true;
}

int encode_bnhd_map(CUtensorMap* map, const void* ptr, const int64_t* shape, const int64_t* stride) {
  // dims innermost first: d, H, N, B; byte strides of H, N, B
  const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(shape[3]), static_cast<cuuint64_t>(shape[2]),
                              static_cast<cuuint64_t>(shape[1]), static_cast<cuuint64_t>(shape[0])};
  const cuuint64_t gstr[3] = {static_cast<cuuint64_t>(stride[2]) * 2,
                              static_cast<cuuint64_t>(stride[1]) * 2,
                              static_cast<cuuint64_t>(stride[0]) * 2};
  const cuuint32_t box[4] = {64, 1, 128, 1};
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), gdim,
                              gstr, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DITANGO_OK : DITANGO_ERR_CUDA;
}

int check_rope(const ditango_rope* r, int64_t N, int64_t d) {
  if (r->dt < 0 || r->dh < 0 || r->dw < 0 || (r->dt | r->dh | r->dw) & 1)
    return DITANGO_ERR_INVALID_ARG;
  if (r->dt + r->dh + r->dw != d) return DITANGO_ERR_SHAPE;
  if (r->Hl < 1 || r->Wl < 1 || r->T_tab < 1 || r->start_frame < 0) return DITANGO_ERR_INVALID_ARG;
  if (N % (r->Hl * r->Wl) != 0) return DITANGO_ERR_SHAPE;
  if (r->start_frame + N / (r->Hl * r->Wl) > r->T_tab) return DITANGO_ERR_SHAPE;
  if ((r->dt && (!r->cos_t || !r->sin_t || !r->cos_t_lo || !r->sin_t_lo)) ||
      (r->dh && (!r->cos_h || !r->sin_h || !r->cos_h_lo || !r->sin_h_lo)) ||
      (r->dw && (!r->cos_w || !r->sin_w || !r->cos_w_lo || !r->sin_w_lo)))
    return DITANGO_ERR_INVALID_ARG;
  return DITANGO_OK;
}

// Bytes of one rotated [B, N, H, d] copy, rounded up to 256.
size_t rope_copy_bytes(int64_t B, int64_t N, int64_t H, int64_t d, int32_t dtype) {
  const size_t one = static_cast<size_t>(B * N * H * d) * elem_size(dtype);
  return (one + 255) & ~static_cast<size_t>(255);
}

// Room for the rotated k and the rotated q. The BF16 pair kernel rotates q itself whenever the
// table rows fit its shared memory and then leaves the second half unused; the size does not
// depend on that, so that a caller's buffer stays valid for any table shape.
size_t rope_workspace_bytes(int64_t B, int64_t N, int64_t H, int64_t d, int32_t dtype) {
  return 2 * rope_copy_bytes(B, N, H, d, dtype);
}


// Validates the state cache's O and lse (device, [B, H, S, N, d] and [B, H, S, N]) and its
// optional host storage ([B, H, P, N, d] and [B, H, P, N], page-locked host memory the device
// can address), and fills `loc` with the pointers and the slot map. S = P without host storage.
int cache_loc(const ditango_state_cache* cache, int64_t B, int64_t H, int64_t P, int64_t N,
              int64_t d, int32_t dtype, CacheLoc* loc) {
  const ditango_tensor& cO = cache->O;
  const ditango_tensor& cL = cache->lse;
  if (cO.ptr == nullptr || cL.ptr == nullptr) return DITANGO_ERR_INVALID_ARG;
  if (cO.dtype != dtype || cL.dtype != DITANGO_F32) return DITANGO_ERR_DTYPE;
  if (cO.ndim != 5 || cL.ndim != 4) return DITANGO_ERR_SHAPE;
  const int64_t S = cO.shape[2];
  const bool host = cache->host_O.ptr != nullptr || cache->host_lse.ptr != nullptr;
  if (S < 1 || S > P || (!host && S != P)) return DITANGO_ERR_SHAPE;
  if (cO.shape[0] != B || cO.shape[1] != H || cO.shape[3] != N || cO.shape[4] != d ||
      !contiguous(&cO))
    return DITANGO_ERR_SHAPE;
  if (cL.shape[0] != B || cL.shape[1] != H || cL.shape[2] != S || cL.shape[3] != N ||
      !contiguous(&cL))
    return DITANGO_ERR_SHAPE;
  if (!aligned16(cO.ptr) || !aligned16(cL.ptr)) return DITANGO_ERR_ALIGN;
  std::memset(loc, 0, sizeof(*loc));
  loc->dO = cO.ptr;
  loc->dL = static_cast<float*>(cL.ptr);
  loc->S = static_cast<int32_t>(S);
  if (host) {
    const ditango_tensor& hO = cache->host_O;
    const ditango_tensor& hL = cache->host_lse;
    if (hO.ptr == nullptr || hL.ptr == nullptr) return DITANGO_ERR_INVALID_ARG;
    if (hO.dtype != dtype || hL.dtype != DITANGO_F32) return DITANGO_ERR_DTYPE;
    if (hO.ndim != 5 || hO.shape[0] != B || hO.shape[1] != H || hO.shape[2] != P ||
        hO.shape[3] != N || hO.shape[4] != d || !contiguous(&hO))
      return DITANGO_ERR_SHAPE;
    if (hL.ndim != 4 || hL.shape[0] != B || hL.shape[1] != H || hL.shape[2] != P ||
        hL.shape[3] != N || !contiguous(&hL))
      return DITANGO_ERR_SHAPE;
    if (!aligned16(hO.ptr) || !aligned16(hL.ptr)) return DITANGO_ERR_ALIGN;
    // the device addresses of page-locked host memory (the same pointers under unified
    // addressing); anything else the kernels could not reach
    void* dev_ptr[2] = {nullptr, nullptr};
    const void* host_ptr[2] = {hO.ptr, hL.ptr};
    for (int x = 0; x < 2; ++x) {
      cudaPointerAttributes attr;
      if (cudaPointerGetAttributes(&attr, host_ptr[x]) != cudaSuccess) {
        (void)cudaGetLastError();
        return DITANGO_ERR_INVALID_ARG;
      }
      if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr)
        return DITANGO_ERR_INVALID_ARG;
      dev_ptr[x] = attr.devicePointer;
    }
    loc->hO = dev_ptr[0];
    loc->hL = static_cast<float*>(dev_ptr[1]);
  }
  cache_slot_map(static_cast<int32_t>(P), static_cast<int32_t>(S), loc->slot);
  return DITANGO_OK;
}

// Validates a plan's state cache (O and lse, and host storage if any; group states are not used
// here) and fills the common planner arguments.
int planner_args(ditango_plan_t plan, const ditango_state_cache* cache, PlannerArgs* a) {
  if (plan == nullptr || cache == nullptr) return DITANGO_ERR_INVALID_ARG;
  const ditango_tensor& cO = cache->O;
  if (cO.ptr == nullptr || cache->lse.ptr == nullptr) return DITANGO_ERR_INVALID_ARG;
  if (cO.dtype != DITANGO_BF16 && cO.dtype != DITANGO_F32) return DITANGO_ERR_DTYPE;
  if (cO.ndim != 5) return DITANGO_ERR_SHAPE;
  const int64_t B = cO.shape[0], H = cO.shape[1], P = plan->P, N = cO.shape[3], d = cO.shape[4];
  if (N != plan->N || B < 1 || H < 1 || (d != 64 && d != 128)) return DITANGO_ERR_SHAPE;
  if (B * H > 65535) return DITANGO_ERR_SHAPE;
  std::memset(a, 0, sizeof(*a));
  const int st = cache_loc(cache, B, H, P, N, d, cO.dtype, &a->cache);
  if (st != DITANGO_OK) return st;
  a->P = static_cast<int32_t>(P);
  a->d = static_cast<int32_t>(d);
  a->dtype = cO.dtype;
  a->B = B; a->H = H; a->N = N;
  for (int64_t i = 0; i <= P; ++i) a->offsets[i] = static_cast<int32_t>(plan->offsets[i]);
  return DITANGO_OK;
}

// The [B, H, N, d] snapshot of the diagonal states: the cache's dtype, contiguous, aligned.
int check_snapshot(const PlannerArgs& a, const ditango_tensor* snap) {
  if (snap == nullptr || snap->ptr == nullptr) return DITANGO_ERR_INVALID_ARG;
  if (snap->dtype != a.dtype) return DITANGO_ERR_DTYPE;
  if (snap->ndim != 4 || snap->shape[0] != a.B || snap->shape[1] != a.H ||
      snap->shape[2] != a.N || snap->shape[3] != a.d || !contiguous(snap))
    return DITANGO_ERR_SHAPE;
  if (!aligned16(snap->ptr)) return DITANGO_ERR_ALIGN;
  return DITANGO_OK;
}

}  // namespace
}  // namespace ditango

using namespace ditango;

extern "C" {

size_t ditango_attn_step_workspace_size(ditango_plan_t plan, int64_t B, int64_t H, int32_t d,
                                        int32_t dtype, int32_t use_rope) {
  if (plan == nullptr || !use_rope) return 0;
  return rope_workspace_bytes(B, plan->N, H, d, dtype);
}

int ditango_attn_step(ditango_plan_t plan, const ditango_tensor* q, const ditango_tensor* k,
                      const ditango_tensor* v, const ditango_rope* rope,
                      const uint8_t* reuse_mask, const ditango_state_cache* cache,
                      const ditango_tensor* out, const ditango_tensor* out_lse,
                      float softmax_scale, void* workspace, size_t workspace_bytes,
                      void* stream) {
  if (plan == nullptr || q == nullptr || k == nullptr || v == nullptr || cache == nullptr ||
      out == nullptr)
    return DITANGO_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale)) return DITANGO_ERR_INVALID_ARG;
  if (q->ndim != 4) return DITANGO_ERR_SHAPE;
  const int64_t B = q->shape[0], N = q->shape[1], H = q->shape[2], d = q->shape[3];
  // an empty batch is refused before its (possibly NULL) pointers are looked at: the step
  // would record every computed pair as fresh without computing one
  if (N != plan->N || B < 1 || H < 1) return DITANGO_ERR_SHAPE;
  if (q->ptr == nullptr) return DITANGO_ERR_INVALID_ARG;
  const int32_t dtype = q->dtype;
  const int64_t P = plan->P;
  if (dtype != DITANGO_BF16 && dtype != DITANGO_F32) return DITANGO_ERR_DTYPE;
  if (d != 64 && d != 128) return DITANGO_ERR_UNSUPPORTED;
  if (B * H * N > (int64_t{1} << 31)) return DITANGO_ERR_SHAPE;
  int st;
  if ((st = check_bnhd(q, B, N, H, d, dtype)) != DITANGO_OK) return st;
  if ((st = check_bnhd(k, B, N, H, d, dtype)) != DITANGO_OK) return st;
  if ((st = check_bnhd(v, B, N, H, d, dtype)) != DITANGO_OK) return st;
  if ((st = check_bnhd(out, B, N, H, d, dtype)) != DITANGO_OK) return st;
  if (out_lse != nullptr) {
    if (out_lse->ptr == nullptr) return DITANGO_ERR_INVALID_ARG;
    if (out_lse->dtype != DITANGO_F32) return DITANGO_ERR_DTYPE;
    if (out_lse->ndim != 3 || out_lse->shape[0] != B || out_lse->shape[1] != H ||
        out_lse->shape[2] != N)
      return DITANGO_ERR_SHAPE;
    if (!positive_strides(out_lse, 3)) return DITANGO_ERR_SHAPE;
  }
  // the cache's pointers are checked here; whether host storage can be reached is asked of
  // the CUDA runtime only after the other arguments passed
  const ditango_tensor& gO = cache->group_O;
  const ditango_tensor& gL = cache->group_lse;
  const bool use_group = gO.ptr != nullptr;
  if ((gO.ptr == nullptr) != (gL.ptr == nullptr)) return DITANGO_ERR_INVALID_ARG;
  if (use_group) {
    if (gO.dtype != DITANGO_F32 || gL.dtype != DITANGO_F32) return DITANGO_ERR_DTYPE;
    if (gO.ndim != 4 || gO.shape[0] != B || gO.shape[1] != H || gO.shape[2] != N ||
        gO.shape[3] != d || !contiguous(&gO))
      return DITANGO_ERR_SHAPE;
    if (gL.ndim != 3 || gL.shape[0] != B || gL.shape[1] != H || gL.shape[2] != N ||
        !contiguous(&gL))
      return DITANGO_ERR_SHAPE;
    if (!aligned16(gO.ptr) || !aligned16(gL.ptr)) return DITANGO_ERR_ALIGN;
  }
  if (rope != nullptr) {
    if ((st = check_rope(rope, N, d)) != DITANGO_OK) return st;
    const size_t need = rope_workspace_bytes(B, N, H, d, dtype);
    if (workspace == nullptr || workspace_bytes < need) return DITANGO_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DITANGO_ERR_ALIGN;
  }
  if ((st = plan_validate(plan, reuse_mask)) != DITANGO_OK) return st;
  const uint8_t* mask = plan_effective_mask(plan, reuse_mask);
  CacheLoc loc;
  if ((st = cache_loc(cache, B, H, P, N, d, dtype, &loc)) != DITANGO_OK) return st;

  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != DITANGO_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  auto mark = [&](int x) -> bool {
    return !plan->profile ||
           cudaEventRecord(static_cast<cudaEvent_t>(plan->events[x]), s) == cudaSuccess;
  };
  if (!mark(0)) return DITANGO_ERR_CUDA;

  // ---- 1. rotary prologue into the workspace: k (and, for F32, q); the BF16 pair kernel
  // rotates each Q tile itself after loading it
  const void* qp = q->ptr;
  const void* kp = k->ptr;
  int64_t qs[4] = {q->stride[0], q->stride[1], q->stride[2], 1};
  int64_t ks[4] = {k->stride[0], k->stride[1], k->stride[2], 1};
  // the BF16 pair kernel rotates Q itself when the table rows fit its shared memory
  RopeQ rq;
  std::memset(&rq, 0, sizeof(rq));
  if (rope != nullptr && dtype == DITANGO_BF16) {
    auto odd = [](int32_t x) { return x | 1; };
    rq.cos_t = rope->cos_t; rq.sin_t = rope->sin_t;
    rq.cos_h = rope->cos_h; rq.sin_h = rope->sin_h;
    rq.cos_w = rope->cos_w; rq.sin_w = rope->sin_w;
    rq.cos_t_lo = rope->cos_t_lo; rq.sin_t_lo = rope->sin_t_lo;
    rq.cos_h_lo = rope->cos_h_lo; rq.sin_h_lo = rope->sin_h_lo;
    rq.cos_w_lo = rope->cos_w_lo; rq.sin_w_lo = rope->sin_w_lo;
    rq.Hl = static_cast<int32_t>(rope->Hl);
    rq.Wl = static_cast<int32_t>(rope->Wl);
    rq.start_frame = static_cast<int32_t>(rope->start_frame);
    rq.dt = rope->dt; rq.dh = rope->dh; rq.dw = rope->dw;
    rq.nT = static_cast<int32_t>(N / (rope->Hl * rope->Wl));
    rq.sT = odd(rope->dt / 2); rq.sH = odd(rope->dh / 2); rq.sW = odd(rope->dw / 2);
    const int64_t pairs = int64_t{rq.nT} * rq.sT + rope->Hl * rq.sH + rope->Wl * rq.sW;
    rq.n_pairs = 8 * pairs <= kRopeSmemMaxBytes ? static_cast<int32_t>(pairs) : 0;
  }
  const bool q_in_kernel = rq.n_pairs > 0;
  if (rope != nullptr) {
    const size_t one = rope_copy_bytes(B, N, H, d, dtype);
    RopeApplyArgs ra;
    std::memset(&ra, 0, sizeof(ra));
    ra.n_tensors = q_in_kernel ? 1 : 2;
    ra.x[0] = k->ptr;
    ra.x[1] = q->ptr;
    for (int a = 0; a < 3; ++a) {
      ra.xs[0][a] = k->stride[a];
      ra.xs[1][a] = q->stride[a];
    }
    ra.y[0] = workspace;
    ra.y[1] = static_cast<uint8_t*>(workspace) + one;
    ra.dtype = dtype;
    ra.B = B; ra.N = N; ra.H = H; ra.d = static_cast<int32_t>(d);
    ra.cos_t = rope->cos_t; ra.sin_t = rope->sin_t;
    ra.cos_h = rope->cos_h; ra.sin_h = rope->sin_h;
    ra.cos_w = rope->cos_w; ra.sin_w = rope->sin_w;
    ra.cos_t_lo = rope->cos_t_lo; ra.sin_t_lo = rope->sin_t_lo;
    ra.cos_h_lo = rope->cos_h_lo; ra.sin_h_lo = rope->sin_h_lo;
    ra.cos_w_lo = rope->cos_w_lo; ra.sin_w_lo = rope->sin_w_lo;
    ra.Hl = rope->Hl; ra.Wl = rope->Wl; ra.start_frame = rope->start_frame;
    ra.dt = rope->dt; ra.dh = rope->dh; ra.dw = rope->dw;
    if (launch_rope_apply(ra, s) != cudaSuccess) return DITANGO_ERR_CUDA;
    const int64_t cs[4] = {N * H * d, H * d, d, 1};
    kp = ra.y[0];
    std::memcpy(ks, cs, sizeof(cs));
    if (!q_in_kernel) {
      qp = ra.y[1];
      std::memcpy(qs, cs, sizeof(cs));
    }
  }

  // ---- 2. fresh states of the computed pairs
  if (!mark(1)) return DITANGO_ERR_CUDA;
  const int32_t block_rows = dtype == DITANGO_BF16 ? 256 : 64;
  PairSchedule sched;
  build_schedule(N, static_cast<int32_t>(P), plan->offsets.data(), mask, B, H, block_rows, &sched);
  if (dtype == DITANGO_BF16) {
    CUtensorMap mq, mk, mv;
    const int64_t shp[4] = {B, N, H, d};
    const int64_t vs[4] = {v->stride[0], v->stride[1], v->stride[2], 1};
    if (encode_bnhd_map(&mq, qp, shp, qs) != DITANGO_OK ||
        encode_bnhd_map(&mk, kp, shp, ks) != DITANGO_OK ||
        encode_bnhd_map(&mv, v->ptr, shp, vs) != DITANGO_OK)
      return DITANGO_ERR_CUDA;
    PairTcArgs pa;
    pa.sched = sched;
    pa.N = N;
    pa.cache = loc;
    pa.scale_log2 = softmax_scale * 1.4426950408889634f;
    pa.err = dev->err_ptr;
    pa.rope = rq;
    pa.inject_fault = plan->inject_fault;
    plan->inject_fault = 0;
    if (launch_pair_tc(static_cast<int>(d), mq, mk, mv, pa, dev->num_sms, s) != cudaSuccess)
      return DITANGO_ERR_CUDA;
  } else {
    PairF32Args pa;
    pa.sched = sched;
    pa.N = N;
    pa.q = static_cast<const float*>(qp);
    pa.k = static_cast<const float*>(kp);
    pa.v = static_cast<const float*>(v->ptr);
    for (int a = 0; a < 3; ++a) {
      pa.qs[a] = qs[a];
      pa.ks[a] = ks[a];
      pa.vs[a] = v->stride[a];
    }
    pa.cache = loc;
    pa.scale = softmax_scale;
    if (launch_pair_f32(static_cast<int>(d), pa, s) != cudaSuccess) return DITANGO_ERR_CUDA;
  }

  // ---- 3. merge: each row's computed states with its reused ones, or with the group state of
  // its partition's reused pairs (built in the same pass where it is missing or out of date)
  if (!mark(2)) return DITANGO_ERR_CUDA;
  uint64_t reused[kMaxP] = {}, rebuild = 0;
  bool any_reuse = false;
  for (int32_t i = 0; i < P; ++i) {
    reused[i] = plan_reused_set(plan, reuse_mask, i);
    any_reuse |= reused[i] != 0;
    if (use_group && reused[i] != 0 && !plan_group_current(plan, gO.ptr, i, reused[i]))
      rebuild |= uint64_t{1} << i;
  }
  // A step that computes every pair, on a plan whose default mask reuses some: the merge, which
  // reads every state anyway, also builds the group states of the default mask's reused sets
  // from this step's states, so that the next step under that mask finds them current.
  uint64_t ahead = 0, ahead_set[kMaxP] = {};
  if (use_group && !any_reuse && reuse_mask != nullptr) {
    for (int32_t i = 0; i < P; ++i) {
      ahead_set[i] = plan_reused_set(plan, nullptr, i);
      if (ahead_set[i] != 0) ahead |= uint64_t{1} << i;
    }
  }
  for (uint64_t m = rebuild | ahead; m; m &= m - 1)
    plan->group_set[__builtin_ctzll(m)] = 0;  // invalid until this build has been launched
  StepMergeArgs ma;
  std::memset(&ma, 0, sizeof(ma));
  ma.P = static_cast<int32_t>(P);
  ma.d = static_cast<int32_t>(d);
  ma.dtype = dtype;
  ma.B = B; ma.H = H; ma.N = N;
  for (int32_t i = 0; i <= P; ++i) ma.offsets[i] = static_cast<int32_t>(plan->offsets[i]);
  for (int32_t i = 0; i < P; ++i) {
    const uint64_t all = P == 64 ? ~uint64_t{0} : (uint64_t{1} << P) - 1;
    const uint64_t set = (ahead >> i) & 1u ? ahead_set[i] : reused[i];
    const bool grp = use_group && set != 0;
    ma.cache_set[i] = grp ? (all & ~set) : all;
    ma.reused_set[i] = set;
    if (grp) ma.group |= uint64_t{1} << i;
  }
  ma.rebuild = rebuild | ahead;
  ma.cache = loc;
  ma.gO = use_group ? static_cast<float*>(gO.ptr) : nullptr;
  ma.gL = use_group ? static_cast<float*>(gL.ptr) : nullptr;
  ma.out = out->ptr;
  ma.outS[0] = out->stride[0]; ma.outS[1] = out->stride[2]; ma.outS[2] = out->stride[1];
  if (out_lse != nullptr) {
    ma.out_lse = static_cast<float*>(out_lse->ptr);
    ma.olS[0] = out_lse->stride[0]; ma.olS[1] = out_lse->stride[1]; ma.olS[2] = out_lse->stride[2];
  }
  if (launch_step_merge(ma, s) != cudaSuccess) return DITANGO_ERR_CUDA;
  if (!mark(3)) return DITANGO_ERR_CUDA;

  for (uint64_t m = rebuild; m; m &= m - 1) {
    const int32_t i = __builtin_ctzll(m);
    plan_group_built(plan, gO.ptr, i, reused[i]);
  }
  plan_commit(plan, reuse_mask);
  // the groups built ahead hold states computed at this step: recorded after the commit
  for (uint64_t m = ahead; m; m &= m - 1) {
    const int32_t i = __builtin_ctzll(m);
    plan_group_built(plan, gO.ptr, i, ahead_set[i]);
  }
  return DITANGO_OK;
}

// ---- anchor-guided planner ---------------------------------------------------------------

int ditango_planner_importance(ditango_plan_t plan, const ditango_state_cache* cache, double* w,
                               void* stream) {
  PlannerArgs a;
  int st = planner_args(plan, cache, &a);
  if (st != DITANGO_OK) return st;
  if (w == nullptr) return DITANGO_ERR_INVALID_ARG;
  a.sums = w;  // summed in place, then divided by the row counts
  a.out = w;
  return launch_planner_importance(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DITANGO_OK
             : DITANGO_ERR_CUDA;
}

int ditango_planner_snapshot(ditango_plan_t plan, const ditango_state_cache* cache,
                             const ditango_tensor* snapshot, void* stream) {
  PlannerArgs a;
  int st = planner_args(plan, cache, &a);
  if (st != DITANGO_OK) return st;
  if ((st = check_snapshot(a, snapshot)) != DITANGO_OK) return st;
  // rows of partition i from the device slot of (i, i) of every (b, h) (the local pair is
  // always on the device), by a copy kernel
  a.snap = snapshot->ptr;
  if (launch_planner_snapshot(a, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DITANGO_ERR_CUDA;
  return DITANGO_OK;
}

int ditango_planner_drift(ditango_plan_t plan, const ditango_state_cache* cache,
                          const ditango_tensor* snapshot, double* delta, void* stream) {
  PlannerArgs a;
  int st = planner_args(plan, cache, &a);
  if (st != DITANGO_OK) return st;
  if ((st = check_snapshot(a, snapshot)) != DITANGO_OK) return st;
  if (delta == nullptr) return DITANGO_ERR_INVALID_ARG;
  a.snap = snapshot->ptr;
  a.sums = delta;      // 2P sums first ...
  a.out = delta;       // ... then the P drifts in the first half
  return launch_planner_drift(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DITANGO_OK
             : DITANGO_ERR_CUDA;
}

int ditango_merge(const ditango_state_list* sl, const ditango_tensor* out,
                  const ditango_tensor* out_lse, void* stream) {
  if (sl == nullptr || out == nullptr || sl->O == nullptr || sl->lse == nullptr)
    return DITANGO_ERR_INVALID_ARG;
  if (sl->n < 1 || sl->n > kMaxStates) return DITANGO_ERR_INVALID_ARG;
  if (sl->dtype != DITANGO_BF16 && sl->dtype != DITANGO_F32) return DITANGO_ERR_DTYPE;
  const int64_t G1 = sl->shape[0], G2 = sl->shape[1], R = sl->shape[2], d = sl->shape[3];
  if (G1 < 0 || G2 < 0 || R < 0 || d < 1) return DITANGO_ERR_SHAPE;
  if (out->ndim != 4 || out->shape[0] != G1 || out->shape[1] != G2 || out->shape[2] != R ||
      out->shape[3] != d)
    return DITANGO_ERR_SHAPE;
  const int64_t vec = 16 / static_cast<int64_t>(elem_size(sl->dtype));
  if (d % vec != 0) return DITANGO_ERR_SHAPE;
  if (G1 == 0 || G2 == 0 || R == 0) return DITANGO_OK;  // no rows: nothing is read or written
  if (out->ptr == nullptr) return DITANGO_ERR_INVALID_ARG;
  for (int a = 0; a < 3; ++a)
    if (sl->O_stride[a] % vec != 0) return DITANGO_ERR_ALIGN;
  for (int a = 0; a < 3; ++a)
    if (sl->O_stride[a] < 1 || sl->lse_stride[a] < 1) return DITANGO_ERR_SHAPE;
  for (int32_t s = 0; s < sl->n; ++s) {
    if (sl->O[s] == nullptr || sl->lse[s] == nullptr) return DITANGO_ERR_INVALID_ARG;
    if (!aligned16(sl->O[s])) return DITANGO_ERR_ALIGN;
  }
  if (out->dtype != sl->dtype) return DITANGO_ERR_DTYPE;
  if (out->stride[3] != 1 || !positive_strides(out, 3)) return DITANGO_ERR_SHAPE;
  if (!aligned16(out->ptr)) return DITANGO_ERR_ALIGN;
  for (int a = 0; a < 3; ++a)
    if (out->stride[a] % vec != 0) return DITANGO_ERR_ALIGN;
  if (out_lse != nullptr) {
    if (out_lse->ptr == nullptr) return DITANGO_ERR_INVALID_ARG;
    if (out_lse->dtype != DITANGO_F32) return DITANGO_ERR_DTYPE;
    if (out_lse->ndim != 3 || out_lse->shape[0] != G1 || out_lse->shape[1] != G2 ||
        out_lse->shape[2] != R)
      return DITANGO_ERR_SHAPE;
    if (!positive_strides(out_lse, 3)) return DITANGO_ERR_SHAPE;
  }
  MergeArgs ma;
  std::memset(&ma, 0, sizeof(ma));
  ma.n = sl->n;
  ma.d = static_cast<int32_t>(d);
  ma.dtype = sl->dtype;
  ma.out_dtype = sl->dtype;
  ma.G1 = G1; ma.G2 = G2; ma.R = R;
  ma.out = out->ptr;
  for (int32_t s = 0; s < sl->n; ++s) {
    ma.O[s] = sl->O[s];
    ma.lse[s] = sl->lse[s];
  }
  for (int a = 0; a < 3; ++a) {
    ma.oS[a] = sl->O_stride[a];
    ma.lS[a] = sl->lse_stride[a];
    ma.outS[a] = out->stride[a];
  }
  if (out_lse != nullptr) {
    ma.out_lse = static_cast<float*>(out_lse->ptr);
    for (int a = 0; a < 3; ++a) ma.olS[a] = out_lse->stride[a];
  }
  return launch_merge(ma, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? DITANGO_OK
                                                                                  : DITANGO_ERR_CUDA;
}

int ditango_rope_build_tables(const ditango_rope* rope, double theta, void* stream) {
  if (rope == nullptr || !(theta > 1.0)) return DITANGO_ERR_INVALID_ARG;
  if (rope->dt < 0 || rope->dh < 0 || rope->dw < 0 || ((rope->dt | rope->dh | rope->dw) & 1))
    return DITANGO_ERR_INVALID_ARG;
  if (rope->T_tab < 0 || rope->Hl < 0 || rope->Wl < 0) return DITANGO_ERR_INVALID_ARG;
  if ((rope->dt && rope->T_tab &&
       (!rope->cos_t || !rope->sin_t || !rope->cos_t_lo || !rope->sin_t_lo)) ||
      (rope->dh && rope->Hl &&
       (!rope->cos_h || !rope->sin_h || !rope->cos_h_lo || !rope->sin_h_lo)) ||
      (rope->dw && rope->Wl &&
       (!rope->cos_w || !rope->sin_w || !rope->cos_w_lo || !rope->sin_w_lo)))
    return DITANGO_ERR_INVALID_ARG;
  return launch_rope_tables(*rope, theta, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DITANGO_OK
             : DITANGO_ERR_CUDA;
}

int ditango_device_status(void* stream, int32_t* code) {
  if (code != nullptr) *code = 0;
  DeviceInfo* dev = nullptr;
  int st = device_info(&dev);
  if (st != DITANGO_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DITANGO_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, dev->err_ptr, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DITANGO_ERR_CUDA;
  if (v == 0) return DITANGO_OK;
  const int zero = 0;
  if (cudaMemcpy(dev->err_ptr, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
    return DITANGO_ERR_CUDA;
  if (code != nullptr) *code = v;
  return DITANGO_ERR_DEVICE_TIMEOUT;
}

const char* ditango_status_string(int status) {
  switch (status) {
    case DITANGO_OK: return "ok";
    case DITANGO_ERR_INVALID_ARG: return "invalid argument";
    case DITANGO_ERR_INVALID_MASK: return "invalid reuse mask (values must be 0/1, diagonal 0)";
    case DITANGO_ERR_NO_CACHE: return "reuse of a pair with no cached state";
    case DITANGO_ERR_SHAPE: return "tensor shape mismatch";
    case DITANGO_ERR_DTYPE: return "unsupported or mismatched dtype";
    case DITANGO_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case DITANGO_ERR_WORKSPACE: return "workspace missing or too small";
    case DITANGO_ERR_CUDA: return "CUDA call or kernel launch failed";
    case DITANGO_ERR_DEVICE_TIMEOUT: return "a kernel barrier wait timed out";
    case DITANGO_ERR_UNSUPPORTED: return "unsupported head dimension";
    default: return "unknown status";
  }
}

int ditango_version(void) { return DITANGO_ABI_VERSION; }

}  // extern "C"
