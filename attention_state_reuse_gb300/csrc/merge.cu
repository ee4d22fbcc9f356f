// Exact merge of attention states (the log-sum-exp rule), memory bound.
//
// Method: DiTango (gist.science/paper/2607.15650), Methodology 2, State Composition: states
// (O_s, lse_s) combine associatively and commutatively into
//   lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s,
// and the result is itself a state (Dynamic Group Compose merges cached states into coarser
// groups without recomputation).
//
// Layout: every state is [G1, G2, R, d] (d contiguous) with shared strides, lse [G1, G2, R].
// Each output row is handled by d/VEC consecutive threads, each owning VEC contiguous
// channels loaded as one 16-byte vector per state, so a warp reads whole rows of every state
// in fully used 32-byte sectors. The lse values of a row are read once per thread (the group of
// threads of a row shares cache lines) and the weights are computed in fp32.
#include <cuda_bf16.h>

#include "ditango_internal.h"

namespace ditango {
namespace {

constexpr int kMergeThreads = 256;

__device__ __forceinline__ void load_vec(const float* p, float (&x)[4]) {
  const float4 v = __ldg(reinterpret_cast<const float4*>(p));
  x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
}
__device__ __forceinline__ void load_vec(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void store_vec(float* p, const float (&x)[4]) {
  *reinterpret_cast<float4*>(p) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void store_vec(__nv_bfloat16* p, const float (&x)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * i], x[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

template <typename T>
__global__ void __launch_bounds__(kMergeThreads)
    merge_kernel(const __grid_constant__ MergeArgs a) {
  constexpr int VEC = 16 / sizeof(T);
  const int tpr = a.d / VEC;  // threads per row
  const int64_t rows = a.G1 * a.G2 * a.R;
  const int64_t gtid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = gtid / tpr;
  if (row >= rows) return;
  const int c0 = static_cast<int>(gtid - row * tpr) * VEC;
  const int64_t r = row % a.R;
  const int64_t g = row / a.R;
  const int64_t g2 = g % a.G2;
  const int64_t g1 = g / a.G2;
  const int64_t lo = g1 * a.lS[0] + g2 * a.lS[1] + r * a.lS[2];
  const int64_t oo = g1 * a.oS[0] + g2 * a.oS[1] + r * a.oS[2] + c0;
  constexpr float kLog2e = 1.4426950408889634f;

  float mx = -INFINITY;
  for (int s = 0; s < a.n; ++s) mx = fmaxf(mx, __ldg(a.lse[s] + lo));
  float sum = 0.f;
  for (int s = 0; s < a.n; ++s) sum += exp2f((__ldg(a.lse[s] + lo) - mx) * kLog2e);
  const float lse = mx + logf(sum);
  const float inv = 1.f / sum;

  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  int s = 0;
  // four states in flight per iteration for memory-level parallelism
  for (; s + 4 <= a.n; s += 4) {
    float x[4][VEC];
    float wgt[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      load_vec(static_cast<const T*>(a.O[s + q]) + oo, x[q]);
      wgt[q] = exp2f((__ldg(a.lse[s + q] + lo) - mx) * kLog2e) * inv;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc[e] = fmaf(wgt[q], x[q][e], acc[e]);
  }
  for (; s < a.n; ++s) {
    float x[VEC];
    load_vec(static_cast<const T*>(a.O[s]) + oo, x);
    const float wg = exp2f((__ldg(a.lse[s] + lo) - mx) * kLog2e) * inv;
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = fmaf(wg, x[e], acc[e]);
  }
  T* out = static_cast<T*>(a.out) + g1 * a.outS[0] + g2 * a.outS[1] + r * a.outS[2] + c0;
  store_vec(out, acc);
  if (a.out_lse != nullptr && c0 == 0) a.out_lse[g1 * a.olS[0] + g2 * a.olS[1] + r * a.olS[2]] = lse;
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int vec = a.dtype == DITANGO_BF16 ? 8 : 4;
  const int64_t threads = a.G1 * a.G2 * a.R * (a.d / vec);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + kMergeThreads - 1) / kMergeThreads;
  if (a.dtype == DITANGO_BF16)
    merge_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(a);
  else
    merge_kernel<float><<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ditango
