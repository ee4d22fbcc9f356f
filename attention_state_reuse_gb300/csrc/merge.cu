// Exact merge of attention states (the log-sum-exp rule), memory bound: merge_kernel for a list
// of states with a common layout (ditango_merge, and building group states), step_merge_kernel
// for the merge that ends an attention step (states found from the cache layout).
//
// Method: DiTango (gist.science/paper/2607.15650), Methodology 2, State Composition: states
// (O_s, lse_s) combine associatively and commutatively into
//   lse = ln sum_s exp(lse_s),   O = sum_s exp(lse_s - lse) O_s,
// and the result is itself a state (Dynamic Group Compose merges cached states into coarser
// groups without recomputation).
//
// Thread layout: grid.y walks the row groups (a (b, h) slab; launched in chunks of at most
// 65535), grid.x the rows of a group; each row is handled by d/VEC consecutive threads, each
// owning VEC contiguous channels loaded as one 16-byte vector per state, so a warp reads whole
// rows of every state in fully used 32-byte sectors. Index arithmetic is 32-bit shifts and
// masks (d/VEC is a power of two); exponentials and the logarithm use the SFU approximations
// (relative error ~2^-22). States are merged online in rounds (eight for a state list, two for
// a step) whose vectors and lse values are all loaded before any is used (a short round repeats
// a state with weight 0), so a round costs one memory round trip.
#include <cuda_bf16.h>

#include <algorithm>

#include "ditango_internal.h"

namespace ditango {
namespace {

constexpr int kMergeThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
// VEC fp32 channels, 16-byte aligned (group states are fp32 whatever the cache dtype).
template <int VEC>
__device__ __forceinline__ void load_f32(const float* p, float (&x)[VEC]) {
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q) {
    const float4 v = __ldg(reinterpret_cast<const float4*>(p) + q);
    x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
  }
}
template <int VEC>
__device__ __forceinline__ void store_f32(float* p, const float (&x)[VEC]) {
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q)
    reinterpret_cast<float4*>(p)[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
}

// One 16-byte vector of a state, kept packed until it is accumulated.
__device__ __forceinline__ uint4 load_raw(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void unpack(const uint4& v, float (&x)[4], const float*) {
  x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
  x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack(const uint4& v, float (&x)[8], const __nv_bfloat16*) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Online merge of one round of up to kRound states (the rest of the round repeats an earlier
// state with use = false): raw[q] and l[q] (lse in log2 units) were loaded together, so the
// whole round is one memory round trip. acc and sum are relative to the running max mx.
template <typename T, int VEC, int kRound>
__device__ __forceinline__ void merge_round(const uint4 (&raw)[kRound], const float (&l)[kRound],
                                            const bool (&use)[kRound], float& mx, float& sum,
                                            float (&acc)[VEC]) {
  float mn = mx;
#pragma unroll
  for (int q = 0; q < kRound; ++q) mn = fmaxf(mn, l[q]);
  const float sc = ex2(mx - mn);  // 0 on the first round (mx = -inf)
  sum *= sc;
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] *= sc;
#pragma unroll
  for (int q = 0; q < kRound; ++q) {
    const float w = use[q] ? ex2(l[q] - mn) : 0.f;
    sum += w;
    float x[VEC];
    unpack(raw[q], x, static_cast<const T*>(nullptr));
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = fmaf(w, x[e], acc[e]);
  }
  mx = mn;
}

// Row and first channel of this thread; false past the group's last row.
__device__ __forceinline__ bool thread_row(int64_t R, int d, int vec_shift, uint32_t& r, int& c0) {
  const int tpr_shift = 31 - __clz(d) - vec_shift;  // log2(d / VEC)
  const uint32_t t = blockIdx.x * kMergeThreads + threadIdx.x;
  r = t >> tpr_shift;
  c0 = static_cast<int>(t & ((1u << tpr_shift) - 1u)) << vec_shift;
  return r < static_cast<uint64_t>(R);
}

// merge_kernel: state list with a common [G1, G2, R, d] layout (MergeArgs). T: the states'
// dtype, TO: the output's (T, or fp32 for group states).
template <typename T, typename TO>
__global__ void __launch_bounds__(kMergeThreads)
    merge_kernel(const __grid_constant__ MergeArgs a, int64_t g_base) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int VEC_SHIFT = VEC == 8 ? 3 : 2;
  uint32_t r;
  int c0;
  if (!thread_row(a.R, a.d, VEC_SHIFT, r, c0)) return;
  const int64_t g = g_base + blockIdx.y;
  const int64_t g1 = g / a.G2, g2 = g - g1 * a.G2;
  const int64_t lo = g1 * a.lS[0] + g2 * a.lS[1] + r * a.lS[2];
  const int64_t oo = g1 * a.oS[0] + g2 * a.oS[1] + r * a.oS[2] + c0;

  constexpr int kRound = 8;  // a whole list of up to eight states in one round trip
  float mx = -INFINITY, sum = 0.f;
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < a.n; s0 += kRound) {
    uint4 raw[kRound];
    float l[kRound];
    bool use[kRound];
#pragma unroll
    for (int q = 0; q < kRound; ++q) {
      use[q] = s0 + q < a.n;
      const int s = use[q] ? s0 + q : s0;
      raw[q] = load_raw(static_cast<const T*>(a.O[s]) + oo);
      l[q] = __ldg(a.lse[s] + lo) * kLog2e;
    }
    merge_round<T, VEC, kRound>(raw, l, use, mx, sum, acc);
  }
  const float lse = (mx + lg2(sum)) * kLn2;
  const float inv = 1.f / sum;
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] *= inv;
  TO* out = static_cast<TO*>(a.out) + g1 * a.outS[0] + g2 * a.outS[1] + r * a.outS[2] + c0;
  if constexpr (sizeof(TO) == sizeof(T))
    store_vec(out, acc);
  else
    store_f32<VEC>(out, acc);
  if (a.out_lse != nullptr && c0 == 0) a.out_lse[g1 * a.olS[0] + g2 * a.olS[1] + r * a.olS[2]] = lse;
}

// step_merge_kernel: the merge that ends a step (StepMergeArgs). Row r of (b, h) = grid.y
// merges the cache slots (b, h, j, r) for j in cache_set[partition(r)] and, if its partition
// has one, its group state.
template <typename T>
__global__ void __launch_bounds__(kMergeThreads)
    step_merge_kernel(const __grid_constant__ StepMergeArgs a, int64_t bh_base) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int VEC_SHIFT = VEC == 8 ? 3 : 2;
  uint32_t r;
  int c0;
  if (!thread_row(a.N, a.d, VEC_SHIFT, r, c0)) return;
  const int64_t bh = bh_base + blockIdx.y;
  int i = 0;
  while (r >= static_cast<uint32_t>(a.offsets[i + 1])) ++i;
  const uint64_t set = a.cache_set[i];
  const bool grp = (a.group >> i) & 1u;
  const float* lrow = a.cL + bh * a.P * a.N + r;  // + j * N: lse of cache state j
  const T* orow = static_cast<const T*>(a.cO) + (bh * a.P * a.N + r) * a.d + c0;
  const int64_t jstride = a.N * a.d;

  // rounds of two: measured faster than rounds of four on the Wan-14B layer (0.371 vs 0.395
  // ms: 48 instead of 62 registers, so more rows in flight per SM)
  constexpr int kRound = 2;
  // the group state starts the online merge (weight 1 relative to its own lse)
  float mx = -INFINITY, sum = 0.f;
  float acc[VEC];
  if (grp) {
    mx = __ldg(a.gL + bh * a.N + r) * kLog2e;
    sum = 1.f;
    load_f32<VEC>(a.gO + (bh * a.N + r) * a.d + c0, acc);
  } else {
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  }
  for (uint64_t m = set; m;) {
    uint4 raw[kRound];
    float l[kRound];
    bool use[kRound];
    int j = __ffsll(m) - 1;
#pragma unroll
    for (int q = 0; q < kRound; ++q) {
      use[q] = m != 0;
      if (use[q]) j = __ffsll(m) - 1;  // else repeat the last state (an L1 hit)
      m &= m - 1;
      raw[q] = load_raw(orow + j * jstride);
      l[q] = __ldg(lrow + j * a.N) * kLog2e;
    }
    merge_round<T, VEC, kRound>(raw, l, use, mx, sum, acc);
  }
  const float lse = (mx + lg2(sum)) * kLn2;
  const float inv = 1.f / sum;
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] *= inv;
  const int64_t b = bh / a.H, h = bh - b * a.H;
  T* out = static_cast<T*>(a.out) + b * a.outS[0] + h * a.outS[1] + r * a.outS[2] + c0;
  store_vec(out, acc);
  if (a.out_lse != nullptr && c0 == 0) a.out_lse[b * a.olS[0] + h * a.olS[1] + r * a.olS[2]] = lse;
}

constexpr int64_t kMaxGridY = 65535;

// Blocks along x for R rows of d channels at `vec` channels per thread (0 when the thread
// index would not fit the kernels' 32-bit arithmetic).
unsigned blocks_x(int64_t R, int d, int vec) {
  const int64_t threads = R * (d / vec);
  if (threads >= (int64_t{1} << 32) - kMergeThreads) return 0;
  return static_cast<unsigned>((threads + kMergeThreads - 1) / kMergeThreads);
}

}  // namespace

cudaError_t launch_step_merge(const StepMergeArgs& a, cudaStream_t stream) {
  const int vec = a.dtype == DITANGO_BF16 ? 8 : 4;
  const int64_t groups = a.B * a.H;
  if (groups == 0 || a.N == 0) return cudaSuccess;
  const unsigned bx = blocks_x(a.N, a.d, vec);
  if (bx == 0) return cudaErrorInvalidValue;
  for (int64_t g0 = 0; g0 < groups; g0 += kMaxGridY) {
    const dim3 grid(bx, static_cast<unsigned>(std::min<int64_t>(kMaxGridY, groups - g0)));
    if (a.dtype == DITANGO_BF16)
      step_merge_kernel<__nv_bfloat16><<<grid, kMergeThreads, 0, stream>>>(a, g0);
    else
      step_merge_kernel<float><<<grid, kMergeThreads, 0, stream>>>(a, g0);
  }
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int vec = a.dtype == DITANGO_BF16 ? 8 : 4;
  const int64_t groups = a.G1 * a.G2;
  if (groups == 0 || a.R == 0) return cudaSuccess;
  const unsigned bx = blocks_x(a.R, a.d, vec);
  if (bx == 0) return cudaErrorInvalidValue;
  for (int64_t g0 = 0; g0 < groups; g0 += kMaxGridY) {
    const dim3 grid(bx, static_cast<unsigned>(std::min<int64_t>(kMaxGridY, groups - g0)));
    if (a.dtype == DITANGO_BF16 && a.out_dtype == DITANGO_BF16)
      merge_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, kMergeThreads, 0, stream>>>(a, g0);
    else if (a.dtype == DITANGO_BF16 && a.out_dtype == DITANGO_F32)
      merge_kernel<__nv_bfloat16, float><<<grid, kMergeThreads, 0, stream>>>(a, g0);
    else if (a.dtype == DITANGO_F32 && a.out_dtype == DITANGO_F32)
      merge_kernel<float, float><<<grid, kMergeThreads, 0, stream>>>(a, g0);
    else
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ditango
