// 3D rotary position embedding keyed by a global time index.
//
// Source: "Accelerating Video Generation Inference with Sequential-Parallel 3D Positional
// Encoding Using a Global Time Index" (gist.science/es/paper/2603.06664), section 2,
// Causal-RoPE SP: a token's temporal index is global, t = t_local + s with s the start frame
// of the block, so it is computed locally; the sin/cos frequencies are precomputed into
// contiguous tensors. The channel groups (temporal, horizontal, vertical) follow "Kaleido"
// (gist.science/es/paper/2607.13770), Methodology 1.
//
// Rotation (plain reading): channel pair m = (2m, 2m+1); the first dt/2 pairs turn with t,
// the next dh/2 with h, the last dw/2 with w; pair k of an axis of width d_a turns by
// angle = pos * theta^(-2k/d_a): (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos).
// Token n sits at t = n / (Hl Wl) + s, h = (n / Wl) mod Hl, w = n mod Wl.
//
// rope_apply_kernel: memory bound; one thread rotates 8 channels (4 pairs) of one (b, n, h),
// reading 16 bytes and writing 16 bytes (bf16). The rotation is evaluated in fp32 as
// y0 = fl(fl(x0 c) - fl(x1 s)), y1 = fl(fl(x0 s) + fl(x1 c)) with fp32 tables c, s, then
// rounded (nearest-even) to the storage dtype.
#include <cuda_bf16.h>

#include "ditango_internal.h"

namespace ditango {
namespace {

constexpr int kRopeThreads = 256;
constexpr int kPairsPerThread = 4;


__device__ __forceinline__ void pair_table(const RopeApplyArgs& a, int m, int64_t t, int64_t h,
                                           int64_t w, float& cs, float& sn) {
  const int ht = a.dt / 2, hh = a.dh / 2, hw = a.dw / 2;
  if (m < ht) {
    cs = __ldg(a.cos_t + t * ht + m);
    sn = __ldg(a.sin_t + t * ht + m);
  } else if (m < ht + hh) {
    cs = __ldg(a.cos_h + h * hh + (m - ht));
    sn = __ldg(a.sin_h + h * hh + (m - ht));
  } else {
    cs = __ldg(a.cos_w + w * hw + (m - ht - hh));
    sn = __ldg(a.sin_w + w * hw + (m - ht - hh));
  }
}

template <typename T>
__global__ void __launch_bounds__(kRopeThreads) rope_apply_kernel(const __grid_constant__ RopeApplyArgs a) {
  const int groups = a.d / (2 * kPairsPerThread);  // threads per (b, n, h)
  const int64_t per_tensor = a.B * a.N * a.H * groups;
  const int64_t total = per_tensor * a.n_tensors;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int which = static_cast<int>(idx / per_tensor);
    int64_t rem = idx - which * per_tensor;
    const int grp = static_cast<int>(rem % groups);
    rem /= groups;
    const int64_t hd = rem % a.H;
    rem /= a.H;
    const int64_t n = rem % a.N;
    const int64_t b = rem / a.N;
    const int64_t hw_tokens = a.Hl * a.Wl;
    const int64_t t = n / hw_tokens + a.start_frame;
    const int64_t hh = (n / a.Wl) % a.Hl;
    const int64_t ww = n % a.Wl;
    const T* src = static_cast<const T*>(a.x[which]) + b * a.xs[which][0] + n * a.xs[which][1] +
                   hd * a.xs[which][2] + grp * 2 * kPairsPerThread;
    T* dst = static_cast<T*>(a.y[which]) + ((b * a.N + n) * a.H + hd) * a.d + grp * 2 * kPairsPerThread;
    float x[2 * kPairsPerThread];
    if constexpr (sizeof(T) == 2) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[2 * i] = __uint_as_float(wv[i] << 16);
        x[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
      }
    } else {
      const float4 v0 = __ldg(reinterpret_cast<const float4*>(src));
      const float4 v1 = __ldg(reinterpret_cast<const float4*>(src) + 1);
      x[0] = v0.x; x[1] = v0.y; x[2] = v0.z; x[3] = v0.w;
      x[4] = v1.x; x[5] = v1.y; x[6] = v1.z; x[7] = v1.w;
    }
    float y[2 * kPairsPerThread];
#pragma unroll
    for (int p = 0; p < kPairsPerThread; ++p) {
      const int m = grp * kPairsPerThread + p;
      float cs, sn;
      pair_table(a, m, t, hh, ww, cs, sn);
      // explicit round-to-nearest products and sums (never contracted into FMA), so that the
      // rotated value rounded to the storage dtype is a reproducible fp32 result
      y[2 * p] = __fsub_rn(__fmul_rn(x[2 * p], cs), __fmul_rn(x[2 * p + 1], sn));
      y[2 * p + 1] = __fadd_rn(__fmul_rn(x[2 * p], sn), __fmul_rn(x[2 * p + 1], cs));
    }
    if constexpr (sizeof(T) == 2) {
      uint32_t wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h2 = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
        wv[i] = *reinterpret_cast<uint32_t*>(&h2);
      }
      *reinterpret_cast<uint4*>(dst) = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    } else {
      reinterpret_cast<float4*>(dst)[0] = make_float4(y[0], y[1], y[2], y[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
  }
}

// cos/sin tables: entry [pos, k] of an axis of width d_a holds cos/sin(pos * theta^(-2k/d_a)),
// evaluated in fp64 and rounded to fp32.
__global__ void rope_tables_kernel(float* c, float* s, int64_t rows, int32_t half, int32_t width,
                                   double theta) {
  const int64_t n = rows * half;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t pos = idx / half;
    const int32_t k = static_cast<int32_t>(idx - pos * half);
    const double inv_freq = pow(theta, -2.0 * static_cast<double>(k) / static_cast<double>(width));
    double sv, cv;
    sincos(static_cast<double>(pos) * inv_freq, &sv, &cv);
    c[idx] = static_cast<float>(cv);
    s[idx] = static_cast<float>(sv);
  }
}

}  // namespace

cudaError_t launch_rope_apply(const RopeApplyArgs& a, cudaStream_t stream) {
  const int64_t total = a.B * a.N * a.H * (a.d / (2 * kPairsPerThread)) * a.n_tensors;
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + kRopeThreads - 1) / kRopeThreads;
  if (blocks > 152 * 32) blocks = 152 * 32;  // grid-stride beyond 32 waves of the SM count
  if (a.dtype == DITANGO_BF16)
    rope_apply_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kRopeThreads, 0, stream>>>(a);
  else
    rope_apply_kernel<float><<<static_cast<unsigned>(blocks), kRopeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_tables(const ditango_rope& r, double theta, cudaStream_t stream) {
  struct Ax { float* c; float* s; int64_t rows; int32_t width; } ax[3] = {
      {r.cos_t, r.sin_t, r.T_tab, r.dt}, {r.cos_h, r.sin_h, r.Hl, r.dh}, {r.cos_w, r.sin_w, r.Wl, r.dw}};
  for (const Ax& x : ax) {
    const int32_t half = x.width / 2;
    const int64_t n = x.rows * half;
    if (n == 0) continue;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    rope_tables_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x.c, x.s, x.rows, half,
                                                                          x.width, theta);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ditango
