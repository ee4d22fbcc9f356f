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
// rope_apply_kernel: memory bound; a thread rotates the 16-byte vector (8 bf16 or 4 fp32
// channels) of one (token, head), reading and writing 16 bytes. The rotation is evaluated in fp32 as
// y0 = fl(fl(x0 c) - fl(x1 s)), y1 = fl(fl(x0 s) + fl(x1 c)) with fp32 tables c, s, then
// rounded (nearest-even) to the storage dtype.
#include <cuda_bf16.h>

#include "ditango_internal.h"

namespace ditango {
namespace {

constexpr int kRopeThreads = 256;
constexpr int kMaxPairs = 64;  // d <= 128

// One block per token at a time (grid-stride over tokens): the token's position (t, h, w) is
// decoded once, the cos/sin of its d/2 channel pairs are staged in shared memory, then the
// block streams every head of q and k for that token with 16-byte vectors (the rows of one
// token are contiguous across heads, so the loads and stores are fully coalesced).
template <typename T>
__global__ void __launch_bounds__(kRopeThreads) rope_apply_kernel(const __grid_constant__ RopeApplyArgs a) {
  constexpr int VEC = 16 / sizeof(T);  // channels per 16-byte vector
  __shared__ float cs_s[kMaxPairs], sn_s[kMaxPairs];
  const int pairs = a.d / 2;
  const int ht = a.dt / 2, hh = a.dh / 2, hw = a.dw / 2;
  const int vpr = a.d / VEC;  // vectors per (token, head)
  const int per_tensor = static_cast<int>(a.H) * vpr;
  const int per_token = a.n_tensors * per_tensor;
  const int64_t tokens = a.B * a.N;
  const int hw_tokens = static_cast<int>(a.Hl * a.Wl);
  for (int64_t tok = blockIdx.x; tok < tokens; tok += gridDim.x) {
    const int64_t b = tok / a.N;
    const int n = static_cast<int>(tok - b * a.N);
    const int t = n / hw_tokens + static_cast<int>(a.start_frame);
    const int hp = (n / static_cast<int>(a.Wl)) % static_cast<int>(a.Hl);
    const int wp = n % static_cast<int>(a.Wl);
    __syncthreads();  // the previous token's tables are no longer read
    for (int m = threadIdx.x; m < pairs; m += blockDim.x) {
      float c, sn;
      if (m < ht) {
        c = __ldg(a.cos_t + t * ht + m);
        sn = __ldg(a.sin_t + t * ht + m);
      } else if (m < ht + hh) {
        c = __ldg(a.cos_h + hp * hh + (m - ht));
        sn = __ldg(a.sin_h + hp * hh + (m - ht));
      } else {
        c = __ldg(a.cos_w + wp * hw + (m - ht - hh));
        sn = __ldg(a.sin_w + wp * hw + (m - ht - hh));
      }
      cs_s[m] = c;
      sn_s[m] = sn;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < per_token; v += blockDim.x) {
      const int which = v >= per_tensor ? 1 : 0;
      const int rem = v - which * per_tensor;
      const int hd = rem / vpr;
      const int grp = rem - hd * vpr;
      const T* __restrict__ src = static_cast<const T*>(a.x[which]) + b * a.xs[which][0] +
                                  static_cast<int64_t>(n) * a.xs[which][1] + hd * a.xs[which][2] +
                                  grp * VEC;
      T* __restrict__ dst = static_cast<T*>(a.y[which]) + (tok * a.H + hd) * a.d + grp * VEC;
      float x[VEC];
      if constexpr (sizeof(T) == 2) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(src));
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[2 * i] = __uint_as_float(wv[i] << 16);
          x[2 * i + 1] = __uint_as_float(wv[i] & 0xFFFF0000u);
        }
      } else {
        const float4 u = __ldg(reinterpret_cast<const float4*>(src));
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
      }
      float y[VEC];
#pragma unroll
      for (int p = 0; p < VEC / 2; ++p) {
        const float c = cs_s[grp * (VEC / 2) + p], sn = sn_s[grp * (VEC / 2) + p];
        // explicit round-to-nearest products and sums (never contracted into FMA), so that the
        // rotated value rounded to the storage dtype is a reproducible fp32 result
        y[2 * p] = __fsub_rn(__fmul_rn(x[2 * p], c), __fmul_rn(x[2 * p + 1], sn));
        y[2 * p + 1] = __fadd_rn(__fmul_rn(x[2 * p], sn), __fmul_rn(x[2 * p + 1], c));
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
        *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
      }
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
  const int64_t tokens = a.B * a.N;
  if (tokens == 0 || a.n_tensors == 0) return cudaSuccess;
  if (a.d / 2 > kMaxPairs) return cudaErrorInvalidValue;
  // up to 16 blocks of 256 threads per SM (152 SMs); each block walks many tokens
  const int64_t blocks = tokens < 152 * 16 ? tokens : 152 * 16;
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
