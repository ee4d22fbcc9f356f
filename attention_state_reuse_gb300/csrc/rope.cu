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
// rope_apply_kernel: memory bound; a warp rotates one token's rows (every head) at a time, a
// lane the 16-byte vectors (8 bf16 or 4 fp32 channels) of one channel group. bf16: every
// output is the nearest-even bf16 of the rotation with fp64 cos/sin (rope_round.cuh: an fp32 fast path with
// an error bound, and an exact slow path from the residual tables when a rounding midpoint is
// too close). fp32: y0 = fma(x0, c, -fl(x1 s)), y1 = fma(x0, s, fl(x1 c)).
#include <cuda_bf16.h>

#include "ditango_internal.h"
#include "rope_round.cuh"

namespace ditango {
namespace {

constexpr int kRopeThreads = 256;
constexpr int kMaxPairs = 64;  // d <= 128
constexpr int kRopeBatch = 2;  // vectors a lane loads before it uses the first

// One warp per token (grid-stride over tokens). A row of d channels is d/VEC 16-byte vectors,
// and d/VEC divides 32, so lane l always owns the same vector slot g = l mod (d/VEC) of heads
// l/(d/VEC), l/(d/VEC) + 32/(d/VEC), ...: its VEC/2 channel pairs are fixed, and it looks up
// their cos/sin once per token (small tables, cached) instead of staging them in shared
// memory. A warp's loads and stores of one head group are contiguous (512 bytes). Four blocks
// of 256 per SM (at most 64 registers) and two vectors in flight per lane: measured 0.373 ms
// on the 720p layer's k against 0.395 ms for blocks that staged four tokens' tables in shared
// memory, 0.39-0.42 ms for four or five vectors per lane at two or three blocks.
template <typename T>
__global__ void __launch_bounds__(kRopeThreads, 4) rope_apply_kernel(const __grid_constant__ RopeApplyArgs a) {
  constexpr int VEC = 16 / sizeof(T);  // channels per 16-byte vector
  constexpr int PPV = VEC / 2;         // channel pairs per vector
  const int lane = threadIdx.x & 31;
  const int vpr = a.d / VEC;           // vectors per (token, head): 8, 16 or 32
  const int g = lane & (vpr - 1);
  const int hd0 = lane / vpr, hstep = 32 / vpr;
  const int ht = a.dt / 2, hh = a.dh / 2;
  const int hw_tokens = static_cast<int>(a.Hl * a.Wl);
  // this lane's pairs: axis (0 t, 1 h, 2 w) and index within the axis
  int axis[PPV], kk[PPV];
#pragma unroll
  for (int p = 0; p < PPV; ++p) {
    const int m = g * PPV + p;
    axis[p] = m < ht ? 0 : (m < ht + hh ? 1 : 2);
    kk[p] = m - (axis[p] == 0 ? 0 : (axis[p] == 1 ? ht : ht + hh));
  }
  const int half_t = ht, half_h = hh, half_w = a.dw / 2;
  const int64_t tokens = a.B * a.N;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kRopeThreads / 32);
  for (int64_t tok = static_cast<int64_t>(blockIdx.x) * (kRopeThreads / 32) + (threadIdx.x >> 5);
       tok < tokens; tok += warps) {
    const int64_t b = tok / a.N;
    const int n = static_cast<int>(tok - b * a.N);
    const int pt = n / hw_tokens + static_cast<int>(a.start_frame);
    const int ph = (n / static_cast<int>(a.Wl)) % static_cast<int>(a.Hl);
    const int pw = n % static_cast<int>(a.Wl);
    float c[PPV], sn[PPV];
    int idx[PPV];
#pragma unroll
    for (int p = 0; p < PPV; ++p) {
      const bool t_ax = axis[p] == 0, h_ax = axis[p] == 1;
      idx[p] = (t_ax ? pt * half_t : (h_ax ? ph * half_h : pw * half_w)) + kk[p];
      c[p] = __ldg((t_ax ? a.cos_t : h_ax ? a.cos_h : a.cos_w) + idx[p]);
      sn[p] = __ldg((t_ax ? a.sin_t : h_ax ? a.sin_h : a.sin_w) + idx[p]);
    }
    for (int which = 0; which < a.n_tensors; ++which) {
      const T* src = static_cast<const T*>(a.x[which]) + b * a.xs[which][0] + n * a.xs[which][1] +
                     g * VEC;
      T* dst = static_cast<T*>(a.y[which]) + tok * a.H * a.d + g * VEC;
      const int64_t hs = a.xs[which][2];
      for (int hd = hd0; hd < a.H; hd += hstep * kRopeBatch) {
        uint4 raw[kRopeBatch];
#pragma unroll
        for (int q = 0; q < kRopeBatch; ++q) {
          const int hq = hd + q * hstep;
          if (hq < a.H) raw[q] = __ldg(reinterpret_cast<const uint4*>(src + hq * hs));
        }
#pragma unroll
        for (int q = 0; q < kRopeBatch; ++q) {
          const int hq = hd + q * hstep;
          if (hq >= a.H) break;
          T* out = dst + static_cast<int64_t>(hq) * a.d;
          if constexpr (sizeof(T) == 2) {
            const uint32_t wv[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
            uint32_t o[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              o[p] = rope_rotate_bf16x2(
                  __uint_as_float(wv[p] << 16), __uint_as_float(wv[p] & 0xFFFF0000u), c[p], sn[p],
                  [&](float& c_lo, float& s_lo) {
                    const bool t_ax = axis[p] == 0, h_ax = axis[p] == 1;
                    c_lo = __ldg((t_ax ? a.cos_t_lo : h_ax ? a.cos_h_lo : a.cos_w_lo) + idx[p]);
                    s_lo = __ldg((t_ax ? a.sin_t_lo : h_ax ? a.sin_h_lo : a.sin_w_lo) + idx[p]);
                  });
            }
            *reinterpret_cast<uint4*>(out) = make_uint4(o[0], o[1], o[2], o[3]);
          } else {
            const float x[4] = {__uint_as_float(raw[q].x), __uint_as_float(raw[q].y),
                                __uint_as_float(raw[q].z), __uint_as_float(raw[q].w)};
            float y[4];
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              y[2 * p] = __fmaf_rn(x[2 * p], c[p], -__fmul_rn(x[2 * p + 1], sn[p]));
              y[2 * p + 1] = __fmaf_rn(x[2 * p], sn[p], __fmul_rn(x[2 * p + 1], c[p]));
            }
            *reinterpret_cast<float4*>(out) = make_float4(y[0], y[1], y[2], y[3]);
          }
        }
      }
    }
  }
}

// cos/sin tables: entry [pos, k] of an axis of width d_a holds cos/sin(pos * theta^(-2k/d_a)),
// evaluated in fp64 and rounded to fp32; the residual tables hold the fp32 rounding of what
// that rounding left out.
__global__ void rope_tables_kernel(float* c, float* s, float* c_lo, float* s_lo, int64_t rows,
                                   int32_t half, int32_t width, double theta) {
  const int64_t n = rows * half;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t pos = idx / half;
    const int32_t k = static_cast<int32_t>(idx - pos * half);
    const double inv_freq = pow(theta, -2.0 * static_cast<double>(k) / static_cast<double>(width));
    double sv, cv;
    sincos(static_cast<double>(pos) * inv_freq, &sv, &cv);
    const float ch = static_cast<float>(cv), sh = static_cast<float>(sv);
    c[idx] = ch;
    s[idx] = sh;
    c_lo[idx] = static_cast<float>(cv - static_cast<double>(ch));
    s_lo[idx] = static_cast<float>(sv - static_cast<double>(sh));
  }
}

}  // namespace

cudaError_t launch_rope_apply(const RopeApplyArgs& a, cudaStream_t stream) {
  const int64_t tokens = a.B * a.N;
  if (tokens == 0 || a.n_tensors == 0) return cudaSuccess;
  if (a.d / 2 > kMaxPairs) return cudaErrorInvalidValue;
  const int vec = a.dtype == DITANGO_BF16 ? 8 : 4;
  if (a.d % vec != 0 || 32 % (a.d / vec) != 0) return cudaErrorInvalidValue;  // d/VEC divides 32
  // one warp per token, eight warps per block, at most 152 x 8 blocks
  const int64_t want = (tokens + kRopeThreads / 32 - 1) / (kRopeThreads / 32);
  const int64_t blocks = want < 152 * 8 ? want : 152 * 8;
  if (a.dtype == DITANGO_BF16)
    rope_apply_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), kRopeThreads, 0, stream>>>(a);
  else
    rope_apply_kernel<float><<<static_cast<unsigned>(blocks), kRopeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_rope_tables(const ditango_rope& r, double theta, cudaStream_t stream) {
  struct Ax { float *c, *s, *c_lo, *s_lo; int64_t rows; int32_t width; } ax[3] = {
      {r.cos_t, r.sin_t, r.cos_t_lo, r.sin_t_lo, r.T_tab, r.dt},
      {r.cos_h, r.sin_h, r.cos_h_lo, r.sin_h_lo, r.Hl, r.dh},
      {r.cos_w, r.sin_w, r.cos_w_lo, r.sin_w_lo, r.Wl, r.dw}};
  for (const Ax& x : ax) {
    const int32_t half = x.width / 2;
    const int64_t n = x.rows * half;
    if (n == 0) continue;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 1024) blocks = 1024;
    rope_tables_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        x.c, x.s, x.c_lo, x.s_lo, x.rows, half, x.width, theta);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ditango
