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
// rope_apply_kernel: memory bound; a thread rotates the 16-byte vectors (8 bf16 or 4 fp32
// channels) of one (head, channel group) for several tokens, reading and writing 16 bytes each. bf16: every output is the
// nearest-even bf16 of the rotation with fp64 cos/sin (rope_round.cuh: an fp32 fast path with
// an error bound, and an exact slow path from the residual tables when a rounding midpoint is
// too close). fp32: y0 = fma(x0, c, -fl(x1 s)), y1 = fma(x0, s, fl(x1 c)).
#include <cuda_bf16.h>

#include "ditango_internal.h"
#include "rope_round.cuh"

namespace ditango {
namespace {

constexpr int kRopeThreads = 256;
constexpr int kMaxPairs = 64;  // d <= 128
constexpr int kRopeTok = 4;    // tokens per block round

// A block takes kRopeTok consecutive tokens per round (grid-stride over rounds): it decodes
// their positions (t, h, w), stages the cos/sin of their d/2 channel pairs in shared memory,
// then each thread takes one 16-byte vector slot (tensor, head, channel group) and handles it
// for all kRopeTok tokens, issuing the kRopeTok loads before using any, so that every thread
// keeps several independent loads in flight. The rows of one token are contiguous across
// heads, so a warp's loads and stores are fully coalesced.
template <typename T>
__global__ void __launch_bounds__(kRopeThreads, 4) rope_apply_kernel(const __grid_constant__ RopeApplyArgs a) {
  constexpr int VEC = 16 / sizeof(T);  // channels per 16-byte vector
  __shared__ float2 cs_s[kRopeTok][kMaxPairs];  // (cos, sin) of pair m of token tt
  __shared__ int idx_s[kRopeTok][kMaxPairs];    // its table index (for the residuals, rarely read)
  __shared__ int64_t src_s[kRopeTok][2];        // element offset of token tt in x[0], x[1]
  const int pairs = a.d / 2;
  const int ht = a.dt / 2, hh = a.dh / 2, hw = a.dw / 2;
  const int vpr_shift = 31 - __clz(a.d / VEC);  // vectors per (token, head): d / VEC = 2^shift
  const int vpr = 1 << vpr_shift;
  const int per_tensor = static_cast<int>(a.H) * vpr;
  const int per_token = a.n_tensors * per_tensor;
  const int64_t tokens = a.B * a.N;
  const int hw_tokens = static_cast<int>(a.Hl * a.Wl);
  for (int64_t tok0 = static_cast<int64_t>(blockIdx.x) * kRopeTok; tok0 < tokens;
       tok0 += static_cast<int64_t>(gridDim.x) * kRopeTok) {
    const int ntok = tokens - tok0 < kRopeTok ? static_cast<int>(tokens - tok0) : kRopeTok;
    __syncthreads();  // the previous round's tables are no longer read
    for (int x = threadIdx.x; x < ntok * pairs; x += blockDim.x) {
      const int tt = x / pairs, m = x - tt * pairs;
      const int n = static_cast<int>((tok0 + tt) % a.N);
      const float *c, *sn;
      int idx;
      if (m < ht) {
        idx = (n / hw_tokens + static_cast<int>(a.start_frame)) * ht + m;
        c = a.cos_t; sn = a.sin_t;
      } else if (m < ht + hh) {
        idx = ((n / static_cast<int>(a.Wl)) % static_cast<int>(a.Hl)) * hh + (m - ht);
        c = a.cos_h; sn = a.sin_h;
      } else {
        idx = (n % static_cast<int>(a.Wl)) * hw + (m - ht - hh);
        c = a.cos_w; sn = a.sin_w;
      }
      cs_s[tt][m] = make_float2(__ldg(c + idx), __ldg(sn + idx));
      idx_s[tt][m] = idx;
    }
    if (threadIdx.x < 2 * ntok) {
      const int tt = threadIdx.x >> 1, which = threadIdx.x & 1;
      const int64_t tok = tok0 + tt, b = tok / a.N, n = tok - b * a.N;
      src_s[tt][which] = b * a.xs[which][0] + n * a.xs[which][1];
    }
    __syncthreads();
    for (int v = threadIdx.x; v < per_token; v += blockDim.x) {
      const int which = v >= per_tensor ? 1 : 0;
      const int rem = v - which * per_tensor;
      const int hd = rem >> vpr_shift;
      const int grp = rem & (vpr - 1);
      const T* src0 = static_cast<const T*>(a.x[which]) + hd * a.xs[which][2] + grp * VEC;
      uint4 raw[kRopeTok];
#pragma unroll
      for (int tt = 0; tt < kRopeTok; ++tt)
        if (tt < ntok) raw[tt] = __ldg(reinterpret_cast<const uint4*>(src0 + src_s[tt][which]));
#pragma unroll
      for (int tt = 0; tt < kRopeTok; ++tt) {
        if (tt >= ntok) break;
        T* dst = static_cast<T*>(a.y[which]) + ((tok0 + tt) * a.H + hd) * a.d + grp * VEC;
        if constexpr (sizeof(T) == 2) {
          const uint32_t wv[4] = {raw[tt].x, raw[tt].y, raw[tt].z, raw[tt].w};
          uint32_t o[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const int m = grp * 4 + p;
            const float2 cs = cs_s[tt][m];
            o[p] = rope_rotate_bf16x2(
                __uint_as_float(wv[p] << 16), __uint_as_float(wv[p] & 0xFFFF0000u), cs.x, cs.y,
                [&](float& c_lo, float& s_lo) {
                  const int idx = idx_s[tt][m];
                  const bool t_ax = m < ht, h_ax = m < ht + hh;
                  c_lo = __ldg((t_ax ? a.cos_t_lo : h_ax ? a.cos_h_lo : a.cos_w_lo) + idx);
                  s_lo = __ldg((t_ax ? a.sin_t_lo : h_ax ? a.sin_h_lo : a.sin_w_lo) + idx);
                });
          }
          *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
          const float x[4] = {__uint_as_float(raw[tt].x), __uint_as_float(raw[tt].y),
                              __uint_as_float(raw[tt].z), __uint_as_float(raw[tt].w)};
          float y[4];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            const float2 cs = cs_s[tt][grp * 2 + p];
            y[2 * p] = __fmaf_rn(x[2 * p], cs.x, -__fmul_rn(x[2 * p + 1], cs.y));
            y[2 * p + 1] = __fmaf_rn(x[2 * p], cs.y, __fmul_rn(x[2 * p + 1], cs.x));
          }
          *reinterpret_cast<float4*>(dst) = make_float4(y[0], y[1], y[2], y[3]);
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
  // four blocks of 256 threads per SM (152 SMs; registers capped for four), each walking many
  // token rounds
  const int64_t rounds = (tokens + kRopeTok - 1) / kRopeTok;
  const int64_t blocks = rounds < 152 * 4 ? rounds : 152 * 4;
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
