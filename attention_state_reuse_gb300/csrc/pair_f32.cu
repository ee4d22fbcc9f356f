// Partition-pair attention states in fp32 on the CUDA cores.
//
// Same definition as the tensor-core kernel (DiTango, gist.science/paper/2607.15650,
// Methodology 2, State Composition): for computed pairs (i, j),
//   lse_ij[r] = ln sum_{c in j} exp(z_c),  O_ij[r] = sum_{c in j} exp(z_c - lse_ij[r]) v_c,
//   z_c = scale <q_r, k_c>.
// This path serves fp32 inputs, whose tolerance (1e-4 absolute) the tf32 tensor-core rate
// cannot meet; it uses fp32 FMA throughout and accurate expf/logf.
//
// One block per unit (64 query rows of partition i for one (b, h)); the block visits every
// computed KV partition j in ascending order and writes one state per j into the cache.
// D/32 consecutive threads share a query row, each owning 32 channels of q and of the running
// output; partial dot products are combined with warp shuffles. K and V are staged through
// shared memory 32 keys at a time.
#include "ditango_internal.h"

namespace ditango {
namespace {

constexpr int kRows = 64;
constexpr int kKeys = 32;

template <int D>
__global__ void __launch_bounds__(kRows * (D / 32))
    pair_f32_kernel(const __grid_constant__ PairF32Args a) {
  constexpr int TPR = D / 32;
  constexpr int NT = kRows * TPR;
  __shared__ float ks[kKeys][D];
  __shared__ float vs[kKeys][D];
  const PairSchedule& sch = a.sched;

  // decode the unit (same numbering as the tensor-core kernel, 64-row blocks)
  const int u = blockIdx.x;
  int kk = 0;
  while (u >= sch.seg_start[kk + 1]) ++kk;
  const int i = sch.order[kk];
  const int local = u - sch.seg_start[kk];
  const int n_i = sch.offsets[i + 1] - sch.offsets[i];
  const int blocks = (n_i + kRows - 1) / kRows;
  const int bh = local / blocks;
  const int qb = local - bh * blocks;
  const int b = bh / sch.H;
  const int h = bh - b * sch.H;

  const int lrow = threadIdx.x / TPR;
  const int part = threadIdx.x % TPR;
  const int prow = qb * kRows + lrow;  // row within partition i
  const bool row_ok = prow < n_i;
  const int64_t r = sch.offsets[i] + (row_ok ? prow : 0);

  float q[32];
  {
    const float* qp = a.q + b * a.qs[0] + r * a.qs[1] + h * a.qs[2] + part * 32;
#pragma unroll
    for (int e = 0; e < 32; ++e) q[e] = qp[e];
  }

  for (uint64_t m = sch.compute_mask[i]; m; m &= m - 1) {
    const int j = __ffsll(static_cast<long long>(m)) - 1;
    const int j0 = sch.offsets[j];
    const int nj = sch.offsets[j + 1] - j0;
    float m_run = -INFINITY, l_run = 0.f;
    float acc[32];
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
    for (int c0 = 0; c0 < nj; c0 += kKeys) {
      const int valid = min(kKeys, nj - c0);
      __syncthreads();
      for (int x = threadIdx.x; x < kKeys * D; x += NT) {
        const int c = x / D, e = x - (x / D) * D;
        float kv = 0.f, vv = 0.f;
        if (c < valid) {
          const int64_t row = j0 + c0 + c;
          kv = a.k[b * a.ks[0] + row * a.ks[1] + h * a.ks[2] + e];
          vv = a.v[b * a.vs[0] + row * a.vs[1] + h * a.vs[2] + e];
        }
        ks[c][e] = kv;
        vs[c][e] = vv;
      }
      __syncthreads();
      float z[kKeys];
      float m_tile = -INFINITY;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) dot = fmaf(q[e], ks[c][part * 32 + e], dot);
#pragma unroll
        for (int o = 1; o < TPR; o <<= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        z[c] = c < valid ? dot * a.scale : -INFINITY;
        m_tile = fmaxf(m_tile, z[c]);
      }
      const float m_new = fmaxf(m_run, m_tile);
      const float alpha = expf(m_run - m_new);  // 0 on the first tile (m_run = -inf)
      l_run *= alpha;
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[e] *= alpha;
#pragma unroll
      for (int c = 0; c < kKeys; ++c) {
        const float p = expf(z[c] - m_new);
        l_run += p;
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] = fmaf(p, vs[c][part * 32 + e], acc[e]);
      }
      m_run = m_new;
    }
    if (row_ok) {
      float* o;
      float* lse_p;
      state_ptrs(a.cache, sch.P, a.N, D, static_cast<int64_t>(b) * sch.H + h, i, j, r, o, lse_p);
      o += part * 32;
      const float inv_l = 1.f / l_run;
#pragma unroll
      for (int e = 0; e < 32; e += 4)
        *reinterpret_cast<float4*>(o + e) =
            make_float4(acc[e] * inv_l, acc[e + 1] * inv_l, acc[e + 2] * inv_l, acc[e + 3] * inv_l);
      if (part == 0) *lse_p = m_run + logf(l_run);
    }
  }
}

}  // namespace

cudaError_t launch_pair_f32(int d, const PairF32Args& a, cudaStream_t stream) {
  if (a.sched.n_units <= 0) return cudaSuccess;
  if (d == 64)
    pair_f32_kernel<64><<<a.sched.n_units, kRows * 2, 0, stream>>>(a);
  else if (d == 128)
    pair_f32_kernel<128><<<a.sched.n_units, kRows * 4, 0, stream>>>(a);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace ditango
