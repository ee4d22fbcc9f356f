// Reductions of the anchor-guided selection planner over a layer's state cache.
//
// Method: DiTango (gist.science/paper/2607.15650), Methodology 1, Anchor-Guided Selection
// Planner, read plainly (the page gives the ingredients, not formulas):
//   importance  w[i][j] = mean over the rows r of partition i (all batch entries and heads) of
//               the merge weight exp(lse_ij[r] - lse_i[r]) of state (i, j), lse_i the
//               log-sum-exp over j: partition j's share of partition i's attention mass at an
//               anchor step (every row's weights sum to 1, so every row of w does);
//   drift       delta[i] = ||O_ii(t) - O_ii(anchor)|| / ||O_ii(anchor)||: the change of the
//               always-computed local states since the anchor, the proxy for how far the
//               reused remote states have drifted.
// Both are small memory-bound reductions run once per step at most. Rows are reduced within a
// warp when the warp's rows lie in one partition (the common case: partitions span thousands
// of rows), else lane by lane, into shared-memory sums, then into fp64 device sums.
#include <cuda_bf16.h>

#include "ditango_internal.h"

namespace ditango {
namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ int partition_of(const PlannerArgs& a, int64_t r) {
  int i = 0;
  while (r >= a.offsets[i + 1]) ++i;
  return i;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Adds v to acc[slot]: once per warp when every lane of the warp targets the same slot.
__device__ __forceinline__ void add_slot(float* acc, int slot, float v, bool uniform) {
  if (uniform) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) atomicAdd(acc + slot, v);
  } else {
    atomicAdd(acc + slot, v);
  }
}

// One thread per query row r of (b, h) = blockIdx.y: the P merge weights of the row, summed
// into row partition(r) of the block's P x P table.
__global__ void __launch_bounds__(kThreads) importance_kernel(const __grid_constant__ PlannerArgs a) {
  __shared__ float acc[kMaxP * kMaxP];
  const int PP = a.P * a.P;
  for (int x = threadIdx.x; x < PP; x += kThreads) acc[x] = 0.f;
  __syncthreads();
  const int64_t r = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const bool live = r < a.N;
  const int64_t rr = live ? r : a.N - 1;
  const int i = partition_of(a, rr);
  const int i0 = __shfl_sync(0xffffffffu, i, 0);  // every lane takes part, live or not
  const bool uniform = __all_sync(0xffffffffu, live && i == i0);
  // lse of state j of the row (a device slot, or its host slot for a state kept in host memory)
  auto lse_of = [&](int j) {
    char* o;
    float* l;
    state_ptrs(a.cache, a.P, a.N, 0, static_cast<int64_t>(blockIdx.y), i, j, rr, o, l);
    return *l;
  };
  float mx = -INFINITY;
  for (int j = 0; j < a.P; ++j) mx = fmaxf(mx, lse_of(j));
  float sum = 0.f;
  for (int j = 0; j < a.P; ++j) sum += exp2f((lse_of(j) - mx) * kLog2e);
  const float inv = 1.f / sum;
  for (int j = 0; j < a.P; ++j) {
    const float wj = live ? exp2f((lse_of(j) - mx) * kLog2e) * inv : 0.f;
    add_slot(acc, i * a.P + j, wj, uniform);
  }
  __syncthreads();
  for (int x = threadIdx.x; x < PP; x += kThreads)
    if (acc[x] != 0.f) atomicAdd(a.sums + x, static_cast<double>(acc[x]));
}

__global__ void importance_finalize(const __grid_constant__ PlannerArgs a) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= a.P * a.P) return;
  const int i = x / a.P;
  const double rows = static_cast<double>(a.B * a.H) * (a.offsets[i + 1] - a.offsets[i]);
  a.out[x] = a.sums[x] / rows;
}

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  const float4 u = __ldg(reinterpret_cast<const float4*>(p));
  const float4 v = __ldg(reinterpret_cast<const float4*>(p) + 1);
  x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
  x[4] = v.x; x[5] = v.y; x[6] = v.z; x[7] = v.w;
}

// Sums of row r's (O_ii - O_ii(anchor))^2 and O_ii(anchor)^2 over this thread's 8 channels
// c0..c0+7 of (b, h) slab bh, i = partition(r).
template <typename T>
__device__ __forceinline__ void drift_terms(const PlannerArgs& a, int64_t bh, int i, int64_t r,
                                            int c0, float& num, float& den) {
  T* o;
  float* l;
  state_ptrs(a.cache, a.P, a.N, a.d, bh, i, i, r, o, l);  // the local state (i, i)
  const T* ref = static_cast<const T*>(a.snap) + (bh * a.N + r) * a.d;
  float x[8], y[8];
  load8(o + c0, x);
  load8(ref + c0, y);
  num = den = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float df = x[k] - y[k];
    num = fmaf(df, df, num);
    den = fmaf(y[k], y[k], den);
  }
}

// A block takes kThreads consecutive rows of (b, h) = blockIdx.y, d/8 threads per row at a
// time (each over 8 channels, so that a warp reads whole rows, coalesced), in d/8 rounds, into
// the block's 2P sums, then once per block into the fp64 device sums. When the block's rows
// lie in at most two partitions (partitions longer than the block), a thread keeps one pair of
// sums per partition in registers and the block reduces them once at the end, so the rounds'
// loads do not wait on reductions; otherwise every round is reduced on its own.
// tpr_shift = log2(d/8).
template <typename T>
__global__ void __launch_bounds__(kThreads) drift_kernel(const __grid_constant__ PlannerArgs a,
                                                         int tpr_shift) {
  __shared__ float acc[2 * kMaxP];
  for (int x = threadIdx.x; x < 2 * a.P; x += kThreads) acc[x] = 0.f;
  __syncthreads();
  const int rows_per_round = kThreads >> tpr_shift;
  const int rounds = 1 << tpr_shift;
  const int c0 = (threadIdx.x & (rounds - 1)) * 8;
  const int64_t bh = blockIdx.y;
  const int64_t r_first = static_cast<int64_t>(blockIdx.x) * kThreads;
  const int64_t r_last = (r_first + kThreads < a.N ? r_first + kThreads : a.N) - 1;
  const int ia = partition_of(a, r_first), ib = partition_of(a, r_last);  // block-uniform
  if (ib - ia <= 1) {
    const int64_t split = a.offsets[ib];  // first row of partition ib
    float na = 0.f, da = 0.f, nb = 0.f, db = 0.f;
#pragma unroll 4
    for (int round = 0; round < rounds; ++round) {
      const int64_t r = r_first + round * rows_per_round + (threadIdx.x >> tpr_shift);
      if (r <= r_last) {
        const bool in_a = ib == ia || r < split;
        float num, den;
        drift_terms<T>(a, bh, in_a ? ia : ib, r, c0, num, den);
        if (in_a) {
          na += num;
          da += den;
        } else {
          nb += num;
          db += den;
        }
      }
    }
    add_slot(acc, 2 * ia, na, true);
    add_slot(acc, 2 * ia + 1, da, true);
    if (ib != ia) {
      add_slot(acc, 2 * ib, nb, true);
      add_slot(acc, 2 * ib + 1, db, true);
    }
  } else {
    for (int round = 0; round < rounds; ++round) {
      const int64_t r = r_first + round * rows_per_round + (threadIdx.x >> tpr_shift);
      const bool live = r <= r_last;
      const int64_t rr = live ? r : r_last;
      const int i = partition_of(a, rr);
      const int i0 = __shfl_sync(0xffffffffu, i, 0);  // every lane takes part, live or not
      const bool uniform = __all_sync(0xffffffffu, live && i == i0);
      float num, den;
      drift_terms<T>(a, bh, i, rr, c0, num, den);
      if (!live) num = den = 0.f;
      add_slot(acc, 2 * i, num, uniform);
      add_slot(acc, 2 * i + 1, den, uniform);
    }
  }
  __syncthreads();
  for (int x2 = threadIdx.x; x2 < 2 * a.P; x2 += kThreads)
    if (acc[x2] != 0.f) atomicAdd(a.sums + x2, static_cast<double>(acc[x2]));
}

// The snapshot: row r of (b, h) = blockIdx.y copied from its local state (i, i) (a device
// slot) into snap [B, H, N, d]. Same thread layout as drift_kernel: 256 rows per block, d/8
// threads per row at a time, 8 elements (16 or 32 bytes) per thread and round.
template <typename T>
__global__ void __launch_bounds__(kThreads) snapshot_kernel(const __grid_constant__ PlannerArgs a,
                                                            int tpr_shift) {
  constexpr int V = 8 * static_cast<int>(sizeof(T)) / 16;  // 16-byte vectors per thread
  const int rows_per_round = kThreads >> tpr_shift;
  const int rounds = 1 << tpr_shift;
  const int c0 = (threadIdx.x & (rounds - 1)) * 8;
  const int64_t bh = blockIdx.y;
  const int64_t r_first = static_cast<int64_t>(blockIdx.x) * kThreads;
#pragma unroll 4
  for (int round = 0; round < rounds; ++round) {
    const int64_t r = r_first + round * rows_per_round + (threadIdx.x >> tpr_shift);
    if (r >= a.N) continue;
    const int i = partition_of(a, r);
    T* o;
    float* l;
    state_ptrs(a.cache, a.P, a.N, a.d, bh, i, i, r, o, l);
    const uint4* src = reinterpret_cast<const uint4*>(o + c0);
    // the snapshot is the one buffer this launch writes (const in the args, shared with drift)
    uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(const_cast<void*>(a.snap)) +
                                          (bh * a.N + r) * a.d + c0);
#pragma unroll
    for (int v = 0; v < V; ++v) dst[v] = __ldg(src + v);
  }
}

// One thread, in ascending i: out[i] may share storage with sums (the caller's buffer holds
// the 2P sums, then the P drifts), and position i is never read again once i is done.
__global__ void drift_finalize(const __grid_constant__ PlannerArgs a) {
  if (threadIdx.x != 0) return;
  for (int i = 0; i < a.P; ++i) {
    const double num = a.sums[2 * i], den = a.sums[2 * i + 1];
    a.out[i] = den > 0.0 ? sqrt(num / den) : 0.0;
  }
}

}  // namespace

cudaError_t launch_planner_importance(const PlannerArgs& a, cudaStream_t stream) {
  const size_t PP = static_cast<size_t>(a.P) * a.P;
  cudaError_t e = cudaMemsetAsync(a.sums, 0, PP * sizeof(double), stream);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>((a.N + kThreads - 1) / kThreads),
                  static_cast<unsigned>(a.B * a.H));
  importance_kernel<<<grid, kThreads, 0, stream>>>(a);
  importance_finalize<<<static_cast<unsigned>((PP + 255) / 256), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_planner_drift(const PlannerArgs& a, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(a.sums, 0, 2 * static_cast<size_t>(a.P) * sizeof(double), stream);
  if (e != cudaSuccess) return e;
  const int tpr = a.d / 8;  // threads per row
  if (a.d % 8 != 0 || tpr < 1 || tpr > 32 || (tpr & (tpr - 1)) != 0) return cudaErrorInvalidValue;
  const int tpr_shift = 31 - __builtin_clz(static_cast<unsigned>(tpr));
  const dim3 grid(static_cast<unsigned>((a.N + kThreads - 1) / kThreads),
                  static_cast<unsigned>(a.B * a.H));
  if (a.dtype == DITANGO_BF16)
    drift_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(a, tpr_shift);
  else
    drift_kernel<float><<<grid, kThreads, 0, stream>>>(a, tpr_shift);
  drift_finalize<<<1, 32, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_planner_snapshot(const PlannerArgs& a, cudaStream_t stream) {
  const int tpr = a.d / 8;  // threads per row
  if (a.d % 8 != 0 || tpr < 1 || tpr > 32 || (tpr & (tpr - 1)) != 0) return cudaErrorInvalidValue;
  const int tpr_shift = 31 - __builtin_clz(static_cast<unsigned>(tpr));
  const dim3 grid(static_cast<unsigned>((a.N + kThreads - 1) / kThreads),
                  static_cast<unsigned>(a.B * a.H));
  if (a.dtype == DITANGO_BF16)
    snapshot_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(a, tpr_shift);
  else
    snapshot_kernel<float><<<grid, kThreads, 0, stream>>>(a, tpr_shift);
  return cudaGetLastError();
}

}  // namespace ditango
