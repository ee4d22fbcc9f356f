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
// owning VEC contiguous channels loaded as VPT 16-byte vectors per state (one for a state list,
// two for a step), so a warp reads whole rows of every state in fully used 32-byte sectors. Index arithmetic is 32-bit (shifts and
// masks when d/VEC is a power of two, a division otherwise); exponentials and the logarithm use
// the SFU approximations (relative error ~2^-22). States are merged online in rounds whose
// vectors and lse values are all loaded before any is used, so a round costs one memory round
// trip: eight states per round for a state list, two for a step (see launch_step_typed).
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

// VEC fp32 channels (VEC / 4 vectors of 16 bytes).
template <int VEC>
__device__ __forceinline__ void store_vec(float* p, const float (&x)[VEC]) {
#pragma unroll
  for (int q = 0; q < VEC / 4; ++q)
    reinterpret_cast<float4*>(p)[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
}
// VEC bf16 channels (VEC / 8 vectors of 16 bytes), each rounded to nearest even.
template <int VEC>
__device__ __forceinline__ void store_vec(__nv_bfloat16* p, const float (&x)[VEC]) {
#pragma unroll
  for (int q = 0; q < VEC / 8; ++q) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 h = __floats2bfloat162_rn(x[8 * q + 2 * i], x[8 * q + 2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&h);
    }
    reinterpret_cast<uint4*>(p)[q] = make_uint4(w[0], w[1], w[2], w[3]);
  }
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

// A row's view of the state cache: where state j of the row lives (device or host slot).
struct RowStates {
  const CacheLoc* c;
  int32_t P, d, i;
  int64_t N, bh, r;
  int c0;
  template <typename T>
  __device__ __forceinline__ void ptrs(int j, const T*& o, const float*& l) const {
    T* op;
    float* lp;
    state_ptrs(*c, P, N, d, bh, i, j, r, op, lp);
    o = op + c0;
    l = lp;
  }
};

// Loads the next round of up to NS states of `m` (a bit set of states j, lowest first): the
// VPT 16-byte vectors of this thread's channels and the lse (log2 units) of each, all issued
// before any is used, so that a round costs one memory round trip. Slots past the set get
// lse = -inf and zero vectors. Returns how many states were loaded; m loses their bits.
template <typename T, int NS, int VPT>
__device__ __forceinline__ int load_round(uint64_t& m, const RowStates& rs,
                                          uint4 (&raw)[NS][VPT], float (&l)[NS]) {
  int cnt = 0;
#pragma unroll
  for (int q = 0; q < NS; ++q) {
    if (m != 0) {
      const int j = __ffsll(static_cast<long long>(m)) - 1;
      m &= m - 1;
      const T* o;
      const float* lp;
      rs.ptrs<T>(j, o, lp);
#pragma unroll
      for (int v = 0; v < VPT; ++v) raw[q][v] = load_raw(o + v * (16 / sizeof(T)));
      l[q] = __ldg(lp) * kLog2e;
      ++cnt;
    } else {
#pragma unroll
      for (int v = 0; v < VPT; ++v) raw[q][v] = make_uint4(0u, 0u, 0u, 0u);
      l[q] = -INFINITY;
    }
  }
  return cnt;
}

// Online merge of one loaded round into (mx, sum, acc), all relative to the running max mx
// (log2 units): acc and sum are rescaled by 2^(mx - mx_new) once per round.
template <typename T, int VEC, int NS, int VPT>
__device__ __forceinline__ void merge_round(const uint4 (&raw)[NS][VPT], const float (&l)[NS],
                                            int cnt, float& mx, float& sum, float (&acc)[VEC]) {
  constexpr int H = VEC / VPT;  // channels per vector
  float mn = mx;
#pragma unroll
  for (int q = 0; q < NS; ++q) mn = fmaxf(mn, l[q]);
  const float sc = ex2(mx - mn);  // 0 on the first round (mx = -inf); cnt >= 1 keeps mn finite
  sum *= sc;
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] *= sc;
#pragma unroll
  for (int q = 0; q < NS; ++q) {
    if (q < cnt) {
      const float w = ex2(l[q] - mn);
      sum += w;
#pragma unroll
      for (int v = 0; v < VPT; ++v) {
        float x[H];
        unpack(raw[q][v], x, static_cast<const T*>(nullptr));
#pragma unroll
        for (int e = 0; e < H; ++e) acc[v * H + e] = fmaf(w, x[e], acc[v * H + e]);
      }
    }
  }
  mx = mn;
}

// Merges every state of the bit set `set` (states j of this row) into (mx, sum, acc).
template <typename T, int VEC, int NS, int VPT>
__device__ __forceinline__ void merge_set(uint64_t set, const RowStates& rs, float& mx, float& sum,
                                          float (&acc)[VEC]) {
  for (uint64_t m = set; m != 0;) {
    uint4 raw[NS][VPT];
    float l[NS];
    const int cnt = load_round<T, NS, VPT>(m, rs, raw, l);
    merge_round<T, VEC, NS, VPT>(raw, l, cnt, mx, sum, acc);
  }
}

// Row and first channel of this thread (tpr = d / VEC threads per row; tpr_shift = log2(tpr)
// when tpr is a power of two, else -1); false past the last of R rows.
__device__ __forceinline__ bool thread_row(int64_t R, int tpr, int tpr_shift, int vec_shift,
                                           uint32_t& r, int& c0) {
  const uint32_t t = blockIdx.x * kMergeThreads + threadIdx.x;
  if (tpr_shift >= 0) {
    r = t >> tpr_shift;
    c0 = static_cast<int>(t & ((1u << tpr_shift) - 1u)) << vec_shift;
  } else {
    r = t / static_cast<uint32_t>(tpr);
    c0 = static_cast<int>(t - r * static_cast<uint32_t>(tpr)) << vec_shift;
  }
  return r < static_cast<uint64_t>(R);
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// merge_kernel: state list with a common [G1, G2, R, d] layout (MergeArgs), d any multiple of
// VEC. T: the states' dtype, TO: the output's (T, or fp32).
template <typename T, typename TO>
__global__ void __launch_bounds__(kMergeThreads)
    merge_kernel(const __grid_constant__ MergeArgs a, int64_t g_base, int tpr_shift) {
  constexpr int VEC = 16 / sizeof(T);
  constexpr int VEC_SHIFT = VEC == 8 ? 3 : 2;
  constexpr int NS = 8;  // a list of up to eight states in one round trip
  uint32_t r;
  int c0;
  if (!thread_row(a.R, a.d / VEC, tpr_shift, VEC_SHIFT, r, c0)) return;
  const int64_t g = g_base + blockIdx.y;
  const int64_t g1 = g / a.G2, g2 = g - g1 * a.G2;
  const int64_t lo = g1 * a.lS[0] + g2 * a.lS[1] + r * a.lS[2];
  const int64_t oo = g1 * a.oS[0] + g2 * a.oS[1] + r * a.oS[2] + c0;

  float mx = -INFINITY, sum = 0.f;
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < a.n; s0 += NS) {
    uint4 raw[NS][1];
    float l[NS];
    const int cnt = min(NS, a.n - s0);
#pragma unroll
    for (int q = 0; q < NS; ++q) {
      if (q < cnt) {
        raw[q][0] = load_raw(static_cast<const T*>(a.O[s0 + q]) + oo);
        l[q] = __ldg(a.lse[s0 + q] + lo) * kLog2e;
      } else {
        raw[q][0] = make_uint4(0u, 0u, 0u, 0u);
        l[q] = -INFINITY;
      }
    }
    merge_round<T, VEC, NS, 1>(raw, l, cnt, mx, sum, acc);
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

// step_merge_kernel: the merge that ends a step (StepMergeArgs). Row r of (b, h) = grid.y, in
// partition i:
//   * if bit i of `rebuild` is set, the row first merges its reused states (reused_set[i]) into
//     its new group state and stores it (fp32 O and lse), then continues from that state;
//   * else if bit i of `group` is set, it starts from its stored group state;
//   * then it merges the states (b, h, j, r) for j in cache_set[i].
// State j of the row lives in a device slot or, when the cache keeps it in host memory, in its
// host slot (CacheLoc).
// Starting from a group state built here or loaded gives the same arithmetic (the same fp32
// values), so a rebuild step and a steady step agree bit for bit on the same states.
// NS: states per round (each round's loads are issued together). Each thread owns two 16-byte
// vectors of a row (VEC = 32 / sizeof(T) channels), which halves the per-state index and
// address work per byte: measured 0.904 ms for the 720p layer's step (6.6 TB/s) against 1.086
// ms with one vector per thread, and 0.299 against 0.349 ms on the Wan-14B layer. At most 64
// registers (four blocks of 256 threads per SM): the cap of 48 (five blocks) spills and
// measured 0.982 ms.
template <typename T, int NS>
__global__ void __launch_bounds__(kMergeThreads, 4)
    step_merge_kernel(const __grid_constant__ StepMergeArgs a, int64_t bh_base) {
  constexpr int VPT = 2;
  constexpr int VEC = VPT * 16 / sizeof(T);
  constexpr int VEC_SHIFT = VEC == 16 ? 4 : 3;
  static_assert(VEC == 1 << VEC_SHIFT, "channels per thread");
  uint32_t r;
  int c0;
  const int tpr_shift = 31 - __clz(a.d) - VEC_SHIFT;  // d / VEC is 4, 8 or 16 (d = 64 or 128)
  const bool live = thread_row(a.N, a.d / VEC, tpr_shift, VEC_SHIFT, r, c0);
  // launched as a programmatic dependent of the pair kernel: everything below reads states it
  // wrote, so wait for that grid to complete (a no-op for an ordinary launch)
  grid_dependency_wait();
  if (!live) return;
  const int64_t bh = bh_base + blockIdx.y;
  int i = 0;
  while (r >= static_cast<uint32_t>(a.offsets[i + 1])) ++i;
  const RowStates rs{&a.cache, a.P, a.d, i, a.N, bh, static_cast<int64_t>(r), c0};

  float mx = -INFINITY, sum = 0.f;
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  if ((a.rebuild >> i) & 1u) {
    // Dynamic Group Compose: the reused states merge into the row's group state
    merge_set<T, VEC, NS, VPT>(a.reused_set[i], rs, mx, sum, acc);
    const float g_lse = (mx + lg2(sum)) * kLn2;
    const float inv = 1.f / sum;
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[e] *= inv;
    store_f32<VEC>(a.gO + (bh * a.N + r) * a.d + c0, acc);
    if (c0 == 0) a.gL[bh * a.N + r] = g_lse;
    mx = g_lse * kLog2e;  // the group state starts the merge (weight 1 relative to its lse)
    sum = 1.f;
  } else if ((a.group >> i) & 1u) {
    mx = __ldg(a.gL + bh * a.N + r) * kLog2e;
    sum = 1.f;
    load_f32<VEC>(a.gO + (bh * a.N + r) * a.d + c0, acc);
  }
  merge_set<T, VEC, NS, VPT>(a.cache_set[i], rs, mx, sum, acc);
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

template <typename T, int NS>
cudaError_t launch_step_chunk(const StepMergeArgs& a, dim3 grid, int64_t g0, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, step_merge_kernel<T, NS>, a, g0);
}

// Rounds of two states: measured faster than whole-row rounds (with one vector per thread,
// Wan-14B layer 0.353 ms against 0.432 ms with rounds of four, 720p layer 1.08 ms against 1.74
// ms with rounds of eight; with two, 0.90 ms against 1.06 ms with rounds of three and 0.92-1.01
// ms with rounds of one): fewer registers per thread keep more rows in flight per SM.
template <typename T>
cudaError_t launch_step_typed(const StepMergeArgs& a, dim3 grid, int64_t g0, cudaStream_t stream) {
  return launch_step_chunk<T, 2>(a, grid, g0, stream);
}

}  // namespace

cudaError_t launch_step_merge(const StepMergeArgs& a, cudaStream_t stream) {
  const int vec = a.dtype == DITANGO_BF16 ? 16 : 8;  // channels per thread (two vectors)
  const int64_t groups = a.B * a.H;
  if (groups == 0 || a.N == 0) return cudaSuccess;
  if (a.d != 64 && a.d != 128) return cudaErrorInvalidValue;
  const unsigned bx = blocks_x(a.N, a.d, vec);
  if (bx == 0) return cudaErrorInvalidValue;
  for (int64_t g0 = 0; g0 < groups; g0 += kMaxGridY) {
    const dim3 grid(bx, static_cast<unsigned>(std::min<int64_t>(kMaxGridY, groups - g0)));
    const cudaError_t e = a.dtype == DITANGO_BF16
                              ? launch_step_typed<__nv_bfloat16>(a, grid, g0, stream)
                              : launch_step_typed<float>(a, grid, g0, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int vec = a.dtype == DITANGO_BF16 ? 8 : 4;
  const int64_t groups = a.G1 * a.G2;
  if (groups == 0 || a.R == 0) return cudaSuccess;
  if (a.d % vec != 0) return cudaErrorInvalidValue;
  const unsigned bx = blocks_x(a.R, a.d, vec);
  if (bx == 0) return cudaErrorInvalidValue;
  const int tpr = a.d / vec;
  const int tpr_shift = (tpr & (tpr - 1)) == 0 ? 31 - __builtin_clz(static_cast<unsigned>(tpr)) : -1;
  for (int64_t g0 = 0; g0 < groups; g0 += kMaxGridY) {
    const dim3 grid(bx, static_cast<unsigned>(std::min<int64_t>(kMaxGridY, groups - g0)));
    if (a.dtype == DITANGO_BF16 && a.out_dtype == DITANGO_BF16)
      merge_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, kMergeThreads, 0, stream>>>(a, g0, tpr_shift);
    else if (a.dtype == DITANGO_BF16 && a.out_dtype == DITANGO_F32)
      merge_kernel<__nv_bfloat16, float><<<grid, kMergeThreads, 0, stream>>>(a, g0, tpr_shift);
    else if (a.dtype == DITANGO_F32 && a.out_dtype == DITANGO_F32)
      merge_kernel<float, float><<<grid, kMergeThreads, 0, stream>>>(a, g0, tpr_shift);
    else
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ditango
