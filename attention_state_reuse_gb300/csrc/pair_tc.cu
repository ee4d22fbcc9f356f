// Partition-pair attention states on the sm_103a tensor cores (bf16 in, fp32 accumulate).
//
// Method: DiTango (gist.science/paper/2607.15650), Methodology 2, State Composition: for a
// query partition i and a KV partition j the state is (O_ij, lse_ij) with
//   lse_ij[r] = ln sum_{c in j} exp(z_c),   O_ij[r] = sum_{c in j} exp(z_c - lse_ij[r]) v_c,
//   z_c = scale <q_r, k_c>.
// Only pairs the step computes are visited (Methodology 1: reused pairs launch nothing).
//
// Kernel design (persistent, one CTA per SM, 320 threads):
//   warps 0-3  softmax warpgroup 0: query tile 0 (rows 0..127 of the unit), one row per thread
//   warps 4-7  softmax warpgroup 1: query tile 1 (rows 128..255)
//   warp  8    TMA producer: Q tiles per unit, then a ring of K and V tiles (128 rows each)
//              (when RoPE is on, the softmax warpgroups rotate their Q tile in shared memory
//              before the first Q K^T of the unit; K arrives already rotated)
//   warp  9    MMA issuer: S_w = Q_w K^T (SS, both K-major) and O_w += P_w V (A from TMEM,
//              V MN-major); owns the TMEM allocation
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+d), O1 [256+d, 256+2d).
// P_w overwrites the first 64 columns of S_w as packed bf16; tcgen05.mma operations issued by
// one thread execute in order, so S_w of the next tile is written only after P_w is consumed.
// The MMA warp runs its loop converged and lets one elected lane issue (see mma_ss in
// ptx_sm103.cuh).
// Online softmax with a lazily updated reference m: the first tile of a partition takes its
// exact row max; later tiles reuse m and check only the row sum of their exponentials, and a
// row whose tile sum exceeds 2^8 (a score above the reference by up to 8 in log2 units, or
// many close to it) takes the exact max of that tile, rescales O and l, and recomputes P.
// The result does not depend on m mathematically; numerically, a reference at the exact max
// makes the largest term of a row exactly 1 in bf16, which keeps the bf16 rounding of P from
// reaching the largest products (measured: letting P grow to 2^12 or beyond roughly doubled
// the worst output error on head-scaled inputs).
// Every barrier wait is bounded (see ptx_sm103.cuh); a timeout makes all roles stop, drain
// their copies, free TMEM and record an error code.
#include <cuda_bf16.h>

#include <cfloat>

#include "ditango_internal.h"
#include "ptx_sm103.cuh"
#include "rope_round.cuh"

namespace ditango {
namespace {

using namespace ptx;

constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kTileRows = 128;               // query rows per tile == KV rows per tile
constexpr int kUnitRows = 2 * kTileRows;     // query rows per unit
constexpr int kChunkBytes = 128 * 128;       // 128 rows x 64 bf16 (one swizzle-atom column)
constexpr float kRescaleSum = 256.0f;  // tile row sum above which m moves to the exact max
constexpr float kLn2 = 0.69314718055994531f;

template <int D>
struct Cfg {
  static constexpr int CH = D / 64;
  static constexpr int TILE_BYTES = CH * kChunkBytes;
  static constexpr int Q_BYTES = 2 * TILE_BYTES;
  static constexpr int STAGES = (D == 128) ? 4 : 8;
  __host__ __device__ static constexpr uint32_t s_col(int w) { return w ? 128u : 0u; }
  __host__ __device__ static constexpr uint32_t o_col(int w) { return 256u + (w ? D : 0); }
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_QK = idesc_bf16_f32(128, 128, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, true);
};

template <int STAGES>
struct SharedCtl {
  uint64_t q_full, q_ready, q_empty;  // Q landed / Q rotated (ready for the MMA) / Q consumed
  uint64_t kv_full[STAGES], kv_empty[STAGES];
  uint64_t s_full[2], p_full[2], o_done[2], o_free[2];
  uint64_t drained;
  uint32_t tmem_base;
  int abort_word;
};

template <int D>
__host__ __device__ constexpr int ctl_bytes() {
  return ((int)sizeof(SharedCtl<Cfg<D>::STAGES>) + 15) & ~15;
}

// Dynamic shared memory: 1 KB alignment slack, Q, the K/V ring, the control block, then the
// RoPE table (rope_pairs (cos, sin) pairs; 0 without RoPE).
template <int D>
constexpr int smem_bytes(int rope_pairs) {
  return 1024 + Cfg<D>::Q_BYTES + Cfg<D>::STAGES * Cfg<D>::TILE_BYTES + ctl_bytes<D>() +
         8 * rope_pairs;
}

struct UnitInfo {
  int b, h, i, qb, row0, n_i;
};

__device__ __forceinline__ UnitInfo decode_unit(const PairSchedule& s, int u) {
  int k = 0;
  while (u >= s.seg_start[k + 1]) ++k;
  UnitInfo ui;
  ui.i = s.order[k];
  const int local = u - s.seg_start[k];
  ui.n_i = s.offsets[ui.i + 1] - s.offsets[ui.i];
  const int blocks = (ui.n_i + s.block_rows - 1) / s.block_rows;
  const int bh = local / blocks;
  ui.qb = local - bh * blocks;
  ui.b = bh / s.H;
  ui.h = bh - ui.b * s.H;
  ui.row0 = s.offsets[ui.i] + ui.qb * s.block_rows;
  return ui;
}

__device__ __forceinline__ int ntiles_of(const PairSchedule& s, int j) {
  return (s.offsets[j + 1] - s.offsets[j] + kTileRows - 1) / kTileRows;
}

// Waits with the CTA's abort word; the result is made uniform across the warp so that
// warp-collective tcgen05 operations are entered by all lanes or by none.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_w) {
  const bool ok = mbar_wait(bar, parity, abort_w);
  return __all_sync(0xffffffffu, ok);
}

// Drain wait: ignores the abort word, bounded by the timeout alone.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity) {
  int dummy = 0;
  (void)mbar_wait(bar, parity, &dummy);
}

// Issues O_w (+)= P_w V for the tile before the current one: waits for P_w of that tile, for
// the epilogue of the previous partition to have read O_w (first tile of a partition), and
// for the V tile; then eight K=16 steps with A read from TMEM (P) and B = V (MN-major).
// v_lo0 is the low descriptor half of ring slot 0 for an MN-major operand.
// Run by the whole MMA warp (converged); one elected lane issues.
template <int D>
__device__ __forceinline__ bool issue_pv(SharedCtl<Cfg<D>::STAGES>* ctl, int w, uint32_t prev_g,
                                         uint32_t prev_v, uint32_t prev_pidx, bool prev_first,
                                         uint32_t v_lo0, uint32_t desc_hi, uint32_t tbase,
                                         volatile int* abort_w) {
  using C = Cfg<D>;
  constexpr int STAGES = C::STAGES;
  if (!warp_wait(&ctl->p_full[w], prev_g & 1u, abort_w)) return false;
  if (prev_first && prev_pidx >= 1 && !warp_wait(&ctl->o_free[w], (prev_pidx - 1) & 1u, abort_w))
    return false;
  if (w == 0 && !warp_wait(&ctl->kv_full[prev_v % STAGES], (prev_v / STAGES) & 1u, abort_w))
    return false;
  tc_fence_after_sync();
  const uint32_t v_lo = v_lo0 + (prev_v % STAGES) * (C::TILE_BYTES >> 4);
  const uint32_t d_t = tbase + C::o_col(w);
  const uint32_t a_t = tbase + C::s_col(w);
  if (prev_first)
    mma_ts<0>(d_t, a_t, v_lo, desc_hi, C::IDESC_PV);
  else
    mma_ts<1>(d_t, a_t, v_lo, desc_hi, C::IDESC_PV);
#pragma unroll
  for (int k = 1; k < kTileRows / 16; ++k)  // 16 KV rows (2048 bytes) per step
    mma_ts<1>(d_t, a_t + k * 8, v_lo + k * (2048 >> 4), desc_hi, C::IDESC_PV);
  tc_commit(&ctl->o_done[w]);
  return true;
}

// Low descriptor-half offset of K step k (16 elements) inside a K-major 128-byte-swizzled
// operand whose K extent is split into 64-element chunks kChunkBytes apart.
__host__ __device__ constexpr uint32_t kstep_off(int k) {
  return static_cast<uint32_t>(((k >> 2) * kChunkBytes + (k & 3) * 32) >> 4);
}

// S_w = Q_w K^T for the K tile at low descriptor half k_lo: D/16 steps, both operands K-major.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_t, uint32_t q_lo, uint32_t k_lo,
                                         uint32_t hi) {
  mma_ss<0>(d_t, q_lo, hi, k_lo, hi, Cfg<D>::IDESC_QK);
#pragma unroll
  for (int k = 1; k < D / 16; ++k)
    mma_ss<1>(d_t, q_lo + kstep_off(k), hi, k_lo + kstep_off(k), hi, Cfg<D>::IDESC_QK);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ float2 ld_shared_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// Copies the RoPE table rows into shared memory as (cos, sin) pairs in the RopeQ layout. Run by
// the `nthreads` threads with index `tid`; padding pairs are left unwritten (never read).
__device__ __forceinline__ void stage_rope_table(const RopeQ& r, float2* tab, int tid, int nthreads) {
  const int ht = r.dt >> 1, hh = r.dh >> 1, hw = r.dw >> 1;
  const int nt_pairs = r.nT * r.sT, nh_pairs = r.Hl * r.sH;
  for (int x = tid; x < r.n_pairs; x += nthreads) {
    const float* c;
    const float* sn;
    int row, m, len;
    if (x < nt_pairs) {
      row = x / r.sT; m = x - row * r.sT; len = ht;
      c = r.cos_t + (r.start_frame + row) * ht; sn = r.sin_t + (r.start_frame + row) * ht;
    } else if (x < nt_pairs + nh_pairs) {
      const int y = x - nt_pairs;
      row = y / r.sH; m = y - row * r.sH; len = hh;
      c = r.cos_h + row * hh; sn = r.sin_h + row * hh;
    } else {
      const int y = x - nt_pairs - nh_pairs;
      row = y / r.sW; m = y - row * r.sW; len = hw;
      c = r.cos_w + row * hw; sn = r.sin_w + row * hw;
    }
    if (m < len) tab[x] = make_float2(__ldg(c + m), __ldg(sn + m));
  }
}

// Rotates one token's row of a Q tile in place in shared memory (3D RoPE keyed by the global
// frame index; "Accelerating Video Generation Inference with Sequential-Parallel 3D Positional
// Encoding Using a Global Time Index", section 2). The row is D bf16 values in 128-byte lines,
// one per 64-channel chunk, with its 16-byte units stored at unit ^ (row mod 8). Channel pair
// m = (2m, 2m+1) turns by the angle of table entry m of the token's frame (m < dt/2), row
// (next dh/2) or column (last dw/2); each output is the nearest-even bf16 of the rotation with
// fp64 cos/sin, as in the rotary pre-pass (rope_round.cuh). A first pass takes the fp32 fast
// path from the staged table and leaves the rare pairs whose rounding it cannot decide
// unrotated, noting them in a bit mask; a second pass recomputes only those exactly, reading
// the residual tables from global memory. Both passes are rolled loops in a function of its
// own: the row rotation runs once per unit, and unrolled or inlined into the softmax loop it
// cost that loop registers (measured: 5.9 ms unrolled and inlined, 5.35 ms this way, against
// 5.2 ms for a plain fp32 rotation, on the Wan-14B layer's reuse step). n is the token's index
// in the sequence; tab is the staged table (shared-space address).
template <int D>
__device__ __noinline__ void rotate_q_row(uint32_t row_addr, uint32_t row_xor, int n,
                                             const RopeQ& r, uint32_t tab) {
  const int hw_tokens = r.Hl * r.Wl;
  const int tl = n / hw_tokens;
  const int rem = n - tl * hw_tokens;
  const int hp = rem / r.Wl;
  const int wp = rem - hp * r.Wl;
  const int ht = r.dt >> 1, hth = ht + (r.dh >> 1);
  // byte addresses of pair 0 of each axis' row, offset so that pair m is at base + 8 m
  const uint32_t bt = tab + 8u * static_cast<uint32_t>(tl * r.sT);
  const uint32_t bh = tab + 8u * static_cast<uint32_t>(r.nT * r.sT + hp * r.sH - ht);
  const uint32_t bw = tab + 8u * static_cast<uint32_t>(r.nT * r.sT + r.Hl * r.sH + wp * r.sW - hth);
  uint64_t unsure = 0;  // bit m: pair m still holds its input, to be rotated exactly below
#pragma unroll 1
  for (int u = 0; u < D / 8; ++u) {  // 16-byte units: chunk u / 8, unit u % 8 of the chunk
    const uint32_t addr = row_addr + (u >> 3) * kChunkBytes + (((u & 7) ^ row_xor) << 4);
    const uint4 v = ld_shared_v4(addr);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int m = u * 4 + p;  // channel pair index
      const uint32_t base = m < ht ? bt : (m < hth ? bh : bw);
      const float2 cs = ld_shared_f2(base + 8u * m);
      bool sure;
      o[p] = rope_rotate_bf16x2_fast(__uint_as_float(wv[p] << 16),
                                     __uint_as_float(wv[p] & 0xFFFF0000u), cs.x, cs.y, sure);
      if (!sure) {
        o[p] = wv[p];
        unsure |= uint64_t{1} << m;
      }
    }
    st_shared_v4(addr, o[0], o[1], o[2], o[3]);
  }
  while (unsure != 0) {  // rare: about one pair in a thousand
    const int m = __ffsll(static_cast<long long>(unsure)) - 1;
    unsure &= unsure - 1;
    const int u = m >> 2;
    const uint32_t addr = row_addr + (u >> 3) * kChunkBytes + (((u & 7) ^ row_xor) << 4) + 4u * (m & 3);
    const uint32_t w = ld_shared_u32(addr);
    const uint32_t base = m < ht ? bt : (m < hth ? bh : bw);
    const float2 cs = ld_shared_f2(base + 8u * m);
    const float *pc, *ps;
    int idx;
    if (m < ht) {
      idx = (r.start_frame + tl) * ht + m;
      pc = r.cos_t_lo; ps = r.sin_t_lo;
    } else if (m < hth) {
      idx = hp * (r.dh >> 1) + (m - ht);
      pc = r.cos_h_lo; ps = r.sin_h_lo;
    } else {
      idx = wp * (r.dw >> 1) + (m - hth);
      pc = r.cos_w_lo; ps = r.sin_w_lo;
    }
    st_shared_u32(addr, rope_rotate_bf16x2_exact(__uint_as_float(w << 16),
                                                 __uint_as_float(w & 0xFFFF0000u), cs.x, cs.y,
                                                 __ldg(pc + idx), __ldg(ps + idx)));
  }
}

// P = 2^(s * scale_log2 - m) for one half row (64 keys) of a 128-key tile, packed to bf16 pairs
// in pk (32 words); returns the sum of the fp32 values. Paired fp32 FMA/add instructions halve
// the ALU issue of the scale-subtract and of the sum; the exponentials go to the SFU.
__device__ __forceinline__ float exp_pack_half(const float (&s)[kTileRows / 2], float sl2, float m,
                                               uint32_t* pk) {
  const float2 sl2x2 = make_float2(sl2, sl2);
  const float2 negm2 = make_float2(-m, -m);
  float2 l4[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                  make_float2(0.f, 0.f)};
#pragma unroll
  for (int c = 0; c < kTileRows / 4; ++c) {
    const float2 x = __ffma2_rn(make_float2(s[2 * c], s[2 * c + 1]), sl2x2, negm2);
    const float p0 = ex2_approx(x.x);
    const float p1 = ex2_approx(x.y);
    l4[c & 3] = __fadd2_rn(l4[c & 3], make_float2(p0, p1));
    pk[c] = pack_bf16x2(p0, p1);
  }
  const float2 l2 = __fadd2_rn(__fadd2_rn(l4[0], l4[1]), __fadd2_rn(l4[2], l4[3]));
  return l2.x + l2.y;
}

// Max of a half row: eight independent three-input max chains, then a short tree.
__device__ __forceinline__ float half_max(const float (&s)[kTileRows / 2]) {
  float m8[8];
#pragma unroll
  for (int x = 0; x < 8; ++x) m8[x] = fmaxf(s[x], s[8 + x]);
#pragma unroll
  for (int c = 16; c < kTileRows / 2; c += 16)
#pragma unroll
    for (int x = 0; x < 8; ++x) m8[x] = fmax3(m8[x], s[c + x], s[c + 8 + x]);
  return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
}

// Reads half h of a row of S (64 fp32 scores per thread) from TMEM; keys at or past `valid`
// (counted from the start of the tile) get -inf.
__device__ __forceinline__ void load_s_half(uint32_t s_taddr, int h, int valid,
                                            float (&s)[kTileRows / 2]) {
  uint32_t r[kTileRows / 2];
  tmem_ld_32x32b_x64(s_taddr + h * (kTileRows / 2), r);
#pragma unroll
  for (int c = 0; c < kTileRows / 2; ++c) s[c] = __uint_as_float(r[c]);
  const int v = valid - h * (kTileRows / 2);
  if (v < kTileRows / 2) {
#pragma unroll
    for (int c = 0; c < kTileRows / 2; ++c)
      if (c >= v) s[c] = -INFINITY;
  }
}

// Exact row max of a tile (both halves).
__device__ __forceinline__ float row_max(uint32_t s_taddr, int valid) {
  float s[kTileRows / 2];
  load_s_half(s_taddr, 0, valid, s);
  const float m0 = half_max(s);
  load_s_half(s_taddr, 1, valid, s);
  return fmaxf(m0, half_max(s));
}

// P of a whole tile row into pk (64 words), half by half: 64 scores live at a time instead of
// 128 keep the softmax within its 168 registers (the whole-row form spilled; measured 2-4%
// slower); returns the row sum.
__device__ __forceinline__ float exp_pack_row(uint32_t s_taddr, int valid, float sl2, float m,
                                              uint32_t (&pk)[kTileRows / 2]) {
  float l = 0.f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    float s[kTileRows / 2];
    load_s_half(s_taddr, h, valid, s);
    l += exp_pack_half(s, sl2, m, pk + h * (kTileRows / 4));
  }
  return l;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    pair_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const __grid_constant__ PairTcArgs args) {
  using C = Cfg<D>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* q_smem = smem;
  uint8_t* kv_smem = smem + C::Q_BYTES;
  auto* ctl = reinterpret_cast<SharedCtl<STAGES>*>(kv_smem + STAGES * C::TILE_BYTES);
  float2* rope_tab = reinterpret_cast<float2*>(kv_smem + STAGES * C::TILE_BYTES + ctl_bytes<D>());
  const bool rope_on = args.rope.n_pairs > 0;
  volatile int* abort_w = &ctl->abort_word;

  const PairSchedule& sch = args.sched;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    ctl->abort_word = 0;
    mbar_init(&ctl->q_full, 1);
    mbar_init(&ctl->q_ready, 2 * kTileRows);
    mbar_init(&ctl->q_empty, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->kv_full[s], 1);
      mbar_init(&ctl->kv_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&ctl->s_full[w], 1);
      mbar_init(&ctl->p_full[w], kTileRows);
      mbar_init(&ctl->o_done[w], 1);
      mbar_init(&ctl->o_free[w], kTileRows);
    }
    mbar_init(&ctl->drained, 1);
    fence_barrier_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_map(&map_q);
    tma_prefetch_map(&map_k);
    tma_prefetch_map(&map_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, C::TMEM_COLS);
    tmem_relinquish_alloc_permit();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tbase = ctl->tmem_base;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t e = 0, uc = 0;  // K/V ring entries and Q loads issued so far
      bool ok = true;
      for (int u = blockIdx.x; ok && u < sch.n_units; u += gridDim.x) {
        const UnitInfo ui = decode_unit(sch, u);
        if (uc > 0) ok = mbar_wait(&ctl->q_empty, (uc - 1) & 1u, abort_w);
        if (!ok) break;
        mbar_arrive_expect_tx(&ctl->q_full, C::Q_BYTES);
        ++uc;
        for (int w = 0; w < 2; ++w)
          for (int c = 0; c < C::CH; ++c)
            tma_load_4d(q_smem + w * C::TILE_BYTES + c * kChunkBytes, &map_q, &ctl->q_full, c * 64,
                        ui.h, ui.row0 + w * kTileRows, ui.b);
        for (uint64_t m = sch.compute_mask[ui.i]; ok && m; m &= m - 1) {
          const int j = __ffsll(static_cast<long long>(m)) - 1;
          const int nt = ntiles_of(sch, j);
          for (int t = 0; ok && t < nt; ++t) {
            const int kvrow = sch.offsets[j] + t * kTileRows;
            for (int kind = 0; kind < 2; ++kind, ++e) {
              const uint32_t slot = e % STAGES;
              if (e >= static_cast<uint32_t>(STAGES)) {
                ok = mbar_wait(&ctl->kv_empty[slot], ((e / STAGES) - 1) & 1u, abort_w);
                if (!ok) break;
              }
              // test hook: the first K tile of CTA 0 never arrives, so the MMA warp's bounded
              // wait for it runs out and the CTA takes its abort path
              if (args.inject_fault && blockIdx.x == 0 && e == 0) continue;
              mbar_arrive_expect_tx(&ctl->kv_full[slot], C::TILE_BYTES);
              const CUtensorMap* mp = kind == 0 ? &map_k : &map_v;
              for (int c = 0; c < C::CH; ++c)
                tma_load_4d(kv_smem + slot * C::TILE_BYTES + c * kChunkBytes, mp, &ctl->kv_full[slot],
                            c * 64, ui.h, kvrow, ui.b);
            }
          }
        }
      }
      if (!ok) {
        // let every copy this thread started land before the CTA can exit
        if (uc > 0) drain_wait(&ctl->q_full, (uc - 1) & 1u);
        const uint32_t lo = e > static_cast<uint32_t>(STAGES) ? e - STAGES : 0u;
        for (uint32_t x = lo; x < e; ++x) drain_wait(&ctl->kv_full[x % STAGES], (x / STAGES) & 1u);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop (converged, waits made warp-uniform); one elected lane
    // issues every MMA and commit.
    {
      uint32_t e = 0, uc = 0, g = 0, pidx = 0;
      bool ok = true;
      const uint32_t desc_hi = sdesc_sw128_hi(1024);  // SBO: 8 rows of 128 bytes
      const uint32_t q_lo0 = sdesc_sw128_lo(smem_u32(q_smem), 16);
      const uint32_t q_lo1 = q_lo0 + (C::TILE_BYTES >> 4);
      const uint32_t k_lo0 = sdesc_sw128_lo(smem_u32(kv_smem), 16);
      const uint32_t v_lo0 = sdesc_sw128_lo(smem_u32(kv_smem), kChunkBytes);  // LBO: next 64 ch
      for (int u = blockIdx.x; ok && u < sch.n_units; u += gridDim.x, ++uc) {
        const UnitInfo ui = decode_unit(sch, u);
        ok = warp_wait(rope_on ? &ctl->q_ready : &ctl->q_full, uc & 1u, abort_w);
        if (!ok) break;
        tc_fence_after_sync();
        // previous tile (for the P V product that trails each S = Q K^T by one tile)
        bool have_prev = false, prev_first = false;
        uint32_t prev_g = 0, prev_v = 0, prev_pidx = 0;
        for (uint64_t m = sch.compute_mask[ui.i]; ok && m; m &= m - 1) {
          const int j = __ffsll(static_cast<long long>(m)) - 1;
          const int nt = ntiles_of(sch, j);
          for (int t = 0; t < nt; ++t, e += 2, ++g) {
            const uint32_t ke = e;
            ok = warp_wait(&ctl->kv_full[ke % STAGES], (ke / STAGES) & 1u, abort_w);
            if (!ok) break;
            tc_fence_after_sync();
            const uint32_t k_lo = k_lo0 + (ke % STAGES) * (C::TILE_BYTES >> 4);
            for (int w = 0; w < 2; ++w) {
              if (have_prev && !(ok = issue_pv<D>(ctl, w, prev_g, prev_v, prev_pidx, prev_first,
                                                  v_lo0, desc_hi, tbase, abort_w)))
                break;
              issue_qk<D>(tbase + C::s_col(w), w ? q_lo1 : q_lo0, k_lo, desc_hi);
              tc_commit(&ctl->s_full[w]);
            }
            if (!ok) break;
            tc_commit(&ctl->kv_empty[ke % STAGES]);
            if (have_prev) tc_commit(&ctl->kv_empty[prev_v % STAGES]);
            have_prev = true;
            prev_first = (t == 0);
            prev_g = g;
            prev_v = ke + 1;
            prev_pidx = pidx;
          }
          ++pidx;
        }
        if (!ok) break;
        tc_commit(&ctl->q_empty);  // every Q K^T of this unit has been issued
        if (!have_prev) continue;  // a unit always visits its own partition; kept for safety
        for (int w = 0; ok && w < 2; ++w)
          ok = issue_pv<D>(ctl, w, prev_g, prev_v, prev_pidx, prev_first, v_lo0, desc_hi, tbase,
                           abort_w);
        if (!ok) break;
        tc_commit(&ctl->kv_empty[prev_v % STAGES]);
      }
      tc_commit(&ctl->drained);
      drain_wait(&ctl->drained, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------------ softmax warpgroups
    const int w = warp >> 2;              // query tile of this warpgroup
    const int lrow = threadIdx.x & 127;   // row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_taddr = tbase + lane_base + C::s_col(w);
    const uint32_t o_taddr = tbase + lane_base + C::o_col(w);
    const float sl2 = args.scale_log2;
    // With RoPE on, the MMA issuer waits for q_ready instead of q_full: once the Q tiles of a
    // unit have landed, each thread rotates its own row of its warpgroup's tile in place and
    // arrives. For the first unit this happens up front; for each later one, right after the
    // last P of the unit before (while the tensor core runs that unit's last P V), so that
    // the next unit's first Q K^T overlaps this unit's epilogue.
    const uint32_t q_row = smem_u32(q_smem) + w * C::TILE_BYTES + lrow * 128;
    const uint32_t tab = smem_u32(rope_tab);
    auto prepare_q = [&](int unit, uint32_t load) -> bool {
      if (!warp_wait(&ctl->q_full, load & 1u, abort_w)) return false;
      const int n_tok = decode_unit(sch, unit).row0 + w * kTileRows + lrow;
      if (n_tok < args.N) rotate_q_row<D>(q_row, lrow & 7, n_tok, args.rope, tab);
      fence_proxy_async_smem();
      mbar_arrive(&ctl->q_ready);
      return true;
    };
    uint32_t g = 0, uc = 0;
    bool ok = true;
    if (rope_on) {
      stage_rope_table(args.rope, rope_tab, threadIdx.x, 2 * kTileRows);
      asm volatile("bar.sync 1, %0;" ::"n"(2 * kTileRows) : "memory");  // softmax warps only
      if (blockIdx.x < sch.n_units) ok = prepare_q(blockIdx.x, 0);
    }
    for (int u = blockIdx.x; ok && u < sch.n_units; u += gridDim.x, ++uc) {
      const UnitInfo ui = decode_unit(sch, u);
      const int qrow = ui.qb * kUnitRows + w * kTileRows + lrow;  // row within partition i
      const bool row_ok = qrow < ui.n_i;
      for (uint64_t m = sch.compute_mask[ui.i]; ok && m; m &= m - 1) {
        const int j = __ffsll(static_cast<long long>(m)) - 1;
        const int nj = sch.offsets[j + 1] - sch.offsets[j];
        const int nt = (nj + kTileRows - 1) / kTileRows;
        float m_run = 0.f, l_run = 0.f;  // reference (log2 units) and row sum of the partition
        for (int t = 0; t < nt; ++t, ++g) {
          ok = warp_wait(&ctl->s_full[w], g & 1u, abort_w);
          if (!ok) break;
          tc_fence_after_sync();
          const int valid = nj - t * kTileRows;
          if (t == 0) m_run = row_max(s_taddr, valid) * sl2;  // first tile: exact max
          uint32_t pk[kTileRows / 2];
          float l_t = exp_pack_row(s_taddr, valid, sl2, m_run, pk);
          const bool redo = t > 0 && !(l_t <= kRescaleSum);
          if (__any_sync(0xffffffffu, redo)) {
            // the rows whose sum left the range move m to the exact max of this tile (S is
            // re-read: it is still intact in TMEM), rescale O and l, and recompute P
            const float m_tile = row_max(s_taddr, valid) * sl2;
            float alpha = 1.f;
            if (redo) {
              const float m_new = fmaxf(m_run, m_tile);
              alpha = ex2_approx(m_run - m_new);
              l_run *= alpha;
              m_run = m_new;
            }
            // O holds the sum over earlier tiles of this partition: wait for the last P V
            ok = warp_wait(&ctl->o_done[w], (g - 1) & 1u, abort_w);
            if (!ok) break;
            tc_fence_after_sync();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t r[32];
              tmem_ld_32x32b_x32(o_taddr + c * 32, r);
#pragma unroll
              for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(__uint_as_float(r[x]) * alpha);
              tmem_st_32x32b_x32(o_taddr + c * 32, r);
            }
            l_t = exp_pack_row(s_taddr, valid, sl2, m_run, pk);
          }
          {
            uint32_t lo[32], hi[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              lo[c] = pk[c];
              hi[c] = pk[32 + c];
            }
            tmem_st_32x32b_x32(s_taddr, lo);
            tmem_st_32x32b_x32(s_taddr + 32, hi);
          }
          l_run = t == 0 ? l_t : l_run + l_t;
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(&ctl->p_full[w]);
          if (rope_on && t == nt - 1 && (m & (m - 1)) == 0 &&
              u + static_cast<int>(gridDim.x) < sch.n_units)
            ok = prepare_q(u + gridDim.x, uc + 1);  // last P of the unit: hand over the next Q
        }
        if (!ok) break;
        // ---- epilogue of pair (i, j): O_ij = O / l, lse_ij = ln 2 * (m_run + log2 l)
        ok = warp_wait(&ctl->o_done[w], (g - 1) & 1u, abort_w);
        if (!ok) break;
        tc_fence_after_sync();
        const float inv_l = 1.f / l_run;
        // the pair's slot: a device slot, or its host slot when the cache keeps it in host
        // memory (the stores then cross the host link)
        __nv_bfloat16* orow;
        float* lse_p;
        state_ptrs(args.cache, sch.P, args.N, D, static_cast<int64_t>(ui.b) * sch.H + ui.h, ui.i, j,
                   static_cast<int64_t>(ui.row0 + w * kTileRows + lrow), orow, lse_p);
        // read the whole row of O in one TMEM load and hand O back to the MMA warp before the
        // packing and the global stores, so that the next partition's first P V can start
        uint32_t r[D];
        if constexpr (D == 128)
          tmem_ld_32x32b_x128(o_taddr, r);
        else
          tmem_ld_32x32b_x64(o_taddr, r);
        tc_fence_before_sync();
        mbar_arrive(&ctl->o_free[w]);
        if (row_ok) {
#pragma unroll
          for (int c = 0; c < D / 8; ++c) {
            const uint32_t p0 = pack_bf16x2(__uint_as_float(r[8 * c]) * inv_l, __uint_as_float(r[8 * c + 1]) * inv_l);
            const uint32_t p1 = pack_bf16x2(__uint_as_float(r[8 * c + 2]) * inv_l, __uint_as_float(r[8 * c + 3]) * inv_l);
            const uint32_t p2 = pack_bf16x2(__uint_as_float(r[8 * c + 4]) * inv_l, __uint_as_float(r[8 * c + 5]) * inv_l);
            const uint32_t p3 = pack_bf16x2(__uint_as_float(r[8 * c + 6]) * inv_l, __uint_as_float(r[8 * c + 7]) * inv_l);
            reinterpret_cast<uint4*>(orow)[c] = make_uint4(p0, p1, p2, p3);
          }
          *lse_p = (m_run + __log2f(l_run)) * kLn2;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tbase, C::TMEM_COLS);
  }
  if (threadIdx.x == 0 && ctl->abort_word) atomicExch(args.err, 1);
}

}  // namespace

cudaError_t launch_pair_tc(int d, const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           const PairTcArgs& args, int num_sms, cudaStream_t stream) {
  if (args.sched.n_units <= 0) return cudaSuccess;
  const int grid = args.sched.n_units < num_sms ? args.sched.n_units : num_sms;
  cudaError_t err;
  if (args.rope.n_pairs < 0 || 8 * args.rope.n_pairs > kRopeSmemMaxBytes) return cudaErrorInvalidValue;
  if (d == 128) {
    const int smem = smem_bytes<128>(args.rope.n_pairs);
    err = cudaFuncSetAttribute(pair_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem_bytes<128>(kRopeSmemMaxBytes / 8));
    if (err != cudaSuccess) return err;
    pair_tc_kernel<128><<<grid, kThreads, smem, stream>>>(mq, mk, mv, args);
  } else if (d == 64) {
    const int smem = smem_bytes<64>(args.rope.n_pairs);
    err = cudaFuncSetAttribute(pair_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               smem_bytes<64>(kRopeSmemMaxBytes / 8));
    if (err != cudaSuccess) return err;
    pair_tc_kernel<64><<<grid, kThreads, smem, stream>>>(mq, mk, mv, args);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ditango
