// Internal declarations shared by the host API (api.cu, plan.cpp) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ditango.h"

namespace ditango {

constexpr int kMaxP = DITANGO_MAX_PARTITIONS;
constexpr int kMaxStates = DITANGO_MAX_STATES;

// Work decomposition of one step for the pair kernels (the mask-driven tile scheduler).
// A unit is one block of `block_rows` query rows of partition i for one (b, h); a unit
// visits every KV partition j with bit j of compute_mask[i] set, in ascending j, and emits one
// state per visited j. Partitions are listed in `order` by decreasing cost (computed KV rows)
// and units are numbered partition by partition in that order, (b, h) major, query block
// minor, so that CTAs running side by side share the K/V tiles of one (b, h) through L2.
struct PairSchedule {
  int32_t P;
  int32_t BH;          // B * H
  int32_t H;
  int32_t block_rows;  // query rows per unit
  int32_t n_units;
  int32_t offsets[kMaxP + 1];
  uint64_t compute_mask[kMaxP];  // bit j of [i]: pair (i, j) is computed this step
  int32_t order[kMaxP];          // partition at position k of the unit numbering
  int32_t seg_start[kMaxP + 1];  // first unit of order[k]; seg_start[P] = n_units
};

// Where the states of a layer's state cache live. The device cache holds S slots per query
// row ([B, H, S, N, d] and [B, H, S, N]); pair (i, j) with slot[i * P + j] = s >= 0 lives in
// device slot s, every other pair in slot j of the host cache ([B, H, P, N, d] and
// [B, H, P, N], page-locked host memory addressed by the device). Without host storage S = P
// and slot[i * P + j] = j.
struct CacheLoc {
  void* dO;
  float* dL;
  void* hO;
  float* hL;
  int32_t S;
  int8_t slot[kMaxP * kMaxP];
};

// O and lse pointers of the state (i, j) of query row r of (b, h) slab bh (d channels of T).
template <typename T>
__host__ __device__ __forceinline__ void state_ptrs(const CacheLoc& c, int32_t P, int64_t N,
                                                    int32_t d, int64_t bh, int32_t i, int32_t j,
                                                    int64_t r, T*& o, float*& l) {
  const int s = c.slot[i * P + j];
  if (s >= 0) {
    const int64_t row = (bh * c.S + s) * N + r;
    o = static_cast<T*>(c.dO) + row * d;
    l = c.dL + row;
  } else {
    const int64_t row = (bh * P + j) * N + r;
    o = static_cast<T*>(c.hO) + row * d;
    l = c.hL + row;
  }
}

// Device slot of every pair when the device cache holds S of the P states per row (host only;
// the rule of ditango_cache_slot_map).
void cache_slot_map(int32_t P, int32_t S, int8_t* map);

// Fills a schedule. `mask` is P*P (1 = reuse). Host only.
void build_schedule(int64_t N, int32_t P, const int64_t* offsets, const uint8_t* mask, int64_t B,
                    int64_t H, int32_t block_rows, PairSchedule* s);

// 3D RoPE tables for rotating Q inside the pair kernel (see rope.cu for the definition). The
// kernel copies the rows it can need into shared memory as (cos, sin) pairs: nT frame rows
// (frames start_frame .. start_frame + nT - 1) of stride sT, then Hl rows of stride sH, then
// Wl rows of stride sW (strides in pairs, odd so that a warp's 32 rows hit distinct banks).
struct RopeQ {
  const float *cos_t, *sin_t, *cos_h, *sin_h, *cos_w, *sin_w;
  const float *cos_t_lo, *sin_t_lo, *cos_h_lo, *sin_h_lo, *cos_w_lo, *sin_w_lo;  // residuals
  int32_t Hl, Wl, start_frame;
  int32_t dt, dh, dw;
  int32_t nT, sT, sH, sW;
  int32_t n_pairs;  // nT*sT + Hl*sH + Wl*sW; 0: q is used as given
};
// Shared memory the pair kernel may give the tables; larger tables keep Q in the pre-pass.
constexpr int kRopeSmemMaxBytes = 32768;

// bf16 pair kernel on tcgen05 (head dim 64 or 128).
struct PairTcArgs {
  PairSchedule sched;
  int64_t N;
  CacheLoc cache;     // bf16 states
  float scale_log2;   // softmax scale * log2(e)
  int* err;           // device error word
  RopeQ rope;         // rotation applied to each Q tile after it lands in shared memory
  int32_t inject_fault;  // 1: CTA 0 skips the copy of its first K tile (test hook)
};
cudaError_t launch_pair_tc(int d, const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const PairTcArgs& args, int num_sms,
                           cudaStream_t stream);

// fp32 pair kernel on CUDA cores (head dim 64 or 128).
struct PairF32Args {
  PairSchedule sched;
  int64_t N;
  const float* q; const float* k; const float* v;
  int64_t qs[3], ks[3], vs[3];  // element strides of b, n, h (d contiguous)
  CacheLoc cache;     // fp32 states
  float scale;
};
cudaError_t launch_pair_f32(int d, const PairF32Args& args, cudaStream_t stream);

// Merge of n states with a common [G1, G2, R, d] layout.
struct MergeArgs {
  int32_t n;
  int32_t d;
  int32_t dtype;      // of the states
  int32_t out_dtype;  // of out: the states' dtype, or F32 (group states)
  int64_t G1, G2, R;
  const void* O[kMaxStates];
  const float* lse[kMaxStates];
  int64_t oS[3], lS[3];
  void* out;
  int64_t outS[3];
  float* out_lse;  // may be null
  int64_t olS[3];
};
cudaError_t launch_merge(const MergeArgs& args, cudaStream_t stream);

// The merge of one attention step: every query row r of partition i merges the cache states
// (i, j) of the pairs in cache_set[i] and, if bit i of `group` is set, the group state of its
// row (the composed state of partition i's reused pairs). If bit i of `rebuild` is set, the
// row first builds that group state from the cache states in reused_set[i] and stores it.
struct StepMergeArgs {
  int32_t P, d, dtype;  // dtype of the cache states and of out
  int64_t B, H, N;
  int32_t offsets[kMaxP + 1];
  uint64_t cache_set[kMaxP];
  uint64_t reused_set[kMaxP];
  uint64_t group;    // partitions whose rows start from their group state
  uint64_t rebuild;  // partitions whose group state is built in this launch (subset of group)
  CacheLoc cache;
  float* gO;        // [B, H, N, d] fp32 (may be null when group == 0)
  float* gL;        // [B, H, N]
  void* out;        // element strides of b, h, r in outS (d contiguous)
  int64_t outS[3];
  float* out_lse;   // may be null
  int64_t olS[3];
};
cudaError_t launch_step_merge(const StepMergeArgs& args, cudaStream_t stream);

// Anchor-guided planner reductions over a state cache (planner.cu). Importance accumulates
// sums[i * P + j] over the rows of partition i and writes w = sums / rows (P*P doubles, in
// place); drift accumulates (num_i, den_i) in sums[0..2P) and writes delta_i = sqrt(num/den).
struct PlannerArgs {
  int32_t P, d, dtype;  // dtype of the cache O and the snapshot
  int64_t B, H, N;
  int32_t offsets[kMaxP + 1];
  CacheLoc cache;
  const void* snap;  // diagonal states at the anchor [B, H, N, d]
  double* sums;      // device scratch: P*P (importance) or 2P (drift) doubles
  double* out;       // device: w [P*P] or delta [P]
};
cudaError_t launch_planner_importance(const PlannerArgs& args, cudaStream_t stream);
cudaError_t launch_planner_drift(const PlannerArgs& args, cudaStream_t stream);
cudaError_t launch_planner_snapshot(const PlannerArgs& args, cudaStream_t stream);

// 3D RoPE applied to up to two [B, N, H, d] tensors, written contiguous.
struct RopeApplyArgs {
  int32_t n_tensors;
  const void* x[2];
  int64_t xs[2][3];  // element strides of b, n, h
  void* y[2];        // contiguous [B, N, H, d], same dtype as x
  int32_t dtype;
  int64_t B, N, H;
  int32_t d;
  const float *cos_t, *sin_t, *cos_h, *sin_h, *cos_w, *sin_w;
  const float *cos_t_lo, *sin_t_lo, *cos_h_lo, *sin_h_lo, *cos_w_lo, *sin_w_lo;  // residuals
  int64_t Hl, Wl, start_frame;
  int32_t dt, dh, dw;
};
cudaError_t launch_rope_apply(const RopeApplyArgs& args, cudaStream_t stream);
cudaError_t launch_rope_tables(const ditango_rope& rope, double theta, cudaStream_t stream);

}  // namespace ditango
