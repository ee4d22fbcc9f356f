/*
 * ditango.h - C ABI of a single-GPU (GB300, sm_103a) library for partitioned attention with
 * attention-state reuse, as used for video diffusion-transformer inference.
 *
 * Method: "DiTango: Cost-Effective Parallel Diffusion Generation with Selective Attention State
 * Reuse" (gist.science/paper/2607.15650), Technical Summary, Methodology:
 *   1. Anchor-Guided Selection Planner - per step, each (query partition i, KV partition j)
 *      pair either computes a fresh attention state or reuses the state cached at an earlier
 *      step; anchor steps compute every pair; local states are always computed.
 *   2. State-Centric Parallel Runtime, State Composition - an attention state is the output
 *      plus the log-sum-exp; states combine associatively and commutatively, and the composed
 *      states are what is cached.
 * Optional rotary prologue: "Accelerating Video Generation Inference with Sequential-Parallel
 * 3D Positional Encoding Using a Global Time Index" (gist.science/es/paper/2603.06664),
 * section 2 (t_global = t_local + s; sin/cos precomputed into contiguous tensors).
 *
 * Definitions used throughout (the pages print no formula; these are the plain readings):
 *   partitions   contiguous slices of the N tokens; the first N mod P partitions hold one
 *                extra row (offsets[p] = p*floor(N/P) + min(p, N mod P)).
 *   pair state   for query row r and KV partition j, with z_c = scale * <q_r, k_c>:
 *                lse_ij[r] = ln sum_{c in j} exp(z_c)     (natural log)
 *                O_ij[r]   = sum_{c in j} exp(z_c - lse_ij[r]) * v_c
 *                i.e. O is normalised within partition j only.
 *   merge        lse = ln sum_j exp(lse_j);  O = sum_j exp(lse_j - lse) * O_j.
 *   reuse mask   P x P bytes, row-major, mask[i*P + j] = 1: reuse the cached state of pair
 *                (i, j); 0: compute it from this step's inputs. The diagonal must be 0.
 *
 * Conventions:
 *   - Every device buffer is allocated and owned by the caller. No entry point allocates or
 *     frees device memory.
 *   - Entry points taking `stream` are asynchronous on that stream (a cudaStream_t passed as
 *     void*; NULL means the legacy default stream). Host-side validation happens before any
 *     launch; on any error nothing is launched and no plan state changes.
 *   - Return value: a ditango_status (0 = success). No C++ exception crosses this boundary.
 *   - Thread safety: a plan must not be used from two threads at once.
 */
#ifndef DITANGO_H_
#define DITANGO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DITANGO_ABI_VERSION 3
#define DITANGO_MAX_PARTITIONS 64 /* P limit of a plan */
#define DITANGO_MAX_STATES 64     /* state limit of one ditango_merge call */

typedef enum {
  DITANGO_OK = 0,
  DITANGO_ERR_INVALID_ARG = 1,     /* null pointer, N < P, P outside [1, 64], ... */
  DITANGO_ERR_INVALID_MASK = 2,    /* a value other than 0/1, or a reused diagonal pair */
  DITANGO_ERR_NO_CACHE = 3,        /* the mask reuses a pair never computed under this plan */
  DITANGO_ERR_SHAPE = 4,           /* tensor shapes disagree with the plan or each other */
  DITANGO_ERR_DTYPE = 5,           /* unsupported or mismatched element type */
  DITANGO_ERR_ALIGN = 6,           /* pointer or stride not 16-byte aligned where required */
  DITANGO_ERR_WORKSPACE = 7,       /* workspace missing or smaller than required */
  DITANGO_ERR_CUDA = 8,            /* a CUDA runtime/driver call or a kernel launch failed */
  DITANGO_ERR_DEVICE_TIMEOUT = 9,  /* a kernel gave up waiting on one of its own barriers */
  DITANGO_ERR_UNSUPPORTED = 10     /* head dim / dtype combination not built */
} ditango_status;

typedef enum { DITANGO_F32 = 0, DITANGO_BF16 = 1 } ditango_dtype;

/* A strided view of device memory. `stride` is in elements. Unused trailing dims ignored. */
typedef struct {
  void* ptr;
  int32_t dtype; /* ditango_dtype */
  int32_t ndim;
  int64_t shape[5];
  int64_t stride[5];
} ditango_tensor;

/* The state cache of one attention layer, owned by the caller and passed unchanged every
 * step. O: [B, H, P, N, d], contiguous, dtype BF16 for bf16 inputs and F32 for f32 inputs.
 * lse: [B, H, P, N], contiguous, F32. Slot [b, h, j, r] holds the state of (partition(r), j)
 * for query row r. Contents are meaningful only for pairs this plan has computed.
 * host_O, host_lse (optional: ptr NULL = not used): host storage for the states that do not
 * fit in device memory (DiTango, closing limitations paragraph: state-cache memory is a
 * constraint, CPU offloading is the remedy it names). With them, O and lse hold only S device
 * slots per row ([B, H, S, N, d] and [B, H, S, N], 1 <= S <= P) and host_O, host_lse are
 * [B, H, P, N, d] and [B, H, P, N] (same dtypes, contiguous) in page-locked host memory that
 * the device can address (cudaHostAlloc / cudaHostRegister). For query partition i the S pairs
 * (i, j) nearest the diagonal (smallest |i - j|, ties to the smaller j; see
 * ditango_cache_slot_map) keep their states in device slots 0..S-1 in ascending j; every other
 * pair keeps its state in host slot [b, h, j, r]. The kernels read and write host states in
 * place over the host link; nothing is copied, and every result is bit-identical to a cache
 * held wholly on the device. With group states and a distance mask |i - j| >= D, S = 2D - 1
 * keeps every pair a steady reuse step computes on the device: host memory is then written
 * when far pairs are computed (anchor steps) and read when group states are rebuilt. Without
 * host storage S must equal P.
 * group_O, group_lse (optional: ptr NULL = not used): one composed state per query row,
 * [B, H, N, d] and [B, H, N], contiguous, both F32 (DiTango, Methodology 2, State Composition
 * and Dynamic Group Compose: cached states merge into a coarser group state without
 * recomputation, and the result is itself a state). When present, a step merges every row's
 * computed states with the single group state of its partition's reused pairs instead of with
 * each reused state. The library builds a partition's group state (one merge of its reused
 * cached states, in the step's merge pass) at a step whose reused set differs from the one the
 * group was built from, or when one of those pairs has been recomputed since; the plan records
 * this, so pass the same buffers with the same plan every step (other buffers make it rebuild).
 * A step that computes every pair (reuse_mask given, all zero) on a plan whose default mask
 * (ditango_plan / ditango_plan_set_mask) reuses pairs builds, in its merge pass, the group
 * states of that default mask's reused sets from its own fresh states: a following step under
 * the default mask then finds them current (DiTango, Methodology 2, Pipeline Orchestration:
 * the reuse work rides on a pass that runs anyway). Its output is the same merge of all states,
 * taken through the group state. */
typedef struct {
  ditango_tensor O;
  ditango_tensor lse;
  ditango_tensor group_O;
  ditango_tensor group_lse;
  ditango_tensor host_O;
  ditango_tensor host_lse;
} ditango_state_cache;

/* Host only: where each pair's state lives when the device cache holds S of the P states per
 * row. map (P*P bytes, row-major [i][j]) receives the device slot (0..S-1) of pair (i, j), or
 * -1 for a pair kept in host storage. S = P maps pair (i, j) to slot j. Errors: INVALID_ARG
 * (P outside [1, 64], S outside [1, P], NULL map). */
int ditango_cache_slot_map(int32_t P, int32_t S, int8_t* map);

/* Precomputed 3D RoPE tables (device memory, fp32, row-major, filled by
 * ditango_rope_build_tables). Channel pairs (2m, 2m+1) of each head: the first dt/2 pairs turn
 * with the global frame index t, the next dh/2 with the row h, the last dw/2 with the column w;
 * pair k of an axis of width d_a turns by pos * theta^(-2k/d_a).
 * Token n of the sequence sits at t = n / (Hl*Wl) + start_frame, h = (n / Wl) % Hl,
 * w = n % Wl, so N must be a multiple of Hl*Wl and start_frame + N/(Hl*Wl) <= T_tab.
 * Each table has a residual table of the same shape: cos_t_lo = fl32(cos - cos_t) with cos in
 * fp64, and so on, so that table + residual carries cos and sin to about 48 bits. The BF16
 * path needs them to round every rotated value as the rotation with fp64 cos/sin rounds
 * (nearest-even); all twelve pointers of a non-empty axis must be set. */
typedef struct {
  float* cos_t; float* sin_t; /* [T_tab, dt/2] */
  float* cos_h; float* sin_h; /* [Hl, dh/2] */
  float* cos_w; float* sin_w; /* [Wl, dw/2] */
  int64_t T_tab, Hl, Wl;
  int32_t dt, dh, dw;       /* even, dt + dh + dw = d */
  int64_t start_frame;      /* s: global frame index of this sequence's first frame */
  float* cos_t_lo; float* sin_t_lo; /* residuals, shapes as above */
  float* cos_h_lo; float* sin_h_lo;
  float* cos_w_lo; float* sin_w_lo;
} ditango_rope;

/* A list of n states with a common layout, for ditango_merge. State s has outputs O[s]
 * ([G1, G2, R, d], strides O_stride for G1, G2, R; d contiguous) and log-sum-exps lse[s]
 * ([G1, G2, R] fp32, strides lse_stride). O and lse are HOST arrays of n DEVICE pointers. */
typedef struct {
  int32_t n;     /* 1 .. DITANGO_MAX_STATES */
  int32_t dtype; /* of every O[s]: F32 or BF16 */
  const void* const* O;
  const float* const* lse;
  int64_t shape[4];      /* G1, G2, R, d */
  int64_t O_stride[3];   /* elements */
  int64_t lse_stride[3]; /* elements */
} ditango_state_list;

typedef struct ditango_plan_s* ditango_plan_t;

/* ---- plan (host only) -------------------------------------------------------------------
 * Source: DiTango, Methodology 1 (per-step compute/reuse decision per partition pair) and the
 * partitioning of the sequence into contiguous context partitions (Problem Statement).
 * Creates a plan for N tokens in P partitions (1 <= P <= 64, N >= P). `mask` (P*P bytes, may
 * be NULL = every pair computed) becomes the plan's default reuse mask; it is validated for
 * values and diagonal only (cache validity is checked per step). The plan also holds the
 * cache bookkeeping: per pair, whether a state has been computed and at which step.
 * Errors: INVALID_ARG, INVALID_MASK. *out_plan is set only on success. */
int ditango_plan(int64_t N, int32_t P, const uint8_t* mask, ditango_plan_t* out_plan);

/* Frees the plan (host memory only). NULL is accepted. */
void ditango_plan_destroy(ditango_plan_t plan);

/* Replaces the default reuse mask (same validation as ditango_plan). The default mask is used
 * by steps given reuse_mask = NULL, and names the group states an all-compute step builds in
 * advance (see ditango_state_cache). */
int ditango_plan_set_mask(ditango_plan_t plan, const uint8_t* mask);

/* Checks `mask` (NULL = default mask) against the bookkeeping without changing anything:
 * INVALID_MASK for bad values / reused diagonal, NO_CACHE for reuse of a never-computed pair. */
int ditango_plan_check_mask(ditango_plan_t plan, const uint8_t* mask);

/* Copies the P+1 partition offsets into `offsets` (host). */
int ditango_plan_get_offsets(ditango_plan_t plan, int64_t* offsets);

/* Writes the pairs computed under `mask` (NULL = default mask), row-major (i ascending, then
 * j ascending), as (i, j) int32 pairs into `pairs` (host, room for 2*P*P) and their number
 * into *count. */
int ditango_plan_get_pairs(ditango_plan_t plan, const uint8_t* mask, int32_t* pairs,
                           int32_t* count);

/* Copies the cache bookkeeping: valid[i*P+j] (1 = a state exists), step_computed[i*P+j]
 * (-1 = never) and the number of steps run so far. Any output pointer may be NULL. */
int ditango_plan_get_cache_state(ditango_plan_t plan, uint8_t* valid, int64_t* step_computed,
                                 int64_t* steps_run);

/* Restores the cache bookkeeping (the counterpart of ditango_plan_get_cache_state), for a
 * caller that restores a saved state cache into its buffers: valid[i*P+j] in {0, 1},
 * step_computed[i*P+j] (-1 exactly where valid is 0, else in [0, steps_run)), steps_run >= 0.
 * The diagonal may be invalid only before the first step (steps_run = 0). Group states built
 * under the plan are forgotten (rebuilt at their next use). Errors: INVALID_ARG (NULL
 * pointers, values out of range); the plan is unchanged on error. */
int ditango_plan_set_cache_state(ditango_plan_t plan, const uint8_t* valid,
                                 const int64_t* step_computed, int64_t steps_run);

/* Optional timing hook. `events` is a host array of 4 cudaEvent_t handles (created by the
 * caller, passed as void*), or NULL to switch the hook off. While set, every
 * ditango_attn_step on this plan records events[0] before the rotary prologue, events[1]
 * before the pair kernel, events[2] before the merge and events[3] after it, on the step's
 * stream, so that the caller can read per-kernel device time with cudaEventElapsedTime. */
int ditango_plan_set_profile_events(ditango_plan_t plan, void* const* events);

/* ---- anchor-guided selection planner ----------------------------------------------------
 * Source: DiTango, Methodology 1, Anchor-Guided Selection Planner. The page names the
 * ingredients (error as a function of partition importance w and temporal error growth delta;
 * anchor steps that recompute everything and update w; the change of the always-computed local
 * states as the online proxy for the drift of the remote ones; decisions per group of
 * spatially adjacent partitions) and leaves the formulas open. These calls take the plainest
 * reading:
 *   w[i][j]  = mean over the rows r of partition i (and batch, heads) of exp(lse_ij - lse_i),
 *              partition j's share of row r's attention mass (each row of w sums to 1);
 *   delta[i] = ||O_ii(t) - O_ii(anchor)|| / ||O_ii(anchor)|| over partition i's rows;
 *   error    = w[i][j] * delta[i], summed over a group's members j != i.
 * cache: the layer's state cache as passed to ditango_attn_step (group states unused). */

/* Importance weights from the cache as it stands (call it after an anchor step, whose every
 * state is fresh). w: device memory for P*P doubles (row-major [i][j]); written
 * asynchronously on `stream`. Errors: INVALID_ARG, SHAPE, DTYPE, ALIGN, CUDA. */
int ditango_planner_importance(ditango_plan_t plan, const ditango_state_cache* cache, double* w,
                               void* stream);

/* Copies every partition's local states (cache slots (i, i) of its rows) into `snapshot`
 * ([B, H, N, d], the cache's dtype, contiguous, 16-byte aligned; owned by the caller), to
 * be compared against later. Call it after the anchor step. Asynchronous on `stream`. */
int ditango_planner_snapshot(ditango_plan_t plan, const ditango_state_cache* cache,
                             const ditango_tensor* snapshot, void* stream);

/* Drift of every partition's local states since the snapshot. delta: device memory for 2*P
 * doubles; on completion delta[0..P) holds the drifts (0 where the snapshot is all zero) and
 * delta[P..2P) is scratch. Asynchronous on `stream`. */
int ditango_planner_drift(ditango_plan_t plan, const ditango_state_cache* cache,
                          const ditango_tensor* snapshot, double* delta, void* stream);

/* Host only: the reuse mask (P*P bytes, 1 = reuse) for the next step from w (host, P*P) and
 * delta (host, P). KV partitions form contiguous groups of `group` (the last may be shorter).
 * For each query partition i and group G with a member j != i, the predicted error is the sum,
 * in ascending j, of w[i][j] * delta[i] over those members. Groups holding a pair this plan
 * never computed are recomputed first; the others go by decreasing error (ties: lower i, then
 * lower G) and are recomputed when their error exceeds tau and the computed pairs, counting
 * the P local ones, stay within `budget` (budget < 0: no limit). The local pairs are always
 * computed. Errors: INVALID_ARG (NULL pointers, group < 1, tau < 0 or NaN, non-finite w or
 * delta). */
int ditango_planner_select(ditango_plan_t plan, const double* w, const double* delta, double tau,
                           int32_t group, int32_t budget, uint8_t* mask);

/* ---- fault injection (a test hook; the paper has no counterpart) ------------------------
 * kind 1 arms a one-shot fault for the next ditango_attn_step on this plan that runs the BF16
 * pair kernel; kind 0 disarms. In that launch the first CTA skips the copy of its first K tile,
 * so the MMA warp's bounded wait for it runs out after about one second: every role of that CTA
 * stops, waits (bounded) for its copies and MMAs in flight, frees its TMEM and sets the device
 * error word. The step itself returns DITANGO_OK (the fault happens on the device);
 * ditango_device_status then reports DITANGO_ERR_DEVICE_TIMEOUT. The outputs of that step and
 * the cache slots of the aborted CTA's work are unspecified; the context stays usable, and a
 * following step that computes every pair restores the cache. Nothing traps, faults or hangs.
 * Errors: DITANGO_ERR_INVALID_ARG for a NULL plan or another kind. */
int ditango_plan_inject_fault(ditango_plan_t plan, int32_t kind);

/* ---- one attention-layer step -----------------------------------------------------------
 * Source: DiTango, Methodology 1-2 (compute or reuse per pair, then compose the states);
 * rotary prologue from the Causal-RoPE SP page, section 2.
 * q, k, v: [B, N, H, d] device tensors of one dtype (BF16 or F32), d contiguous; for BF16 the
 *   other strides must be multiples of 8 elements and the pointers 16-byte aligned.
 *   Supported d: 64 and 128 (UNSUPPORTED otherwise). B and H must be at least 1: an empty
 *   batch returns SHAPE, whatever its pointers, and leaves the plan unchanged.
 * rope: NULL = no rotation; else q and k are rotated before attention and the attention reads
 *   them in the input dtype: for BF16 each rotated value is the nearest-even bf16 of the
 *   rotation with fp64 cos/sin (exact up to ~2^-46 relative), for F32 the rotation evaluated
 *   in fp32 (within a few fp32 ulps); v is never rotated.
 * reuse_mask: host P*P bytes; NULL = the plan's default mask.
 * cache: the layer's state cache (see ditango_state_cache). Pairs with mask 0 are computed
 *   from this step's inputs and overwrite their slots; pairs with mask 1 are read as cached.
 * out: [B, N, H, d], same dtype as q, d contiguous. out_lse: [B, H, N] F32 with strides of
 *   at least 1 (SHAPE otherwise), or NULL.
 * softmax_scale: the `scale` of the pair-state definition (commonly 1/sqrt(d)).
 * workspace: device memory of at least ditango_attn_step_workspace_size(...) bytes, 256-byte
 *   aligned (may be NULL when that size is 0). Its contents need not be preserved. It holds
 *   the rotated k, and the rotated q unless the BF16 pair kernel rotates each Q tile itself
 *   (it does when the table rows of the sequence, as (cos, sin) pairs, fit in 32 KB).
 * On success the computed pairs are recorded in the plan as valid at this step. The result
 * is complete when the stream reaches this point. Kernel-side barrier timeouts are reported
 * by ditango_device_status, not here. */
int ditango_attn_step(ditango_plan_t plan, const ditango_tensor* q, const ditango_tensor* k,
                      const ditango_tensor* v, const ditango_rope* rope,
                      const uint8_t* reuse_mask, const ditango_state_cache* cache,
                      const ditango_tensor* out, const ditango_tensor* out_lse,
                      float softmax_scale, void* workspace, size_t workspace_bytes,
                      void* stream);

/* The same step for callers that cannot allocate device memory (the paper has no counterpart
 * to this entry point; it exists for the library's users). Some callers cannot call cudaMalloc:
 * plugins whose host framework forbids device allocation during execution, processes whose
 * memory pool already holds the GPU's free memory, latency-critical loops that cannot take
 * cudaMalloc's implicit synchronisation. Arguments and errors are those of ditango_attn_step,
 * without the workspace: the step's scratch (the rotated q and k when rope != NULL) lives in
 * a 64 MiB device array inside the library, held on every GPU where the library's device code
 * is loaded until the process exits. Steps whose scratch exceeds 64 MiB
 * (ditango_attn_step_workspace_size > 64 MiB, i.e. more than 2^24 bf16 or 2^23 fp32 elements
 * per rotated tensor) return DITANGO_ERR_WORKSPACE before launching anything; shapes that
 * ditango_attn_step refuses (a dimension below 1, N other than the plan's, B*N*H above 2^31)
 * return DITANGO_ERR_SHAPE first. Allocates nothing (no
 * cudaMalloc/cudaFree). The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress), so make it before any stream capture on that device. Every call
 * shares the one array and it keeps the last call's contents; nothing in it needs to start
 * at zero (each call writes every byte it reads), but calls whose work overlaps on the GPU
 * (other streams, other threads) race on it. */
int ditango_attn_step_static_workspace(ditango_plan_t plan, const ditango_tensor* q,
                                       const ditango_tensor* k, const ditango_tensor* v,
                                       const ditango_rope* rope, const uint8_t* reuse_mask,
                                       const ditango_state_cache* cache, const ditango_tensor* out,
                                       const ditango_tensor* out_lse, float softmax_scale,
                                       void* stream);

/* Bytes of workspace ditango_attn_step needs for these shapes (0 without RoPE). */
size_t ditango_attn_step_workspace_size(ditango_plan_t plan, int64_t B, int64_t H, int32_t d,
                                        int32_t dtype, int32_t use_rope);

/* ---- state merge -------------------------------------------------------------------------
 * Source: DiTango, Methodology 2, State Composition and Dynamic Group Compose (cached states
 * merge into coarser groups without recomputation; the result is itself a state).
 * Merges the n states of `states` row by row into out ([G1, G2, R, d], same dtype as the
 * states, d contiguous, other strides at least 1) and out_lse ([G1, G2, R] F32, strides at least
 * 1, or NULL); the list's O and lse strides must be at least 1 too. Any d that is a multiple of
 * the 16-byte vector (8 BF16 or 4 F32 channels) is supported. Reads only the
 * listed states. With no rows (G1, G2 or R = 0) it returns DITANGO_OK without touching memory,
 * and the data pointers may be NULL. Errors: INVALID_ARG, SHAPE, DTYPE, ALIGN (O pointers / row
 * strides of BF16 states must allow 16-byte vector access), CUDA. */
int ditango_merge(const ditango_state_list* states, const ditango_tensor* out,
                  const ditango_tensor* out_lse, void* stream);

/* ---- RoPE tables -------------------------------------------------------------------------
 * Source: Causal-RoPE SP page, section 2 (frequencies precomputed into contiguous tensors, so
 * inference moves no positional data between host and GPU). Fills the six fp32 tables of
 * `rope` and their six residual tables (caller-allocated device buffers of the sizes given
 * there) on the device: cos/sin(pos * theta^(-2k/d_a)) computed in fp64, rounded to fp32, and
 * the fp32 rounding of what that rounding left out. */
int ditango_rope_build_tables(const ditango_rope* rope, double theta, void* stream);

/* ---- diagnostics --------------------------------------------------------------------------- */

/* Synchronises `stream`, then reports and clears the device-side error word that kernels set
 * when a bounded barrier wait gives up: DITANGO_OK or DITANGO_ERR_DEVICE_TIMEOUT (with the
 * kernel's code in *code if code != NULL), or DITANGO_ERR_CUDA.
 * The library looks up the device addresses of its own device variables (this error word, the
 * static workspace) once per device and keeps them; after cudaDeviceReset the process must
 * reload the library before calling it on that device again. */
int ditango_device_status(void* stream, int32_t* code);

/* Static description of a status code. */
const char* ditango_status_string(int status);

/* DITANGO_ABI_VERSION of the loaded library. */
int ditango_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DITANGO_H_ */
