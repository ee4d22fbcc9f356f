// The plan object behind the opaque ditango_plan_t handle (host memory only).
#pragma once
#include <cstdint>
#include <vector>

#include "ditango.h"

struct ditango_plan_s {
  int64_t N = 0;
  int32_t P = 0;
  std::vector<int64_t> offsets;       // P + 1
  std::vector<uint8_t> mask;          // default reuse mask, P * P
  std::vector<uint8_t> valid;         // a state exists for pair (i, j)
  std::vector<int64_t> step_computed; // step at which pair (i, j) was last computed, -1 never
  int64_t steps = 0;                  // steps run so far
  void* events[4] = {nullptr, nullptr, nullptr, nullptr};  // optional timing hook
  bool profile = false;
  int32_t inject_fault = 0;  // one-shot test hook for the next bf16 pair kernel (0 = none)
  // Group states (one composed state per query row of partition i, over its reused pairs):
  // the reused set each partition's group state was built from (0 = none built), the step at
  // which each of those pairs had been computed then, and the buffer it was built in.
  std::vector<uint64_t> group_set;       // P
  std::vector<int64_t> group_src_step;   // P * P
  const void* group_buf = nullptr;
};

namespace ditango {
const uint8_t* plan_effective_mask(const ditango_plan_s* p, const uint8_t* mask);
// DITANGO_OK, DITANGO_ERR_INVALID_MASK or DITANGO_ERR_NO_CACHE; changes nothing.
int plan_validate(const ditango_plan_s* p, const uint8_t* mask);
// Records the pairs computed under `mask` as valid at the current step and advances the step.
void plan_commit(ditango_plan_s* p, const uint8_t* mask);
// Reused set of query partition i under `mask` (bit j = pair (i, j) reused).
uint64_t plan_reused_set(const ditango_plan_s* p, const uint8_t* mask, int32_t i);
// True when partition i's group state in `buf` was built from exactly `set` and none of those
// pairs has been recomputed since.
bool plan_group_current(const ditango_plan_s* p, const void* buf, int32_t i, uint64_t set);
// Records that partition i's group state in `buf` now holds the merge of `set` (as cached now).
void plan_group_built(ditango_plan_s* p, const void* buf, int32_t i, uint64_t set);
}  // namespace ditango
