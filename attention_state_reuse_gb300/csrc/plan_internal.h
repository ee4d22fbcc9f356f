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
};

namespace ditango {
const uint8_t* plan_effective_mask(const ditango_plan_s* p, const uint8_t* mask);
// DITANGO_OK, DITANGO_ERR_INVALID_MASK or DITANGO_ERR_NO_CACHE; changes nothing.
int plan_validate(const ditango_plan_s* p, const uint8_t* mask);
// Records the pairs computed under `mask` as valid at the current step and advances the step.
void plan_commit(ditango_plan_s* p, const uint8_t* mask);
}  // namespace ditango
