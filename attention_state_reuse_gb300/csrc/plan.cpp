// Host planner: contiguous partitions, reuse-mask validation, cache bookkeeping, and the work
// decomposition (schedule) handed to the pair kernels.
//
// Source: DiTango (gist.science/paper/2607.15650), Problem Statement (the sequence is split
// into context partitions) and Methodology 1, Anchor-Guided Selection Planner (per step each
// partition pair computes fresh or reuses an earlier state; local states are always computed,
// so the diagonal of a reuse mask must be 0; a pair can only be reused once a state for it
// exists, so the first step computes every pair).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <numeric>
#include <vector>

#include "ditango_internal.h"
#include "plan_internal.h"

using ditango::kMaxP;

namespace {

int check_values(int32_t P, const uint8_t* mask) {
  if (mask == nullptr) return DITANGO_OK;
  for (int32_t i = 0; i < P; ++i) {
    for (int32_t j = 0; j < P; ++j) {
      const uint8_t m = mask[i * P + j];
      if (m > 1) return DITANGO_ERR_INVALID_MASK;
      if (i == j && m != 0) return DITANGO_ERR_INVALID_MASK;
    }
  }
  return DITANGO_OK;
}

}  // namespace

namespace ditango {

// Device slots of a cache that keeps S of the P states of a row on the device: for query
// partition i, the S pairs nearest the diagonal (smallest |i - j|, ties to the smaller j) take
// slots 0..S-1 in ascending j; the others are kept in host memory (-1). These are the pairs a
// distance mask computes, and the local pair (i, i) is always on the device.
void cache_slot_map(int32_t P, int32_t S, int8_t* map) {
  for (int32_t i = 0; i < P; ++i) {
    std::vector<int32_t> js(P);
    std::iota(js.begin(), js.end(), 0);
    std::stable_sort(js.begin(), js.end(), [i](int32_t a, int32_t b) {
      return std::abs(a - i) < std::abs(b - i);  // stable: ties keep the smaller j first
    });
    std::vector<uint8_t> on_dev(P, 0);
    for (int32_t k = 0; k < S; ++k) on_dev[js[k]] = 1;
    int8_t next = 0;
    for (int32_t j = 0; j < P; ++j) map[i * P + j] = on_dev[j] ? next++ : int8_t{-1};
  }
}

const uint8_t* plan_effective_mask(const ditango_plan_s* p, const uint8_t* mask) {
  return mask != nullptr ? mask : p->mask.data();
}

int plan_validate(const ditango_plan_s* p, const uint8_t* mask) {
  const uint8_t* m = plan_effective_mask(p, mask);
  const int st = check_values(p->P, m);
  if (st != DITANGO_OK) return st;
  for (size_t x = 0; x < p->valid.size(); ++x)
    if (m[x] == 1 && !p->valid[x]) return DITANGO_ERR_NO_CACHE;
  return DITANGO_OK;
}

uint64_t plan_reused_set(const ditango_plan_s* p, const uint8_t* mask, int32_t i) {
  const uint8_t* m = plan_effective_mask(p, mask);
  uint64_t set = 0;
  for (int32_t j = 0; j < p->P; ++j)
    if (m[i * p->P + j] == 1) set |= uint64_t{1} << j;
  return set;
}

bool plan_group_current(const ditango_plan_s* p, const void* buf, int32_t i, uint64_t set) {
  if (set == 0 || buf != p->group_buf || p->group_set[i] != set) return false;
  for (int32_t j = 0; j < p->P; ++j) {
    const size_t x = static_cast<size_t>(i) * p->P + j;
    if (((set >> j) & 1u) && p->group_src_step[x] != p->step_computed[x]) return false;
  }
  return true;
}

void plan_group_built(ditango_plan_s* p, const void* buf, int32_t i, uint64_t set) {
  if (buf != p->group_buf) {  // a new buffer holds none of the old groups
    std::fill(p->group_set.begin(), p->group_set.end(), 0);
    p->group_buf = buf;
  }
  p->group_set[i] = set;
  for (int32_t j = 0; j < p->P; ++j) {
    const size_t x = static_cast<size_t>(i) * p->P + j;
    p->group_src_step[x] = p->step_computed[x];
  }
}

void plan_commit(ditango_plan_s* p, const uint8_t* mask) {
  const uint8_t* m = plan_effective_mask(p, mask);
  for (size_t x = 0; x < p->valid.size(); ++x) {
    if (m[x] == 0) {
      p->valid[x] = 1;
      p->step_computed[x] = p->steps;
    }
  }
  ++p->steps;
}

void build_schedule(int64_t N, int32_t P, const int64_t* offsets, const uint8_t* mask, int64_t B,
                    int64_t H, int32_t block_rows, PairSchedule* s) {
  (void)N;
  std::memset(s, 0, sizeof(*s));
  s->P = P;
  s->BH = static_cast<int32_t>(B * H);
  s->H = static_cast<int32_t>(H);
  s->block_rows = block_rows;
  std::vector<int64_t> cost(P, 0);
  for (int32_t i = 0; i <= P; ++i) s->offsets[i] = static_cast<int32_t>(offsets[i]);
  for (int32_t i = 0; i < P; ++i) {
    uint64_t bits = 0;
    for (int32_t j = 0; j < P; ++j) {
      if (mask[i * P + j] == 0) {
        bits |= uint64_t{1} << j;
        cost[i] += offsets[j + 1] - offsets[j];
      }
    }
    s->compute_mask[i] = bits;
  }
  std::vector<int32_t> order(P);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return cost[a] > cost[b]; });
  int64_t acc = 0;
  for (int32_t k = 0; k < P; ++k) {
    const int32_t i = order[k];
    s->order[k] = i;
    s->seg_start[k] = static_cast<int32_t>(acc);
    const int64_t n_i = offsets[i + 1] - offsets[i];
    acc += ((n_i + block_rows - 1) / block_rows) * B * H;
  }
  s->seg_start[P] = static_cast<int32_t>(acc);
  s->n_units = static_cast<int32_t>(acc);
}

}  // namespace ditango

extern "C" {

int ditango_plan(int64_t N, int32_t P, const uint8_t* mask, ditango_plan_t* out_plan) {
  if (out_plan == nullptr || P < 1 || P > kMaxP || N < P || N > (int64_t{1} << 30))
    return DITANGO_ERR_INVALID_ARG;
  const int st = check_values(P, mask);
  if (st != DITANGO_OK) return st;
  auto* p = new (std::nothrow) ditango_plan_s;
  if (p == nullptr) return DITANGO_ERR_INVALID_ARG;
  p->N = N;
  p->P = P;
  p->offsets.resize(P + 1);
  const int64_t base = N / P, extra = N % P;
  p->offsets[0] = 0;
  for (int32_t i = 0; i < P; ++i) p->offsets[i + 1] = p->offsets[i] + base + (i < extra ? 1 : 0);
  p->mask.assign(static_cast<size_t>(P) * P, 0);
  if (mask != nullptr) std::memcpy(p->mask.data(), mask, p->mask.size());
  p->valid.assign(static_cast<size_t>(P) * P, 0);
  p->step_computed.assign(static_cast<size_t>(P) * P, -1);
  p->steps = 0;
  p->group_set.assign(P, 0);
  p->group_src_step.assign(static_cast<size_t>(P) * P, -1);
  *out_plan = p;
  return DITANGO_OK;
}

void ditango_plan_destroy(ditango_plan_t plan) { delete plan; }

int ditango_plan_set_mask(ditango_plan_t plan, const uint8_t* mask) {
  if (plan == nullptr || mask == nullptr) return DITANGO_ERR_INVALID_ARG;
  const int st = check_values(plan->P, mask);
  if (st != DITANGO_OK) return st;
  std::memcpy(plan->mask.data(), mask, plan->mask.size());
  return DITANGO_OK;
}

int ditango_plan_check_mask(ditango_plan_t plan, const uint8_t* mask) {
  if (plan == nullptr) return DITANGO_ERR_INVALID_ARG;
  return ditango::plan_validate(plan, mask);
}

int ditango_plan_get_offsets(ditango_plan_t plan, int64_t* offsets) {
  if (plan == nullptr || offsets == nullptr) return DITANGO_ERR_INVALID_ARG;
  std::copy(plan->offsets.begin(), plan->offsets.end(), offsets);
  return DITANGO_OK;
}

int ditango_plan_get_pairs(ditango_plan_t plan, const uint8_t* mask, int32_t* pairs,
                           int32_t* count) {
  if (plan == nullptr || pairs == nullptr || count == nullptr) return DITANGO_ERR_INVALID_ARG;
  const int st = check_values(plan->P, mask);
  if (st != DITANGO_OK) return st;
  const uint8_t* m = ditango::plan_effective_mask(plan, mask);
  int32_t n = 0;
  for (int32_t i = 0; i < plan->P; ++i)
    for (int32_t j = 0; j < plan->P; ++j)
      if (m[i * plan->P + j] == 0) {
        pairs[2 * n] = i;
        pairs[2 * n + 1] = j;
        ++n;
      }
  *count = n;
  return DITANGO_OK;
}

int ditango_planner_select(ditango_plan_t plan, const double* w, const double* delta, double tau,
                           int32_t group, int32_t budget, uint8_t* mask) {
  if (plan == nullptr || w == nullptr || delta == nullptr || mask == nullptr || group < 1 ||
      !(tau >= 0.0))
    return DITANGO_ERR_INVALID_ARG;
  const int32_t P = plan->P;
  for (int32_t x = 0; x < P * P; ++x)
    if (!std::isfinite(w[x])) return DITANGO_ERR_INVALID_ARG;
  for (int32_t i = 0; i < P; ++i)
    if (!std::isfinite(delta[i])) return DITANGO_ERR_INVALID_ARG;
  struct Cand {
    double err;
    int32_t i, k;
  };
  std::vector<Cand> forced, ranked;
  for (int32_t i = 0; i < P; ++i) {
    for (int32_t k = 0; k * group < P; ++k) {
      const int32_t j0 = k * group, j1 = std::min(P, j0 + group);
      double err = 0.0;
      bool any = false, never = false;
      for (int32_t j = j0; j < j1; ++j) {  // ascending j: the summation order is part of the rule
        if (j == i) continue;
        any = true;
        const double e = w[i * P + j] * delta[i];
        err = err + e;
        if (!plan->valid[static_cast<size_t>(i) * P + j]) never = true;
      }
      if (!any) continue;
      (never ? forced : ranked).push_back({err, i, k});
    }
  }
  std::memset(mask, 1, static_cast<size_t>(P) * P);
  for (int32_t i = 0; i < P; ++i) mask[i * P + i] = 0;
  int64_t computed = P;
  auto take = [&](const Cand& c) {
    const int32_t j0 = c.k * group, j1 = std::min(P, j0 + group);
    for (int32_t j = j0; j < j1; ++j)
      if (j != c.i) {
        mask[c.i * P + j] = 0;
        ++computed;
      }
  };
  auto size_of = [&](const Cand& c) {
    const int32_t j0 = c.k * group, j1 = std::min(P, j0 + group);
    return (j1 - j0) - ((c.i >= j0 && c.i < j1) ? 1 : 0);
  };
  for (const Cand& c : forced) take(c);
  std::stable_sort(ranked.begin(), ranked.end(), [](const Cand& a, const Cand& b) {
    if (a.err != b.err) return a.err > b.err;
    if (a.i != b.i) return a.i < b.i;
    return a.k < b.k;
  });
  for (const Cand& c : ranked) {
    if (!(c.err > tau)) continue;
    if (budget >= 0 && computed + size_of(c) > budget) continue;
    take(c);
  }
  return DITANGO_OK;
}

int ditango_plan_inject_fault(ditango_plan_t plan, int32_t kind) {
  if (plan == nullptr || kind < 0 || kind > 1) return DITANGO_ERR_INVALID_ARG;
  plan->inject_fault = kind;
  return DITANGO_OK;
}

int ditango_plan_set_profile_events(ditango_plan_t plan, void* const* events) {
  if (plan == nullptr) return DITANGO_ERR_INVALID_ARG;
  if (events == nullptr) {
    plan->profile = false;
    for (auto& e : plan->events) e = nullptr;
    return DITANGO_OK;
  }
  for (int x = 0; x < 4; ++x)
    if (events[x] == nullptr) return DITANGO_ERR_INVALID_ARG;
  for (int x = 0; x < 4; ++x) plan->events[x] = events[x];
  plan->profile = true;
  return DITANGO_OK;
}

int ditango_plan_get_cache_state(ditango_plan_t plan, uint8_t* valid, int64_t* step_computed,
                                 int64_t* steps_run) {
  if (plan == nullptr) return DITANGO_ERR_INVALID_ARG;
  if (valid != nullptr) std::copy(plan->valid.begin(), plan->valid.end(), valid);
  if (step_computed != nullptr)
    std::copy(plan->step_computed.begin(), plan->step_computed.end(), step_computed);
  if (steps_run != nullptr) *steps_run = plan->steps;
  return DITANGO_OK;
}

int ditango_plan_set_cache_state(ditango_plan_t plan, const uint8_t* valid,
                                 const int64_t* step_computed, int64_t steps_run) {
  if (plan == nullptr || valid == nullptr || step_computed == nullptr || steps_run < 0)
    return DITANGO_ERR_INVALID_ARG;
  const int32_t P = plan->P;
  for (int32_t x = 0; x < P * P; ++x) {
    if (valid[x] > 1) return DITANGO_ERR_INVALID_ARG;
    if (valid[x] == 0 && step_computed[x] != -1) return DITANGO_ERR_INVALID_ARG;
    if (valid[x] == 1 && (step_computed[x] < 0 || step_computed[x] >= steps_run))
      return DITANGO_ERR_INVALID_ARG;
    if (steps_run > 0 && x / P == x % P && valid[x] == 0) return DITANGO_ERR_INVALID_ARG;
  }
  std::copy(valid, valid + static_cast<size_t>(P) * P, plan->valid.begin());
  std::copy(step_computed, step_computed + static_cast<size_t>(P) * P, plan->step_computed.begin());
  plan->steps = steps_run;
  std::fill(plan->group_set.begin(), plan->group_set.end(), 0);
  return DITANGO_OK;
}

}  // extern "C"

extern "C" int ditango_cache_slot_map(int32_t P, int32_t S, int8_t* map) {
  if (map == nullptr || P < 1 || P > kMaxP || S < 1 || S > P) return DITANGO_ERR_INVALID_ARG;
  ditango::cache_slot_map(P, S, map);
  return DITANGO_OK;
}
