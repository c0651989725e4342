// Planner entry used by the C ABI (pure host code).
#pragma once
#include <cstdint>

#include "split_kv_decode.h"

namespace skv {

struct PlanOut {
    int32_t chunk[DA_MAX_BATCH];
    int32_t n_splits[DA_MAX_BATCH];
    int32_t n_items;
    int32_t grid;
    int64_t est_cost;
};

// Returns 0 on success, 1 for invalid input, 2 if no split fits max_items.
int plan_splits(const int32_t *lens, int batch, int hkv, int tile, int slots, int force_splits,
                int max_items, PlanOut *out);

} // namespace skv
