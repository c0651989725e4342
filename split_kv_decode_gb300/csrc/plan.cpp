// Host planner: how the context is cut into work items and how many CTAs
// run them. Pure host code, no CUDA calls.
//
// The split rule follows aprender issue 3725 design note §2 -- chunk =
// ceil(L / S), n_splits = ceil(L / chunk), so no split is ever empty -- with
// the split budget taken on the product (sequences x KV heads x splits), as
// "Attention at 128k" §5.1 prescribes, so that the grid fills every SM
// whatever the batch and head counts. On GB300 the split kernel is
// persistent (one CTA per SM, static round-robin over the items), so the
// planner scores each candidate chunk by simulating that assignment and
// keeps the one with the smallest makespan; ties go to the larger chunk
// (fewer partials for the combine to read).
#include <algorithm>
#include <cstdint>
#include <vector>

#include "plan_internal.h"

namespace skv {

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
static int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Makespan (in positions, plus `overhead` per item) of the static round-robin
// assignment of the items of `chunk` over min(items, slots) CTAs.
static int64_t simulate(const int32_t *lens, int batch, int hkv, int64_t chunk, int slots,
                        int64_t overhead, int64_t *n_items_out)
{
    int64_t items = 0;
    for (int b = 0; b < batch; ++b) items += ceil_div(lens[b], chunk) * hkv;
    *n_items_out = items;
    const int64_t grid = std::min<int64_t>(items, slots);
    std::vector<int64_t> cost((size_t)grid, 0);
    int64_t item = 0;
    for (int b = 0; b < batch; ++b) {
        const int64_t ns = ceil_div(lens[b], chunk);
        for (int64_t s = 0; s < ns; ++s) {
            const int64_t len = std::min<int64_t>(chunk, lens[b] - s * chunk);
            for (int h = 0; h < hkv; ++h, ++item) cost[(size_t)(item % grid)] += len + overhead;
        }
    }
    return *std::max_element(cost.begin(), cost.end());
}

int plan_splits(const int32_t *lens, int batch, int hkv, int tile, int slots, int force_splits,
                int max_items, PlanOut *out)
{
    if (batch < 1 || batch > DA_MAX_BATCH || hkv < 1 || tile < 1 || slots < 1) return 1;
    for (int b = 0; b < batch; ++b)
        if (lens[b] < 1) return 1;
    const int64_t overhead = tile; // per-item merge and partial write, in positions
    if (force_splits > 0) {
        int64_t items = 0, cost = 0;
        for (int b = 0; b < batch; ++b) {
            const int64_t chunk = round_up(ceil_div(lens[b], force_splits), tile);
            out->chunk[b] = (int32_t)chunk;
            out->n_splits[b] = (int32_t)ceil_div(lens[b], chunk);
            items += (int64_t)out->n_splits[b] * hkv;
        }
        if (items > max_items) return 2;
        // cost of the round-robin assignment with per-sequence chunks
        const int64_t grid = std::min<int64_t>(items, slots);
        std::vector<int64_t> c((size_t)grid, 0);
        int64_t item = 0;
        for (int b = 0; b < batch; ++b)
            for (int s = 0; s < out->n_splits[b]; ++s) {
                const int64_t len =
                    std::min<int64_t>(out->chunk[b], lens[b] - (int64_t)s * out->chunk[b]);
                for (int h = 0; h < hkv; ++h, ++item) c[(size_t)(item % grid)] += len + overhead;
            }
        cost = *std::max_element(c.begin(), c.end());
        out->n_items = (int32_t)items;
        out->grid = (int32_t)grid;
        out->est_cost = cost;
        return 0;
    }
    int64_t total = 0, maxlen = 0;
    for (int b = 0; b < batch; ++b) {
        total += (int64_t)lens[b] * hkv;
        maxlen = std::max<int64_t>(maxlen, lens[b]);
    }
    // candidate chunks: the even share of 1..32 waves over all slots, and powers
    // of two times the tile; every candidate a multiple of the tile
    std::vector<int64_t> cand;
    for (int w = 1; w <= 32; ++w) cand.push_back(round_up(ceil_div(total, (int64_t)w * slots), tile));
    for (int64_t c = tile; c < round_up(maxlen, tile) * 2; c *= 2) cand.push_back(c);
    cand.push_back(round_up(maxlen, tile));
    std::sort(cand.begin(), cand.end());
    cand.erase(std::unique(cand.begin(), cand.end()), cand.end());
    struct Cand { int64_t chunk, cost, items; };
    std::vector<Cand> ok;
    int64_t min_cost = -1;
    for (int64_t c : cand) {
        int64_t items = 0;
        const int64_t cost = simulate(lens, batch, hkv, c, slots, overhead, &items);
        if (items > max_items) continue;
        ok.push_back({c, cost, items});
        if (min_cost < 0 || cost < min_cost) min_cost = cost;
    }
    // the largest chunk whose makespan is within 0.5% of the best one
    int64_t best_chunk = -1, best_cost = 0, best_items = 0;
    for (const Cand &x : ok)
        if (x.cost * 1000 <= min_cost * 1005 && x.chunk > best_chunk) {
            best_chunk = x.chunk;
            best_cost = x.cost;
            best_items = x.items;
        }
    if (best_chunk < 0) return 2;
    for (int b = 0; b < batch; ++b) {
        out->chunk[b] = (int32_t)best_chunk;
        out->n_splits[b] = (int32_t)ceil_div(lens[b], best_chunk);
    }
    out->n_items = (int32_t)best_items;
    out->grid = (int32_t)std::min<int64_t>(best_items, slots);
    out->est_cost = best_cost;
    return 0;
}

} // namespace skv
