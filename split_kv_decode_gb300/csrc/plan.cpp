// Host planner: how the context is cut into work items and how many CTAs
// run them. Pure host code, no CUDA calls.
//
// The split rule follows aprender issue 3725 design note §2 -- chunk =
// ceil(L / S), n_splits = ceil(L / chunk), so no split is ever empty -- with
// the split budget taken on the product (sequences x KV heads x splits), as
// "Attention at 128k" §5.1 prescribes, so that the grid fills every SM
// whatever the batch and head counts. On GB300 the split kernel is
// persistent (one CTA per SM, static round-robin over the items), so the
// planner scores each candidate by simulating that assignment and keeps the
// one with the smallest makespan; near-ties go to fewer items (fewer
// partials for the combine to read). Candidates are one chunk for the whole
// batch, or -- for ragged batches -- a chunk per sequence chosen so that all
// items have about the same length and fill a whole number of waves.
#include <algorithm>
#include <cstdint>
#include <vector>

#include "plan_internal.h"

namespace skv {

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
static int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Makespan (in positions, plus `overhead` per item) of the static round-robin
// assignment of the items (sequence b cut into chunks of chunk[b]; items in
// the kernel's order: sequence, split, KV head) over min(items, slots) CTAs.
// Item i goes to CTA i % grid. A sequence's full splits are one contiguous run
// of equal items, which adds a whole number of items to every CTA plus one
// more item to a circular range of CTAs (a difference array), so the cost is
// O(batch * hkv + grid), not O(items).
static int64_t simulate(const int32_t *lens, int batch, int hkv, const int64_t *chunk, int slots,
                        int64_t overhead, int64_t *n_items_out, std::vector<int64_t> &diff)
{
    int32_t full[DA_MAX_BATCH], rem[DA_MAX_BATCH];
    int64_t items = 0;
    for (int b = 0; b < batch; ++b) {
        full[b] = (int32_t)(lens[b] / chunk[b]);               // chunks may exceed 2^31
        rem[b] = (int32_t)(lens[b] - (int64_t)full[b] * chunk[b]);
        items += (int64_t)(full[b] + (rem[b] > 0)) * hkv;
    }
    *n_items_out = items;
    const int64_t grid = std::min<int64_t>(items, slots);
    const uint32_t g = (uint32_t)grid;
    diff.assign((size_t)grid + 1, 0);
    int64_t all = 0;
    uint32_t st = 0; // (index of the next item) mod grid
    auto run = [&](int64_t len, int64_t w) { // the next len items, each of cost w
        const uint64_t q = (uint64_t)len / g;
        const uint32_t r = (uint32_t)((uint64_t)len - q * g);
        all += (int64_t)q * w;
        if (r > 0) {
            diff[st] += w;
            if (st + r <= g) {
                diff[st + r] -= w;
            } else {
                diff[g] -= w;
                diff[0] += w;
                diff[st + r - g] -= w;
            }
            st += r;
            if (st >= g) st -= g;
        }
    };
    for (int b = 0; b < batch; ++b) {
        run((int64_t)full[b] * hkv, chunk[b] + overhead);
        if (rem[b] > 0) run(hkv, rem[b] + overhead);
    }
    int64_t best = 0, acc = 0;
    for (uint32_t c = 0; c < g; ++c) {
        acc += diff[c];
        best = std::max(best, all + acc);
    }
    return best;
}

int plan_splits(const int32_t *lens, int batch, int hkv, int tile, int slots, int force_splits,
                int max_items, PlanOut *out)
{
    if (batch < 1 || batch > DA_MAX_BATCH || hkv < 1 || tile < 1 || slots < 1) return 1;
    for (int b = 0; b < batch; ++b)
        if (lens[b] < 1) return 1;
    // per-item cost in positions: the warps' merge, the partial write and the
    // wait for the slowest warp take about as long as three tiles
    const int64_t overhead = 3 * (int64_t)tile;
    if (force_splits > 0) {
        int64_t items = 0, cost = 0;
        for (int b = 0; b < batch; ++b) {
            const int64_t chunk = round_up(ceil_div(lens[b], force_splits), tile);
            out->chunk[b] = (int32_t)chunk;
            out->n_splits[b] = (int32_t)ceil_div(lens[b], chunk);
            items += (int64_t)out->n_splits[b] * hkv;
        }
        if (items > max_items) return 2;
        std::vector<int64_t> ch((size_t)batch), diff;
        for (int b = 0; b < batch; ++b) ch[(size_t)b] = out->chunk[b];
        cost = simulate(lens, batch, hkv, ch.data(), slots, overhead, &items, diff);
        const int64_t grid = std::min<int64_t>(items, slots);
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
    // candidates:
    //  (a) one chunk for every sequence: the even share of w waves over all
    //      slots (w from 1 to 32), and powers of two times the tile;
    //  (b) a chunk per sequence: sequence b gets about L_b / target splits, so
    //      that the items are of about equal length, target = the even share
    //      of w waves; every chunk a multiple of the tile
    // candidates live in one flat array, `batch` chunks each
    std::vector<int64_t> cand;
    cand.reserve((size_t)batch * 96);
    auto uniform = [&](int64_t c) { cand.insert(cand.end(), (size_t)batch, c); };
    static const int kWaves[] = {1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15, 16, 20, 24, 28, 32};
    for (int w : kWaves) uniform(round_up(ceil_div(total, (int64_t)w * slots), tile));
    for (int64_t c = tile; c < round_up(maxlen, tile) * 2; c *= 2) uniform(c);
    uniform(round_up(maxlen, tile));
    if (batch > 1)
        for (int w : kWaves) {
            const int64_t target = std::max<int64_t>(tile, ceil_div(total, (int64_t)w * slots));
            for (int b = 0; b < batch; ++b) {
                const int64_t ns = std::max<int64_t>(1, (lens[b] + target / 2) / target);
                cand.push_back(round_up(ceil_div(lens[b], ns), tile));
            }
        }
    const size_t n_cand = cand.size() / (size_t)batch;
    std::vector<int64_t> diff, cost_of(n_cand), items_of(n_cand);
    int64_t min_cost = -1;
    for (size_t i = 0; i < n_cand; ++i) {
        cost_of[i] = simulate(lens, batch, hkv, &cand[i * (size_t)batch], slots, overhead,
                              &items_of[i], diff);
        if (items_of[i] > max_items) continue;
        if (min_cost < 0 || cost_of[i] < min_cost) min_cost = cost_of[i];
    }
    // the fewest items whose makespan is within 0.5% of the best one
    size_t best = n_cand;
    for (size_t i = 0; i < n_cand; ++i)
        if (items_of[i] <= max_items && cost_of[i] * 1000 <= min_cost * 1005 &&
            (best == n_cand || items_of[i] < items_of[best] ||
             (items_of[i] == items_of[best] && cost_of[i] < cost_of[best])))
            best = i;
    if (best == n_cand) return 2;
    for (int b = 0; b < batch; ++b) {
        const int64_t c = cand[best * (size_t)batch + (size_t)b];
        out->chunk[b] = (int32_t)c;
        out->n_splits[b] = (int32_t)ceil_div(lens[b], c);
    }
    out->n_items = (int32_t)items_of[best];
    out->grid = (int32_t)std::min<int64_t>(items_of[best], slots);
    out->est_cost = cost_of[best];
    return 0;
}

} // namespace skv
