// costmodel.cpp -- expected-latency model of one msa_attention launch
// (msa_plan_estimate) and the plan-order accessor.  Host only.
//
// AsymCache decides what to evict and how to chunk by weighing a block's
// recompute cost and hit rate against the attention kernel's expected
// latency (MSA paper abstract; AsymCache explainer, "核心方法 2" and "3").
// The model below prices each work item from its shape and replays the
// kernel's work queue over the launch's CTAs.
#include <algorithm>
#include <cstdint>
#include <queue>
#include <utility>
#include <vector>

#include "plan.h"

namespace {

using msa::kBlock;
using msa::kTileKeys;

// TMA boxes the producer issues for the tiles of one item beyond one per
// tile: a full 128-key window inside one segment is one rectangle; any other
// tile is fetched per 16-key block of each segment piece.
int64_t extra_boxes(const msa_plan_s* P, const msa::Item& it) {
    const int32_t rb = P->run_indptr[it.seq + 1];
    int32_t r = it.first_run;
    int64_t extra = 0;
    for (int32_t t0 = it.kb; t0 < it.ke; t0 += kTileKeys) {
        const int32_t t1 = std::min(t0 + kTileKeys, it.ke);
        int64_t boxes = 0;
        int32_t cur = t0;
        while (cur < t1 && r < rb) {
            const msa::Run& R = P->runs[r];
            const int32_t rend = R.log_start + R.n_tok;
            if (cur >= rend) { ++r; continue; }
            const int32_t pend = std::min(t1, rend);
            if (cur == t0 && pend - cur == kTileKeys) boxes += 1;
            else boxes += (pend - cur + kBlock - 1) / kBlock;
            cur = pend;
        }
        if (boxes > 1) extra += boxes - 1;
    }
    return extra;
}

}  // namespace

extern "C" {

int msa_plan_get_order(msa_plan_t plan, int32_t* order, int32_t* n_items) {
    if (!plan || !n_items) return MSA_ERR_INVALID_ARG;
    *n_items = (int32_t)plan->order.size();
    if (order)
        for (size_t q = 0; q < plan->order.size(); ++q) order[q] = plan->order[q];
    return MSA_OK;
}

int msa_plan_estimate(msa_plan_t plan, const msa_cost_params* c, msa_cost_estimate* e) {
    if (!plan || !c || !e) return MSA_ERR_INVALID_ARG;
    const msa_plan_s* P = plan;
    msa_cost_estimate out{};
    std::vector<double> cost(P->items.size(), 0.0);
    for (size_t i = 0; i < P->items.size(); ++i) {
        const msa::Item& it = P->items[i];
        const msa::Group& g = P->groups[it.group];
        const int64_t tiles = it.pad;
        const int64_t boxes = extra_boxes(P, it);
        const bool split = g.n_parts > 1;
        double ci;
        if (it.kind == msa::kDecode) {
            ci = c->dec_item_us + c->dec_tile_us * (double)tiles;
            out.decode_tiles += tiles;
        } else {
            ci = c->pre_item_us + c->pre_tile_us * (double)(tiles * g.pad);
            out.prefill_tile_heads += tiles * g.pad;
        }
        ci += c->box_us * (double)boxes + (split ? c->merge_us : 0.0);
        out.extra_boxes += boxes;
        out.n_split_items += split ? 1 : 0;
        cost[i] = ci;
        out.busy_us += ci;
    }
    // replay the queue: the earliest-free CTA (lowest index on ties) takes
    // the next item of the plan's order
    using Slot = std::pair<double, int32_t>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
    const int32_t grid = std::max(1, P->grid);
    for (int32_t b = 0; b < grid; ++b) free_at.push({0.0, b});
    double makespan = 0.0;
    for (int32_t idx : P->order) {
        Slot s = free_at.top();
        free_at.pop();
        s.first += cost[idx];
        if (s.first > makespan) makespan = s.first;
        free_at.push(s);
    }
    out.makespan_us = makespan;
    out.time_us = c->launch_us + makespan;
    out.n_items = (int64_t)P->items.size();
    out.decode_kv_bytes = P->info.decode_kv_bytes;
    out.prefill_flops = P->info.prefill_flops;
    *e = out;
    return MSA_OK;
}

}  // extern "C"
