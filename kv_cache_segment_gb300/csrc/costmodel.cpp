// costmodel.cpp -- expected-latency model of one msa_attention launch
// (msa_plan_estimate) and the plan-order accessor.  Host only.
//
// AsymCache decides what to evict and how to chunk by weighing a block's
// recompute cost and hit rate against the attention kernel's expected
// latency (MSA paper abstract; AsymCache explainer, "核心方法 2" and "3").
// The model below prices each work item from its shape and replays the
// kernel's work queue over the launch's CTAs, with the decode streams
// sharing HBM bandwidth.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <utility>
#include <vector>

#include "plan.h"

namespace {

using msa::kBlock;
using msa::kTileKeys;

// TMA boxes the producer issues for the tile [t0, t1) of sequence `seq`
// beyond one: a full 128-key window inside one segment is one rectangle; any
// other tile is fetched piece by piece (one piece per segment it touches),
// each piece's whole 16-key blocks in boxes of 4, 2 and 1 blocks.
int64_t tile_extra_boxes(const msa_plan_s* P, int32_t seq, int32_t t0, int32_t t1) {
    const int32_t ra = P->run_indptr[seq], rb = P->run_indptr[seq + 1];
    // first run that ends after t0 (runs are in logical order)
    int32_t lo = ra, hi = rb;
    while (lo < hi) {
        const int32_t mid = (lo + hi) / 2;
        if (P->runs[mid].log_start + P->runs[mid].n_tok <= t0) lo = mid + 1;
        else hi = mid;
    }
    int64_t boxes = 0;
    int32_t cur = t0;
    for (int32_t r = lo; r < rb && cur < t1; ++r) {
        const msa::Run& R = P->runs[r];
        const int32_t pend = std::min(t1, R.log_start + R.n_tok);
        if (pend <= cur) continue;
        if (cur == t0 && pend - cur == kTileKeys) {
            boxes += 1;
        } else {
            const int64_t nb = (pend - cur + kBlock - 1) / kBlock;
            boxes += nb / 4 + (nb % 4) / 2 + nb % 2;
        }
        cur = pend;
    }
    return boxes > 1 ? boxes - 1 : 0;
}

// Per sequence, prefix sums of the extra boxes of its full 128-key tiles:
// items start on tile boundaries, so an item's count is a difference of two
// prefix sums plus, when its end is not on a boundary, its partial last tile.
// One pass per sequence walks its tiles and runs together (both in logical
// order); the sums of all sequences share one array.
struct BoxCounts {
    std::vector<int64_t> prefix;  // prefix[base[s] + i] = sum over full tiles j < i of sequence s
    std::vector<size_t> base;
    explicit BoxCounts(const msa_plan_s* P) : base(P->seq_lens.size() + 1, 0) {
        const size_t S = P->seq_lens.size();
        for (size_t s = 0; s < S; ++s) base[s + 1] = base[s] + (size_t)(P->seq_lens[s] / kTileKeys) + 1;
        prefix.assign(base[S], 0);
        for (size_t s = 0; s < S; ++s) {
            const int32_t full = P->seq_lens[s] / kTileKeys;
            const int32_t rb = P->run_indptr[s + 1];
            int32_t r = P->run_indptr[s];  // first run that ends after the current tile's start
            int64_t* pf = prefix.data() + base[s];
            for (int32_t i = 0; i < full; ++i) {
                const int32_t t0 = i * kTileKeys, t1 = t0 + kTileKeys;
                while (r < rb && P->runs[r].log_start + P->runs[r].n_tok <= t0) ++r;
                int64_t boxes = 0;
                int32_t cur = t0;
                for (int32_t q = r; q < rb && cur < t1; ++q) {
                    const msa::Run& R = P->runs[q];
                    const int32_t pend = std::min(t1, R.log_start + R.n_tok);
                    if (pend <= cur) continue;
                    if (cur == t0 && pend - cur == kTileKeys) {
                        boxes += 1;
                    } else {
                        const int64_t nb = (pend - cur + kBlock - 1) / kBlock;
                        boxes += nb / 4 + (nb % 4) / 2 + nb % 2;
                    }
                    cur = pend;
                }
                pf[i + 1] = pf[i] + (boxes > 1 ? boxes - 1 : 0);
            }
        }
    }
    int64_t item(const msa_plan_s* P, const msa::Item& it) const {
        if (it.ke <= it.kb) return 0;
        const int64_t* pf = prefix.data() + base[it.seq];
        const size_t last = base[it.seq + 1] - base[it.seq] - 1;
        const int32_t i0 = it.kb / kTileKeys, i1 = it.ke / kTileKeys;  // full tiles [i0, i1)
        int64_t n = pf[std::min<size_t>(i1, last)] - pf[std::min<size_t>(i0, last)];
        if (it.ke % kTileKeys) n += tile_extra_boxes(P, it.seq, i1 * kTileKeys, it.ke);
        return n;
    }
};

// Binary min-heap of (key, CTA) pairs in lexicographic order (the CTA index
// breaks ties, so the order in which entries leave it is fixed), with room
// for every CTA reserved up front and a replace-top for "pop, then push".
// Keys are finite and non-negative (times and byte counts that start at +0
// and only grow), so the IEEE bit pattern of a key, as an unsigned integer,
// orders like its value: an entry is stored as one 128-bit integer, key bits
// above the CTA index, and compared in one step.
class MinHeap {
public:
    using Ev = std::pair<double, int32_t>;
    explicit MinHeap(size_t cap) { h_.reserve(cap); }
    bool empty() const { return h_.empty(); }
    size_t size() const { return h_.size(); }
    Ev top() const { return decode(h_[0]); }
    void push(Ev v) {
        const K key = encode(v);
        size_t i = h_.size();
        h_.push_back(key);
        while (i > 0) {
            const size_t p = (i - 1) / 2;
            if (!(key < h_[p])) break;
            h_[i] = h_[p];
            i = p;
        }
        h_[i] = key;
    }
    void pop() {
        const K last = h_.back();
        h_.pop_back();
        if (!h_.empty()) sift_down(last);
    }
    void replace_top(Ev v) { sift_down(encode(v)); }

private:
    using K = unsigned __int128;
    static K encode(Ev v) {
        uint64_t bits;
        std::memcpy(&bits, &v.first, sizeof bits);
        return ((K)bits << 32) | (uint32_t)v.second;
    }
    static Ev decode(K k) {
        const uint64_t bits = (uint64_t)(k >> 32);
        double d;
        std::memcpy(&d, &bits, sizeof d);
        return {d, (int32_t)(uint32_t)k};
    }
    // place v at the root and move it down to where it belongs
    void sift_down(K v) {
        const size_t n = h_.size();
        size_t i = 0;
        for (;;) {
            size_t c = 2 * i + 1;
            if (c >= n) break;
            c += (size_t)((c + 1 < n) & (h_[c + 1] < h_[c]));
            if (!(h_[c] < v)) break;
            h_[i] = h_[c];
            i = c;
        }
        h_[i] = v;
    }
    std::vector<K> h_;
};

bool params_ok(const msa_cost_params* c) {
    const double prm[10] = {c->launch_us, c->dec_item_us, c->dec_gbs,     c->dec_cta_gbs,  c->pre_item_us,
                            c->pre_tile_us, c->box_us, c->dec_merge_us, c->pre_merge_us, c->pre_tile_dfrac};
    for (double v : prm)
        if (!(v >= 0.0) || !std::isfinite(v)) return false;
    return c->pre_tile_dfrac <= 1.0;
}

// Time of one (128-key tile x 128-row query tile) at head dim D: the share
// pre_tile_dfrac of the D = 128 time scales with D, the rest does not.
double tile_us(const msa_cost_params* c, int32_t head_dim) {
    return c->pre_tile_us * (1.0 - c->pre_tile_dfrac + c->pre_tile_dfrac * (double)head_dim / 128.0);
}

int estimate(const msa_plan_s* P, const msa_cost_params* c, const BoxCounts& box_counts, msa_cost_estimate* e) {
    const size_t n = P->items.size();
    msa_cost_estimate out{};
    std::vector<double> fixed(n, 0.0), bytes(n, 0.0);
    const double tile_bytes = 2.0 * kTileKeys * P->dims.head_dim * 2.0;  // K and V, bf16
    const double t_tile = tile_us(c, P->dims.head_dim);
    for (size_t i = 0; i < n; ++i) {
        const msa::Item& it = P->items[i];
        const msa::Group& g = P->groups[it.group];
        const int64_t tiles = it.pad;
        const int64_t boxes = box_counts.item(P, it);
        const bool split = g.n_parts > 1;
        double f;
        if (it.kind == msa::kDecode) {
            f = c->dec_item_us;
            bytes[i] = tile_bytes * (double)tiles;
            out.decode_tiles += tiles;
            out.stream_bytes += (int64_t)bytes[i];
        } else {
            f = c->pre_item_us + t_tile * (double)(tiles * g.pad);
            out.prefill_tile_heads += tiles * g.pad;
        }
        f += c->box_us * (double)boxes +
             (split ? (it.kind == msa::kDecode ? c->dec_merge_us : c->pre_merge_us) : 0.0);
        fixed[i] = f;
        out.extra_boxes += boxes;
        out.n_split_items += split ? 1 : 0;
        out.fixed_us += f;
    }
    if (out.stream_bytes > 0 && (c->dec_gbs <= 0.0 || c->dec_cta_gbs <= 0.0)) return MSA_ERR_INVALID_ARG;

    // Event-by-event replay.  A CTA's item is a fixed phase (time) then a
    // stream phase (bytes); a CTA that finishes takes the next item of the
    // order at once.  All streaming CTAs advance at the same rate, so their
    // progress is one clock `sigma` (bytes per streaming CTA so far) and a
    // CTA's stream ends when sigma reaches its target: two min-heaps, one in
    // time (fixed phases) and one in sigma (streams).  Which of several CTAs
    // freed at the same instant takes which item does not change the finish
    // times, the CTAs being alike.
    const int32_t grid = std::max(1, P->grid);
    MinHeap fixed_q((size_t)grid), stream_q((size_t)grid);
    std::vector<int32_t> item(grid, -1);
    size_t next = 0;
    double t = 0.0, sigma = 0.0;
    auto rate_of = [&](size_t n_stream) {
        return n_stream > 0 ? std::min(c->dec_cta_gbs, c->dec_gbs / (double)n_stream) * 1e3 : 0.0;  // B/us
    };
    // start the next item on CTA b at time t (its fixed phase)
    auto take = [&](int32_t b) {
        if (next >= P->order.size()) { item[b] = -1; return; }
        item[b] = P->order[next++];
        fixed_q.push({t + fixed[item[b]], b});
    };
    for (int32_t b = 0; b < grid; ++b) take(b);
    while (!fixed_q.empty() || !stream_q.empty()) {
        const double r = rate_of(stream_q.size());
        const double t_fixed = fixed_q.empty() ? INFINITY : fixed_q.top().first;
        const double t_stream = stream_q.empty() ? INFINITY : t + (stream_q.top().first - sigma) / r;
        if (t_fixed <= t_stream) {
            const int32_t b = fixed_q.top().second;
            if (r > 0.0) sigma += (t_fixed - t) * r;
            t = t_fixed;
            if (bytes[item[b]] > 0.0) {
                fixed_q.pop();
                stream_q.push({sigma + bytes[item[b]], b});
            } else if (next < P->order.size()) {  // the CTA's next item, in place of this one
                item[b] = P->order[next++];
                fixed_q.replace_top({t + fixed[item[b]], b});
            } else {
                item[b] = -1;
                fixed_q.pop();
            }
        } else {
            const int32_t b = stream_q.top().second;
            sigma = stream_q.top().first;
            stream_q.pop();
            t = t_stream;
            take(b);
        }
    }
    out.makespan_us = t;
    out.time_us = c->launch_us + t;
    out.n_items = (int64_t)n;
    out.decode_kv_bytes = P->info.decode_kv_bytes;
    out.prefill_flops = P->info.prefill_flops;
    *e = out;
    return MSA_OK;
}

}  // namespace

namespace msa {

// Adaptive chunking (AsymCache explainer, "核心方法 3": chunk sizes adjusted
// so the attention kernel stays busy without per-chunk overheads dominating):
// the decode split, then the prefill split, with the lowest expected launch
// time under the latency model.
void choose_split(msa_plan_s* P, const std::vector<Pending>& pend, const msa_cost_params& c, double* dec_split,
                  double* pre_split) {
    bool has[2] = {false, false};
    for (auto& pd : pend) has[pd.g.kind] = true;
    const BoxCounts box_counts(P);
    auto time_of = [&](double d, double p) {
        split_items(P, pend, d, p);
        msa_cost_estimate e{};
        return estimate(P, &c, box_counts, &e) == MSA_OK ? e.time_us : INFINITY;
    };
    static const double kDec[] = {1.0, 1.5, 2.0, 3.0, 4.0};
    static const double kPre[] = {1.0, 2.0, 4.0};
    double best = INFINITY;
    if (has[kDecode]) {
        const double p = *pre_split;
        for (double d : kDec) {
            const double t = time_of(d, p);
            if (t < best) { best = t; *dec_split = d; }
        }
    }
    if (has[kPrefill]) {
        const double d = *dec_split;
        for (double p : kPre) {
            const double t = time_of(d, p);
            if (t < best) { best = t; *pre_split = p; }
        }
    }
}

}  // namespace msa

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
    if (!params_ok(c)) return MSA_ERR_INVALID_ARG;
    try {
        const BoxCounts box_counts(plan);
        return estimate(plan, c, box_counts, e);
    } catch (...) {  // allocation failure: no exception leaves the C ABI
        return MSA_ERR_INVALID_ARG;
    }
}

// Adaptive prefill chunk size: the candidate chunk sizes in ascending order
// (multiples of the granularity up to the largest pending remainder, capped
// at max_chunk, thinned to at most 63 multiples, plus the cap itself), a
// plan and a latency-model prediction of the step for each, and the lowest
// predicted time per prefill token within the budget.
static int choose_prefill_chunk(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks_per_seq,
                                const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_range_indptr,
                                const int32_t* q_ranges, const msa_pending_prefill* pending, int32_t n_pending,
                                const msa_plan_options* opts, const msa_cost_params* params, double budget_us,
                                int32_t granularity, int32_t max_chunk, msa_chunk_choice* choice,
                                int32_t* cand_chunk, double* cand_time_us) {
    if (!dims || !seq_lens || !q_range_indptr || !pending || !params || !choice) return MSA_ERR_INVALID_ARG;
    if (num_seqs <= 0 || n_pending <= 0 || n_pending > num_seqs || granularity < 0 || max_chunk < 0 ||
        !std::isfinite(budget_us) || !params_ok(params))
        return MSA_ERR_INVALID_ARG;
    const int32_t g = granularity > 0 ? granularity : msa::kTileRows;
    std::vector<int32_t> remain(num_seqs, -1), start(num_seqs, 0);
    int32_t cmax = 0;
    for (int32_t i = 0; i < n_pending; ++i) {
        const msa_pending_prefill& pp = pending[i];
        if (pp.seq < 0 || pp.seq >= num_seqs || remain[pp.seq] >= 0) return MSA_ERR_INVALID_ARG;
        if (pp.start < 0 || pp.end <= pp.start) return MSA_ERR_BAD_Q_RANGE;
        // a pending sequence's rows come from the chunk only
        if (q_range_indptr[pp.seq + 1] != q_range_indptr[pp.seq]) return MSA_ERR_INVALID_ARG;
        remain[pp.seq] = pp.end - pp.start;
        start[pp.seq] = pp.start;
        cmax = std::max(cmax, pp.end - pp.start);
    }
    if (max_chunk > 0) cmax = std::min(cmax, max_chunk);
    std::vector<int32_t> cands;
    const int32_t n_mult = cmax / g;
    const int32_t step = std::max(1, (n_mult + 62) / 63);
    for (int32_t k = 1; k <= n_mult; k += step) cands.push_back(k * g);
    if (cands.empty() || cands.back() != cmax) cands.push_back(cmax);

    // The SM count is resolved here: a worker thread would see the CUDA
    // runtime's default device rather than the caller's current one.
    msa_plan_options o = opts ? *opts : msa_plan_options{0, 0.0, 0.0, nullptr};
    if (o.num_sms == 0) {
        o.num_sms = msa::device_sm_count();
        if (o.num_sms <= 0) return MSA_ERR_CUDA;
    }
    const size_t n_cand = cands.size();
    std::vector<double> time_us(n_cand, 0.0);
    std::vector<int64_t> tokens(n_cand, 0);
    std::vector<int> status(n_cand, MSA_OK);
    // Candidate ci: the step's batch with min(c, remainder) rows of every
    // pending prefill, planned and priced.  Candidates are independent.
    auto evaluate = [&](size_t ci) {
      try {
        const int32_t c = cands[ci];
        std::vector<int32_t> lens(num_seqs), indptr(num_seqs + 1), ranges;
        ranges.reserve(2 * ((size_t)q_range_indptr[num_seqs] + n_pending));
        int64_t tok = 0;
        indptr[0] = 0;
        for (int32_t s = 0; s < num_seqs; ++s) {
            if (remain[s] >= 0) {
                const int32_t n = std::min(c, remain[s]);
                lens[s] = start[s] + n;
                ranges.push_back(start[s]);
                ranges.push_back(start[s] + n);
                tok += n;
            } else {
                lens[s] = seq_lens[s];
                for (int32_t r = q_range_indptr[s]; r < q_range_indptr[s + 1]; ++r) {
                    ranges.push_back(q_ranges[2 * r]);
                    ranges.push_back(q_ranges[2 * r + 1]);
                }
            }
            indptr[s + 1] = (int32_t)(ranges.size() / 2);
        }
        tokens[ci] = tok;
        msa_plan_t plan = nullptr;
        int rc = msa_plan_create_ex(dims, num_seqs, max_blocks_per_seq, block_table, lens.data(), indptr.data(),
                                    ranges.data(), &o, &plan);
        if (rc == MSA_OK) {
            msa_cost_estimate e{};
            rc = msa_plan_estimate(plan, params, &e);
            time_us[ci] = e.time_us;
        }
        msa_plan_destroy(plan);
        status[ci] = rc;
      } catch (...) {  // allocation failure in this candidate
        status[ci] = MSA_ERR_INVALID_ARG;
      }
    };
    // Up to 8 host threads share the candidates (each plans with its own
    // scratch); if threads cannot be started, this thread does the rest.
    const unsigned hw = std::thread::hardware_concurrency();
    const size_t n_thr = std::min<size_t>(n_cand, std::max<unsigned>(1u, std::min(hw, 8u)));
    std::vector<std::thread> pool;
    size_t started = 1;
    if (n_thr > 1) {
        try {
            pool.reserve(n_thr - 1);
            for (size_t k = 1; k < n_thr; ++k) {
                pool.emplace_back([&, k] {
                    for (size_t ci = k; ci < n_cand; ci += n_thr) evaluate(ci);
                });
                ++started;
            }
        } catch (...) {
        }
    }
    for (size_t ci = 0; ci < n_cand; ci += n_thr) evaluate(ci);
    for (auto& th : pool) th.join();
    // candidates of workers that never started
    for (size_t k = started; k < n_thr; ++k)
        for (size_t ci = k; ci < n_cand; ci += n_thr) evaluate(ci);

    int best = -1;
    double best_per = INFINITY;
    for (size_t ci = 0; ci < n_cand; ++ci) {
        if (status[ci] != MSA_OK) return status[ci];
        const int32_t c = cands[ci];
        if (cand_chunk) cand_chunk[ci] = c;
        if (cand_time_us) cand_time_us[ci] = time_us[ci];
        const double per = time_us[ci] / (double)tokens[ci];
        const bool ok = budget_us <= 0.0 || time_us[ci] <= budget_us;
        // ascending c, so "<=" gives equal per-token costs to the larger chunk
        if (ok && per <= best_per) {
            best_per = per;
            best = (int)ci;
        }
        if (ci == 0 || (int)ci == best) {
            choice->chunk = c;
            choice->tokens = (int32_t)tokens[ci];
            choice->time_us = time_us[ci];
            choice->us_per_token = per;
        }
    }
    // with nothing inside the budget the smallest chunk stands (set above)
    choice->within_budget = best >= 0 ? 1 : 0;
    choice->n_candidates = (int32_t)cands.size();
    return MSA_OK;
}

int msa_choose_prefill_chunk(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks_per_seq,
                             const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_range_indptr,
                             const int32_t* q_ranges, const msa_pending_prefill* pending, int32_t n_pending,
                             const msa_plan_options* opts, const msa_cost_params* params, double budget_us,
                             int32_t granularity, int32_t max_chunk, msa_chunk_choice* choice, int32_t* cand_chunk,
                             double* cand_time_us) {
    try {
        return choose_prefill_chunk(dims, num_seqs, max_blocks_per_seq, block_table, seq_lens, q_range_indptr,
                                    q_ranges, pending, n_pending, opts, params, budget_us, granularity, max_chunk,
                                    choice, cand_chunk, cand_time_us);
    } catch (...) {  // allocation failure: no exception leaves the C ABI
        return MSA_ERR_INVALID_ARG;
    }
}

}  // extern "C"

// ---------------------------------------------------------------- eviction --

static int select_evictions(const msa_dims* dims, int32_t seq_len, const float* hit_prob, int32_t mode,
                            double alpha, double beta, const msa_cost_params* params, int32_t n_evict,
                            int32_t* evicted, double* cost_us) {
    if (!dims || !params || seq_len < 0) return MSA_ERR_INVALID_ARG;
    if (mode & ~(MSA_EVICT_EXPECTED_COST | MSA_EVICT_PREFIX_COST)) return MSA_ERR_INVALID_ARG;
    const bool expected = (mode & MSA_EVICT_EXPECTED_COST) != 0;
    const bool prefix = (mode & MSA_EVICT_PREFIX_COST) != 0;
    if (!(alpha >= 0.0) || !(beta >= 0.0) || !std::isfinite(alpha) || !std::isfinite(beta)) return MSA_ERR_INVALID_ARG;
    if (!(params->pre_tile_us >= 0.0) || !std::isfinite(params->pre_tile_us)) return MSA_ERR_INVALID_ARG;
    if (!(params->pre_tile_dfrac >= 0.0 && params->pre_tile_dfrac <= 1.0)) return MSA_ERR_INVALID_ARG;
    const double t_tile = tile_us(params, dims->head_dim);
    const int32_t nb = (seq_len + kBlock - 1) / kBlock;
    if (n_evict < 0 || n_evict > nb) return MSA_ERR_INVALID_ARG;
    if (nb > 0 && !hit_prob) return MSA_ERR_INVALID_ARG;
    if (n_evict > 0 && !evicted) return MSA_ERR_INVALID_ARG;
    for (int32_t b = 0; b < nb; ++b)
        if (!(hit_prob[b] >= 0.0f && hit_prob[b] <= 1.0f)) return MSA_ERR_INVALID_ARG;
    std::vector<double> cost(nb);
    for (int32_t b = 0; b < nb; ++b) {
        const int64_t p0 = (int64_t)b * kBlock, p1 = std::min<int64_t>(p0 + kBlock, seq_len);
        // sum over p in [p0, p1) of min(p + 1, seq_len) = p + 1 (p < seq_len)
        const double keys = (double)((p0 + 1 + p1) * (p1 - p0) / 2);
        cost[b] = t_tile * dims->num_q_heads * keys / (double)(msa::kTileKeys * msa::kTileRows);
    }
    // prefix reading: evicting b leaves blocks b .. end to recompute
    if (prefix)
        for (int32_t b = nb - 2; b >= 0; --b) cost[b] += cost[b + 1];
    double cmax = 0.0;
    for (int32_t b = 0; b < nb; ++b) {
        cmax = std::max(cmax, cost[b]);
        if (cost_us) cost_us[b] = cost[b];
    }
    std::vector<std::pair<double, int32_t>> sc(nb);
    for (int32_t b = 0; b < nb; ++b)
        sc[b] = {expected ? (double)hit_prob[b] * cost[b]
                          : alpha * (double)hit_prob[b] + (cmax > 0.0 ? beta * cost[b] / cmax : 0.0),
                 b};
    std::stable_sort(sc.begin(), sc.end(), [](const auto& x, const auto& y) { return x.first < y.first; });
    std::vector<int32_t> out(n_evict);
    for (int32_t i = 0; i < n_evict; ++i) out[i] = sc[i].second;
    std::sort(out.begin(), out.end());
    for (int32_t i = 0; i < n_evict; ++i) evicted[i] = out[i];
    return MSA_OK;
}

extern "C" int msa_select_evictions(const msa_dims* dims, int32_t seq_len, const float* hit_prob, int32_t mode,
                                    double alpha, double beta, const msa_cost_params* params, int32_t n_evict,
                                    int32_t* evicted, double* cost_us) {
    try {
        return select_evictions(dims, seq_len, hit_prob, mode, alpha, beta, params, n_evict, evicted, cost_us);
    } catch (...) {  // allocation failure: no exception leaves the C ABI
        return MSA_ERR_INVALID_ARG;
    }
}
