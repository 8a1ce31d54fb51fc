// planner.cpp -- host planner of libmsa: validates the block table and the
// query ranges, splits every sequence's live blocks into physically
// contiguous segments (runs), forms output groups (GQA-packed decode rows or
// 128-row prefill tiles per query head), splits long key ranges for SM
// balance and orders the work items (longest first) for the dynamic queue of
// one persistent launch.
//
// Segment rule (AsymCache explainer, "核心方法 1. Multi-Segment Attention"):
// live blocks are regrouped by physical contiguity; an eviction hole, or any
// block that is not the physical successor of the previous logical block,
// starts a new segment.  Runs are therefore maximal, left to right, and
// unique.  Two runs that touch physically but not in logical order stay
// separate, because inside a run the logical->physical map must be a shift.
//
// The work list replaces the per-segment kernel launches the pages discuss
// (MSA summary: one kernel over many disjoint segments removes launch
// overhead) by one list consumed by a persistent grid.
#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "msa_internal.h"
#include "plan.h"

namespace msa {

static int validate_dims(const msa_dims* d) {
    if (!d) return MSA_ERR_INVALID_ARG;
    if (d->block_size != kBlock) return MSA_ERR_UNSUPPORTED_DIMS;
    if (d->head_dim != 64 && d->head_dim != 128) return MSA_ERR_UNSUPPORTED_DIMS;
    if (d->num_q_heads <= 0 || d->num_kv_heads <= 0) return MSA_ERR_UNSUPPORTED_DIMS;
    if (d->num_q_heads % d->num_kv_heads != 0) return MSA_ERR_UNSUPPORTED_DIMS;
    if (d->num_q_heads / d->num_kv_heads > kDecRows) return MSA_ERR_UNSUPPORTED_DIMS;
    if (!(d->softmax_scale > 0.0f) || !std::isfinite(d->softmax_scale)) return MSA_ERR_UNSUPPORTED_DIMS;
    return MSA_OK;
}

namespace {
constexpr size_t kRecycledPlans = 2;
thread_local std::vector<std::unique_ptr<msa_plan_s>> t_recycled;
// scratch of plan_create / split_items, kept per thread for the same reason
thread_local std::vector<Pending> t_pend;
thread_local std::vector<double> t_cost;
thread_local std::vector<uint64_t> t_keys;  // queue-order sort keys
thread_local std::vector<unsigned __int128> t_ord;  // (key, item) pairs being sorted
}  // namespace

// Number of KV tiles the kernels walk over keys [kb, ke): 128-key windows
// of the logical key range starting at kb (a window may span segments).
static int64_t count_tiles(int32_t kb, int32_t ke) {
    return ke > kb ? (ke - kb + kTileKeys - 1) / kTileKeys : 0;
}

// Index of the run (within runs[r0..r1)) holding logical key k.
static int32_t run_of(const Run* runs, int32_t r0, int32_t r1, int32_t k) {
    int32_t lo = r0, hi = r1 - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) / 2;
        if (runs[mid].log_start <= k) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Cut every group's key range into parts and order the items (longest
// first).  A part holds about (work per CTA) / split of a group's tiles:
// `dec_split` for decode groups, `pre_split` for prefill groups.  Rebuilds
// P->groups, items, order and the partial-slot counts from scratch.
void split_items(msa_plan_s* P, const std::vector<Pending>& pend, double dec_split, double pre_split) {
    P->groups.clear();
    P->items.clear();
    P->order.clear();
    P->n_dec_slots = 0;
    P->n_pre_slots = 0;
    // Cost of an item ~ its KV tiles (a decode tile moves 2*128*D*2 bytes, a
    // prefill tile does 4*128*128*D flops; on GB300 both take ~1.3-1.5 us per
    // SM) plus a fixed per-item cost.
    const double w_tile[2] = {1.1, 1.0};
    const double w_item[2] = {0.5, 2.0};
    double total = 0.0;
    for (auto& pd : pend) total += pd.tiles * w_tile[pd.g.kind] + w_item[pd.g.kind];
    const double per_cta = total / P->grid;
    const int64_t min_tiles[2] = {4, 8};

    std::vector<double>& cost = t_cost;
    cost.clear();
    P->groups.reserve(pend.size());
    P->items.reserve(pend.size() * 2);
    cost.reserve(pend.size() * 2);
    for (size_t gi = 0; gi < pend.size(); ++gi) {
        const Pending& pd = pend[gi];
        const int32_t kind = pd.g.kind;
        const double per_item = per_cta / (kind == kDecode ? dec_split : pre_split);
        int64_t chunk = std::max<int64_t>(min_tiles[kind], (int64_t)std::ceil(per_item / w_tile[kind]));
        int32_t parts = (int32_t)std::max<int64_t>(1, (pd.tiles + chunk - 1) / chunk);
        const int32_t s = pd.g.seq;
        const int32_t ra = P->run_indptr[s], rb = P->run_indptr[s + 1];
        Group g = pd.g;
        g.n_parts = parts;
        const int32_t gid = (int32_t)P->groups.size();
        if (parts > 1) {
            if (kind == kDecode) { g.slot = P->n_dec_slots; P->n_dec_slots += parts; }
            else { g.slot = P->n_pre_slots; P->n_pre_slots += parts; }
        }
        P->groups.push_back(g);
        // cut the key range into `parts` runs of whole tiles
        if (pd.ke <= 0 || ra == rb) {
            Item it{gid, 0, 0, ra, 0, kind, s, 0};
            P->items.push_back(it);
            cost.push_back(w_item[kind]);
            continue;
        }
        const int64_t per = (pd.tiles + parts - 1) / parts;
        int32_t part = 0;
        for (int64_t t = 0; t < pd.tiles; t += per) {
            const int32_t kb = (int32_t)(t * kTileKeys);
            const int32_t ke = (int32_t)std::min<int64_t>((t + per) * kTileKeys, pd.ke);
            Item it{gid, kb, ke, run_of(P->runs.data(), ra, rb, kb), part, kind, s, 0};
            P->items.push_back(it);
            cost.push_back(std::min<int64_t>(per, pd.tiles - t) * w_tile[kind] + w_item[kind]);
            ++part;
        }
        P->groups[gid].n_parts = part;
        if (part == 1) P->groups[gid].slot = -1;
    }

    // KV tiles of every item (the kernels walk exactly these)
    for (auto& it : P->items) it.pad = (int32_t)count_tiles(it.kb, it.ke);

    // One global queue, longest first: every CTA of the persistent launch
    // takes the next item when it is free (list scheduling in LPT order), so
    // the load balances itself on the device.  Costs within a 1.6-3 % bucket
    // count as equal, and equal-cost items are ordered by (sequence, kv head), then
    // in generation order: the CTAs that run at the same time then stream the same K/V
    // tiles, which L2 serves to all of them after one read from HBM (all
    // prefill items of a sequence and kv head read the same keys).  Measured:
    // -3 % on a long-context launch against cost order alone.
    const int32_t n_items = (int32_t)P->items.size();
    std::vector<uint64_t>& keys = t_keys;
    keys.resize(n_items);
    for (int32_t i = 0; i < n_items; ++i) {
        // bucket: the cost's exponent and top 5 mantissa bits (monotone in
        // the cost for positive doubles; buckets 1.6-3.1 % wide), largest
        // first; then sequence and kv head (generation order -- row tile,
        // head, part -- breaks the remaining ties)
        uint64_t bits;
        const double c = std::max(cost[i], 1e-30);
        std::memcpy(&bits, &c, sizeof bits);
        const Item& it = P->items[i];
        const Group& g = P->groups[it.group];
        const uint64_t kvh = (uint64_t)(g.kind == kDecode ? g.head : g.head / P->G);
        keys[i] = ((0x1FFFFull - (bits >> 47)) << 46) | (((uint64_t)it.seq & 0x3FFFFFFull) << 20) | (kvh & 0xFFFFFull);
    }
    // sort (key, generation index) as one 128-bit integer: the same order as a
    // stable sort by key, on contiguous values
    std::vector<unsigned __int128>& ord = t_ord;
    ord.resize(n_items);
    for (int32_t i = 0; i < n_items; ++i) ord[i] = ((unsigned __int128)keys[i] << 32) | (uint32_t)i;
    std::sort(ord.begin(), ord.end());
    P->order.resize(n_items);
    for (int32_t i = 0; i < n_items; ++i) P->order[i] = (int32_t)(uint32_t)ord[i];
}


msa_plan_s* plan_alloc() {
    if (!t_recycled.empty()) {
        msa_plan_s* P = t_recycled.back().release();
        t_recycled.pop_back();
        return P;
    }
    return new (std::nothrow) msa_plan_s();
}

void plan_release(msa_plan_s* P) {
    if (!P) return;
    if (t_recycled.size() >= kRecycledPlans) {
        delete P;
        return;
    }
    P->reset();
    try {
        t_recycled.emplace_back(P);
    } catch (...) {  // no room to keep it: free it instead
        delete P;
    }
}

int plan_create(const msa_dims* dims, int32_t num_seqs, int32_t max_blocks,
                const int32_t* table, const int32_t* seq_lens, const int32_t* q_range_indptr,
                const int32_t* q_ranges, int32_t num_sms, const msa_plan_options* opts, msa_plan_s** out) {
    auto t0 = std::chrono::steady_clock::now();
    if (!out) return MSA_ERR_INVALID_ARG;
    *out = nullptr;
    int rc = validate_dims(dims);
    if (rc != MSA_OK) return rc;
    if (num_seqs < 0 || max_blocks < 0 || num_sms < 0) return MSA_ERR_INVALID_ARG;
    if (opts && (!(opts->decode_split >= 0.0) || !(opts->prefill_split >= 0.0) ||
                 !std::isfinite(opts->decode_split) || !std::isfinite(opts->prefill_split)))
        return MSA_ERR_INVALID_ARG;
    if (num_seqs > 0 && (!seq_lens || !q_range_indptr)) return MSA_ERR_INVALID_ARG;
    if (num_seqs > 0 && max_blocks > 0 && !table) return MSA_ERR_INVALID_ARG;
    if (num_sms == 0) {
        num_sms = device_sm_count();
        if (num_sms <= 0) return MSA_ERR_CUDA;
    }

    msa_plan_s* P = plan_alloc();
    if (!P) return MSA_ERR_INVALID_ARG;
    std::unique_ptr<msa_plan_s, void (*)(msa_plan_s*)> guard(P, plan_release);
    P->dims = *dims;
    P->num_seqs = num_seqs;
    P->G = dims->num_q_heads / dims->num_kv_heads;
    P->dec_rows = kDecRows / P->G;
    const int32_t D = dims->head_dim;
    const int32_t Hq = dims->num_q_heads, Hkv = dims->num_kv_heads, G = P->G;

    // ---- sequences and segment runs -------------------------------------
    P->seq_lens.assign(seq_lens, seq_lens + num_seqs);
    P->run_indptr.assign(1, 0);
    int64_t max_row = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t L = seq_lens[s];
        if (L < 0) return MSA_ERR_INVALID_ARG;
        const int32_t nb = (L + kBlock - 1) / kBlock;
        if (nb > max_blocks) return MSA_ERR_INVALID_ARG;
        const int32_t* row = table + (int64_t)s * max_blocks;
        int32_t b = 0;
        while (b < nb) {
            if (row[b] < 0) return MSA_ERR_MISSING_BLOCK;
            if (row[b] >= (1 << 27)) return MSA_ERR_BAD_BLOCK_ID;
            int32_t e = b + 1;
            while (e < nb && row[e] >= 0 && row[e] < (1 << 27) && row[e] == row[e - 1] + 1) ++e;
            Run r;
            r.log_start = b * kBlock;
            r.phys_row = row[b] * kBlock;
            r.n_tok = std::min(e * kBlock, L) - b * kBlock;
            r.pad = 0;
            P->runs.push_back(r);
            max_row = std::max<int64_t>(max_row, (int64_t)row[e - 1] * kBlock + kBlock);
            b = e;
        }
        P->run_indptr.push_back((int32_t)P->runs.size());
    }
    P->max_pool_row = max_row;

    // ---- query rows -------------------------------------------------------
    if (num_seqs > 0) {
        if (q_range_indptr[0] != 0) return MSA_ERR_BAD_Q_RANGE;
        if (q_range_indptr[num_seqs] > 0 && !q_ranges) return MSA_ERR_INVALID_ARG;
    }
    // validate the ranges and count the rows, then lay the positions out
    int64_t n_rows = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t a = q_range_indptr[s], b = q_range_indptr[s + 1];
        if (b < a) return MSA_ERR_BAD_Q_RANGE;
        int64_t prev_end = 0;
        for (int32_t i = a; i < b; ++i) {
            const int32_t st = q_ranges[2 * i], en = q_ranges[2 * i + 1];
            if (st < 0 || en <= st || (int64_t)en > (int64_t)seq_lens[s] + 1 || st < prev_end)
                return MSA_ERR_BAD_Q_RANGE;
            prev_end = en;
            n_rows += en - st;
            if (n_rows > (int64_t)INT32_MAX / 2) return MSA_ERR_INVALID_ARG;
        }
    }
    P->row_indptr.assign(1, 0);
    P->row_indptr.reserve((size_t)num_seqs + 1);
    P->pos.reserve((size_t)n_rows);
    for (int32_t s = 0; s < num_seqs; ++s) {
        for (int32_t i = q_range_indptr[s]; i < q_range_indptr[s + 1]; ++i)
            for (int32_t p = q_ranges[2 * i]; p < q_ranges[2 * i + 1]; ++p) P->pos.push_back(p);
        P->row_indptr.push_back((int32_t)P->pos.size());
    }
    const int32_t n_q = (int32_t)P->pos.size();

    // ---- output groups ----------------------------------------------------
    // A sequence's trailing rows go to the GQA-packed decode path when they
    // number at most kDecRows / G; everything else is cut into 128-row tiles.
    std::vector<Pending>& pend = t_pend;
    pend.clear();
    {
        size_t n_groups = 0;  // capacity hint: at most one decode group per kv head plus the 128-row tiles
        for (int32_t s = 0; s < num_seqs; ++s) {
            const int32_t n = P->row_indptr[s + 1] - P->row_indptr[s];
            n_groups += (size_t)(n / kTileRows + 2) * (size_t)std::max(Hkv, Hq);
        }
        pend.reserve(n_groups);
    }
    double prefill_flops = 0.0;
    int64_t dec_kv = 0, dec_qo = 0;
    int32_t dec_rows_total = 0, pre_rows_total = 0;
    for (int32_t s = 0; s < num_seqs; ++s) {
        const int32_t r0 = P->row_indptr[s], r1 = P->row_indptr[s + 1];
        const int32_t n = r1 - r0;
        if (n == 0) continue;
        const int32_t L = seq_lens[s];
        const int32_t ra = P->run_indptr[s], rb = P->run_indptr[s + 1];
        // Groups over rows [row0, row0 + nrows).  decode: one group per kv
        // head (all G query heads packed), Group.pad = G.  prefill: two
        // query tiles of 128 rows x one head that share a kv head, Group.pad
        // = the number of query tiles (1 or 2) -- `pairs`: query heads 2i
        // and 2i + 1 of every kv head over <= 128 rows (all heads for even
        // G, all but the last for odd G); otherwise the last query head of
        // every kv head (odd G: no second head left to pair with) over two
        // consecutive row tiles (<= 256 rows).  The kernel tells the two
        // prefill forms apart by pad == 2 with nrows <= 128.
        auto add_groups = [&](int32_t kind, int32_t row0, int32_t nrows, bool pairs) {
            const int32_t pmax = P->pos[row0 + nrows - 1];  // rows ascend within a sequence
            const int32_t ke = std::min(pmax + 1, L);
            const int64_t tiles = count_tiles(0, ke);
            auto push = [&](int32_t head, int32_t pad) {
                Pending pd;
                pd.g = Group{kind, s, head, row0, nrows, 1, -1, pad};
                pd.ke = ke;
                pd.tiles = tiles;
                pend.push_back(pd);
            };
            int32_t heads = 0;  // query heads these groups cover
            if (kind == kDecode) {
                for (int32_t h = 0; h < Hkv; ++h) push(h, G);
                heads = Hq;
            } else if (pairs) {
                for (int32_t kv = 0; kv < Hkv; ++kv)
                    for (int32_t i = 0; 2 * i + 1 < G; ++i) push(kv * G + 2 * i, 2);
                heads = Hkv * (G - (G & 1));
            } else {
                for (int32_t kv = 0; kv < Hkv; ++kv) push(kv * G + G - 1, (nrows + kTileRows - 1) / kTileRows);
                heads = Hkv;
            }
            if (kind == kDecode) {
                dec_kv += (int64_t)ke * Hkv * D * 2 * 2;
                dec_qo += (int64_t)nrows * Hq * (D * 2 + D * 2 + 4);
                dec_rows_total += nrows;
            } else {
                for (int32_t r = row0; r < row0 + nrows; ++r)
                    prefill_flops += 4.0 * D * heads * (double)std::min(P->pos[r] + 1, L);
                if (!pairs || G % 2 == 0) pre_rows_total += nrows;  // each row once
            }
        };
        if (n <= P->dec_rows) {
            add_groups(kDecode, r0, n, false);
        } else {
            // 128-row tiles (the remainder too, unless the decode path takes
            // it); for odd G the last query head of each kv head takes two
            // consecutive tiles per group
            const int32_t full = n / kTileRows, rem = n % kTileRows;
            const int32_t pre_rows = full * kTileRows + (rem > P->dec_rows ? rem : 0);
            if (G >= 2)
                for (int32_t a = 0; a < pre_rows; a += kTileRows)
                    add_groups(kPrefill, r0 + a, std::min(kTileRows, pre_rows - a), true);
            if (G & 1)
                for (int32_t a = 0; a < pre_rows; a += 2 * kTileRows)
                    add_groups(kPrefill, r0 + a, std::min(2 * kTileRows, pre_rows - a), false);
            if (rem > 0 && rem <= P->dec_rows) add_groups(kDecode, r0 + full * kTileRows, rem, false);
        }
    }

    // ---- work items and their order ----------------------------------------
    P->grid = std::max(1, num_sms);
    double dec_split = opts && opts->decode_split > 0.0 ? opts->decode_split : kDefaultDecodeSplit;
    double pre_split = opts && opts->prefill_split > 0.0 ? opts->prefill_split : kDefaultPrefillSplit;
    if (opts && opts->choose_with) choose_split(P, pend, *opts->choose_with, &dec_split, &pre_split);
    split_items(P, pend, dec_split, pre_split);
    const int32_t n_items = (int32_t)P->items.size();

    // ---- info ---------------------------------------------------------------
    msa_plan_info& I = P->info;
    std::memset(&I, 0, sizeof I);
    I.num_seqs = num_seqs;
    I.num_q_rows = n_q;
    I.num_runs = (int32_t)P->runs.size();
    I.num_groups = (int32_t)P->groups.size();
    I.num_items = n_items;
    for (auto& it : P->items) (it.kind == kDecode ? I.num_decode_items : I.num_prefill_items)++;
    I.num_decode_rows = dec_rows_total;
    I.num_prefill_rows = pre_rows_total;
    I.grid = P->grid;
    I.decode_kv_bytes = dec_kv;
    I.decode_qo_bytes = dec_qo;
    I.prefill_flops = prefill_flops;
    I.max_pool_row = P->max_pool_row;
    I.decode_split = dec_split;
    I.prefill_split = pre_split;

    build_image(P);
    I.counters_offset = (int64_t)P->lay.counters;
    I.counters_bytes = (int64_t)(P->lay.counters_end - P->lay.counters);
    I.host_plan_us = std::chrono::duration<double, std::micro>(std::chrono::steady_clock::now() - t0).count();
    *out = guard.release();
    return MSA_OK;
}

// Lay out the workspace and serialise the int sections into the host image.
void build_image(msa_plan_s* P) {
    WsLayout& W = P->lay;
    const size_t D = (size_t)P->dims.head_dim;
    size_t o = 0;
    auto sec = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 256); return at; };
    W.error = sec(64 * sizeof(int32_t));
    W.items = sec(P->items.size() * sizeof(Item));
    W.groups = sec(P->groups.size() * sizeof(Group));
    W.runs = sec(P->runs.size() * sizeof(Run));
    W.pos = sec(P->pos.size() * sizeof(int32_t));
    W.order = sec(P->order.size() * sizeof(int32_t));
    W.image_end = o;
    W.counters = sec(2 * P->groups.size() * sizeof(int32_t));
    W.sched = sec(2 * sizeof(int32_t));
    W.counters_end = o;
    W.dec_part = sec((size_t)P->n_dec_slots * kDecRows * D * sizeof(float));
    W.dec_lse = sec((size_t)P->n_dec_slots * kDecRows * sizeof(float));
    W.pre_part = sec((size_t)P->n_pre_slots * 2 * kTileRows * D * sizeof(float));
    W.pre_lse = sec((size_t)P->n_pre_slots * 2 * kTileRows * sizeof(float));
    W.total = align_up(o, 256);

    P->image.assign(W.image_end, 0);
    auto put = [&](size_t at, const void* src, size_t bytes) {
        if (bytes) std::memcpy(P->image.data() + at, src, bytes);
    };
    put(W.items, P->items.data(), P->items.size() * sizeof(Item));
    put(W.groups, P->groups.data(), P->groups.size() * sizeof(Group));
    put(W.runs, P->runs.data(), P->runs.size() * sizeof(Run));
    put(W.pos, P->pos.data(), P->pos.size() * sizeof(int32_t));
    put(W.order, P->order.data(), P->order.size() * sizeof(int32_t));
}

}  // namespace msa
